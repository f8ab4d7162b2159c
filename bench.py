"""Benchmark: batched row-wise top-k on GB300.

One step = one ``topk_select`` call over the whole batch (every stage of the
selection: visiting order, streaming filter, compaction, tray sorts, split-row
merge, final write).  The default workload is 64 rows x 1,048,576 fp32
Normal(0,1) scores with k = 512, the decode shape the throughput metric is
quoted on.  Prints ONE JSON line on rank 0.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl gb300|reference]
                  [--workload NAME] [--pool P,Q] [--timeline]

``--gpus N`` must match the number of ranks: N = 1 runs in this process, N > 1
runs under torchrun (one rank per GPU).  ``--timeline`` also records one launch
with the instrumented build of the library (per-CTA stamps; see
``sparse_attention_indexer_row_gb300/timeline.py``) and adds its summary.

Under torchrun each rank runs the same per-GPU batch on its own GPU (weak
scaling, no collective on the data path); the timed region is bracketed by a
barrier and the slowest rank's time is reported.

``--impl reference`` times the CPU oracle (test infrastructure) on the host's
cores on a bounded sample of the same workload: the only other place this
script runs the oracle is the ``cpu_baseline`` leg of the default arm.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from sparse_attention_indexer_row_gb300 import synth  # noqa: E402

METRIC = "rows/s and achieved HBM GB/s (fraction of GB300 peak) at n=1M, k=512"
UNIT = "rows/s"
FALLBACK_HBM_GBS = 6800.0
KERNEL_SRC = os.path.join(ROOT, "sparse_attention_indexer_row_gb300", "csrc", "topk_select.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "topk_select_kernel_traffic.json")
N_INPUT_BUFFERS = 3   # rotated so consecutive steps never re-read L2-resident scores
L2_BYTES = 129 * 10**6
FLUSH_BYTES = 512 << 20  # written before each timed launch when the inputs fit in L2


def _dist():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def _launches_per_call(rows: int, n: int, has_lengths: bool, pool: bool, plan_sms: int) -> int:
    """Kernels one call launches: the selection kernel; before it, for a
    batch of at least as many rows as the plan has CTAs (the device's SM
    count, at most 256) with per-row lengths and rows of at most 4096 units of
    8192 elements, the kernel that orders the shared queue by row length;
    after it, with a block pool, the pool kernel."""
    per = 1
    if has_lengths and rows >= plan_sms and -(-n // 8192) <= 4096:
        per += 1
    if pool:
        per += 1
    return per


def _workload(name: str) -> synth.Workload:
    return synth.make(name)


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(path))
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def _kernel_hash() -> str:
    return hashlib.sha256(open(KERNEL_SRC, "rb").read()).hexdigest()[:16]


def _kernel_name(rows: int, n: int, pool: bool, sms: int) -> str:
    """The selection kernel a call runs (the library's routing rule: batches of
    at least as many rows as SMs with rows of at most 65,536 scores take the
    short-row kernel)."""
    if pool:
        return "topk_select_kernel (+ pool_select_kernel)"
    if rows >= min(256, sms) and n <= 65536:
        return "short_select_kernel"
    return "topk_select_kernel"


def _traffic_per_launch(workload: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches the
    current kernel source and workload; else None."""
    try:
        d = json.load(open(TRAFFIC_FILE))
    except Exception:
        return None
    if d.get("kernel_sha256_16") != _kernel_hash() or d.get("workload") != workload:
        return None
    return d.get("dram_bytes_per_launch")


class ClockSampler:
    """nvidia-smi clock/throttle sampling while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            return
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out = ""
        self.out = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.out:
            f = [t.strip() for t in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def run_gb300(args, world, rank, local):
    import torch

    from sparse_attention_indexer_row_gb300 import binding as B
    from sparse_attention_indexer_row_gb300 import dist as D

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    w = _workload(args.workload)
    rows, n, k, stride = w.rows, w.n, w.k, w.row_stride
    stream = torch.cuda.current_stream(dev)

    host = torch.from_numpy(w.scores)
    bufs = [host.to(dev) for _ in range(N_INPUT_BUFFERS)]
    lengths = None if w.lengths is None else torch.from_numpy(w.lengths).to(dev)
    vals = torch.empty((rows, k), dtype=torch.float32, device=dev)
    idx = torch.empty((rows, k), dtype=torch.int32, device=dev)
    split = B.topk_split_plan(rows, n)
    pool = None
    if args.pool:
        # the layer-20 block pool in the same pass: pool_blocks, pinned_blocks
        pool = tuple(int(t) for t in args.pool.split(","))
        ws = torch.zeros(B.topk_pool_ws_bytes(rows, n, k, *pool), dtype=torch.uint8, device=dev)
        out_pool = torch.empty((rows, pool[0]), dtype=torch.int32, device=dev)
    else:
        ws = torch.zeros(B.topk_ws_bytes(rows, n, k), dtype=torch.uint8, device=dev)

    def select(x):
        if pool:
            rc = B.topk_select_pool(x, rows, n, stride, lengths, k, vals, idx, pool[0], pool[1],
                                    out_pool, ws, stream)
        else:
            rc = B.topk_select(x, rows, n, stride, lengths, k, vals, idx, ws, stream)
        if rc != 0:
            raise RuntimeError(f"selection returned {rc}")

    def step(i):
        select(bufs[i % N_INPUT_BUFFERS])

    barrier = D.barrier

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    # Device-timed region on the launching stream.  Inputs larger than L2
    # (together): K back-to-back launches between one event pair (the kernel
    # is the only work in the region, so the region's length over K is also
    # the kernel's average launch duration).  Inputs that fit in L2: before
    # each launch an untimed write of FLUSH_BYTES evicts them, and each launch
    # sits between its own event pair.
    flush = N_INPUT_BUFFERS * host.numel() * 4 < 2 * L2_BYTES
    scratch = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev) if flush else None
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    pairs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(args.steps)] if flush else []
    with ClockSampler(local) as clocks:
        barrier()
        torch.cuda.synchronize()
        if flush:
            for i in range(args.steps):
                scratch.fill_(i & 0xFF)
                pairs[i][0].record(stream)
                step(i)
                pairs[i][1].record(stream)
        else:
            t0.record(stream)
            for i in range(args.steps):
                step(i)
            t1.record(stream)
        torch.cuda.synchronize()
        barrier()
    per_launch = [a.elapsed_time(b) for a, b in pairs]
    local_ms = sum(per_launch) if flush else t0.elapsed_time(t1)
    total_ms = D.max_over_ranks(local_ms, device=dev)
    ms_per_step = total_ms / args.steps
    value = world * rows / (ms_per_step / 1e3)
    launch_stats = None
    if flush:
        # the same launches back to back on one buffer, no flush: L2-resident
        # scores after the first (a latency figure beside the HBM one)
        h0 = torch.cuda.Event(enable_timing=True)
        h1 = torch.cuda.Event(enable_timing=True)
        select(bufs[0])
        h0.record(stream)
        for _ in range(args.steps):
            select(bufs[0])
        h1.record(stream)
        torch.cuda.synchronize()
        q = np.percentile(per_launch, [10, 50, 90])
        launch_stats = {"flushed_ms": {"p10": round(float(q[0]), 5), "median": round(float(q[1]), 5),
                                       "p90": round(float(q[2]), 5), "launches": len(per_launch)},
                        "hot_l2_ms": round(h0.elapsed_time(h1) / args.steps, 5)}

    # End to end through the same C call: pinned host scores in, results out.
    host_pin = host.pin_memory()
    len_pin = None if w.lengths is None else torch.from_numpy(w.lengths).pin_memory()
    vals_h = torch.empty((rows, k), dtype=torch.float32).pin_memory()
    idx_h = torch.empty((rows, k), dtype=torch.int32).pin_memory()
    pool_h = torch.empty((rows, pool[0]), dtype=torch.int32).pin_memory() if pool else None
    dev_in = bufs[0]

    def e2e_step():
        dev_in.copy_(host_pin, non_blocking=True)
        if len_pin is not None:
            lengths.copy_(len_pin, non_blocking=True)
        select(dev_in)
        vals_h.copy_(vals, non_blocking=True)
        idx_h.copy_(idx, non_blocking=True)
        if pool:
            pool_h.copy_(out_pool, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        e2e_step()
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = D.max_over_ranks(e0.elapsed_time(e1), device=dev)
    e2e_value = world * rows / (e2e_ms / args.steps / 1e3)
    # the host-to-device copy alone (what the e2e figure spends outside the kernel)
    e0.record(stream)
    for _ in range(args.steps):
        dev_in.copy_(host_pin, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    h2d_ms = e0.elapsed_time(e1) / args.steps
    h2d = host.numel() * 4 + (0 if w.lengths is None else rows * 4)
    d2h = rows * k * 8 + (rows * pool[0] * 4 if pool else 0)

    # Survivor counters for one call (elements that reached a tray sort).
    B.topk_ws_stats(ws, rows, n, k, 0, stream)
    step(0)
    rc, surv, sorts, adm = B.topk_ws_stats(ws, rows, n, k, 0, stream)
    rc2, status = B.topk_ws_status(ws, stream)

    if rank != 0:
        return None

    # torch.topk on the same device tensor, as context.
    tk_ms = None
    if w.lengths is None:
        x = bufs[0][:, :n]
        for _ in range(3):
            torch.topk(x, k, dim=1, sorted=True)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        reps = max(3, min(args.steps, 10))
        a.record(stream)
        for _ in range(reps):
            torch.topk(x, k, dim=1, sorted=True)
        b.record(stream)
        torch.cuda.synchronize()
        tk_ms = a.elapsed_time(b) / reps

    alg_bytes = w.algorithmic_bytes() + (rows * pool[0] * 4 if pool else 0)
    avg_launch_ms = local_ms / args.steps
    peak, peak_kind = _peaks()
    achieved = alg_bytes / (avg_launch_ms / 1e3) / 1e9
    traffic = None if pool else _traffic_per_launch(args.workload)
    T = k + 2 * 1024
    m = (n + 1023) // 1024
    harmonic = sum(1.0 / j for j in range(1, m + 1))

    line = {
        "metric": METRIC,
        "value": round(value, 1),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64)",
        "config": {
            "workload": w.name,
            "rows": rows, "n": n, "k": k, "row_stride": stride,
            "values": w.meta,
            "split_per_row": split,
            "l2": (f"inputs fit in L2: a {FLUSH_BYTES >> 20} MiB write before each timed launch, "
                   "each launch between its own event pair") if flush else
                  (f"{N_INPUT_BUFFERS} rotating input buffers of "
                   f"{host.numel() * 4 / 2**20:.0f} MiB (> 129 MB L2), no flush"),
            "parallelism": f"weak: {world} GPU(s), each its own batch",
            **({"pool_blocks": pool[0], "pinned_blocks": pool[1],
                "pool_block_positions": 8} if pool else {}),
        },
        "gbs": round(alg_bytes / (ms_per_step / 1e3) / 1e9, 1),
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peak,
            "unit": "GB/s",
            "frac": round(achieved / peak, 4),
            "traffic": traffic,
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs, copy bandwidth)"
                           if peak_kind == "measured" else "fallback 6.8 TB/s",
            "kernel": _kernel_name(rows, n, bool(pool), torch.cuda.get_device_properties(dev).multi_processor_count),
            "algorithmic_bytes_per_launch": alg_bytes,
            "avg_launch_ms": round(avg_launch_ms, 5),
        },
        "e2e": {
            "value": round(e2e_value, 1), "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": round(e2e_ms / args.steps, 4), "h2d_copy_ms_per_step": round(h2d_ms, 4),
            "path": "pinned host -> device copy, " + ("topk_select_pool" if pool else "topk_select") +
                    " (C ABI), device -> pinned host",
        },
        "gpu_launches": args.steps * _launches_per_call(
            rows, n, w.lengths is not None, bool(pool),
            min(256, torch.cuda.get_device_properties(dev).multi_processor_count)),
        "clocks": clocks.summary(),
        "survivors": {
            "mean_per_row": round(float(np.mean(surv)), 1), "max_per_row": int(max(surv)),
            "sorts_per_row_mean": round(float(np.mean(sorts)), 2),
            "admitted_per_row_mean": round(float(np.mean(adm)), 1),
            "bound_unsplit_row": round(1.5 * T * harmonic, 1),
            "split_per_row": split,
        },
        "status_word": status,
        "torch_topk": None if tk_ms is None else {
            "ms": round(tk_ms, 4), "gbs": round(alg_bytes / (tk_ms / 1e3) / 1e9, 1)},
    }
    if launch_stats:
        line["launch_ms"] = launch_stats
    if args.timeline:
        line["timeline"] = timeline_of(B, bufs[0], w, lengths, vals, idx, ws, stream, pool,
                                       out_pool if pool else None, line["clocks"].get("sm_mhz"))
    if args.cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    return line


def timeline_of(B, x, w, lengths, vals, idx, ws, stream, pool, out_pool, sm_mhz):
    """One launch of the same call through the instrumented build, summarised
    per CTA (stamps in µs after the earliest CTA start; cycles at the clock the
    timed region saw)."""
    from sparse_attention_indexer_row_gb300 import timeline as TLM
    lib = TLM.load()
    P, S = B._ptr, B._stream

    def call(l):
        if pool:
            rc = l.topk_select_pool(P(x), w.rows, w.n, w.row_stride, P(lengths), w.k, P(vals),
                                    P(idx), pool[0], pool[1], P(out_pool), P(ws), S(stream))
        else:
            rc = l.topk_select(P(x), w.rows, w.n, w.row_stride, P(lengths), w.k, P(vals), P(idx),
                               P(ws), S(stream))
        if rc != 0:
            raise RuntimeError(f"instrumented selection returned {rc}")

    for _ in range(3):
        call(lib)
    table = TLM.record(lib, call, stream)
    out = TLM.summarize(table, float(sm_mhz or 2070.0))
    out["build"] = "libtopk_gb300_timeline.so (-DTOPK_TIMELINE=1), one launch after three"
    return out


def cpu_baseline(w: synth.Workload, cpu_seconds: float, rows_per_pass=None):
    """The oracle as it stands, spread over the host's cores, on whole passes
    over the batch until about `cpu_seconds` of CPU time has accumulated."""
    import oracle
    orc = oracle.load()
    cores = os.cpu_count() or 1
    sample = w.scores if rows_per_pass is None else w.scores[:rows_per_pass]
    lens = w.lengths if (w.lengths is None or rows_per_pass is None) else w.lengths[:rows_per_pass]
    passes, t_total = 0, 0.0
    while True:
        t = time.perf_counter()
        _, _, st = orc.topk(sample, w.k, lengths=lens, n=w.n, nthreads=cores)
        t_total += time.perf_counter() - t
        passes += 1
        if st != 0:
            raise RuntimeError(f"oracle status {st}")
        if t_total * min(cores, sample.shape[0]) >= cpu_seconds or passes >= 50:
            break
    rows_done = passes * sample.shape[0]
    # the same oracle on one thread, over the first few rows of the sample
    few = min(4, sample.shape[0])
    t = time.perf_counter()
    _, _, st = orc.topk(sample[:few], w.k, lengths=None if lens is None else lens[:few], n=w.n,
                        nthreads=1)
    t_one = time.perf_counter() - t
    if st != 0:
        raise RuntimeError(f"oracle status {st}")
    return {"value": round(rows_done / t_total, 2), "unit": UNIT,
            "cores": min(cores, sample.shape[0]), "kind": "oracle",
            "sample": f"{passes} pass(es) over {sample.shape[0]} rows of {w.name} "
                      f"({t_total:.2f} s wall)",
            "single_thread": {"value": round(few / t_one, 2), "unit": UNIT, "cores": 1,
                              "sample": f"the first {few} rows of the batch, once"}}


def run_reference(args, world, rank):
    if rank != 0:
        return None
    import oracle
    w = _workload(args.workload)
    orc = oracle.load()
    cores = os.cpu_count() or 1
    per_step = min(w.rows, max(1, args.ref_rows))
    rng_rows = [(i * per_step) % w.rows for i in range(args.warmup + args.steps)]

    def step(i):
        r0 = rng_rows[i]
        sel = np.arange(r0, r0 + per_step) % w.rows
        lens = None if w.lengths is None else w.lengths[sel]
        _, _, st = orc.topk(w.scores[sel], w.k, lengths=lens, n=w.n, nthreads=cores)
        if st != 0:
            raise RuntimeError(f"oracle status {st}")

    for i in range(args.warmup):
        step(i)
    t = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = time.perf_counter() - t
    value = per_step * args.steps / dt
    used = min(cores, per_step)
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded numpy PCG64)", "impl": "reference",
        "config": {"workload": w.name, "rows": w.rows, "n": w.n, "k": w.k,
                   "values": w.meta, "reference_step": f"{per_step} rows per step"},
        "cpu_baseline": {"value": round(value, 2), "unit": UNIT, "cores": used,
                         "kind": "oracle",
                         "sample": f"{per_step} of {w.rows} rows per step, "
                                   f"{args.steps} timed steps"},
        "e2e": {"value": round(value, 2), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--workload", default="c4_normal_k512", choices=sorted(synth.CONFIGS))
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--pool", default=None,
                    help="POOL,PINNED: also build the layer-20 block pool in the same pass "
                         "(topk_select_pool; e.g. 2048,64)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--ref-rows", type=int, default=16)
    ap.add_argument("--timeline", action="store_true",
                    help="also record one launch with the instrumented build and summarise it")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world, rank, local = _dist()
    if args.gpus != world:
        ap.error(f"--gpus {args.gpus} but {world} rank(s): for N > 1 launch one rank per GPU "
                 "with torchrun (python -m torch.distributed.run --nproc-per-node N bench.py "
                 "--gpus N ...)")
    if world > 1:
        import torch.distributed as dist
        if args.impl == "reference":
            # rank 0 alone times the CPU oracle; the other ranks have no work
            if rank != 0:
                return
        else:
            dist.init_process_group("nccl")
    if args.impl == "reference":
        line = run_reference(args, world, rank)
    else:
        line = run_gb300(args, world, rank, local)
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if line is not None and rank == 0:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

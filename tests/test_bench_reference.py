"""The bench's reference arm (the CPU oracle timed on the host's cores) runs
without a GPU: its JSON line carries every key of the bench contract, and
under several ranks only rank 0 works and prints."""

from __future__ import annotations

import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run_reference(extra_env=None, workload="c1", gpus=1):
    env = dict(os.environ)
    for name in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        env.pop(name, None)
    env.update(extra_env or {})
    return subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
         workload, "--steps", "2", "--warmup", "3", "--gpus", str(gpus)],
        cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def _json_lines(stdout):
    return [json.loads(s) for s in stdout.splitlines() if s.startswith("{")]


def test_reference_line_has_the_contract_keys():
    out = _run_reference()
    assert out.returncode == 0, out.stderr[-2000:]
    lines = _json_lines(out.stdout)
    assert len(lines) == 1, out.stdout
    d = lines[0]
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 3
    assert d["value"] > 0 and d["ms_per_step"] > 0 and d["higher_is_better"] is True
    assert d["config"]["workload"] and d["config"]["rows"] >= 1 and d["config"]["k"] >= 1
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["unit"] == d["unit"]
    assert cb["cores"] >= 1 and cb["sample"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_under_two_ranks_prints_on_rank_zero_only():
    base = {"WORLD_SIZE": "2", "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": "29581"}
    r1 = _run_reference({**base, "RANK": "1", "LOCAL_RANK": "1"}, gpus=2)
    assert r1.returncode == 0, r1.stderr[-2000:]
    assert _json_lines(r1.stdout) == []
    r0 = _run_reference({**base, "RANK": "0", "LOCAL_RANK": "0"}, gpus=2)
    assert r0.returncode == 0, r0.stderr[-2000:]
    lines = _json_lines(r0.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2 and lines[0]["impl"] == "reference"


def test_bench_gpus_must_match_the_ranks():
    """--gpus N names the ranks the run has: N > 1 without torchrun's ranks
    (or a rank count that differs) is an error, not a silent one-GPU run."""
    out = _run_reference(gpus=2)
    assert out.returncode != 0 and "--gpus" in out.stderr
    out = _run_reference({"WORLD_SIZE": "2", "RANK": "1", "LOCAL_RANK": "1"}, gpus=4)
    assert out.returncode != 0 and "--gpus" in out.stderr


def test_bench_rejects_fewer_than_three_warmup_steps():
    out = subprocess.run(
        [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "c1",
         "--steps", "1", "--warmup", "2"],
        cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert out.returncode != 0 and "warmup" in out.stderr


def test_cpu_baseline_leg_reports_all_cores_and_one_thread():
    import bench
    from sparse_attention_indexer_row_gb300 import synth
    w = synth.make("c1")
    cb = bench.cpu_baseline(w, 0.2)
    assert cb["kind"] == "oracle" and cb["unit"] == bench.UNIT
    assert cb["value"] > 0 and 1 <= cb["cores"] <= w.rows and w.name in cb["sample"]
    one = cb["single_thread"]
    assert one["value"] > 0 and one["cores"] == 1 and one["unit"] == bench.UNIT

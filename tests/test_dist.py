"""Multi-rank host logic on CPU: two gloo ranks, no GPU."""

import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

from sparse_attention_indexer_row_gb300 import dist as D  # noqa: E402


def test_row_range_partitions_rows():
    for rows in (0, 1, 7, 64, 8192):
        for world in (1, 2, 3, 8):
            cover = []
            for r in range(world):
                a, b = D.row_range(rows, world, r)
                assert 0 <= a <= b <= rows
                cover.extend(range(a, b))
                assert b - a in (rows // world, rows // world + 1)
            assert cover == list(range(rows))
    with pytest.raises(ValueError):
        D.row_range(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from sparse_attention_indexer_row_gb300 import synth
        # each rank selects its own batch: rows are independent, no data exchange
        w = synth.uniform_pool(rows=2, n=4096, k=64, seed=D.rank_seed(1, rank))
        vals, idx, st = oracle.topk(w.scores, w.k)
        assert st == 0
        D.barrier()
        t = D.max_over_ranks(10.0 * (rank + 1))
        # gather a fingerprint of every rank's result on rank 0 (test only)
        fp = torch.tensor([float(idx.sum()), float(vals.sum())], dtype=torch.float64)
        got = [torch.zeros(2, dtype=torch.float64) for _ in range(world)]
        dist.all_gather(got, fp)
        out[rank] = (t, [g.tolist() for g in got])
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 20.0          # max over ranks
    assert out[0][1] == out[1][1]                   # both ranks see the same gather
    assert out[0][1][0] != out[0][1][1]             # per-rank batches differ

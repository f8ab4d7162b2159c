"""GPU parity of the layer-20 block pool (topk_select_pool) against the oracle.

The same pass returns the row's top-k (compared with the oracle's top-k) and
the block pool: blocks of eight positions scored by their largest value, the
newest blocks pinned, the best others added, ascending block indices
(compared with the oracle's block pool, bit for bit).
"""

from __future__ import annotations

import numpy as np
import pytest

import oracle
from tests.gpu_util import assert_bit_exact, host_threads, oracle_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def run_pool(x: np.ndarray, k: int, pool: int, pinned: int, lengths=None, ws=None):
    from sparse_attention_indexer_row_gb300 import binding as B
    rows, n = x.shape
    xt = torch.from_numpy(np.ascontiguousarray(x)).cuda()
    lt = None if lengths is None else torch.from_numpy(np.asarray(lengths, np.int32)).cuda()
    vals = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    out = torch.full((rows * pool + 64,), -777, dtype=torch.int32, device="cuda")
    if ws is None:
        nbytes = B.topk_pool_ws_bytes(rows, n, k, pool, pinned)
        assert nbytes > 0
        ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    rc = B.topk_select_pool(xt, rows, n, n, lt, k, vals, idx, pool, pinned, out, ws)
    assert rc == 0, rc
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert np.all(o[rows * pool:] == -777), "pool writes past rows * pool"
    rc, status = B.topk_ws_status(ws)
    assert rc == 0
    return vals.cpu().numpy(), idx.cpu().numpy(), o[:rows * pool].reshape(rows, pool), status, ws


def check(x, k, pool, pinned, lengths=None, what=""):
    v, i, got, status, ws = run_pool(x, k, pool, pinned, lengths=lengths)
    assert status == 0, status
    ov, oi = oracle_rows(x, k, lengths=lengths)
    assert_bit_exact(v, i, ov, oi, what + " top-k")
    want, st = oracle.block_pool(x, 8, pool, pinned, lengths=lengths, nthreads=host_threads())
    assert st == 0
    bad = np.nonzero(got != want)
    assert bad[0].size == 0, (f"{what}: {bad[0].size} pool slots differ; first row {bad[0][0]} "
                              f"slot {bad[1][0]}: gpu {got[bad[0][0], bad[1][0]]} vs oracle "
                              f"{want[bad[0][0], bad[1][0]]}")
    return ws


def test_pool_small_rows():
    rng = np.random.default_rng(31)
    x = rng.uniform(-1, 1, size=(4, 16384)).astype(np.float32)
    check(x, 512, 64, 8, what="4x16384")
    check(x, 512, 2048, 0, what="no pin")
    check(x, 64, 2048 + 40, 40, what="largest selection")
    check(x, 512, 3000, 1000, what="whole row (2048 blocks) in the pool")
    check(x, 512, 10, 10, what="pins only")


def test_pool_long_rows_1m():
    rng = np.random.default_rng(32)
    x = rng.standard_normal((8, 1 << 20)).astype(np.float32)
    check(x, 512, 2048, 64, what="8x1M")


def test_pool_variable_lengths():
    rng = np.random.default_rng(33)
    rows, n = 24, 131072
    x = rng.standard_normal((rows, n)).astype(np.float32)
    lengths = rng.integers(0, n + 1, size=rows).astype(np.int32)
    lengths[:6] = [0, 1, 7, 8, 9, 8 * 33 + 3]
    check(x, 512, 256, 32, lengths=lengths, what="varlen")


def test_pool_ties_and_special_values():
    rng = np.random.default_rng(34)
    rows, n = 6, 65536
    x = np.round(rng.standard_normal((rows, n)) * 2).astype(np.float32)   # heavy ties
    x[1] = np.where(rng.random(n) < 0.5, np.float32(0.0), np.float32(-0.0))  # signed zeros only
    x[2][rng.random(n) < 0.01] = np.inf
    x[3][rng.random(n) < 0.3] = -np.inf
    x[4] = -np.inf
    x[4][::4096] = -0.0
    x[5] = np.sort(x[5])
    check(x, 512, 700, 20, what="ties")


def test_pool_argument_errors():
    from sparse_attention_indexer_row_gb300 import binding as B
    x = torch.zeros((2, 1024), dtype=torch.float32, device="cuda")
    v = torch.empty((2, 8), dtype=torch.float32, device="cuda")
    i = torch.empty((2, 8), dtype=torch.int32, device="cuda")
    out = torch.empty((2 * 4000,), dtype=torch.int32, device="cuda")
    ws = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    for pool, pinned in [(0, 0), (4, 5), (4, -1), (2100, 10)]:
        assert B.topk_pool_ws_bytes(2, 1024, 8, pool, pinned) == 0
        assert B.topk_select_pool(x, 2, 1024, 1024, None, 8, v, i, pool, pinned, out, ws) == \
            B.TOPK_ERR_ARG
    assert B.topk_select_pool(x, 2, 1024, 1024, None, 8, v, i, 4, 1, None, ws) == B.TOPK_ERR_NULL


def test_pool_workspace_reuse():
    rng = np.random.default_rng(35)
    x = rng.standard_normal((3, 1 << 18)).astype(np.float32)
    _, _, first, _, ws = run_pool(x, 256, 512, 16)
    y = rng.standard_normal((3, 1 << 18)).astype(np.float32)
    v, i, got, status, _ = run_pool(y, 256, 512, 16, ws=ws)
    assert status == 0
    want, st = oracle.block_pool(y, 8, 512, 16, nthreads=host_threads())
    assert st == 0 and np.array_equal(got, want)
    ov, oi = oracle_rows(y, 256)
    assert_bit_exact(v, i, ov, oi, "reuse top-k")

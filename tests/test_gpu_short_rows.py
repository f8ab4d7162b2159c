"""GPU parity of the short-row path: batches of at least as many rows as the
device has SMs, rows of at most 65,536 elements, go to one CTA per row (the
same threshold-and-tray method without the role split, the causal prefill's
shape).  Every case is compared bit for bit with the oracle.

Each row of that path is sorted exactly once (the workspace's per-row sort
count is 1), which the first test also checks: the cases below do run the
short-row kernel, not the selection kernel's queue plan.
"""

from __future__ import annotations

import numpy as np
import pytest

from tests.gpu_util import assert_bit_exact, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROWS = 300  # (at least the SM count: the queue plan's batches)


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


@pytest.mark.parametrize("n", [1, 100, 4095, 4096, 4097, 20000, 65536])
@pytest.mark.parametrize("k", [1, 33, 512, 2048])
def test_short_rows_lengths_and_k(n, k):
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(n * 7 + k)
    x = rng.standard_normal((ROWS, n)).astype(np.float32)
    lengths = rng.integers(0, n + 1, size=ROWS).astype(np.int32)
    lengths[:4] = [0, 1, min(n, k), n]
    gv, gi, ws = run_gpu(x, k, lengths=lengths, return_ws=True)
    ov, oi = oracle_rows(x, k, lengths=lengths)
    assert_bit_exact(gv, gi, ov, oi, f"short rows n={n} k={k}")
    rc, surv, sorts, adm = B.topk_ws_stats(ws, ROWS, n, k, 0)
    assert rc == 0 and all(s == 1 for s in sorts), "every row sorted once (the short-row path)"
    rc, status = B.topk_ws_status(ws)
    assert rc == 0 and status == 0


@pytest.mark.parametrize("layout", ["ascending", "descending", "levels", "specials"])
@pytest.mark.parametrize("k", [64, 512, 2048])
def test_short_rows_layouts(layout, k):
    """Rows that flood the tray (ascending: every chunk sets a record), heavy
    ties (a few levels, the smaller index first), and the special values."""
    rng = np.random.default_rng(["ascending", "descending", "levels", "specials"].index(layout) * 10000 + k)
    n = 50000
    if layout == "ascending":
        x = np.sort(rng.standard_normal((ROWS, n)).astype(np.float32), axis=1)
    elif layout == "descending":
        x = -np.sort(rng.standard_normal((ROWS, n)).astype(np.float32), axis=1)
    elif layout == "levels":
        x = (rng.integers(0, 4, size=(ROWS, n)) - 1.5).astype(np.float32)
    else:
        vals = np.array([-np.inf, -1.0, -0.0, 0.0, 1.0, np.inf, np.float32(3.4e38)], np.float32)
        x = vals[rng.integers(0, len(vals), size=(ROWS, n))]
    lengths = rng.integers(n // 2, n + 1, size=ROWS).astype(np.int32)
    gv, gi = run_gpu(x, k, lengths=lengths)
    ov, oi = oracle_rows(x, k, lengths=lengths)
    assert_bit_exact(gv, gi, ov, oi, f"short rows {layout} k={k}")


@pytest.mark.parametrize("pad", [1, 3, 16])
def test_short_rows_misaligned_strides(pad):
    """Row starts off the 16-byte grid take scalar loads; the gaps between
    rows hold NaN that no row may read."""
    n, k = 9000, 512
    rng = np.random.default_rng(pad)
    x = np.full((ROWS, n + pad), np.nan, np.float32)
    x[:, :n] = rng.standard_normal((ROWS, n)).astype(np.float32)
    gv, gi = run_gpu(x, k, n=n)
    ov, oi = oracle_rows(x[:, :n], k)
    assert_bit_exact(gv, gi, ov, oi, f"short rows stride pad {pad}")


def test_short_rows_nan_and_bad_lengths():
    """NaN is left out of the selection and flagged; lengths outside [0, n]
    are clamped and flagged."""
    from sparse_attention_indexer_row_gb300 import binding as B
    n, k = 30000, 256
    rng = np.random.default_rng(5)
    x = rng.standard_normal((ROWS, n)).astype(np.float32)
    nan_rows = [3, 100, 299]
    for r in nan_rows:
        x[r, rng.choice(n, size=50, replace=False)] = np.nan
    lengths = np.full(ROWS, n, np.int32)
    lengths[7] = n + 5
    lengths[8] = -2
    gv, gi, ws = run_gpu(x, k, lengths=lengths, return_ws=True)
    rc, status = B.topk_ws_status(ws)
    assert rc == 0 and status == (B.TOPK_STATUS_NAN | B.TOPK_STATUS_BAD_LENGTH), status
    clamped = np.clip(lengths, 0, n)
    clean = [r for r in range(ROWS) if r not in nan_rows]
    ov, oi = oracle_rows(x, k, lengths=clamped, rows=clean)
    assert_bit_exact(gv[clean], gi[clean], ov, oi, "short rows without NaN")
    for r in nan_rows:
        keep = np.nonzero(~np.isnan(x[r]))[0]
        v1, i1 = oracle_rows(x[r, keep][None, :], k)
        i1 = np.where(i1[0] >= 0, keep[np.maximum(i1[0], 0)], -1).astype(np.int32)
        assert_bit_exact(gv[r:r + 1], gi[r:r + 1], v1, i1[None], f"NaN row {r}")


def test_short_rows_repeated_calls_one_workspace():
    """The shared queue is empty again after every call."""
    from sparse_attention_indexer_row_gb300 import binding as B
    rows, n, k = 400, 65536, 512
    rng = np.random.default_rng(9)
    ws = torch.zeros(B.topk_ws_bytes_ex(rows, n, k, 0), dtype=torch.uint8, device="cuda")
    for call in range(3):
        x = rng.standard_normal((rows, n)).astype(np.float32)
        lengths = (8 * (np.arange(rows) + 1) * (1 + call)).astype(np.int32).clip(0, n)
        gv, gi = run_gpu(x, k, lengths=lengths, ws=ws)
        ov, oi = oracle_rows(x, k, lengths=lengths)
        assert_bit_exact(gv, gi, ov, oi, f"call {call}")

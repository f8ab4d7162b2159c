"""GPU parity of the speculative start and its rescan.

A long piece may start from a threshold that its first 8192-element units
(three for k <= 512, four above) only make likely.  These inputs are built so that, with units visited in
address order, every piece's sample promises more large scores than the row
holds: the start misses, the row must be selected again from global memory,
and the result must still equal the oracle bit for bit (with the status word's
rescan bit set).  A control on i.i.d. data checks that the speculation does
not miss there.
"""

from __future__ import annotations

import numpy as np
import pytest

from tests.gpu_util import assert_bit_exact, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

UNIT = 8192


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _warp_slot(w: int, lane: int) -> int:
    """Offset inside a unit of the first element a selector warp `w`, lane
    `lane` reads during the warm start (thread 32 w + lane reads float4
    32 w + lane first)."""
    return 4 * (32 * w + lane)


def _plant_piece(x, row, u0, base_value, per_unit_after=2, per_warp=2):
    """Large scores in a piece whose first unit is u0: `per_warp` per selector
    warp share of unit u0, then `per_unit_after` in each of the next three
    units, all above the first unit's (a sample of three units sees the
    first two of those)."""
    for w in range(8):
        for lane in range(per_warp):
            x[row, u0 * UNIT + _warp_slot(w, lane)] = base_value + 100 + per_warp * w + lane
    for q in range(1, 4):
        for j in range(per_unit_after):
            x[row, (u0 + q) * UNIT + 1000 + 37 * j] = base_value + 200 + 10 * q + j


def _status(ws):
    from sparse_attention_indexer_row_gb300 import binding as B
    rc, status = B.topk_ws_status(ws)
    assert rc == 0
    return status


@pytest.mark.parametrize("quantised", [False, True])
def test_unsplit_row_rescan(quantised):
    """One row of 16 units (one piece, no split), k = 64: the three sample
    units hold 39 scores at or above the speculative bound (the need is 30),
    the row only 53 < 64."""
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(11)
    n, k = 16 * UNIT, 64
    if quantised:   # heavy ties among the small scores
        x = (rng.integers(0, 16, size=(1, n)).astype(np.float32) / 8 - 2).astype(np.float32)
    else:
        x = (rng.standard_normal((1, n)).astype(np.float32) * 0.1 - 1).astype(np.float32)
    _plant_piece(x, 0, 0, 0.0, per_unit_after=14)
    gv, gi, ws = run_gpu(x, k, split=1, flags=B.TOPK_FLAG_IDENTITY_ORDER, return_ws=True)
    ov, oi = oracle_rows(x, k)
    assert_bit_exact(gv, gi, ov, oi, "unsplit rescan")
    assert _status(ws) == B.TOPK_STATUS_RESCAN


@pytest.mark.parametrize("split", [0, 8])
def test_split_row_rescan(split):
    """One row of 128 units in eight pieces of 16 (the flat plan, or eight
    explicit segments), k = 64: each piece's sample supports a bound that
    only 17 scores of the row reach; the leader finds the merged 64th word
    below the largest bound and selects the row again."""
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(12)
    n, k = 128 * UNIT, 64
    x = (rng.standard_normal((1, n)).astype(np.float32) * 0.1 - 1).astype(np.float32)
    for piece in range(8):
        _plant_piece(x, 0, 16 * piece, 1000.0 * piece)
    gv, gi, ws = run_gpu(x, k, split=split, flags=B.TOPK_FLAG_IDENTITY_ORDER, return_ws=True)
    ov, oi = oracle_rows(x, k)
    assert_bit_exact(gv, gi, ov, oi, f"split rescan (split={split})")
    assert _status(ws) == B.TOPK_STATUS_RESCAN
    # the workspace is clean again: a second call on i.i.d. data of the same
    # shape neither misses nor inherits the row's bounds
    y = rng.standard_normal((1, n)).astype(np.float32)
    gv, gi = run_gpu(y, k, split=split, ws=ws)
    ov, oi = oracle_rows(y, k)
    assert_bit_exact(gv, gi, ov, oi, "after rescan")
    assert _status(ws) == 0


@pytest.mark.parametrize("split", [1, 0])
def test_k2048_row_rescan(split):
    """k = 2048 on a 1M row (one piece, or eight): the speculative candidates
    are the warps' 7th-largest-key bounds; eight planted scores per warp share
    of each piece's first unit and fifty in each of the next three give the
    sample 214 scores above them (the need is 160), the row fewer than 2048."""
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(14)
    n, k = 128 * UNIT, 2048
    x = (rng.standard_normal((1, n)).astype(np.float32) * 0.1 - 1).astype(np.float32)
    starts = [0] if split == 1 else [16 * p for p in range(8)]
    for piece, u0 in enumerate(starts):
        _plant_piece(x, 0, u0, 1000.0 * piece, per_unit_after=50, per_warp=8)
    gv, gi, ws = run_gpu(x, k, split=split, flags=B.TOPK_FLAG_IDENTITY_ORDER, return_ws=True)
    ov, oi = oracle_rows(x, k)
    assert_bit_exact(gv, gi, ov, oi, f"k2048 rescan (split={split})")
    assert _status(ws) == B.TOPK_STATUS_RESCAN


def test_k2048_iid_rows_start_speculatively():
    """k = 2048 on i.i.d. 1M rows: far fewer admitted words than a proven
    start gives (about 43,000 per row), and no rescan."""
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(15)
    rows, n, k = 8, 1 << 20, 2048
    x = rng.standard_normal((rows, n)).astype(np.float32)
    gv, gi, ws = run_gpu(x, k, return_ws=True)
    ov, oi = oracle_rows(x, k)
    assert_bit_exact(gv, gi, ov, oi, "k2048 iid")
    assert _status(ws) == 0
    rc, surv, _, adm = B.topk_ws_stats(ws, rows, n, k, 0)
    assert rc == 0 and min(surv) >= k
    assert max(adm) < 8 * k, adm


@pytest.mark.parametrize("rows,split", [(4, 0), (4, 1), (16, 0)])
def test_iid_rows_start_speculatively_without_rescan(rows, split):
    """On i.i.d. Normal rows of 1M the speculative start is taken (far fewer
    elements are admitted than the row's 3.6 k target plus the warm-start
    window would allow without it) and never misses."""
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(13 + rows)
    n, k = 1 << 20, 512
    x = rng.standard_normal((rows, n)).astype(np.float32)
    gv, gi, ws = run_gpu(x, k, split=split, return_ws=True)
    ov, oi = oracle_rows(x, k)
    assert_bit_exact(gv, gi, ov, oi, "iid speculative")
    assert _status(ws) == 0
    rc, surv, _, adm = B.topk_ws_stats(ws, rows, n, k, split)
    assert rc == 0
    assert min(surv) >= k
    assert max(adm) < 16 * k, adm

"""GPU parity of the queue plan: batches of many rows take (row, segment)
items from a shared queue, longest rows first, instead of a fixed deal.

Results must equal the oracle whatever order the CTAs take the items in, and
the queue must be empty again after every call (a second call on the same
workspace would otherwise skip items).
"""

from __future__ import annotations

import numpy as np
import pytest

from tests.gpu_util import assert_bit_exact, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def test_queue_varlen_many_rows_longest_first():
    """600 rows of up to 12 units with random lengths (some empty, some
    shorter than k): a shared queue sorted by length."""
    rng = np.random.default_rng(41)
    rows, n, k = 600, 12 * 8192 - 5, 256
    x = rng.standard_normal((rows, n)).astype(np.float32)
    lengths = rng.integers(0, n + 1, size=rows).astype(np.int32)
    lengths[:5] = [0, 1, 255, 256, n]
    gv, gi = run_gpu(x, k, lengths=lengths)
    ov, oi = oracle_rows(x, k, lengths=lengths)
    assert_bit_exact(gv, gi, ov, oi, "queue varlen")


def test_queue_full_rows_and_repeated_calls():
    """300 full rows (queue in index order), three calls on one workspace:
    each call must see every item."""
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(42)
    rows, n, k = 300, 40000, 512
    ws = torch.zeros(B.topk_ws_bytes_ex(rows, n, k, 0), dtype=torch.uint8, device="cuda")
    for call in range(3):
        x = rng.standard_normal((rows, n)).astype(np.float32)
        gv, gi = run_gpu(x, k, ws=ws)
        ov, oi = oracle_rows(x, k)
        assert_bit_exact(gv, gi, ov, oi, f"queue call {call}")
    rc, status = B.topk_ws_status(ws)
    assert rc == 0 and status == 0


def test_queue_with_explicit_segments():
    """Many rows split into explicit segments: segments of a row are
    separate queue items that meet in the leader merge."""
    rng = np.random.default_rng(43)
    rows, n, k = 160, 5 * 8192, 128
    x = rng.standard_normal((rows, n)).astype(np.float32)
    lengths = rng.integers(1, n + 1, size=rows).astype(np.int32)
    gv, gi = run_gpu(x, k, lengths=lengths, split=2)
    ov, oi = oracle_rows(x, k, lengths=lengths)
    assert_bit_exact(gv, gi, ov, oi, "queue segments")

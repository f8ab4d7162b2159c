"""Bounded waits that run out: the call finishes, reports TOPK_STATUS_TIMEOUT,
and the same workspace then serves a normal call bit-exactly.

TOPK_FLAG_TEST_STALL makes the copy producer of every CTA stop for good in
front of its fourth ring stage: that stage's full barrier never completes and
the producer publishes no end marker.  No copy is left in flight (the producer
waits for the ones it issued before it leaves).  What runs out, by k:

* k = 512 on rows of 32 units: the warm start uses the first three units, the
  filter warps take stages 0-2 and then wait on stage 3's barrier until the
  wait gives up; the selectors' poll for the piece's end gives up after it.
* k = 1024 on a row of 64 units: the warm start needs four units, so the
  starting threshold is never published; the filter warps' wait for it gives
  up, then the selectors' poll.

Every wait in the kernel is bounded (the failure-detection design of the
selector: a status bit, never a trap), so these calls end by themselves.
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


@pytest.mark.parametrize("rows,n,k", [(2, 1 << 18, 512), (1, 1 << 19, 1024)])
def test_stalled_copies_time_out_and_the_workspace_stays_usable(rows, n, k):
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(rows * 1000 + k)
    x = rng.standard_normal((rows, n)).astype(np.float32)
    nbytes = B.topk_ws_bytes_ex(rows, n, k, 1)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    # the stalled call: it must return, with the timeout bit set
    run_gpu(x, k, split=1, ws=ws, flags=B.TOPK_FLAG_TEST_STALL)
    rc, status = B.topk_ws_status(ws)
    assert rc == 0
    assert status & B.TOPK_STATUS_TIMEOUT, status
    # the status word is read and cleared; a normal call on the same
    # workspace is exact and clean
    gv, gi = run_gpu(x, k, split=1, ws=ws)
    ov, oi = oracle_rows(x, k)
    assert_bit_exact(gv, gi, ov, oi, "after a timed-out call")
    rc, status = B.topk_ws_status(ws)
    assert rc == 0 and (status & B.TOPK_STATUS_TIMEOUT) == 0, status
    # the tickets (u32[rows] from byte 256) are still zero
    assert torch.all(ws[256:256 + 4 * rows] == 0)

"""topk_select_noalloc: the entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc where they select: real-time paths that
forbid allocation once running, and plug-ins whose host framework owns all
device memory and hands them only input and output buffers.
topk_select_noalloc takes no workspace and uses the library's built-in device
array instead.  This test calls it through the C ABI twice in a row (a batch
of split long rows with a leader merge, then a batch with per-row lengths and
another k, on the same array) and checks each result bit for bit (the
tolerance every parity test here uses) against topk_select with a
caller-owned workspace and against the CPU oracle.  It sits in its own file,
collected last, and holds no state between tests, so it passes alone or after
the rest of the suite.
"""

import numpy as np
import pytest

from tests.gpu_util import assert_bit_exact, oracle_rows

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _with_workspace(B, x, lengths, n, k):
    rows = x.shape[0]
    ws = torch.zeros(B.topk_ws_bytes(rows, n, k), dtype=torch.uint8, device="cuda")
    v = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    i = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    assert B.topk_select(x, rows, n, x.stride(0), lengths, k, v, i, ws) == B.TOPK_OK
    return v, i


def _no_alloc(B, x, lengths, n, k):
    rows = x.shape[0]
    v = torch.full((rows, k), 7.0, dtype=torch.float32, device="cuda")
    i = torch.full((rows, k), 7, dtype=torch.int32, device="cuda")
    status = torch.full((1,), 0xFFFF, dtype=torch.int32, device="cuda")
    assert B.topk_select_noalloc(x, rows, n, x.stride(0), lengths, k, v, i, status) == B.TOPK_OK
    return v, i, int(status.item())


def _check(B, x_host, lengths_host, n, k, what):
    x = torch.from_numpy(x_host).cuda()
    lengths = None if lengths_host is None else torch.from_numpy(lengths_host).cuda()
    v, i, st = _no_alloc(B, x, lengths, n, k)
    vw, iw = _with_workspace(B, x, lengths, n, k)
    torch.cuda.synchronize()
    assert st == 0, st
    # against the entry point with a caller-owned workspace
    assert torch.equal(i, iw), what
    assert torch.equal(v.view(torch.int32), vw.view(torch.int32)), what
    # and against the oracle
    ov, oi = oracle_rows(x_host, k, lengths=lengths_host, n=n)
    assert_bit_exact(v.cpu().numpy(), i.cpu().numpy(), ov, oi, what)


def test_two_calls_match_the_workspace_entry_point_and_the_oracle():
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(2024)
    # call 1: a short batch of long rows (persistent plan, split rows, leader merge)
    x1 = rng.standard_normal((8, 300_000)).astype(np.float32)
    _check(B, x1, None, 300_000, 512, "no-alloc call 1")
    # call 2, straight after on the same array: varying lengths and another k
    x2 = np.round(rng.standard_normal((40, 70_000)) * 3).astype(np.float32)
    lengths = rng.integers(0, 70_001, size=40).astype(np.int32)
    _check(B, x2, lengths, 70_000, 1000, "no-alloc call 2")


def test_rejects_shapes_beyond_the_built_in_workspace():
    from sparse_attention_indexer_row_gb300 import binding as B
    rows = 1 << 20          # one CTA per row: about 20 bytes of workspace per row
    assert B.topk_ws_bytes(rows, 64, 8) > (16 << 20)
    assert B.topk_select_noalloc(1 << 12, rows, 64, 64, None, 8, 1 << 12, 1 << 12) == \
        B.TOPK_ERR_NOSPACE

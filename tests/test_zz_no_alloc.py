"""topk_select_noalloc: the entry point for callers that cannot allocate.

Some callers cannot call cudaMalloc where they select (code running under
CUDA-graph capture that must not allocate, allocation-free real-time paths,
plug-ins whose host framework owns all device memory).  topk_select_noalloc
takes no workspace and uses the library's built-in device array instead.  This
test calls it through the C ABI twice in a row and checks each result against
topk_select with a caller-owned workspace, bit for bit (the tolerance every
parity test here uses).  It sits in its own file, collected last, and holds no
state between tests, so it passes alone or after the rest of the suite.
"""

import numpy as np
import pytest

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


def _same(a, b):
    (va, ia), (vb, ib) = a, b
    torch.cuda.synchronize()
    assert torch.equal(ia, ib)
    assert torch.equal(va.view(torch.int32), vb.view(torch.int32))


def test_two_calls_match_the_workspace_entry_point():
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(2024)
    # call 1: a short batch of long rows (persistent plan, split rows, leader merge)
    x1 = torch.from_numpy(rng.standard_normal((8, 300_000)).astype(np.float32)).cuda()
    v, i, st = _no_alloc(B, x1, None, 300_000, 512)
    _same((v, i), _with_workspace(B, x1, None, 300_000, 512))
    assert st == 0
    # call 2, straight after on the same array: varying lengths and another k
    x2 = torch.from_numpy(np.round(rng.standard_normal((40, 70_000)) * 3).astype(np.float32)).cuda()
    lengths = torch.from_numpy(rng.integers(0, 70_001, size=40).astype(np.int32)).cuda()
    v, i, st = _no_alloc(B, x2, lengths, 70_000, 1000)
    _same((v, i), _with_workspace(B, x2, lengths, 70_000, 1000))
    assert st == 0


def test_rejects_shapes_beyond_the_built_in_workspace():
    from sparse_attention_indexer_row_gb300 import binding as B
    rows = 1 << 20          # one CTA per row: about 20 bytes of workspace per row
    assert B.topk_ws_bytes(rows, 64, 8) > (16 << 20)
    assert B.topk_select_noalloc(1 << 12, rows, 64, 64, None, 8, 1 << 12, 1 << 12) == \
        B.TOPK_ERR_NOSPACE

"""The instrumented builds of the library on the GPU.

* ``libtopk_gb300_debug.so`` (``-DTOPK_DEBUG_BOUNDS=1``) checks every shared-
  and global-memory write index the selection computes at run time (tray,
  kept list, leader-merge area, partial lists, outputs, block maxima, pool
  output).  A failed check sets TOPK_STATUS_BOUNDS and skips the write.  It
  stands in for a memory checker: on a spread of shapes that reach every plan
  and path (flat shares with leader merges, round-robin items, the queue,
  ragged and misaligned rows, k up to 2048, the rescan, the block pool) no
  check may fail, and the results must still equal the oracle bit for bit.
* ``libtopk_gb300_timeline.so`` (``-DTOPK_TIMELINE=1``) stamps per-CTA events;
  its table must describe the launch consistently and its results must be
  exact as well.
"""

from __future__ import annotations

import numpy as np
import pytest

from sparse_attention_indexer_row_gb300 import synth
from tests.gpu_util import assert_bit_exact, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _variant(name):
    from sparse_attention_indexer_row_gb300 import binding as B
    from sparse_attention_indexer_row_gb300 import build
    path = build.variant_path(name)
    if build.needs_build(path):
        build.build_variant(name)
    return B.load_library(path)


@pytest.fixture(scope="module")
def debug_lib():
    return _variant("debug")


def _cases():
    """(name, scores, lengths, n, k, split, flags)"""
    from tests.test_gpu_speculative import UNIT, _plant_piece
    rng = np.random.default_rng(404)
    x = rng.standard_normal((3, 300_000)).astype(np.float32)
    yield "3 x 300K split rows k512", x, None, 300_000, 512, 0, 0
    yield "3 x 300K split=7 k2048", x, None, 300_000, 2048, 7, 0
    w = synth.normal_varlen()
    yield "64 x 131072 varlen", w.scores, w.lengths, w.n, w.k, 0, 0
    w = synth.relu_mix(rows=4)
    yield "4 x 1M decode mix", w.scores, None, w.n, w.k, 0, 0
    w = synth.long_rows("sorted", rows=16, k=512)
    yield "16 x 1M sorted", w.scores, None, w.n, 512, 0, 0
    w = synth.long_rows("quant", rows=16, k=2048)
    yield "16 x 1M quant k2048", w.scores, None, w.n, 2048, 0, 0
    y = rng.standard_normal((300, 20_000)).astype(np.float32)
    lengths = rng.integers(0, 20_001, size=300).astype(np.int32)
    yield "300 rows queue plan", y, lengths, 20_000, 1000, 0, 0
    yield "300 rows short-row path k2048", y, lengths, 20_000, 2048, 0, 0
    c = rng.standard_normal((600, 65536)).astype(np.float32)
    yield "600 causal rows k512 (short-row path)", c, \
        np.minimum(104 * (np.arange(600) + 1), 65536).astype(np.int32), 65536, 512, 0, 0
    buf = np.full((5, 9003), np.nan, dtype=np.float32)
    buf[:, :9000] = rng.standard_normal((5, 9000))
    yield "misaligned rows", buf, np.array([9000, 8999, 4097, 1025, 3], np.int32), 9000, 300, 0, 0
    # eight pieces whose samples promise too much: the leader selects the row again
    z = (rng.standard_normal((1, 128 * UNIT)).astype(np.float32) * 0.1 - 1).astype(np.float32)
    for piece in range(8):
        _plant_piece(z, 0, 16 * piece, 1000.0 * piece)
    yield "planted speculative misses", z, None, 128 * UNIT, 64, 0, 1


def test_debug_build_no_bound_fails_and_exact(debug_lib):
    from sparse_attention_indexer_row_gb300 import binding as B
    for name, x, lengths, n, k, split, flags in _cases():
        gv, gi, ws = run_gpu(x, k, lengths=lengths, n=n, split=split, flags=flags,
                             return_ws=True, lib=debug_lib)
        rc, status = B.topk_ws_status(ws)
        assert rc == 0
        assert (status & B.TOPK_STATUS_BOUNDS) == 0, (name, status)
        if name == "planted speculative misses":
            assert status & B.TOPK_STATUS_RESCAN, status
        ov, oi = oracle_rows(x, k, lengths=lengths, n=n)
        assert_bit_exact(gv, gi, ov, oi, name)


def test_debug_build_pool(debug_lib):
    import oracle
    from sparse_attention_indexer_row_gb300 import binding as B
    w = synth.long_rows("quant", rows=8, k=512)
    x = torch.from_numpy(w.scores).cuda()
    pool, pinned = 2048, 64
    ws = torch.zeros(B.topk_pool_ws_bytes(w.rows, w.n, w.k, pool, pinned), dtype=torch.uint8,
                     device="cuda")
    v = torch.empty((w.rows, w.k), dtype=torch.float32, device="cuda")
    i = torch.empty((w.rows, w.k), dtype=torch.int32, device="cuda")
    out = torch.empty((w.rows, pool), dtype=torch.int32, device="cuda")
    rc = debug_lib.topk_select_pool(x.data_ptr(), w.rows, w.n, w.n, None, w.k, v.data_ptr(),
                                    i.data_ptr(), pool, pinned, out.data_ptr(), ws.data_ptr(), None)
    assert rc == 0
    torch.cuda.synchronize()
    rc, status = B.topk_ws_status(ws)
    assert rc == 0 and (status & B.TOPK_STATUS_BOUNDS) == 0, status
    want, st = oracle.block_pool(w.scores, 8, pool, pinned, nthreads=8)
    assert np.array_equal(out.cpu().numpy(), want)


def test_timeline_build_records_the_launch():
    from sparse_attention_indexer_row_gb300 import timeline as TLM
    lib = _variant("timeline")
    w = synth.long_rows("normal", rows=64, k=512)
    x = torch.from_numpy(w.scores).cuda()
    v = torch.empty((w.rows, w.k), dtype=torch.float32, device="cuda")
    i = torch.empty((w.rows, w.k), dtype=torch.int32, device="cuda")
    from sparse_attention_indexer_row_gb300 import binding as B
    ws = torch.zeros(B.topk_ws_bytes(w.rows, w.n, w.k), dtype=torch.uint8, device="cuda")

    def call(l):
        assert l.topk_select(x.data_ptr(), w.rows, w.n, w.n, None, w.k, v.data_ptr(),
                             i.data_ptr(), ws.data_ptr(), None) == 0

    table = TLM.record(lib, call)
    ov, oi = oracle_rows(w.scores[:4], w.k)
    assert_bit_exact(v.cpu().numpy()[:4], i.cpu().numpy()[:4], ov, oi, "timeline build")
    s = TLM.summarize(table, 2000.0)
    assert s["ctas"] >= 64
    t = table.astype(np.int64)[:s["ctas"]]
    start, setup, exit_ = t[:, 0], t[:, 1], t[:, 7]
    assert np.all(start > 0) and np.all(setup >= start) and np.all(exit_ >= setup)
    # every CTA of the flat plan took at least one piece; its first piece's
    # threshold came before the selectors finished it
    assert np.all((t[:, 8] >> 32) >= 1)
    theta0, done0 = t[:, TLM.PIECE0], t[:, TLM.PIECE0 + 3]
    assert np.all(theta0 > 0) and np.all(done0 >= theta0)
    assert 0 < s["span_us"] < 10_000
    # the normal build has no table
    assert B.LIB.topk_timeline_read(np.zeros(4, np.uint64).ctypes.data, None) == B.TOPK_ERR_ARG

"""The C-ABI library loads, exports every declared symbol, and validates
arguments on the host (no kernel launches: these run without a GPU)."""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER_DIR = os.path.join(ROOT, "include")


def _declared_functions():
    names = set()
    for fn in os.listdir(HEADER_DIR):
        if fn.endswith(".h"):
            text = open(os.path.join(HEADER_DIR, fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            for m in re.finditer(r"^\s*[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M):
                if not m.group(0).lstrip().startswith("#"):
                    names.add(m.group(1))
    return names


@pytest.fixture(scope="module")
def B():
    from sparse_attention_indexer_row_gb300 import build
    if build.needs_build():
        build.build_library()
    from sparse_attention_indexer_row_gb300 import binding
    return binding


def test_every_declared_symbol_is_exported(B):
    declared = _declared_functions()
    assert {"topk_ws_bytes", "topk_select"} <= declared
    lib = ctypes.CDLL(str(B._LIB_PATH))
    for name in declared:
        assert hasattr(lib, name), name
    assert declared == set(B.SIGNATURES), declared ^ set(B.SIGNATURES)


def test_ws_bytes_and_plan(B):
    assert B.topk_ws_bytes(0, 1, 1) > 0
    assert B.topk_ws_bytes(4, 0, 512) == 0
    assert B.topk_ws_bytes(4, 16, 0) == 0
    assert B.topk_ws_bytes(4, 16, 2049) == 0
    assert B.topk_ws_bytes(4, 1 << 31, 8) == 0
    # long rows in a short batch are split; big batches are not
    assert B.topk_split_plan(64, 1 << 20) > 1
    assert B.topk_split_plan(8192, 65536) == 1
    # partial lists: rows * split * next_pow2(k) * 8 bytes on top of the counters
    s = B.topk_split_plan(64, 1 << 20)
    assert B.topk_ws_bytes(64, 1 << 20, 512) >= 64 * s * 512 * 8
    assert B.topk_ws_bytes_ex(64, 1 << 20, 1000, 1) < 64 * 1024 * 8
    assert B.topk_ws_bytes_ex(64, 1 << 20, 1000, 65) == 0


def test_host_validation_returns_codes(B):
    # rows = 0 enqueues nothing and succeeds
    assert B.topk_select(0, 0, 100, 100, None, 5, 0, 0, 0) == B.TOPK_OK
    assert B.topk_select(0, 2, 100, 99, None, 5, 0, 0, 0) == B.TOPK_ERR_SHAPE
    assert B.topk_select(0, 2, 100, 100, None, 0, 0, 0, 0) == B.TOPK_ERR_SHAPE
    assert B.topk_select(0, 2, 100, 100, None, 2049, 0, 0, 0) == B.TOPK_ERR_SHAPE
    assert B.topk_select(0, -1, 100, 100, None, 5, 0, 0, 0) == B.TOPK_ERR_SHAPE
    assert B.topk_select(0, 2, 100, 100, None, 5, 0, 0, 0) == B.TOPK_ERR_NULL
    assert B.topk_select(4096, 2, 100, 100, None, 5, 4096, 4096, 0) == B.TOPK_ERR_WS
    assert B.topk_select(4096, 2, 100, 100, None, 5, 4096, 4096, 4096 + 16) == B.TOPK_ERR_WS
    assert B.topk_select_ex(4096, 2, 100, 100, None, 5, 4096, 4096, 4096, None, 65) == \
        B.TOPK_ERR_SHAPE
    assert B.topk_visit_order(0, 0, 0, 1, 4096) == B.TOPK_ERR_ARG
    assert B.topk_visit_order(257, 0, 0, 1, 4096) == B.TOPK_ERR_ARG
    assert B.topk_ws_status(0)[0] == B.TOPK_ERR_WS


def test_pool_sizes_and_argument_codes(B):
    """The block pool's workspace size and its host-side checks (no launch)."""
    plain = B.topk_ws_bytes_ex(64, 1 << 20, 512, 0)
    pool = B.topk_pool_ws_bytes(64, 1 << 20, 512, 2048, 64)
    # the selection's own workspace plus one fp32 block maximum per 8 scores
    assert pool >= plain + 64 * (1 << 17) * 4
    assert B.topk_pool_ws_bytes(64, 1 << 20, 512, 2048 + 64, 64) == pool
    for p, q in [(0, 0), (4, 5), (4, -1), (2100, 10)]:
        assert B.topk_pool_ws_bytes(4, 1000, 8, p, q) == 0
        assert B.topk_select_pool(4096, 4, 1000, 1000, None, 8, 4096, 4096, p, q, 4096, 4096) == \
            B.TOPK_ERR_ARG
    assert B.topk_pool_ws_bytes(4, 0, 8, 4, 1) == 0
    assert B.topk_select_pool(0, 0, 1000, 1000, None, 8, 0, 0, 4, 1, 0, 0) == B.TOPK_OK
    assert B.topk_select_pool(4096, 4, 1000, 999, None, 8, 4096, 4096, 4, 1, 4096, 4096) == \
        B.TOPK_ERR_SHAPE
    assert B.topk_select_pool(4096, 4, 1000, 1000, None, 8, 4096, 4096, 4, 1, None, 4096) == \
        B.TOPK_ERR_NULL
    assert B.topk_select_pool(4096, 4, 1000, 1000, None, 8, 4096, 4096, 4, 1, 4096, 4096 + 16) == \
        B.TOPK_ERR_WS

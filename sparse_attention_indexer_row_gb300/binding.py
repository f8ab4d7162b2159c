"""ctypes binding to the C ABI declared in ``include/topk_select.h``.

Argument marshalling only: every step of the selection runs in the CUDA
library.  Pointer arguments accept either integers (raw device addresses) or
torch tensors (their ``data_ptr()``); streams accept an integer handle, a
``torch.cuda.Stream`` or None (the legacy default stream).  If the compiled
library is missing this module raises at import time: there is no fallback.
"""

from __future__ import annotations

import ctypes
from pathlib import Path

_LIB_PATH = Path(__file__).resolve().parent / "libtopk_gb300.so"

TOPK_OK = 0
TOPK_ERR_SHAPE = 1
TOPK_ERR_NULL = 2
TOPK_ERR_WS = 3
TOPK_ERR_LAUNCH = 4
TOPK_ERR_ARG = 5
TOPK_ERR_NOSPACE = 6
TOPK_STATUS_NAN = 1
TOPK_STATUS_BAD_LENGTH = 2
TOPK_STATUS_TIMEOUT = 4
TOPK_STATUS_RESCAN = 8
TOPK_STATUS_BOUNDS = 16
TOPK_POOL_BLOCK = 8
TOPK_FLAG_IDENTITY_ORDER = 1
TOPK_FLAG_TEST_STALL = 256
TOPK_TIMELINE_CTAS = 512
TOPK_TIMELINE_SLOTS = 128
TOPK_MAX_K = 2048

# Every symbol the header exports, with (restype, argtypes).
_I32, _I64, _U32, _U64, _SZ, _P = (ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32,
                                   ctypes.c_uint64, ctypes.c_size_t, ctypes.c_void_p)
SIGNATURES = {
    "topk_ws_bytes": (_SZ, [_I32, _I64, _I32]),
    "topk_select": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _I32, _P, _P, _P, _P]),
    "topk_split_plan": (_I32, [_I32, _I64]),
    "topk_ws_bytes_ex": (_SZ, [_I32, _I64, _I32, _I32]),
    "topk_select_ex": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _I32, _P, _P, _P, _P,
                                      _I32, _U64, _U32]),
    "topk_ws_status": (ctypes.c_int, [_P, ctypes.POINTER(_U32), _P]),
    "topk_ws_stats": (ctypes.c_int, [_P, _I32, _I64, _I32, _I32, _P, _P, _P, _P]),
    "topk_visit_order": (ctypes.c_int, [_I32, _I32, _I64, _U64, _P, _P]),
    "topk_timeline_read": (ctypes.c_int, [_P, _P]),
    "topk_select_noalloc": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _I32, _P, _P, _P, _P]),
    "topk_pool_ws_bytes": (_SZ, [_I32, _I64, _I32, _I32, _I32]),
    "topk_select_pool": (ctypes.c_int, [_P, _I32, _I64, _I64, _P, _I32, _P, _P, _I32, _I32,
                                        _P, _P, _P]),
}


def load_library(path: Path = _LIB_PATH) -> ctypes.CDLL:
    """Load one build of the library (the product one by default, or an
    instrumented variant) with every exported signature declared."""
    if not path.exists():
        raise ImportError(
            f"{path.name} is not built; run __graft_entry__.build() "
            "(nvcc for sm_103a) first -- there is no CPU fallback")
    lib = ctypes.CDLL(str(path))
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


LIB = load_library()


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    raise TypeError(f"cannot pass {type(x).__name__} as a pointer")


def _stream(s):
    if s is None:
        return None
    if isinstance(s, int):
        return s
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    raise TypeError(f"cannot pass {type(s).__name__} as a stream")


def topk_ws_bytes(rows: int, n: int, k: int) -> int:
    return int(LIB.topk_ws_bytes(rows, n, k))


def topk_ws_bytes_ex(rows: int, n: int, k: int, split: int) -> int:
    return int(LIB.topk_ws_bytes_ex(rows, n, k, split))


def topk_split_plan(rows: int, n: int) -> int:
    return int(LIB.topk_split_plan(rows, n))


def topk_select(scores, rows, n, row_stride, lengths_or_null, k, out_vals, out_idx, ws,
                stream=None) -> int:
    return int(LIB.topk_select(_ptr(scores), rows, n, row_stride, _ptr(lengths_or_null), k,
                               _ptr(out_vals), _ptr(out_idx), _ptr(ws), _stream(stream)))


def topk_select_ex(scores, rows, n, row_stride, lengths_or_null, k, out_vals, out_idx, ws,
                   stream=None, split=0, seed=0x5EEDC0DE1234ABCD, flags=0) -> int:
    return int(LIB.topk_select_ex(_ptr(scores), rows, n, row_stride, _ptr(lengths_or_null), k,
                                  _ptr(out_vals), _ptr(out_idx), _ptr(ws), _stream(stream),
                                  split, seed & 0xFFFFFFFFFFFFFFFF, flags))


def topk_ws_status(ws, stream=None) -> tuple[int, int]:
    out = ctypes.c_uint32(0)
    rc = int(LIB.topk_ws_status(_ptr(ws), ctypes.byref(out), _stream(stream)))
    return rc, int(out.value)


def topk_ws_stats(ws, rows, n, k, split=0, stream=None):
    """Returns (rc, survivors, sorts, admitted) per row and clears the counters."""
    arrs = [(ctypes.c_uint32 * max(rows, 1))() for _ in range(3)]
    rc = int(LIB.topk_ws_stats(_ptr(ws), rows, n, k, split, *[ctypes.addressof(a) for a in arrs],
                               _stream(stream)))
    return (rc, *[list(a)[:rows] for a in arrs])


def topk_visit_order(m, row, first_unit, seed, order_out, stream=None) -> int:
    return int(LIB.topk_visit_order(m, row, first_unit, seed & 0xFFFFFFFFFFFFFFFF,
                                    _ptr(order_out), _stream(stream)))


def topk_select_noalloc(scores, rows, n, row_stride, lengths_or_null, k, out_vals, out_idx,
                        status_or_null=None, stream=None) -> int:
    """topk_select without a workspace argument, for callers that cannot
    allocate device memory (the library's built-in 16 MiB array is used)."""
    return int(LIB.topk_select_noalloc(_ptr(scores), rows, n, row_stride, _ptr(lengths_or_null),
                                       k, _ptr(out_vals), _ptr(out_idx), _ptr(status_or_null),
                                       _stream(stream)))


class TopK:
    """Convenience holder: device outputs and a zeroed workspace from torch.

    Memory comes from torch's allocator (plumbing); the selection itself is the
    library's ``topk_select_ex``.
    """

    def __init__(self, rows: int, n: int, k: int, device="cuda", split: int = 0):
        import torch
        self.rows, self.n, self.k, self.split = rows, n, k, split
        nbytes = topk_ws_bytes_ex(rows, n, k, split)
        if nbytes == 0:
            raise ValueError("invalid shape")
        # 256-byte alignment: torch's CUDA allocator returns 512-byte aligned blocks
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.vals = torch.empty((rows, k), dtype=torch.float32, device=device)
        self.idx = torch.empty((rows, k), dtype=torch.int32, device=device)

    def __call__(self, scores, lengths=None, n=None, stream=None, seed=0x5EEDC0DE1234ABCD,
                 flags=0):
        n = self.n if n is None else n
        rc = topk_select_ex(scores, self.rows, n, scores.stride(0), lengths, self.k, self.vals,
                            self.idx, self.ws, stream, self.split, seed, flags)
        if rc != TOPK_OK:
            raise RuntimeError(f"topk_select_ex returned {rc}")
        return self.vals, self.idx


def topk_pool_ws_bytes(rows: int, n: int, k: int, pool_blocks: int, pinned_blocks: int) -> int:
    return int(LIB.topk_pool_ws_bytes(rows, n, k, pool_blocks, pinned_blocks))


def topk_select_pool(scores, rows, n, row_stride, lengths_or_null, k, out_vals, out_idx,
                     pool_blocks, pinned_blocks, out_pool, ws, stream=None) -> int:
    return int(LIB.topk_select_pool(_ptr(scores), rows, n, row_stride, _ptr(lengths_or_null), k,
                                    _ptr(out_vals), _ptr(out_idx), pool_blocks, pinned_blocks,
                                    _ptr(out_pool), _ptr(ws), _stream(stream)))

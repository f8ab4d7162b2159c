"""Row-wise top-k oracle: TEST INFRASTRUCTURE ONLY.

A ctypes loader for ``topk_oracle.cpp``, the plain single-threaded C++
statement of the selection (sort every valid row prefix by value descending,
ties to the smaller index; pad short rows with (-inf, -1)) and of the
layer-20 block pool (blocks of consecutive positions scored by their largest
value; the newest blocks pinned, then the best others; ascending indices).  Only the tests,
``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg may use it;
the library under ``sparse_attention_indexer_row_gb300`` never does.

Parity status: pinned, both functions.  ``tests/test_oracle.py`` checks them
against brute-force enumeration, repeated argmax, closed forms, numpy's
lexsort and invariants, and compiles mutants of them to show that each pin
bites.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SRC = _HERE / "topk_oracle.cpp"
_BUILD = _HERE / "_build"

ORACLE_NAN = 5
ORACLE_BAD_LENGTH = 6


def compile_oracle(mutant: int = 0, out: Path | None = None) -> Path:
    """Compile the oracle (optionally with one planted mistake) with g++."""
    _BUILD.mkdir(exist_ok=True)
    if out is None:
        out = _BUILD / ("liboracle.so" if mutant == 0 else f"liboracle_m{mutant}.so")
    tmp = out.with_suffix(f".{os.getpid()}.tmp")
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread",
           f"-DORACLE_MUTANT={int(mutant)}", str(_SRC), "-o", str(tmp)]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


class Oracle:
    """Thin wrapper over one compiled oracle library."""

    def __init__(self, path: Path):
        lib = ctypes.CDLL(str(path))
        lib.oracle_topk.restype = ctypes.c_int
        lib.oracle_topk.argtypes = [
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p,
            ctypes.c_int32,
        ]
        lib.oracle_hardware_threads.restype = ctypes.c_int32
        lib.oracle_block_pool.restype = ctypes.c_int
        lib.oracle_block_pool.argtypes = [
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
            ctypes.c_void_p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
            ctypes.c_void_p, ctypes.c_int32,
        ]
        self._lib = lib

    def hardware_threads(self) -> int:
        return int(self._lib.oracle_hardware_threads())

    def topk(self, scores: np.ndarray, k: int, lengths: np.ndarray | None = None,
             n: int | None = None, nthreads: int = 1):
        """Top-k of every row of a 2-D float32 array.

        ``scores`` is [rows, row_stride]; ``n`` (default row_stride) is the
        logical row width; ``lengths`` (int32[rows]) the valid prefix per row.
        Returns (vals float32[rows, k], idx int32[rows, k], status int).
        """
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        assert scores.ndim == 2
        rows, stride = scores.shape
        n = stride if n is None else int(n)
        vals = np.empty((rows, k), dtype=np.float32)
        idx = np.empty((rows, k), dtype=np.int32)
        lp = None
        if lengths is not None:
            lengths = np.ascontiguousarray(lengths, dtype=np.int32)
            assert lengths.shape == (rows,)
            lp = lengths.ctypes.data
        st = self._lib.oracle_topk(scores.ctypes.data, rows, n, stride, lp, k,
                                   vals.ctypes.data, idx.ctypes.data, nthreads)
        return vals, idx, int(st)


    def block_pool(self, scores: np.ndarray, block: int, pool: int, pinned: int,
                   lengths: np.ndarray | None = None, n: int | None = None, nthreads: int = 1):
        """Block pool of every row (see oracle_block_pool in topk_oracle.cpp).

        Returns (blocks int32[rows, pool], status int).
        """
        scores = np.ascontiguousarray(scores, dtype=np.float32)
        assert scores.ndim == 2
        rows, stride = scores.shape
        n = stride if n is None else int(n)
        out = np.empty((rows, pool), dtype=np.int32)
        lp = None
        if lengths is not None:
            lengths = np.ascontiguousarray(lengths, dtype=np.int32)
            assert lengths.shape == (rows,)
            lp = lengths.ctypes.data
        st = self._lib.oracle_block_pool(scores.ctypes.data, rows, n, stride, lp, block, pool,
                                         pinned, out.ctypes.data, nthreads)
        return out, int(st)


_DEFAULT: Oracle | None = None


def load(mutant: int = 0) -> Oracle:
    """Load (compiling first if needed) the oracle, or one of its mutants."""
    global _DEFAULT
    if mutant == 0:
        if _DEFAULT is None:
            path = _BUILD / "liboracle.so"
            if not path.exists() or path.stat().st_mtime < _SRC.stat().st_mtime:
                compile_oracle(0)
            _DEFAULT = Oracle(path)
        return _DEFAULT
    return Oracle(compile_oracle(mutant))


def topk(scores, k, lengths=None, n=None, nthreads=1):
    return load().topk(scores, k, lengths=lengths, n=n, nthreads=nthreads)


def block_pool(scores, block, pool, pinned, lengths=None, n=None, nthreads=1):
    return load().block_pool(scores, block, pool, pinned, lengths=lengths, n=n, nthreads=nthreads)

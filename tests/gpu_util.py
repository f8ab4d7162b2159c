"""Helpers shared by the GPU tests: run the library, compare with the oracle."""

from __future__ import annotations

import os

import numpy as np

import oracle

CANARY = 64          # guard elements before and after every output buffer
CANARY_F = np.float32(1234.5)
CANARY_I = np.int32(-777)


def host_threads() -> int:
    return max(1, min(os.cpu_count() or 1, 32))


def run_gpu(scores: np.ndarray, k: int, lengths=None, n=None, split=0, seed=None, flags=0,
            device="cuda", ws=None, check_canaries=True, return_ws=False, lib=None):
    """Select on the GPU through the C ABI; outputs sit between canary zones.
    `lib`: another build of the library (a ctypes handle from
    binding.load_library), else the product one."""
    import torch

    from sparse_attention_indexer_row_gb300 import binding as B

    rows, stride = scores.shape
    n = stride if n is None else n
    x = torch.from_numpy(np.ascontiguousarray(scores)).to(device)
    lt = None if lengths is None else torch.from_numpy(np.asarray(lengths, np.int32)).to(device)
    total = rows * k
    vbuf = torch.full((total + 2 * CANARY,), float(CANARY_F), dtype=torch.float32, device=device)
    ibuf = torch.full((total + 2 * CANARY,), int(CANARY_I), dtype=torch.int32, device=device)
    if ws is None:
        nbytes = B.topk_ws_bytes_ex(rows, n, k, split)
        assert nbytes > 0
        ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)
    kw = {} if seed is None else {"seed": seed}
    vptr = vbuf[CANARY:].data_ptr() if total else vbuf.data_ptr()
    iptr = ibuf[CANARY:].data_ptr() if total else ibuf.data_ptr()
    if lib is None:
        rc = B.topk_select_ex(x, rows, n, stride, lt, k, vptr, iptr, ws, None, split,
                              flags=flags, **kw)
    else:
        rc = int(lib.topk_select_ex(x.data_ptr(), rows, n, stride, B._ptr(lt), k, vptr, iptr,
                                    ws.data_ptr(), None, split,
                                    kw.get("seed", 0x5EEDC0DE1234ABCD), flags))
    assert rc == 0, f"topk_select_ex returned {rc}"
    torch.cuda.synchronize()
    v = vbuf.cpu().numpy()
    i = ibuf.cpu().numpy()
    if check_canaries:
        assert np.all(v[:CANARY] == CANARY_F) and np.all(v[CANARY + total:] == CANARY_F), \
            "value writes outside [0, rows*k)"
        assert np.all(i[:CANARY] == CANARY_I) and np.all(i[CANARY + total:] == CANARY_I), \
            "index writes outside [0, rows*k)"
    vals = v[CANARY:CANARY + total].reshape(rows, k)
    idx = i[CANARY:CANARY + total].reshape(rows, k)
    if return_ws:
        return vals, idx, ws
    return vals, idx


def oracle_rows(scores, k, lengths=None, n=None, rows=None):
    """Oracle on all rows, or on the listed row numbers only."""
    if rows is None:
        v, i, st = oracle.topk(scores, k, lengths=lengths, n=n, nthreads=host_threads())
        assert st == 0, st
        return v, i
    rows = np.asarray(rows)
    sub = scores[rows]
    lsub = None if lengths is None else np.asarray(lengths)[rows]
    v, i, st = oracle.topk(sub, k, lengths=lsub, n=n, nthreads=host_threads())
    assert st == 0, st
    return v, i


def assert_bit_exact(gv, gi, ov, oi, what=""):
    gv = np.asarray(gv, np.float32)
    ov = np.asarray(ov, np.float32)
    bad = np.nonzero((gv.view(np.uint32) != ov.view(np.uint32)) | (np.asarray(gi) != oi))
    if bad[0].size:
        r, j = bad[0][0], bad[1][0] if len(bad) > 1 else 0
        raise AssertionError(
            f"{what}: {bad[0].size} mismatching slots; first at row {r} slot {j}: "
            f"gpu ({gv[r, j]!r}, {gi[r, j]}) vs oracle ({ov[r, j]!r}, {oi[r, j]})")

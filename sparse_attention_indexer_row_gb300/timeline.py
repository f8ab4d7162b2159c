"""Where a selection launch spends its time, from the instrumented build.

``libtopk_gb300_timeline.so`` is the library compiled with
``-DTOPK_TIMELINE=1``: every CTA of the selection kernel stamps the global
timer at its start, set-up, first and last copy, the exit of each role and four
events of each of its first eight pieces, and counts SM cycles per activity of
one thread of each role.  ``record`` runs one call through that library and
``summarize`` turns the table into per-CTA figures relative to the earliest
CTA start (medians, 90th percentiles and maxima over the CTAs, in µs).

The stamps cost a few global stores per piece and one clock read per activity,
so an instrumented launch runs slightly slower than the product one; its
figures explain a product measurement, they do not replace it.
"""

from __future__ import annotations

import numpy as np

from . import binding as B
from . import build

SLOT = {"start": 0, "setup": 1, "first_copy": 2, "last_copy": 3, "prod_exit": 4,
        "filt_first": 5, "filt_exit": 6, "sel_exit": 7, "info": 8, "prod_piece": 9,
        "prod_order": 10, "warm_enter": 11, "warm_unit0": 12, "warm_count": 13,
        "warm_second": 14}
PIECE0 = 16
PIECES = 4
PER_PIECE = 16
CYC0 = PIECE0 + PIECES * PER_PIECE
CYC = ["filt_wait_full", "filt_wait_theta", "filt_cand", "filt_stages", "filt_cand_stages",
       "sel_warm", "sel_take", "sel_prune", "sel_sort", "sel_end", "sel_poll", "sel_leaders",
       "prod_wait_empty", "sel_rescans", "filt_body", "cand_classify", "cand_reserve",
       "cand_write", "cand_words", "filt_load"]
COUNTS = {"filt_stages", "filt_cand_stages", "sel_leaders", "sel_rescans", "cand_words"}
# per-piece events: +0 threshold published, +1 filters' first stage, +2 filter
# group 0's last release, +3 selectors done, +4 final sort and merge done,
# +5 ticket taken, +6 leader's merge done, +7 pre-final sort done, +8 selectors
# see the filters done, +9 pre-final started, +10 final sort done (before its
# merge), +11 partial list published, +12 filter group 1's last release,
# +13 producer's last copy of the piece


def load():
    """The instrumented library (built first if it is missing or stale)."""
    path = build.variant_path("timeline")
    if build.needs_build(path):
        build.build_variant("timeline")
    return B.load_library(path)


def read(lib, stream=None) -> np.ndarray:
    out = np.zeros((B.TOPK_TIMELINE_CTAS, B.TOPK_TIMELINE_SLOTS), dtype=np.uint64)
    rc = lib.topk_timeline_read(out.ctypes.data, B._stream(stream))
    if rc != B.TOPK_OK:
        raise RuntimeError(f"topk_timeline_read returned {rc}")
    return out


def record(lib, call, stream=None) -> np.ndarray:
    """Clear the table, run ``call(lib)`` once, return the table."""
    read(lib, stream)
    call(lib)
    return read(lib, stream)


def _stats(x):
    x = np.asarray(x, dtype=np.float64)
    if x.size == 0:
        return None
    return {"median": round(float(np.median(x)), 2), "p90": round(float(np.percentile(x, 90)), 2),
            "max": round(float(x.max()), 2)}


def summarize(table: np.ndarray, sm_mhz: float) -> dict:
    """Per-CTA figures of one recorded launch, in µs after the earliest start."""
    t = table.astype(np.int64)
    used = np.nonzero(t[:, SLOT["start"]] > 0)[0]
    if used.size == 0:
        return {"ctas": 0}
    t = t[used]
    t0 = t[:, SLOT["start"]].min()

    def rel(col):
        v = t[:, col]
        return (v[v > 0] - t0) / 1e3

    out = {"ctas": int(used.size)}
    for name in ("start", "setup", "prod_piece", "prod_order", "first_copy", "warm_enter",
                 "warm_unit0", "warm_count", "warm_second", "filt_first", "last_copy",
                 "filt_exit", "sel_exit", "prod_exit"):
        out[name] = _stats(rel(SLOT[name]))
    ends = np.maximum.reduce([t[:, SLOT["filt_exit"]], t[:, SLOT["sel_exit"]],
                              t[:, SLOT["prod_exit"]]])
    out["span_us"] = round(float((ends.max() - t0) / 1e3), 2)
    pieces = (t[:, SLOT["info"]] >> 32).astype(np.int64)
    out["pieces_per_cta"] = _stats(pieces)
    theta_first = []
    lag = {"prefinal_before_last": [], "final": [], "ticket": [], "leader": [], "done": []}
    for p in range(PIECES):
        base = PIECE0 + PER_PIECE * p
        th, ff, fl0, sd, fs, tk, ld, pf = (t[:, base + i] for i in range(8))
        fl = np.maximum(fl0, t[:, base + 12])  # both filter groups' last releases
        ok = (fl > 0) & (pf > 0)
        lag["prefinal_before_last"].extend(((fl[ok] - pf[ok]) / 1e3).tolist())
        if p == 0:
            ok = th > 0
            theta_first.extend(((th[ok] - t0) / 1e3).tolist())
        ok = (fl > 0) & (fs > 0)
        lag["final"].extend(((fs[ok] - fl[ok]) / 1e3).tolist())
        ok = (fs > 0) & (tk > 0)
        lag["ticket"].extend(((tk[ok] - fs[ok]) / 1e3).tolist())
        ok = (tk > 0) & (ld > 0)
        lag["leader"].extend(((ld[ok] - tk[ok]) / 1e3).tolist())
        ok = (fl > 0) & (sd > 0)
        lag["done"].extend(((sd[ok] - fl[ok]) / 1e3).tolist())
    out["first_theta"] = _stats(theta_first)
    out["piece_end"] = {name: _stats(v) for name, v in lag.items()}
    cyc = {}
    for i, name in enumerate(CYC):
        v = t[:, CYC0 + i].astype(np.float64)
        if name in COUNTS:
            cyc[name] = round(float(v.mean()), 2)
        else:
            cyc[name + "_us"] = round(float(v.mean() / sm_mhz), 2)
    out["per_cta_mean"] = cyc
    return out

"""Pins for the CPU oracle: checks that do not go through the oracle's own code.

Each pin takes an ``oracle.Oracle`` and raises ``AssertionError`` when the
oracle disagrees with something fixed independently of it:

* brute-force enumeration of the unique k-subset that dominates its complement,
  with output positions found by counting (tiny rows, every value class);
* repeated argmax (pick the best remaining element k times);
* closed forms (ascending rows, constant rows, quantised rows with +/-inf);
* numpy's ``lexsort`` on rows without signed zeros or NaN;
* invariants on random rows (count, domination, tie rule, uniqueness, order);
* the contract around lengths, strides, padding, NaN and bad shapes.

The selection these pins define: value descending under the total order
-inf < negatives < -0.0 < +0.0 < positives < +inf, ties to the smaller in-row
index, rows shorter than k padded with (-inf, -1) (The Secret GPU Kernel
Behind DeepSeek V4.1 Flash, video transcript 2:28-4:08; the bit-exact packed
words of DeepSeek V4.1 Flash, kernelbench model page, entry "Single-launch
CUDA bitonic selection").

``tests/test_oracle.py`` runs every pin against the oracle, and against
mutants of it that each plant one plausible mistake, to show that each
mistake is caught.
"""

from __future__ import annotations

import itertools
import math

import numpy as np

NINF = float("-inf")
PINF = float("inf")
ALPHABET = [NINF, -1.5, -0.0, 0.0, 1.5, PINF]


# ---- an independent statement of the order (pure Python) ------------------

def _key(x: float):
    """Total-order key: the value, then +0.0 above -0.0."""
    return (x, 1 if (x == 0.0 and math.copysign(1.0, x) > 0) else 0)


def _before(row, i, j):
    ki, kj = _key(row[i]), _key(row[j])
    return ki > kj or (ki == kj and i < j)


def brute_force(row, k):
    """Unique dominating subset, positions by counting."""
    L = len(row)
    t = min(k, L)
    found = None
    for sub in itertools.combinations(range(L), t):
        s = set(sub)
        if all(_before(row, i, j) for i in s for j in range(L) if j not in s):
            assert found is None, "dominating subset must be unique"
            found = sub
    assert found is not None
    pos = {i: sum(1 for j in found if _before(row, j, i)) for i in found}
    vals = [NINF] * k
    idx = [-1] * k
    for i in found:
        vals[pos[i]] = row[i]
        idx[pos[i]] = i
    return vals, idx


def repeated_argmax(row, k):
    left = list(range(len(row)))
    vals, idx = [], []
    for _ in range(min(k, len(row))):
        best = next(i for i in left if all(_before(row, i, j) for j in left if j != i))
        left.remove(best)
        vals.append(row[best])
        idx.append(best)
    pad = k - len(idx)
    return vals + [NINF] * pad, idx + [-1] * pad


def _bits(a):
    return np.asarray(a, dtype=np.float32).view(np.uint32)


def assert_same(vals, idx, ev, ei, what=""):
    ev = np.asarray(ev, dtype=np.float32)
    ei = np.asarray(ei, dtype=np.int32)
    assert np.array_equal(np.asarray(idx), ei), f"{what}: indices {np.asarray(idx)} != {ei}"
    assert np.array_equal(_bits(vals), _bits(ev)), f"{what}: value bits differ"


# ---- invariants (numpy, no sorting of the whole row) ------------------------

def _order_key64(x: np.ndarray) -> np.ndarray:
    """Map float32 to int64 ranks consistent with the total order (for tests)."""
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.int32).astype(np.int64)
    # for negatives (sign set) reverse the magnitude order
    return np.where(b < 0, -(b & 0x7FFFFFFF) - 1, b)


def check_invariants(row: np.ndarray, k: int, vals: np.ndarray, idx: np.ndarray):
    L = row.shape[0]
    t = min(k, L)
    idx = np.asarray(idx)
    vals = np.asarray(vals, dtype=np.float32)
    assert np.all(idx[t:] == -1), "padding indices"
    assert np.all(np.isneginf(vals[t:])), "padding values"
    sel = idx[:t]
    assert np.all((sel >= 0) & (sel < L)), "indices in range"
    assert np.unique(sel).size == t, "indices unique"
    assert np.array_equal(_bits(vals[:t]), _bits(row[sel])), "values are the row's"
    key = _order_key64(row)
    ks = key[sel]
    # strictly descending in (key desc, index asc)
    if t > 1:
        a, b = ks[:-1], ks[1:]
        ia, ib = sel[:-1], sel[1:]
        assert np.all((a > b) | ((a == b) & (ia < ib))), "output order"
    if t < L:
        mask = np.ones(L, dtype=bool)
        mask[sel] = False
        rest_key = key[mask]
        rest_idx = np.nonzero(mask)[0]
        kk, ki = ks[-1], sel[-1]
        assert np.all((rest_key < kk) | ((rest_key == kk) & (rest_idx > ki))), \
            "a dropped element outranks the k-th"


# ---- the pins ---------------------------------------------------------------

def pin_brute_force_exhaustive(orc):
    """Every row of length <= 4 over the six value classes, several k."""
    for L in range(1, 5):
        rows = np.array(list(itertools.product(ALPHABET, repeat=L)), dtype=np.float32)
        for k in sorted({1, 2, L, L + 2}):
            v, i, st = orc.topk(rows, k)
            assert st == 0
            for r in range(rows.shape[0]):
                ev, ei = brute_force([float(x) for x in rows[r]], k)
                assert_same(v[r], i[r], ev, ei, f"L={L} k={k} row={rows[r]}")


def pin_brute_force_random(orc, cases=120, seed=11):
    rng = np.random.default_rng(seed)
    for c in range(cases):
        L = int(rng.integers(5, 10))
        k = int(rng.integers(1, L + 3))
        row = np.array(rng.choice(ALPHABET, size=L), dtype=np.float32)
        v, i, st = orc.topk(row[None, :], k)
        assert st == 0
        ev, ei = brute_force([float(x) for x in row], k)
        assert_same(v[0], i[0], ev, ei, f"case {c}")


def pin_repeated_argmax(orc, cases=60, seed=12):
    rng = np.random.default_rng(seed)
    fmax = float(np.finfo(np.float32).max)
    levels = np.array([NINF, -fmax, -2.0, -0.5, -0.0, 0.0, 0.25, 3.0, fmax, PINF],
                      dtype=np.float32)
    for c in range(cases):
        L = int(rng.integers(1, 40))
        k = int(rng.integers(1, 45))
        row = levels[rng.integers(0, levels.size, size=L)]
        v, i, st = orc.topk(row[None, :], k)
        assert st == 0
        ev, ei = repeated_argmax([float(x) for x in row], k)
        assert_same(v[0], i[0], ev, ei, f"case {c}")


def pin_ascending_rows(orc):
    """Distinct ascending values: winners are L-1, L-2, ..., L-k."""
    for L, k in [(1000, 10), (4096, 512), (300, 512), (5000, 2048)]:
        row = np.linspace(-3.0, 7.0, L, dtype=np.float32)
        assert np.all(np.diff(row) > 0)
        v, i, st = orc.topk(row[None, :], k)
        assert st == 0
        t = min(k, L)
        ei = np.concatenate([np.arange(L - 1, L - 1 - t, -1), -np.ones(k - t)]).astype(np.int32)
        ev = np.concatenate([row[ei[:t]], np.full(k - t, -np.inf, np.float32)])
        assert_same(v[0], i[0], ev, ei, f"ascending L={L} k={k}")


def pin_constant_rows(orc):
    """Every value tied: winners are 0..k-1 in order."""
    for c in [0.0, -0.0, 1.0, -7.5, np.inf, -np.inf]:
        row = np.full(3000, c, dtype=np.float32)
        v, i, st = orc.topk(row[None, :], 512)
        assert st == 0
        assert_same(v[0], i[0], row[:512], np.arange(512), f"constant {c}")


def pin_quantised_levels(orc, seed=13):
    """256 levels plus +/-inf: +inf first in index order, then whole levels
    from the top, then the lowest indices of the boundary level."""
    rng = np.random.default_rng(seed)
    L, k = 20000, 700
    lvl = rng.integers(0, 256, size=L)
    row = ((lvl - 127.5) / 32.0).astype(np.float32)
    hit = rng.random(L) < 0.01
    sgn = rng.random(L) < 0.5
    row[hit & sgn] = np.inf
    row[hit & ~sgn] = -np.inf
    expect = []
    for level in [np.inf] + [(j - 127.5) / 32.0 for j in range(255, -1, -1)] + [-np.inf]:
        where = np.nonzero(row == np.float32(level))[0]   # ascending index order
        expect.extend(where.tolist())
        if len(expect) >= k:
            break
    ei = np.array(expect[:k], dtype=np.int32)
    v, i, st = orc.topk(row[None, :], k)
    assert st == 0
    assert_same(v[0], i[0], row[ei], ei, "quantised")


def pin_numpy_lexsort(orc, seed=14):
    """Library special case: rows with no -0.0 and no NaN sort like lexsort."""
    rng = np.random.default_rng(seed)
    for r in range(6):
        L = int(rng.integers(1, 6000))
        k = int(rng.integers(1, 2049))
        row = np.round(rng.standard_normal(L) * 4).astype(np.float32)  # many ties
        row[row == 0] = 0.0                                           # +0 only
        row[rng.random(L) < 0.01] = np.inf
        order = np.lexsort((np.arange(L), -row.astype(np.float64)))
        t = min(k, L)
        ei = np.concatenate([order[:t], -np.ones(k - t)]).astype(np.int32)
        ev = np.concatenate([row[order[:t]], np.full(k - t, -np.inf, np.float32)])
        v, i, st = orc.topk(row[None, :], k)
        assert st == 0
        assert_same(v[0], i[0], ev, ei, f"lexsort case {r}")


def pin_invariants_random(orc, seed=15):
    rng = np.random.default_rng(seed)
    rows, n = 6, 9000
    x = rng.standard_normal((rows, n)).astype(np.float32)
    x[1] = np.round(x[1] * 3)             # heavy ties including zeros
    x[1][rng.random(n) < 0.5] *= -1       # produces -0.0 as well as +0.0
    x[2][rng.random(n) < 0.02] = -np.inf
    x[3] = np.sort(x[3])
    x[4] = np.where(rng.random(n) < 0.5, np.float32(0.0), np.float32(-0.0))
    for k in (1, 33, 512, 1000, 2048):
        v, i, st = orc.topk(x, k)
        assert st == 0
        for r in range(rows):
            check_invariants(x[r], k, v[r], i[r])


def pin_lengths_and_stride(orc, seed=16):
    """Only the valid prefix counts; the stride gap and the tail are ignored."""
    rng = np.random.default_rng(seed)
    rows, n, stride, k = 5, 3000, 3013, 64
    buf = np.full((rows, stride), np.nan, dtype=np.float32)   # poison outside
    body = rng.standard_normal((rows, n)).astype(np.float32)
    lengths = np.array([0, 1, 63, 64, 2500], dtype=np.int32)
    for r in range(rows):
        buf[r, :lengths[r]] = body[r, :lengths[r]]
        buf[r, lengths[r]:n] = np.inf                          # past the length
    v, i, st = orc.topk(buf, k, lengths=lengths, n=n)
    assert st == 0
    for r in range(rows):
        L = int(lengths[r])
        ev, ei = repeated_argmax([float(t) for t in body[r, :L]], k) if L <= 64 else (None, None)
        if ev is not None:
            assert_same(v[r], i[r], ev, ei, f"length row {r}")
        check_invariants(body[r, :L], k, v[r], i[r])
    # L = 0 gives an all-padding row
    assert np.all(i[0] == -1) and np.all(np.isneginf(v[0]))


def pin_contract_errors(orc):
    x = np.zeros((2, 16), dtype=np.float32)
    assert orc.topk(x, 0)[2] == 1
    assert orc.topk(x, 2049)[2] == 1
    assert orc.topk(x, 4, lengths=np.array([3, 17], np.int32))[2] == 6
    assert orc.topk(x, 4, lengths=np.array([-1, 2], np.int32))[2] == 6
    y = x.copy()
    y[1, 5] = np.nan
    assert orc.topk(y, 4)[2] == 5
    # a NaN outside the valid prefix is not looked at
    assert orc.topk(y, 4, lengths=np.array([16, 5], np.int32))[2] == 0


# ---- the block pool (layer-20 sweep, video transcript 7:22-7:46) ----------
#
# Blocks of `block` consecutive positions of the valid prefix (the last one
# may be short) score the largest value inside them; the pool keeps the
# `pinned` newest blocks and then the best other blocks (value descending,
# ties to the smaller block index), emitted as ascending block indices padded
# with -1.  Stated again here in plain Python with the order key above.

def pool_brute_force(row, block, pool, pinned):
    L = len(row)
    nb = -(-L // block)
    pe = min(pinned, nb)
    cand = list(range(nb - pe))
    score = {b: max((row[i] for i in range(b * block, min(L, (b + 1) * block))), key=_key)
             for b in cand}
    kept = set(range(nb - pe, nb))
    left = list(cand)
    while len(kept) < pool and left:
        # the block no other remaining block beats
        best = next(b for b in left
                    if all(_key(score[b]) > _key(score[c]) or
                           (_key(score[b]) == _key(score[c]) and b < c) for c in left if c != b))
        left.remove(best)
        kept.add(best)
    out = sorted(kept)
    return out + [-1] * (pool - len(out))


def pin_pool_brute_force(orc, cases=150, seed=17):
    rng = np.random.default_rng(seed)
    for c in range(cases):
        block = int(rng.choice([1, 2, 3, 8]))
        L = int(rng.integers(0, 33))
        pool = int(rng.integers(1, 7))
        pinned = int(rng.integers(0, pool + 1))
        row = [float(ALPHABET[j]) for j in rng.integers(0, len(ALPHABET), size=L)]
        n = max(L, 1)
        x = np.full((1, n), 7.0, dtype=np.float32)     # past the length: ignored
        x[0, :L] = np.array(row, dtype=np.float32)
        got, st = orc.block_pool(x, block, pool, pinned, lengths=np.array([L], np.int32), n=n)
        assert st == 0
        want = pool_brute_force(row, block, pool, pinned)
        assert list(got[0]) == want, f"pool case {c}: {list(got[0])} != {want} (block {block}, L {L}, pool {pool}, pinned {pinned}, row {row})"


def pin_pool_closed_forms(orc, seed=18):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((3, 1000)).astype(np.float32)
    nb = 125
    # a pool at least as large as the row: every block, ascending
    got, st = orc.block_pool(x, 8, 200, 10)
    assert st == 0 and all(list(r) == list(range(nb)) + [-1] * 75 for r in got)
    # every place pinned: the newest blocks only
    got, st = orc.block_pool(x, 8, 40, 40)
    assert st == 0 and all(list(r) == list(range(nb - 40, nb)) for r in got)
    # ascending rows: the best blocks are the newest ones anyway
    asc = np.sort(x, axis=1)
    got, st = orc.block_pool(asc, 8, 30, 3)
    assert st == 0 and all(list(r) == list(range(nb - 30, nb)) for r in got)
    # descending rows, nothing pinned: the oldest blocks
    got, st = orc.block_pool(asc[:, ::-1].copy(), 8, 30, 0)
    assert st == 0 and all(list(r) == list(range(30)) for r in got)
    # one large score per chosen block, zeros elsewhere: exactly those blocks
    y = np.zeros((1, 1000), np.float32)
    chosen = [3, 17, 40, 41, 99]
    for j, b in enumerate(chosen):
        y[0, 8 * b + (j % 8)] = 10.0 + j
    got, st = orc.block_pool(y, 8, 6, 1)
    assert st == 0 and list(got[0]) == sorted(chosen) + [124]


def pin_pool_invariants(orc, seed=19):
    rng = np.random.default_rng(seed)
    rows, n, block, pool, pinned = 4, 5000, 8, 100, 10
    x = rng.standard_normal((rows, n)).astype(np.float32)
    x[1] = np.round(x[1] * 2)                     # ties between blocks
    lengths = np.array([5000, 4999, 17, 801], np.int32)
    got, st = orc.block_pool(x, block, pool, pinned, lengths=lengths)
    assert st == 0
    for r in range(rows):
        L = int(lengths[r])
        nb = -(-L // block)
        pe = min(pinned, nb)
        kept = [int(b) for b in got[r] if b >= 0]
        assert kept == sorted(set(kept)), "ascending and unique"
        assert all(0 <= b < nb for b in kept)
        assert len(kept) == min(pool, nb)
        assert set(range(nb - pe, nb)) <= set(kept), "the newest blocks are pinned"
        score = {b: max((float(v) for v in x[r, b * block:min(L, (b + 1) * block)]), key=_key)
                 for b in range(nb)}
        sel = [b for b in kept if b < nb - pe]
        out = [b for b in range(nb - pe) if b not in set(kept)]
        for b in sel:            # every chosen block beats every left-out one
            for c in out:
                assert _key(score[b]) > _key(score[c]) or (_key(score[b]) == _key(score[c]) and b < c)


def pin_pool_contract(orc):
    x = np.zeros((2, 16), dtype=np.float32)
    assert orc.block_pool(x, 0, 4, 0)[1] == 1
    assert orc.block_pool(x, 8, 0, 0)[1] == 1
    assert orc.block_pool(x, 8, 4, 5)[1] == 1
    assert orc.block_pool(x, 8, 2100, 10)[1] == 1
    assert orc.block_pool(x, 8, 2058, 10)[1] == 0
    assert orc.block_pool(x, 8, 4, 1, lengths=np.array([3, 17], np.int32))[1] == 6
    y = x.copy()
    y[1, 5] = np.nan
    out, st = orc.block_pool(y, 8, 4, 1)
    assert st == 5 and np.all(out[1] == -1)


ALL_PINS = [
    pin_pool_brute_force,
    pin_pool_closed_forms,
    pin_pool_invariants,
    pin_pool_contract,
    pin_brute_force_exhaustive,
    pin_brute_force_random,
    pin_repeated_argmax,
    pin_ascending_rows,
    pin_constant_rows,
    pin_quantised_levels,
    pin_numpy_lexsort,
    pin_invariants_random,
    pin_lengths_and_stride,
    pin_contract_errors,
]

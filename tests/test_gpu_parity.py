"""GPU parity: the CUDA selector against the CPU oracle, bit for bit.

Values are compared as uint32 bit patterns and indices exactly, padding
included; every output buffer sits between canary zones that must survive.
"""

from __future__ import annotations

import numpy as np
import pytest

from sparse_attention_indexer_row_gb300 import synth
from tests import oracle_pins as P
from tests.gpu_util import assert_bit_exact, oracle_rows, run_gpu

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)


def _check(w: synth.Workload, split=0, rows=None, seed=None, flags=0):
    gv, gi = run_gpu(w.scores, w.k, lengths=w.lengths, n=w.n, split=split, seed=seed,
                     flags=flags)
    ov, oi = oracle_rows(w.scores, w.k, lengths=w.lengths, n=w.n, rows=rows)
    if rows is not None:
        gv, gi = gv[rows], gi[rows]
    assert_bit_exact(gv, gi, ov, oi, w.name)
    return gv, gi


# ---- the five workload families ---------------------------------------------

def test_uniform_pool_4x16384():
    _check(synth.uniform_pool())


def test_normal_varlen_64x131072():
    w = synth.normal_varlen()
    assert np.any(w.lengths < 512)   # some rows shorter than k
    _check(w)


@pytest.mark.parametrize("rows", [1, 4])
def test_relu_mix_1m(rows):
    _check(synth.relu_mix(rows=rows))


@pytest.mark.parametrize("layout", ["normal", "sorted", "quant"])
@pytest.mark.parametrize("k", [512, 2048])
def test_long_rows_64x1m(layout, k):
    _check(synth.long_rows(layout, k=k))


def test_causal_prefill_8192x65536_all_rows():
    """Every one of the 8,192 rows (the queue plan at full size: items handed
    out longest first, short rows returning all their positions)."""
    _check(synth.causal_prefill())


# ---- edge shapes --------------------------------------------------------------

@pytest.mark.parametrize("k", [1, 2, 31, 32, 33, 511, 512, 513, 1000, 2047, 2048])
def test_k_sweep(k):
    rng = np.random.default_rng(100 + k)
    x = rng.standard_normal((3, 20000)).astype(np.float32)
    x[1] = np.round(x[1] * 2)                   # heavy ties incl. zeros
    x[1][rng.random(20000) < 0.5] *= -1         # -0.0 as well as +0.0
    gv, gi = run_gpu(x, k)
    ov, oi = oracle_rows(x, k)
    assert_bit_exact(gv, gi, ov, oi, f"k={k}")


@pytest.mark.parametrize("n", [1, 3, 1023, 1024, 1025, 4097, 129000])
@pytest.mark.parametrize("k", [1, 512, 1000])
def test_n_sweep(n, k):
    rng = np.random.default_rng(n * 7 + k)
    x = rng.standard_normal((3, n)).astype(np.float32)
    gv, gi = run_gpu(x, k)
    ov, oi = oracle_rows(x, k)
    assert_bit_exact(gv, gi, ov, oi, f"n={n} k={k}")


def test_lengths_zero_one_and_short():
    rng = np.random.default_rng(3)
    n, k = 5000, 512
    x = rng.standard_normal((6, n)).astype(np.float32)
    lengths = np.array([0, 1, 2, 511, 512, 513], np.int32)
    gv, gi = run_gpu(x, k, lengths=lengths)
    ov, oi = oracle_rows(x, k, lengths=lengths)
    assert_bit_exact(gv, gi, ov, oi, "short lengths")
    assert np.all(gi[0] == -1) and np.all(np.isneginf(gv[0]))


@pytest.mark.parametrize("stride_pad", [1, 2, 3, 5, 16])
def test_misaligned_and_padded_rows(stride_pad):
    """row_stride > n and not a multiple of 4: rows start off 16-byte bounds."""
    rng = np.random.default_rng(stride_pad)
    rows, n, k = 5, 9000, 300
    buf = np.full((rows, n + stride_pad), np.nan, dtype=np.float32)  # poison the gap
    buf[:, :n] = rng.standard_normal((rows, n))
    lengths = np.array([9000, 8999, 4097, 1025, 3], np.int32)
    gv, gi = run_gpu(buf, k, lengths=lengths, n=n)
    ov, oi = oracle_rows(buf, k, lengths=lengths, n=n)
    assert_bit_exact(gv, gi, ov, oi, f"stride pad {stride_pad}")


def test_multi_chunk_segments():
    """Pieces longer than one shuffle chunk (256 units of 8192 elements), split
    and unsplit, and many variable-length rows dealt round-robin."""
    rng = np.random.default_rng(31)
    x = rng.standard_normal((2, 2_500_003)).astype(np.float32)
    gv, gi = run_gpu(x, 512, split=1)                 # two 2-chunk pieces
    ov, oi = oracle_rows(x, 512)
    assert_bit_exact(gv, gi, ov, oi, "2 x 2.5M unsplit")
    y = rng.standard_normal((160, 1_100_005)).astype(np.float32)
    lengths = rng.integers(0, 1_100_006, size=160).astype(np.int32)
    lengths[:4] = [1_100_005, 1_048_577, 1_048_576, 0]
    gv, gi = run_gpu(y, 1000, lengths=lengths)        # many rows, one item each
    ov, oi = oracle_rows(y, 1000, lengths=lengths)
    assert_bit_exact(gv, gi, ov, oi, "160 x 1.1M")


def test_rows_zero_is_noop():
    from sparse_attention_indexer_row_gb300 import binding as B
    assert B.topk_select(0, 0, 100, 100, None, 5, 0, 0, 0) == 0


def test_special_values():
    """+/-inf, +/-0.0, extreme finite values and heavy ties in long rows."""
    rng = np.random.default_rng(44)
    alphabet = np.array([-np.inf, -3.4e38, -1.5, -0.0, 0.0, 1.5, 3.4e38, np.inf], np.float32)
    x = alphabet[rng.integers(0, alphabet.size, size=(4, 50000))]
    for k in (1, 7, 512, 2048):
        gv, gi = run_gpu(x, k)
        ov, oi = oracle_rows(x, k)
        assert_bit_exact(gv, gi, ov, oi, f"special k={k}")


def test_constant_and_ascending_rows():
    n = 70000
    x = np.stack([np.full(n, 0.5, np.float32), np.full(n, -np.inf, np.float32),
                  np.linspace(-1, 1, n, dtype=np.float32),
                  np.linspace(1, -1, n, dtype=np.float32)])
    for k in (512, 2048):
        gv, gi = run_gpu(x, k)
        ov, oi = oracle_rows(x, k)
        assert_bit_exact(gv, gi, ov, oi, f"closed forms k={k}")
        assert np.array_equal(gi[0], np.arange(k))
        assert np.array_equal(gi[2], np.arange(n - 1, n - 1 - k, -1))


# ---- result invariance: split, seed, order ----------------------------------

@pytest.mark.parametrize("split", [1, 2, 3, 7, 16, 64])
def test_split_invariance(split):
    rng = np.random.default_rng(split)
    x = rng.standard_normal((3, 300000)).astype(np.float32)
    x[2] = np.round(x[2] * 4)
    lengths = np.array([300000, 123457, 700], np.int32)
    gv, gi = run_gpu(x, 512, lengths=lengths, split=split)
    ov, oi = oracle_rows(x, 512, lengths=lengths)
    assert_bit_exact(gv, gi, ov, oi, f"split={split}")


def test_seed_and_identity_invariance():
    w = synth.long_rows("quant", rows=4, n=1 << 18, k=512)
    base = run_gpu(w.scores, w.k)
    for seed in (1, 2, 0xFFFFFFFFFFFFFFFF):
        v, i = run_gpu(w.scores, w.k, seed=seed)
        assert_bit_exact(v, i, *base, f"seed {seed}")
    v, i = run_gpu(w.scores, w.k, flags=1)
    assert_bit_exact(v, i, *base, "identity order")


def test_repeated_calls_reuse_workspace():
    """Tickets return to zero, so one workspace serves many calls."""
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(9)
    x = rng.standard_normal((2, 200000)).astype(np.float32)
    ov, oi = oracle_rows(x, 512)
    nbytes = B.topk_ws_bytes_ex(2, 200000, 512, 8)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    for _ in range(3):
        gv, gi = run_gpu(x, 512, split=8, ws=ws)
        assert_bit_exact(gv, gi, ov, oi, "reuse")
    # tickets (u32[rows] at byte 256) are back at zero
    assert torch.all(ws[256:256 + 8] == 0)


# ---- cross-checks with library routines --------------------------------------

def test_torch_sort_and_topk_agree():
    w = synth.relu_mix(rows=4, n=1 << 18)
    x = torch.from_numpy(w.scores).cuda()
    gv, gi = run_gpu(w.scores, w.k)
    # stable descending sort: same order wherever there is no -0.0
    assert not np.any((w.scores == 0) & np.signbit(w.scores))
    sv, si = torch.sort(x, dim=1, descending=True, stable=True)
    assert np.array_equal(si[:, :w.k].cpu().numpy(), gi)
    tv, _ = torch.topk(x, w.k, dim=1, sorted=True)
    assert np.array_equal(tv.cpu().numpy().view(np.uint32), gv.view(np.uint32))


def test_invariants_at_scale():
    w = synth.long_rows("normal", rows=8, k=2048)
    gv, gi = run_gpu(w.scores, w.k)
    for r in range(w.rows):
        P.check_invariants(w.scores[r], w.k, gv[r], gi[r])


# ---- status word, survivors, visiting order ----------------------------------

def test_nan_sets_status_and_kernel_finishes():
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(5)
    x = rng.standard_normal((2, 30000)).astype(np.float32)
    x[1, 777] = np.nan
    x[0, 29990] = np.nan                     # beyond row 0's length: not looked at
    lengths = np.array([29000, 30000], np.int32)
    gv, gi, ws = run_gpu(x, 64, lengths=lengths, return_ws=True)
    rc, status = B.topk_ws_status(ws)
    assert rc == 0 and status == B.TOPK_STATUS_NAN
    ov, oi = oracle_rows(x[:1], 64, lengths=lengths[:1])
    assert_bit_exact(gv[:1], gi[:1], ov, oi, "row without NaN")
    rc, status = B.topk_ws_status(ws)
    assert rc == 0 and status == 0           # read-and-clear


def _oracle_without_nan(x, k, length):
    """The selection of a row's valid non-NaN scores, by the oracle: the row
    with its NaN positions taken out, indices mapped back.  Taking positions
    out keeps the others in index order, so the smaller-index tie rule maps
    over unchanged."""
    row = x[:length]
    keep = np.nonzero(~np.isnan(row))[0]
    ov, oi = oracle_rows(row[keep][None, :], k)
    oi = np.where(oi[0] >= 0, keep[np.maximum(oi[0], 0)], -1).astype(np.int32)
    return ov[0], oi


@pytest.mark.parametrize("n,k,split", [(30000, 64, 0), (300000, 512, 0), (300000, 512, 1),
                                       (50000, 2048, 0), (2000, 512, 0)])
def test_nan_is_left_out_of_the_selection(n, k, split):
    """The header's contract for a row holding NaN: the result is the
    selection over the row's other valid scores (TOPK_STATUS_NAN is set).
    Pinned against the oracle run on the row with the NaN positions removed;
    the NaNs sit in the warm-start sample, in later units, in a short row and
    next to +/-inf and ties."""
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(n + k + split)
    x = rng.standard_normal((3, n)).astype(np.float32)
    x[1] = np.round(x[1] * 2)                              # ties
    for r in range(3):
        pos = rng.choice(n, size=max(3, n // 1000), replace=False)
        x[r, pos] = np.nan
    x[2, :16] = np.nan                                     # the row's first positions
    x[2, rng.choice(n, size=20, replace=False)] = np.inf
    x[0, 0:4] = [np.nan, np.inf, -np.inf, np.nan]
    lengths = np.array([n, n - 7, n // 2], np.int32)
    gv, gi, ws = run_gpu(x, k, lengths=lengths, split=split, return_ws=True)
    rc, status = B.topk_ws_status(ws)
    assert rc == 0 and status & B.TOPK_STATUS_NAN
    for r in range(3):
        ov, oi = _oracle_without_nan(x[r], k, lengths[r])
        assert_bit_exact(gv[r:r + 1], gi[r:r + 1], ov[None], oi[None], f"NaN row {r}")


def test_bad_length_sets_status():
    from sparse_attention_indexer_row_gb300 import binding as B
    x = np.ones((3, 1000), np.float32)
    lengths = np.array([5, 1001, -3], np.int32)
    gv, gi, ws = run_gpu(x, 8, lengths=lengths, return_ws=True)
    rc, status = B.topk_ws_status(ws)
    assert rc == 0 and status == B.TOPK_STATUS_BAD_LENGTH
    assert np.array_equal(gi[0], [0, 1, 2, 3, 4, -1, -1, -1])


def _harmonic(m):
    return sum(1.0 / j for j in range(1, m + 1))


@pytest.mark.parametrize("layout", ["normal", "sorted", "quant"])
@pytest.mark.parametrize("k", [512, 2048])
def test_survivor_bound_unsplit(layout, k):
    """Elements reaching a sort stay under 1.5 x tray x H(blocks) per row
    (video transcript 4:32-4:55), for unsplit rows in the shuffled order."""
    from sparse_attention_indexer_row_gb300 import binding as B
    w = synth.long_rows(layout, rows=8, k=k)
    gv, gi, ws = run_gpu(w.scores, w.k, split=1, return_ws=True)
    rc, surv, sorts, adm = B.topk_ws_stats(ws, w.rows, w.n, w.k, 1)
    assert rc == 0
    T = k + 2 * 1024
    bound = 1.5 * T * _harmonic(w.n // 1024)
    assert max(surv) <= bound, (max(surv), bound)
    assert min(surv) >= k
    assert all(a >= s for a, s in zip(adm, surv))
    # Every element that passed the threshold test and went to the tray.  The
    # pages' argument bounds it per visited block: a block that sets a record
    # can send all its elements before the line rises.  This build visits
    # 8192-element units, so the same bound, with the unit as the block
    # (tray k + 2 units, H over the units), covers the admitted words.
    unit = 8192
    bound_adm = 1.5 * (k + 2 * unit) * _harmonic(-(-w.n // unit))
    assert max(adm) <= bound_adm, (max(adm), bound_adm)


def test_identity_order_on_ascending_rows_admits_everything():
    """Without the shuffle an ascending row sends every element past the
    warm-start window (for k <= 512 the first three 8192-element units of the
    row, 96 KB) to the tray."""
    from sparse_attention_indexer_row_gb300 import binding as B
    x = np.sort(np.random.default_rng(1).standard_normal((2, 1 << 18)).astype(np.float32), axis=1)
    gv, gi, ws = run_gpu(x, 512, split=1, flags=B.TOPK_FLAG_IDENTITY_ORDER, return_ws=True)
    rc, surv, _, adm = B.topk_ws_stats(ws, 2, 1 << 18, 512, 1)
    assert rc == 0 and min(adm) >= (1 << 18) - 3 * 8192
    gv2, gi2, ws2 = run_gpu(x, 512, split=1, return_ws=True)
    rc, surv2, _, adm2 = B.topk_ws_stats(ws2, 2, 1 << 18, 512, 1)
    assert max(adm2) < (1 << 18) // 4
    assert_bit_exact(gv, gi, gv2, gi2, "identity vs shuffled")


def test_visit_order_matches_philox():
    from sparse_attention_indexer_row_gb300 import binding as B
    from tests.philox_ref import philox4x32_10
    for m, row, first, seed in [(256, 3, 0, 0x1234), (205, 17, 410, 0xDEADBEEFCAFEF00D), (1, 0, 5, 7)]:
        out = torch.empty(m, dtype=torch.int32, device="cuda")
        assert B.topk_visit_order(m, row, first, seed, out) == 0
        got = out.cpu().numpy()
        keys = []
        for j in range(m):
            r = philox4x32_10((first + j, row, 0, 0), (seed & 0xFFFFFFFF, seed >> 32))
            keys.append(((r[0] & ~255) & 0xFFFFFFFF) | j)
        want = np.argsort(np.array(keys, dtype=np.uint64), kind="stable")
        assert np.array_equal(got, want)
        assert np.array_equal(np.sort(got), np.arange(m))


@pytest.mark.slow
def test_large_offsets():
    """row_stride = 2^29 + 16: element offsets beyond 2^31 (needs ~8.6 GB)."""
    stride = (1 << 29) + 16
    rows, n, k = 4, 1 << 20, 512
    free, _ = torch.cuda.mem_get_info()
    if free < rows * stride * 4 + (1 << 30):
        pytest.skip("not enough device memory")
    from sparse_attention_indexer_row_gb300 import binding as B
    rng = np.random.default_rng(77)
    body = rng.standard_normal((rows, n)).astype(np.float32)
    big = torch.full((rows, stride), float("nan"), dtype=torch.float32, device="cuda")
    big[:, :n] = torch.from_numpy(body).cuda()
    vals = torch.empty((rows, k), dtype=torch.float32, device="cuda")
    idx = torch.empty((rows, k), dtype=torch.int32, device="cuda")
    ws = torch.zeros(B.topk_ws_bytes(rows, n, k), dtype=torch.uint8, device="cuda")
    assert B.topk_select(big, rows, n, stride, None, k, vals, idx, ws) == 0
    torch.cuda.synchronize()
    ov, oi = oracle_rows(body, k)
    assert_bit_exact(vals.cpu().numpy(), idx.cpu().numpy(), ov, oi, "large offsets")
    del big

"""The seeded input generators: determinism and the recipe of each workload."""

import numpy as np

from sparse_attention_indexer_row_gb300 import synth


def test_deterministic():
    a = synth.uniform_pool(rows=2, n=4096)
    b = synth.uniform_pool(rows=2, n=4096)
    assert np.array_equal(a.scores.view(np.uint32), b.scores.view(np.uint32))


def test_uniform_range():
    w = synth.uniform_pool(rows=4, n=16384)
    assert w.scores.dtype == np.float32 and w.scores.shape == (4, 16384)
    assert w.scores.min() >= -1.0 and w.scores.max() < 1.0
    assert not np.any(np.signbit(w.scores) & (w.scores == 0))   # no -0.0


def test_varlen_lengths():
    w = synth.normal_varlen(rows=64, n=131072)
    assert w.lengths.dtype == np.int32
    assert w.lengths.min() >= 256 and w.lengths.max() <= 131072
    assert np.sum(w.lengths < 512) >= 2      # rows that return every valid position


def test_relu_mix_shape():
    w = synth.relu_mix(rows=2, n=1 << 16)
    frac_small = np.mean(np.abs(w.scores) < 0.05)
    assert 0.4 < frac_small < 0.6          # about half the rows are noise only


def test_long_layouts():
    s = synth.long_rows("sorted", rows=2, n=1 << 15)
    assert np.all(np.diff(s.scores, axis=1) >= 0)
    q = synth.long_rows("quant", rows=2, n=1 << 16)
    fin = q.scores[np.isfinite(q.scores)]
    assert np.unique(fin).size == 256 and not np.any(fin == 0)
    frac_inf = np.mean(np.isinf(q.scores))
    assert 0.0005 < frac_inf < 0.0015
    assert np.any(q.scores == np.inf) and np.any(q.scores == -np.inf)


def test_causal_lengths():
    w = synth.causal_prefill(rows=64, n=512)
    assert np.array_equal(w.lengths, np.minimum(8 * (np.arange(64) + 1), 512))


def test_algorithmic_bytes():
    w = synth.uniform_pool(rows=4, n=16384, k=512)
    assert w.algorithmic_bytes() == 4 * 4 * 16384 + 8 * 4 * 512

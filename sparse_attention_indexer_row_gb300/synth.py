"""Seeded synthetic score rows for the selector's workloads.

This module only draws inputs.  It holds none of the selection arithmetic and
is shared by the tests, the smoke check and the benchmark, so that the CUDA
path and the CPU oracle always see the same bytes.

Every workload mirrors a shape the pages describe for the indexer's top-k:
* ~16K-candidate pool rows (the layer-20 block pool of 8-position blocks that
  leaves about 16,000 candidates: The Secret GPU Kernel Behind DeepSeek V4.1
  Flash, video transcript 7:22-7:46);
* decode rows of up to a million cached positions with k = 512 ("index top k
  512", 2:00-2:13; "a million tokens", 2:13-2:40);
* a causal prefill indexer, where query row r can see the first 8(r+1)
  positions.

All draws use numpy's PCG64 ``Generator`` seeded with the workload's seed, in
float64 where a transform is applied, rounded once to float32.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

M1 = 1 << 20


@dataclass
class Workload:
    name: str
    scores: np.ndarray              # float32 [rows, row_stride]
    k: int
    n: int
    lengths: np.ndarray | None      # int32 [rows] or None (all rows full)
    meta: dict = field(default_factory=dict)

    @property
    def rows(self) -> int:
        return int(self.scores.shape[0])

    @property
    def row_stride(self) -> int:
        return int(self.scores.shape[1])

    def valid_elements(self) -> int:
        if self.lengths is None:
            return self.rows * self.n
        return int(self.lengths.astype(np.int64).sum())

    def algorithmic_bytes(self) -> int:
        """Each valid score read once (4 B) plus the k (value, index) outputs."""
        return 4 * self.valid_elements() + 8 * self.rows * self.k


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    return rng.standard_normal(shape, dtype=np.float32)


def uniform_pool(rows=4, n=16384, k=512, seed=1) -> Workload:
    """i.i.d. Uniform[-1, 1) rows, all full length."""
    rng = np.random.default_rng(seed)
    u = rng.random((rows, n), dtype=np.float32)           # j * 2^-24, j < 2^24
    x = (u * np.float32(2.0) - np.float32(1.0)).astype(np.float32)  # exact
    return Workload(f"uniform_pool_{rows}x{n}_k{k}", x, k, n, None,
                    {"dist": "Uniform[-1,1)", "seed": seed})


def normal_varlen(rows=64, n=131072, k=512, seed=2, lo=256, short_rows=2) -> Workload:
    """i.i.d. Normal(0,1) rows with valid length L_r ~ UniformInt[lo, n].

    A uniform draw over [256, 131072] almost never lands below k, so the first
    ``short_rows`` rows draw L_r ~ UniformInt[lo, k - 1] instead: the batch
    always holds rows that return every valid position.
    """
    rng = np.random.default_rng(seed)
    x = _normal(rng, (rows, n))
    lengths = rng.integers(lo, n, size=rows, endpoint=True).astype(np.int32)
    ns = min(short_rows, rows)
    if ns and k - 1 >= lo:
        lengths[:ns] = rng.integers(lo, k - 1, size=ns, endpoint=True)
    return Workload(f"normal_varlen_{rows}x{n}_k{k}", x, k, n, lengths,
                    {"dist": "Normal(0,1)",
                     "lengths": f"UniformInt[{lo},{n}], first {ns} rows UniformInt[{lo},{k - 1}]",
                     "seed": seed})


def relu_mix(rows=1, n=M1, k=512, seed=3) -> Workload:
    """ReLU(N1) * 0.5 + 0.01 * N2 with two independent standard normals."""
    rng = np.random.default_rng(seed)
    a = rng.standard_normal((rows, n))
    b = rng.standard_normal((rows, n))
    x = (np.maximum(a, 0.0) * 0.5 + 0.01 * b).astype(np.float32)
    return Workload(f"relu_mix_{rows}x{n}_k{k}", x, k, n, None,
                    {"dist": "ReLU(N)*0.5+N(0,0.01)", "seed": seed})


def long_rows(layout="normal", rows=64, n=M1, k=512, seed=4) -> Workload:
    """Long decode rows in one of three value layouts.

    normal: i.i.d. Normal(0,1).
    sorted: the same draws sorted ascending in every row (the visiting order
            that makes an unshuffled threshold admit every element).
    quant:  256 exact levels (lvl - 127.5) / 32 with lvl ~ UniformInt[0, 255]
            (heavy ties, no zero), then each entry independently with
            probability 0.001 replaced by +inf or -inf (probability 1/2 each).
    """
    rng = np.random.default_rng(seed)
    if layout in ("normal", "sorted"):
        x = _normal(rng, (rows, n))
        if layout == "sorted":
            x.sort(axis=1)
    elif layout == "quant":
        lvl = rng.integers(0, 256, size=(rows, n), dtype=np.int16)
        x = ((lvl.astype(np.float32) - np.float32(127.5)) / np.float32(32.0)).astype(np.float32)
        hit = rng.random((rows, n), dtype=np.float32) < np.float32(0.001)
        sign = rng.random((rows, n), dtype=np.float32) < np.float32(0.5)
        x[hit & sign] = np.inf
        x[hit & ~sign] = -np.inf
    else:
        raise ValueError(layout)
    return Workload(f"long_{layout}_{rows}x{n}_k{k}", x, k, n, None,
                    {"layout": layout, "seed": seed})


def causal_prefill(rows=8192, n=65536, k=512, seed=5) -> Workload:
    """Prefill indexer: Normal(0,1), row r valid for its first 8(r+1) entries."""
    rng = np.random.default_rng(seed)
    x = _normal(rng, (rows, n))
    lengths = np.minimum(8 * (np.arange(rows, dtype=np.int64) + 1), n).astype(np.int32)
    return Workload(f"causal_prefill_{rows}x{n}_k{k}", x, k, n, lengths,
                    {"dist": "Normal(0,1)", "lengths": "8(r+1)", "seed": seed})


# The five workload families at their full sizes.
CONFIGS = {
    "c1": lambda: uniform_pool(),
    "c2": lambda: normal_varlen(),
    "c3_1": lambda: relu_mix(rows=1),
    "c3_4": lambda: relu_mix(rows=4),
    "c4_normal_k512": lambda: long_rows("normal", k=512),
    "c4_sorted_k512": lambda: long_rows("sorted", k=512),
    "c4_quant_k512": lambda: long_rows("quant", k=512),
    "c4_normal_k2048": lambda: long_rows("normal", k=2048),
    "c4_sorted_k2048": lambda: long_rows("sorted", k=2048),
    "c4_quant_k2048": lambda: long_rows("quant", k=2048),
    "c5": lambda: causal_prefill(),
}


def make(name: str) -> Workload:
    return CONFIGS[name]()

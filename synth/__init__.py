"""Seeded synthetic workloads for the training path and its parity tests.

This module only draws inputs: features, labels, pre-binned columns, node
assignments and gradients.  It holds none of the training method's arithmetic
(no binning, gradients, histograms, gains or partitions), so the CUDA path and
the CPU oracle can both consume its arrays without sharing method code.

Every generator takes ``seed`` (default 0) and an optional row count ``n`` so
that tests can draw the same *shape* of workload at a size the oracle finishes
in seconds.  Features are returned column-major as a C-contiguous ``(F, N)``
float32 array; labels as ``(N,)`` float32.

Workloads (the real datasets the pages measure on are not available; these
stand in for their shapes):

``tiny``    2,000 x 8, U(0,1) features, y = 3x0 - 2x1 + x2*x3 + N(0, 0.1).
``mid``     100,000 x 28, N(0,1) features,
            y = sum_{j<10} sin x_j + 0.5 x10 x11 + N(0, 0.1).
``covtype`` 581,012 x 54 (the shape of the forest-cover data): 3 uniform
            integers in [0, 4000), 7 rounded 100*N(0,1), a 4-way and a 40-way
            one-hot block of Zipf(1.2) categories; label in 1..7 with
            P(k) ~ k^-1.2, independent of the features.
``large``   10,000,000 x 100: 50 N(0,1), 30 LogNormal(0, 1.5), 20 integer
            columns with 2..16 distinct values; label = sum of 20 random full
            depth-3 step trees + N(0, 0.5).
``make_binary(name)``: the same features with a 0/1 label, 1 where the
            workload's label exceeds its median (input of the logistic
            objective).
``micro``   one tree level: 50,000,000 x 64 pre-binned uint8 columns with
            P(b) ~ (b+1)^-1.1 on 0..255, 256 nodes (sibling pairs 2k, 2k+1),
            g ~ N(0,1) float32.
"""
from __future__ import annotations

import numpy as np

__all__ = ["CONFIGS", "make", "make_binary", "binary_label", "make_tiny", "make_mid", "make_covtype", "make_large", "make_micro"]

# Training parameters of each workload.  Unspecified ones take the readings
# recorded in the design notes: gamma 0, min_child_weight 0, lambda 1.
CONFIGS = {
    "tiny": dict(n=2_000, f=8, max_bins=32, max_depth=3, n_trees=5, learning_rate=0.3,
                 reg_lambda=1.0, gamma=0.0, min_samples_leaf=1, min_child_weight=0.0),
    "mid": dict(n=100_000, f=28, max_bins=255, max_depth=6, n_trees=100, learning_rate=0.1,
                reg_lambda=1.0, gamma=0.0, min_samples_leaf=20, min_child_weight=0.0),
    "covtype": dict(n=581_012, f=54, max_bins=255, max_depth=10, n_trees=100, learning_rate=0.1,
                    reg_lambda=1.0, gamma=0.0, min_samples_leaf=1, min_child_weight=0.0),
    "large": dict(n=10_000_000, f=100, max_bins=255, max_depth=8, n_trees=200, learning_rate=0.05,
                  reg_lambda=1.0, gamma=0.1, min_samples_leaf=20, min_child_weight=0.0),
    "micro": dict(n=50_000_000, f=64, n_nodes=256, reg_lambda=1.0, gamma=0.0,
                  min_samples_leaf=1, min_child_weight=0.0),
}


def _rng(seed: int, *stream: int) -> np.random.Generator:
    """Independent stream per (seed, stream ids), so columns do not depend on N."""
    return np.random.default_rng(np.random.SeedSequence([seed, *stream]))


def make_tiny(seed: int = 0, n: int | None = None):
    n = CONFIGS["tiny"]["n"] if n is None else n
    f = CONFIGS["tiny"]["f"]
    X = np.empty((f, n), dtype=np.float32)
    for j in range(f):
        X[j] = _rng(seed, 1, j).random(n, dtype=np.float32)
    x = X.astype(np.float64)
    noise = _rng(seed, 2).normal(0.0, 0.1, n)
    y = 3.0 * x[0] - 2.0 * x[1] + x[2] * x[3] + noise
    return X, y.astype(np.float32)


def make_mid(seed: int = 0, n: int | None = None):
    n = CONFIGS["mid"]["n"] if n is None else n
    f = CONFIGS["mid"]["f"]
    X = np.empty((f, n), dtype=np.float32)
    for j in range(f):
        X[j] = _rng(seed, 1, j).standard_normal(n, dtype=np.float32)
    x = X.astype(np.float64)
    y = np.sin(x[:10]).sum(axis=0) + 0.5 * x[10] * x[11] + _rng(seed, 2).normal(0.0, 0.1, n)
    return X, y.astype(np.float32)


def _zipf_categories(rng: np.random.Generator, n: int, k: int, s: float) -> np.ndarray:
    p = (np.arange(1, k + 1, dtype=np.float64)) ** (-s)
    p /= p.sum()
    return rng.choice(k, size=n, p=p)


def make_covtype(seed: int = 0, n: int | None = None):
    n = CONFIGS["covtype"]["n"] if n is None else n
    X = np.zeros((54, n), dtype=np.float32)
    for j in range(3):
        X[j] = _rng(seed, 1, j).integers(0, 4000, n).astype(np.float32)
    for j in range(3, 10):
        X[j] = np.rint(100.0 * _rng(seed, 1, j).standard_normal(n)).astype(np.float32)
    c4 = _zipf_categories(_rng(seed, 3, 0), n, 4, 1.2)
    c40 = _zipf_categories(_rng(seed, 3, 1), n, 40, 1.2)
    X[10 + c4, np.arange(n)] = 1.0
    X[14 + c40, np.arange(n)] = 1.0
    y = 1 + _zipf_categories(_rng(seed, 2), n, 7, 1.2)
    return X, y.astype(np.float32)


def _random_step_tree(rng: np.random.Generator, X: np.ndarray) -> np.ndarray:
    """A full depth-3 axis-aligned tree with random features and thresholds."""
    f, n = X.shape
    feats = rng.integers(0, f, 7)
    rows = rng.integers(0, n, 7)
    thr = X[feats, rows]
    leaves = rng.standard_normal(8)
    node = np.zeros(n, dtype=np.int64)  # heap index 0..6 for internal nodes
    for _ in range(3):
        go_right = X[feats[node], np.arange(n)] > thr[node]
        node = 2 * node + 1 + go_right
    return leaves[node - 7]


def make_large(seed: int = 0, n: int | None = None):
    n = CONFIGS["large"]["n"] if n is None else n
    X = np.empty((100, n), dtype=np.float32)
    for j in range(50):
        X[j] = _rng(seed, 1, j).standard_normal(n, dtype=np.float32)
    for j in range(50, 80):
        X[j] = _rng(seed, 1, j).lognormal(0.0, 1.5, n).astype(np.float32)
    for k in range(20):
        X[80 + k] = _rng(seed, 1, 80 + k).integers(0, 2 + (k % 15), n).astype(np.float32)
    y = _rng(seed, 2).normal(0.0, 0.5, n)
    trees = _rng(seed, 4)
    for _ in range(20):
        y += _random_step_tree(trees, X)
    return X, y.astype(np.float32)


def _zipf_lut(n_bins: int = 256, s: float = 1.1, bits: int = 16) -> np.ndarray:
    """Lookup table mapping a uniform `bits`-bit integer to a Zipf(s) bin."""
    p = (np.arange(1, n_bins + 1, dtype=np.float64)) ** (-s)
    cdf = np.cumsum(p / p.sum())
    u = (np.arange(1 << bits, dtype=np.float64) + 0.5) / (1 << bits)
    return np.minimum(np.searchsorted(cdf, u, side="right"), n_bins - 1).astype(np.uint8)


def make_micro(seed: int = 0, n: int | None = None, f: int | None = None, n_nodes: int = 256,
               grouped: bool = True):
    """Pre-binned level: returns (bins [F][N] uint8, node [N] uint16, g [N] float32).

    Each row's node is uniform on 0..n_nodes-1; sibling pairs are (2k, 2k+1).
    With ``grouped`` the rows are stored grouped by parent k (the order a
    trainer that keeps node segments contiguous holds them in); rows are i.i.d.
    so this is the same distribution as an ungrouped draw, only reordered.
    """
    n = CONFIGS["micro"]["n"] if n is None else n
    f = CONFIGS["micro"]["f"] if f is None else f
    lut = _zipf_lut()
    bins = np.empty((f, n), dtype=np.uint8)
    for j in range(f):
        u = _rng(seed, 1, j).integers(0, 1 << 16, n, dtype=np.uint16)
        bins[j] = lut[u]
    r = _rng(seed, 5)
    if grouped:
        counts = r.multinomial(n, np.full(n_nodes // 2, 1.0 / (n_nodes // 2)))
        parent = np.repeat(np.arange(n_nodes // 2, dtype=np.uint16), counts)
        node = (2 * parent + r.integers(0, 2, n, dtype=np.uint16)).astype(np.uint16)
    else:
        node = r.integers(0, n_nodes, n, dtype=np.uint16)
    g = _rng(seed, 6).standard_normal(n, dtype=np.float32)
    return bins, node, g


def make(name: str, seed: int = 0, n: int | None = None):
    return {"tiny": make_tiny, "mid": make_mid, "covtype": make_covtype, "large": make_large}[name](seed, n)


def binary_label(y: np.ndarray) -> np.ndarray:
    """0/1 float32 label: 1 where y exceeds its median."""
    return (y > np.median(y)).astype(np.float32)


def make_binary(name: str, seed: int = 0, n: int | None = None):
    """Features of workload ``name`` with the 0/1 label of binary_label."""
    X, y = make(name, seed, n)
    return X, binary_label(y)

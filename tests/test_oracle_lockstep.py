"""Pins of the oracle's parity-harness options (no GPU): starting from given predictions, and the
lockstep guide's tie rule.

The guide lets the oracle take another program's (feature, bin) at a node only where the two are
tied: gains within 1e-12 relative, or -- given that program's per-row rounding of g -- within a bound
on how far rounding the same rows' sums can move the gains.  These tests check that the bound covers
what such rounding really does (another program is simulated by rounding every g to a coarse fixed
point grid and letting the oracle's own split search choose on those sums), that it does not let a
clearly worse candidate through, and that a run started from given predictions is the run it continues.
"""
import numpy as np
import pytest

import oracle


def _data(seed, N=3000, F=6, nb=24, dup=False):
    rng = np.random.default_rng(seed)
    bins = rng.integers(0, nb, (F, N)).astype(np.uint8)
    if dup:
        bins[1] = bins[0]  # two identical features: every split of one ties with the other's exactly
    w = rng.normal(size=F)
    y = (bins.astype(np.float64).T @ w / nb + rng.normal(0, 0.3, N)).astype(np.float32)
    return bins, np.full(F, nb, np.int32), y


P = dict(max_depth=1, learning_rate=0.3, reg_lambda=1.0, gamma=0.0, min_samples_leaf=1, min_child_weight=0.0)


def test_start_from_predictions_continues_the_same_run():
    bins, nb, y = _data(0)
    two = oracle.train(bins, nb, y, n_trees=2, **dict(P, max_depth=3))
    first = oracle.train(bins, nb, y, n_trees=1, **dict(P, max_depth=3))
    second = oracle.train(bins, nb, y, n_trees=1, pred_in=first["pred"], **dict(P, max_depth=3))
    assert np.array_equal(second["nodes"][0], two["nodes"][1])
    assert np.array_equal(second["pred"], two["pred"])
    assert second["init_pred"] == two["init_pred"]


def _guide(feature, bin_, M=3):
    g = np.full((1, M, 2), -1, np.int32)
    g[0, 0] = (feature, bin_)
    return g


def test_exact_ties_are_adopted_and_worse_candidates_are_not():
    rng = np.random.default_rng(1)
    N, F, nb = 3000, 6, 24
    bins = rng.integers(0, nb, (F, N)).astype(np.uint8)
    bins[1] = bins[0]  # feature 1 is feature 0: every split of one is the same partition as the other's
    y = (bins[0] / nb + rng.normal(0, 0.1, N)).astype(np.float32)
    nbins = np.full(F, nb, np.int32)
    own = oracle.train(bins, nbins, y, n_trees=1, **P)
    f, b = own["nodes"][0][0]["feature"], own["nodes"][0][0]["threshold_bin"]
    assert f == 0  # the smaller feature wins the exact tie
    tied = oracle.train(bins, nbins, y, n_trees=1, guide=_guide(1, b), **P)
    assert tied["info"][0][0]["adopted"] == 1 and tied["nodes"][0][0]["feature"] == 1
    assert tied["info"][0][0]["guide_gap"] == 0.0
    # a candidate far from the best (a feature the label ignores) is a mismatch, with or without quanta
    for tq in (None, np.array([[2.0 ** -30, 0.0]])):
        r = oracle.train(bins, nbins, y, n_trees=1, guide=_guide(F - 1, nb // 2), tie_quanta=tq, **P)
        assert r["info"][0][0]["guide_mismatch"] == 1
        assert (r["nodes"][0][0]["feature"], r["nodes"][0][0]["threshold_bin"]) == (f, b)


def _close_data(seed, N=2000, F=8, nb=16):
    """Features that are copies of one base column with 0.5% .. 4% of their rows redrawn: every feature's
    best split has nearly the same gain, so rounding can reorder them."""
    rng = np.random.default_rng(seed)
    base = rng.integers(0, nb, N)
    bins = np.empty((F, N), np.uint8)
    for j in range(F):
        col = base.copy()
        m = rng.random(N) < 0.005 * (j + 1)
        col[m] = rng.integers(0, nb, int(m.sum()))
        bins[j] = col
    y = (np.sin(base / 3.0) + rng.normal(0, 0.5, N)).astype(np.float32)
    return bins, np.full(F, nb, np.int32), y


def _rounded_program_choice(bins, nb, y, S):
    """The root split another program would choose if it summed round(g * 2^S) * 2^-S per row."""
    pred = np.full(bins.shape[1], float(np.float64(y).mean()))
    g, _ = oracle.gradients(pred, y, 0)
    gq = np.ldexp(np.rint(np.ldexp(g, S)), -S)
    h = oracle.histograms(bins, gq, np.zeros(bins.shape[1], np.int32), 1)
    sp = oracle.best_split(h["cnt"][0], h["G"][0], h["H"][0], nb, bins.shape[1], float(h["Gt"][0]), float(h["Ht"][0]),
                           **P)
    return sp


@pytest.mark.parametrize("S", [1, 2, 4, 8])
def test_rounding_bound_covers_a_coarse_fixed_point_program(S):
    """Over many seeds a program rounding g to 2^-S per row chooses differently at some roots; with its
    quantum 2^-(S+1) every such choice is adopted (never a mismatch), and without it they mismatch."""
    differ = 0
    for seed in range(60):
        bins, nb, y = _close_data(100 + seed)
        sp = _rounded_program_choice(bins, nb, y, S)
        if not sp.valid:
            continue
        guide = _guide(sp.feature, sp.bin)
        with_q = oracle.train(bins, nb, y, n_trees=1, guide=guide, tie_quanta=np.array([[2.0 ** -(S + 1), 0.0]]),
                              **P)
        info = with_q["info"][0][0]
        assert info["guide_mismatch"] == 0, (seed, info["guide_gap"], info["guide_bound"])
        assert (with_q["nodes"][0][0]["feature"], with_q["nodes"][0][0]["threshold_bin"]) == (sp.feature, sp.bin)
        if info["adopted"] == 2:
            differ += 1
            assert 0 <= info["guide_gap"] <= info["guide_bound"]
            without = oracle.train(bins, nb, y, n_trees=1, guide=guide, **P)
            assert without["info"][0][0]["guide_mismatch"] == 1
    if S <= 2:
        assert differ >= 2  # the coarse program does reorder some roots: the bound is what admits them

"""Pins of the oracle's logistic objective ("Gradient boosted trees
(spec model)": binary cross-entropy with a sigmoid, whose gradient in the
margin is sigmoid(pred) - target; the second derivative p(1 - p) weighs H).
"""
import math

import numpy as np
import pytest

import oracle


def test_gradients_closed_form(o=oracle):
    y = np.array([0, 1, 0, 1, 0, 1], np.float32)
    pred = np.array([0.0, 0.0, math.log(3.0), math.log(3.0), 40.0, -40.0])
    g, h = o.gradients(pred, y, objective=1)
    assert g[0] == 0.5 and g[1] == -0.5 and h[0] == 0.25 and h[1] == 0.25  # p = 1/2 exactly
    assert abs(g[2] - 0.75) < 1e-15 and abs(g[3] + 0.25) < 1e-15 and abs(h[2] - 0.1875) < 1e-15
    assert g[4] == pytest.approx(1.0, abs=1e-16) and g[5] == pytest.approx(-1.0, abs=1e-16)
    # saturated: at +40 the sigmoid rounds to 1 and h to exactly 0; at -40 p = e^-40 stays positive
    assert h[4] == 0.0 and h[5] == pytest.approx(math.exp(-40.0), rel=1e-12)
    assert np.all(np.isfinite(g)) and np.all(np.isfinite(h))
    gs, hs = o.gradients(pred, y, objective=0)
    assert np.array_equal(gs, pred - y) and np.all(hs == 1.0)


def _hand_data():
    X = np.array([[0.0, 0.0, 1.0, 1.0]], np.float32)
    y = np.array([0, 0, 1, 1], np.float32)
    return X, y


def test_hand_tree_depth_one(o=oracle):
    """Margin 0: g = 0.5 - y, h = 1/4.  Root G = 0, H = 1; the split x <= 0 has G_L = 1, H_L = 1/2,
    G_R = -1, H_R = 1/2: gain = 0.5 * (1/(1/2 + 1) + 1/(1/2 + 1) - 0) = 2/3; leaves -G/(H + 1) = -/+ 2/3."""
    X, y = _hand_data()
    bins, _, n_bins = o.quantize(X, 4)
    r = o.train(bins, n_bins, y, n_trees=1, max_depth=1, learning_rate=1.0, reg_lambda=1.0, objective=1)
    assert r["init_pred"] == 0.0
    nd = r["nodes"][0]
    assert nd[0]["feature"] == 0 and nd[0]["threshold_bin"] == 0
    assert nd[0]["gain"] == pytest.approx(2.0 / 3.0, rel=1e-15)
    assert nd[1]["leaf_value"] == pytest.approx(-2.0 / 3.0, rel=1e-15)
    assert nd[2]["leaf_value"] == pytest.approx(2.0 / 3.0, rel=1e-15)
    assert np.allclose(r["pred"], [-2 / 3, -2 / 3, 2 / 3, 2 / 3], rtol=1e-15, atol=0)
    info = r["info"][0]
    assert info[0]["H"] == 1.0 and info[1]["H"] == 0.5 and info[2]["H"] == 0.5


def test_second_tree_uses_new_margins(o=oracle):
    """After one depth-0 tree (lambda 0: the Newton step -G/H of a constant margin) the second
    tree's gradients are taken at the new margin m: g = sigmoid(m) - y, h = p(1 - p)."""
    X, y = _hand_data()
    y = np.array([0, 1, 1, 1], np.float32)
    bins, _, n_bins = o.quantize(X, 4)
    r = o.train(bins, n_bins, y, n_trees=2, max_depth=0, learning_rate=1.0, reg_lambda=0.0, objective=1)
    w0 = (3 - 4 * 0.5) / (4 * 0.25)  # first step from margin 0: -G/H with G = 4*(1/2) - 3, H = 4/4
    p = 1.0 / (1.0 + math.exp(-w0))
    w1 = (3 - 4 * p) / (4 * p * (1 - p))
    assert r["nodes"][0][0]["leaf_value"] == pytest.approx(w0, rel=1e-15)
    assert r["nodes"][1][0]["leaf_value"] == pytest.approx(w1, rel=1e-13)
    assert np.allclose(r["pred"], w0 + w1, rtol=1e-13)


def test_logistic_needs_binary_labels(o=oracle):
    X, y = _hand_data()
    bins, _, n_bins = o.quantize(X, 4)
    with pytest.raises(o.OracleError):
        o.train(bins, n_bins, np.array([0, 0.5, 1, 1], np.float32), n_trees=1, max_depth=1, objective=1)
    assert o.validate_params(objective=2) != 0 and o.validate_params(objective=1) == 0


def test_histograms_with_hessians_brute_force(o=oracle):
    """H of a (slot, feature, bin) entry is the sum of h over its rows, visited one by one here."""
    rng = np.random.default_rng(11)
    F, N, n_slots = 3, 40, 3
    bins = rng.integers(0, 5, size=(F, N)).astype(np.uint8)
    g = rng.normal(size=N)
    h = rng.uniform(0.0, 0.25, size=N)
    slot = rng.integers(-1, n_slots, size=N).astype(np.int32)
    out = o.histograms(bins, g, slot, n_slots, h=h)
    for s in range(n_slots):
        for j in range(F):
            for b in range(5):
                rows = [r for r in range(N) if slot[r] == s and bins[j, r] == b]
                assert out["cnt"][s, j, b] == len(rows)
                assert out["H"][s, j, b] == pytest.approx(sum(h[r] for r in rows), rel=1e-14, abs=1e-300)
                assert out["G"][s, j, b] == pytest.approx(sum(g[r] for r in rows), rel=1e-14, abs=1e-15)
        assert out["Ht"][s] == pytest.approx(sum(h[r] for r in range(N) if slot[r] == s), rel=1e-14)
    unit = o.histograms(bins, g, slot, n_slots)
    assert np.array_equal(unit["H"], unit["cnt"].astype(np.float64))

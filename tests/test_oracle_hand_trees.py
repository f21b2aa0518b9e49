"""Hand-computed trees ("Module Design: Training Core", s.8 Acceptance: small
trees computed by hand agree node by node).  Every expected number below was
worked out on paper from s.2 (g = pred - label, h = 1, score G^2/(H+lambda),
weight -G/(H+lambda), gain 0.5(s_L + s_R - s_P) - gamma) and s.3 (validity,
frozen tie-break, bin <= threshold goes left); the derivation is in comments.
"""
import numpy as np
import pytest

TOL = 1e-12


def _tree(out, t):
    n = out["nodes_per_tree"][t]
    return out["nodes"][t][:n]


def test_hand_tree_single_split(orc):
    # 4 rows, 1 feature with bins 0..3, labels 0,0,4,4; lambda=gamma=0, depth 1, lr 1.
    # init = 2, g = [2, 2, -2, -2], G_P = 0, H_P = 4.
    # b=0: G_L=2,H_L=1 | G_R=-2,H_R=3: gain = .5(4 + 4/3) = 8/3
    # b=1: G_L=4,H_L=2 | G_R=-4,H_R=2: gain = .5(8 + 8) = 8      <- best
    # b=2: G_L=2,H_L=3 | G_R=-2,H_R=1: gain = 8/3
    # leaves: -4/2 = -2 and 4/2 = 2; predictions 2-2 = 0 and 2+2 = 4.
    bins = np.array([[0, 1, 2, 3]], np.uint8)
    y = np.array([0, 0, 4, 4], np.float32)
    out = orc.train(bins, [4], y, n_trees=1, max_depth=1, learning_rate=1.0, reg_lambda=0.0, gamma=0.0)
    assert out["init_pred"] == 2.0
    t = _tree(out, 0)
    assert len(t) == 3
    assert (t[0]["feature"], t[0]["threshold_bin"], t[0]["left"], t[0]["right"], t[0]["is_leaf"]) == (0, 1, 1, 2, 0)
    assert t[0]["gain"] == pytest.approx(8.0, abs=TOL)
    assert t[1]["is_leaf"] == 1 and t[1]["leaf_value"] == pytest.approx(-2.0, abs=TOL)
    assert t[2]["is_leaf"] == 1 and t[2]["leaf_value"] == pytest.approx(2.0, abs=TOL)
    np.testing.assert_allclose(out["pred"], [0, 0, 4, 4], atol=TOL)


@pytest.mark.parametrize(
    "kw,expect_split",
    [
        (dict(min_samples_leaf=2), (0, 1)),  # b=0 and b=2 leave one row on a side
        (dict(min_samples_leaf=3), None),  # no threshold leaves 3 rows on both sides
        (dict(min_child_weight=2.0), (0, 1)),  # H_L = H_R = 2 meets >= 2
        (dict(min_child_weight=2.5), None),  # b=1 has H = 2 < 2.5; b=0/b=2 have H = 1 on one side
        (dict(gamma=8.0), None),  # gain 8 - 8 = 0 is not strictly positive: leaf
        (dict(gamma=7.5), (0, 1)),  # gain 0.5 > 0
    ],
)
def test_hand_tree_validity_rules(orc, kw, expect_split):
    bins = np.array([[0, 1, 2, 3]], np.uint8)
    y = np.array([0, 0, 4, 4], np.float32)
    params = dict(n_trees=1, max_depth=1, learning_rate=1.0, reg_lambda=0.0, gamma=0.0)
    params.update(kw)
    out = orc.train(bins, [4], y, **params)
    t = _tree(out, 0)
    if expect_split is None:
        assert len(t) == 1 and t[0]["is_leaf"] == 1
        assert t[0]["leaf_value"] == 0.0  # -0/(4+0)
    else:
        assert (t[0]["feature"], t[0]["threshold_bin"]) == expect_split
        assert t[0]["gain"] == pytest.approx(8.0 - kw.get("gamma", 0.0), abs=TOL)


def test_hand_tree_two_trees_lambda_one(orc):
    # 6 rows; f0 bins [0,0,1,1,2,2] (3 bins), f1 bins [1,0,1,0,1,0] (2 bins);
    # labels [0,2,6,6,10,12]; lambda = 1, gamma = 0, depth 2, lr 0.5, 2 trees.
    # Tree 1: init 6, g = [6,4,0,0,-4,-6], G_P = 0, H_P = 6.
    #   f0 b0: G_L=10,H_L=2 | -10,4 -> .5(100/3 + 100/5) = 80/3
    #   f0 b1: G_L=10,H_L=4 | -10,2 -> same value, bit-identical: tie -> smaller bin b0
    #   f1 b0: rows {1,3,5} G_L=-2,H_L=3 | 2,3 -> .5(4/4 + 4/4) = 1
    #   root: f0 b0, left = rows {0,1}, right = rows {2,3,4,5}.
    #   node1 rows {0,1}: f0 has one occupied bin (no valid threshold);
    #     f1 b0: 4,1 | 6,1 vs s_P = 100/3: .5(8 + 18 - 100/3) < 0 -> leaf -10/3.
    #   node2 rows {2..5}: G=-10,H=4, s_P = 20.
    #     f0 b0: empty left -> invalid; f0 b1: 0,2 | -10,2 -> .5(0 + 100/3 - 20) = 20/3
    #     f1 b0: rows {3,5} -6,2 | -4,2 -> .5(12 + 16/3 - 20) < 0
    #     split f0 b1 -> node3 rows {2,3} leaf -0/3 = 0, node4 rows {4,5} leaf 10/3.
    #   preds: 6 - 5/3 = 13/3 (rows 0,1), 6 (rows 2,3), 6 + 5/3 = 23/3 (rows 4,5).
    # Tree 2: g = [13/3, 7/3, 0, 0, -7/3, -13/3], G_P = 0.
    #   f0 b0 and b1 tie at .5(400/27 + 400/45) = 320/27 -> b0; f1 b0 gives 1.
    #   node1 rows {0,1}: G = 20/3, H = 2, leaf -(20/3)/3 = -20/9 (f1 b0 gain < 0).
    #   node2 rows {2..5}: G = -20/3, s_P = 80/9; f0 b1: .5(400/27 - 240/27) = 80/27;
    #     f1 b0: .5(169/27 + 49/27 - 240/27) < 0. leaves 0 and 20/9.
    #   preds: 13/3 - 10/9 = 29/9, 6, 23/3 + 10/9 = 79/9.
    bins = np.array([[0, 0, 1, 1, 2, 2], [1, 0, 1, 0, 1, 0]], np.uint8)
    y = np.array([0, 2, 6, 6, 10, 12], np.float32)
    out = orc.train(bins, [3, 2], y, n_trees=2, max_depth=2, learning_rate=0.5, reg_lambda=1.0, gamma=0.0)
    assert out["init_pred"] == 6.0
    expect = [
        dict(gains=(80 / 3, 20 / 3), leaves=(-10 / 3, 0.0, 10 / 3)),
        dict(gains=(320 / 27, 80 / 27), leaves=(-20 / 9, 0.0, 20 / 9)),
    ]
    for ti, e in enumerate(expect):
        t = _tree(out, ti)
        assert len(t) == 5
        assert [(n["feature"], n["threshold_bin"], n["left"], n["right"]) for n in t] == [
            (0, 0, 1, 2), (-1, -1, -1, -1), (0, 1, 3, 4), (-1, -1, -1, -1), (-1, -1, -1, -1)]
        assert list(t["is_leaf"]) == [0, 1, 0, 1, 1]
        assert t[0]["gain"] == pytest.approx(e["gains"][0], rel=1e-13)
        assert t[2]["gain"] == pytest.approx(e["gains"][1], rel=1e-13)
        for idx, v in zip((1, 3, 4), e["leaves"]):
            assert t[idx]["leaf_value"] == pytest.approx(v, abs=1e-13)
    np.testing.assert_allclose(out["pred"], [29 / 9, 29 / 9, 6, 6, 79 / 9, 79 / 9], rtol=0, atol=1e-13)


def test_tie_break_prefers_smaller_feature(orc):
    # Two identical columns give bit-identical gains: feature 0 must win.
    col = np.array([0, 1, 2, 3], np.uint8)
    bins = np.stack([col, col])
    y = np.array([0, 0, 4, 4], np.float32)
    out = orc.train(bins, [4, 4], y, n_trees=1, max_depth=1, learning_rate=1.0, reg_lambda=0.0)
    assert _tree(out, 0)[0]["feature"] == 0
    # Swap in a strictly better second column: the larger gain wins regardless of index.
    worse = np.array([0, 1, 1, 1], np.uint8)  # best threshold isolates one row only
    out = orc.train(np.stack([worse, col]), [2, 4], y, n_trees=1, max_depth=1, learning_rate=1.0,
                    reg_lambda=0.0)
    assert (_tree(out, 0)[0]["feature"], _tree(out, 0)[0]["threshold_bin"]) == (1, 1)


def test_constant_labels_single_leaf(orc):
    rng = np.random.default_rng(3)
    bins = rng.integers(0, 8, (3, 40)).astype(np.uint8)
    y = np.full(40, 1.75, np.float32)
    out = orc.train(bins, [8, 8, 8], y, n_trees=3, max_depth=4, learning_rate=0.3, reg_lambda=1.0)
    for t in range(3):
        tr = _tree(out, t)
        assert len(tr) == 1 and tr[0]["is_leaf"] == 1 and tr[0]["leaf_value"] == 0.0
    assert np.all(out["pred"] == 1.75)


def test_max_depth_zero_is_a_leaf(orc):
    bins = np.array([[0, 1, 2, 3]], np.uint8)
    y = np.array([0, 0, 4, 4], np.float32)
    out = orc.train(bins, [4], y, n_trees=1, max_depth=0, learning_rate=1.0, reg_lambda=1.0)
    t = _tree(out, 0)
    assert len(t) == 1 and t[0]["is_leaf"] == 1


def test_parameter_rules(orc):
    # "Module Design: Training Core", s.3: min_samples_leaf >= 1, min_child_weight >= 0,
    # reg_lambda >= 0, gamma >= 0, every floating parameter finite.
    assert orc.validate_params() == orc.OK
    for bad in (dict(min_samples_leaf=0), dict(min_child_weight=-1e-300), dict(reg_lambda=-1.0),
                dict(gamma=-0.5), dict(learning_rate=float("nan")), dict(reg_lambda=float("inf")),
                dict(gamma=float("inf")), dict(min_child_weight=float("nan")), dict(max_depth=-1)):
        assert orc.validate_params(**bad) == orc.EINVAL, bad
    bins = np.zeros((1, 4), np.uint8)
    with pytest.raises(orc.OracleError) as e:
        orc.train(bins, [1], np.array([0, 1, 2, np.nan], np.float32), n_trees=1, max_depth=1)
    assert e.value.code == orc.ENONFINITE

"""Batched prediction on raw features (gbdt_predict through the C ABI) against the oracle.

"Gradient boosted trees (spec model)", Forward pass and Tree representation:
predictions are init + learning_rate * sum of tree outputs, x > edges[j][b]
goes right.  Predicting the training rows must give gbdt_train's own
predictions bit for bit; new rows (values exactly at edges, +-0, NaN, +-inf,
huge magnitudes) must equal the oracle bit for bit.
"""
import math

import numpy as np
import pytest

from tests.gpu_util import g, needs_gpu, oracle, torch
import synth

pytestmark = [pytest.mark.gpu, needs_gpu]


def _train(name, n, depth, trees):
    X, y = synth.make(name, n=n)
    cfg = dict(synth.CONFIGS[name], max_depth=depth, n_trees=trees)
    Xd = torch.from_numpy(X).cuda()
    bins, edges, n_bins = g.quantize(Xd, cfg["max_bins"])
    out = g.train(bins, n_bins, torch.from_numpy(y).cuda(), **cfg)
    return X, Xd, edges, out, cfg


@pytest.mark.parametrize("name,n,depth,trees", [("mid", 50_021, 6, 12), ("covtype", 30_011, 8, 5),
                                                ("large", 20_003, 8, 6), ("tiny", None, 0, 3)])
def test_training_rows_give_training_predictions(name, n, depth, trees):
    X, Xd, edges, out, cfg = _train(name, n, depth, trees)
    p = g.predict(Xd, edges, out["nodes"], out["init_pred"], cfg["learning_rate"], out["nodes_per_tree"])
    assert torch.equal(p, out["pred"])
    ref = oracle.predict(X, edges.cpu().numpy(), out["nodes"], out["init_pred"], cfg["learning_rate"])
    assert np.array_equal(p.cpu().numpy(), ref)


def test_new_rows_with_special_values_match_oracle():
    X, Xd, edges, out, cfg = _train("mid", 40_009, 7, 10)
    rng = np.random.default_rng(5)
    F = X.shape[0]
    N2 = 100_003  # not a multiple of the CTA's rows
    X2 = rng.normal(0, 2, (F, N2)).astype(np.float32)
    e = edges.cpu().numpy()
    for j in range(F):  # values exactly at thresholds go left
        fin = e[j][np.isfinite(e[j])]
        idx = rng.choice(N2, 2000, replace=False)
        X2[j, idx] = rng.choice(fin, 2000)
    specials = np.array([0.0, -0.0, math.nan, math.inf, -math.inf, 1e38, -1e38, 1e-38], np.float32)
    X2[:, :8] = specials[None, :]
    p = g.predict(torch.from_numpy(X2).cuda(), edges, out["nodes"], out["init_pred"], cfg["learning_rate"],
                  out["nodes_per_tree"])
    ref = oracle.predict(X2, e, out["nodes"], out["init_pred"], cfg["learning_rate"])
    assert np.array_equal(p.cpu().numpy(), ref)


def test_many_features_read_directly():
    """More features than the staged shared-memory tile holds: the rows are read from global memory."""
    rng = np.random.default_rng(9)
    F, N = 400, 6_007
    X = rng.normal(size=(F, N)).astype(np.float32)
    y = (X[3] - 2 * X[377] + 0.5 * X[200] * X[201]).astype(np.float32)
    Xd = torch.from_numpy(X).cuda()
    bins, edges, n_bins = g.quantize(Xd, 64)
    cfg = dict(n_trees=4, max_depth=4, learning_rate=0.3, reg_lambda=1.0)
    out = g.train(bins, n_bins, torch.from_numpy(y).cuda(), **cfg)
    p = g.predict(Xd, edges, out["nodes"], out["init_pred"], 0.3, out["nodes_per_tree"])
    assert torch.equal(p, out["pred"])
    X2 = rng.normal(size=(F, 1_001)).astype(np.float32)
    p2 = g.predict(torch.from_numpy(X2).cuda(), edges, out["nodes"], out["init_pred"], 0.3, out["nodes_per_tree"])
    assert np.array_equal(p2.cpu().numpy(), oracle.predict(X2, edges.cpu().numpy(), out["nodes"], out["init_pred"], 0.3))


def test_one_row_and_no_trees():
    X, Xd, edges, out, cfg = _train("tiny", None, 3, 2)
    one = Xd[:, 5:6].contiguous()
    p = g.predict(one, edges, out["nodes"], out["init_pred"], cfg["learning_rate"], out["nodes_per_tree"])
    assert p.item() == out["pred"][5].item()
    p0 = g.predict(Xd, edges, out["nodes"][:0], 1.25, 0.3)
    assert torch.all(p0 == 1.25)


def test_bad_model_is_rejected():
    X, Xd, edges, out, cfg = _train("tiny", None, 3, 2)
    assert out["nodes"][1, 0]["is_leaf"] == 0
    nodes = out["nodes"].copy()
    nodes[1, 0]["feature"] = X.shape[0]  # an internal node pointing past the features
    with pytest.raises(g.GbdtError) as e:
        g.predict(Xd, edges, nodes, out["init_pred"], cfg["learning_rate"], out["nodes_per_tree"])
    assert e.value.code == g.ERR_INVALID_ARG

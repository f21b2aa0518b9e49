"""Pins of the oracle's prediction on raw features (no GPU).

"Gradient boosted trees (spec model)", Forward pass and Tree representation:
init + learning_rate * sum of tree outputs, x > threshold goes right; the
threshold of a split (feature j, bin b) on raw values is the quantize edge
edges[j][b].
"""
import math

import numpy as np
import pytest

import oracle
import synth


def _node(feature=-1, thr=-1, left=-1, right=-1, leaf=0.0):
    return (feature, thr, left, right, leaf, 0.0, 1 if feature < 0 else 0, 0)


def test_hand_model(o=oracle):
    # one feature, edges 1, 2, 3 (max_bins 4).  Tree 0: x > 2 ? (x > 3 ? 2.0 : -1.0) : 0.5.  Tree 1: leaf 0.25.
    edges = np.array([[1.0, 2.0, 3.0]], np.float32)
    nodes = np.zeros((2, 7), oracle.NODE_DTYPE)
    nodes[0, 0] = _node(0, 1, 1, 2)
    nodes[0, 1] = _node(leaf=0.5)
    nodes[0, 2] = _node(0, 2, 3, 4)
    nodes[0, 3] = _node(leaf=-1.0)
    nodes[0, 4] = _node(leaf=2.0)
    nodes[1, 0] = _node(leaf=0.25)
    x = np.array([[2.0, 2.5, 3.0, 3.5, -0.0, math.nan, -7.0, 1e30]], np.float32)
    leaf0 = [0.5, -1.0, -1.0, 2.0, 0.5, 0.5, 0.5, 2.0]  # at a threshold: left; -0.0 and NaN: left
    init, lr = 1.0, 0.1
    want = np.array([(init + (lr * w)) + (lr * 0.25) for w in leaf0])
    got = o.predict(x, edges, nodes, init, lr)
    assert np.array_equal(got, want)
    assert np.array_equal(o.predict(x, edges, nodes[:0], init, lr), np.full(8, init))


@pytest.mark.parametrize("name,depth,trees", [("tiny", 3, 4), ("mid", 4, 3), ("covtype", 5, 2), ("tiny", 0, 2)])
def test_prediction_of_training_rows_equals_training_predictions(name, depth, trees, o=oracle):
    """Routing on raw values against the edges is the training's routing on bins, and the sum is
    taken in the same order: predicting the training rows reproduces the training predictions
    bit for bit (covers features with few distinct values, whose edges are the values themselves)."""
    X, y = synth.make(name, n=3000)
    cfg = dict(synth.CONFIGS[name], max_depth=depth, n_trees=trees)
    bins, edges, n_bins = o.quantize(X, cfg["max_bins"])
    r = o.train(bins, n_bins, y, want_info=False, **cfg)
    got = o.predict(X, edges, r["nodes"], r["init_pred"], cfg["learning_rate"])
    assert np.array_equal(got, r["pred"])


def test_predict_rejects_a_node_outside_the_features(o=oracle):
    edges = np.array([[0.0]], np.float32)
    nodes = np.zeros((1, 3), oracle.NODE_DTYPE)
    nodes[0, 0] = _node(5, 0, 1, 2)
    with pytest.raises(oracle.OracleError):
        o.predict(np.zeros((1, 4), np.float32), edges, nodes, 0.0, 1.0)

"""Pins of the oracle's leaf budget (the ExaBoost page's "depth-capped
final partial level"): levels split while every valid split fits the budget;
at the first level where applying all of them would exceed num_leaves, only
the top K = num_leaves - (leaves so far + the level's nodes) candidates by
(gain desc, node index asc) split, and their children are leaves.
"""
import numpy as np
import pytest

import oracle
import synth


def _levels(nodes, n):
    """BFS levels of a tree: list of lists of node indices."""
    out, cur = [], [0]
    while cur:
        out.append(cur)
        nxt = []
        for v in cur:
            if not nodes[v]["is_leaf"]:
                nxt += [nodes[v]["left"], nodes[v]["right"]]
        cur = nxt
    assert sum(map(len, out)) == n
    return out


def _expected_budget_tree(U, budget):
    """From the unbudgeted tree U: the binding level, the nodes kept there, by the rule written out."""
    levels = _levels(U, len(U))
    leaves_done = 0
    for d, lv in enumerate(levels):
        cand = [i for i, v in enumerate(lv) if not U[v]["is_leaf"]]
        K = budget - (leaves_done + len(lv))
        if len(cand) > K:
            order = sorted(cand, key=lambda i: (-U[lv[i]]["gain"], i))
            return d, set(order[:max(K, 0)])
        leaves_done += len(lv) - len(cand)
    return None, None


def _train_one(name, n, depth, budget, seed=0):
    X, y = synth.make(name, n=n, seed=seed)
    cfg = dict(synth.CONFIGS[name], max_depth=depth, n_trees=1, num_leaves=budget)
    bins, _, n_bins = oracle.quantize(X, cfg["max_bins"])
    r = oracle.train(bins, n_bins, y, want_info=False, **cfg)
    return r["nodes"][0][: r["nodes_per_tree"][0]]


@pytest.mark.parametrize("name,n,depth,budget", [("tiny", None, 3, 5), ("mid", 4000, 5, 12), ("covtype", 6000, 6, 40),
                                                 ("mid", 4000, 4, 15), ("tiny", None, 4, 2)])
def test_budget_tree_is_the_truncated_level_wise_tree(name, n, depth, budget, o=oracle):
    U = _train_one(name, n, depth, 0)
    V = _train_one(name, n, depth, budget)
    dstar, kept = _expected_budget_tree(U, budget)
    LU, LV = _levels(U, len(U)), _levels(V, len(V))
    if dstar is None:  # the budget never binds: the same tree
        assert np.array_equal(U, V)
        return
    fields = ["feature", "threshold_bin", "gain", "leaf_value", "is_leaf"]
    for d in range(dstar):
        assert len(LU[d]) == len(LV[d])
        for a, b in zip(LU[d], LV[d]):
            assert all(U[a][f] == V[b][f] for f in fields), (d, a, b)
    for i, (a, b) in enumerate(zip(LU[dstar], LV[dstar])):
        assert U[a]["leaf_value"] == V[b]["leaf_value"]
        if i in kept:
            assert all(U[a][f] == V[b][f] for f in ["feature", "threshold_bin", "gain"]) and not V[b]["is_leaf"]
        else:
            assert V[b]["is_leaf"]
    assert all(V[v]["is_leaf"] for v in (LV[dstar + 1] if len(LV) > dstar + 1 else []))
    assert len(LV) <= dstar + 2
    assert sum(int(v["is_leaf"]) for v in V) <= budget


def test_budget_at_least_the_full_tree_changes_nothing(o=oracle):
    X, y = synth.make("mid", n=3000)
    cfg = dict(synth.CONFIGS["mid"], max_depth=4, n_trees=3)
    bins, _, n_bins = o.quantize(X, cfg["max_bins"])
    a = o.train(bins, n_bins, y, want_info=False, **cfg)
    b = o.train(bins, n_bins, y, want_info=False, num_leaves=16, **cfg)
    assert np.array_equal(a["nodes"], b["nodes"]) and np.array_equal(a["pred"], b["pred"])


def test_every_tree_respects_the_budget(o=oracle):
    X, y = synth.make("covtype", n=5000)
    cfg = dict(synth.CONFIGS["covtype"], max_depth=7, n_trees=4, num_leaves=23)
    bins, _, n_bins = o.quantize(X, cfg["max_bins"])
    r = o.train(bins, n_bins, y, want_info=False, **cfg)
    for t in range(4):
        nd = r["nodes"][t][: r["nodes_per_tree"][t]]
        assert 1 <= int(nd["is_leaf"].sum()) <= 23


def test_budget_one_is_invalid(o=oracle):
    assert o.validate_params(num_leaves=1) != 0
    assert o.validate_params(num_leaves=0) == 0 and o.validate_params(num_leaves=2) == 0

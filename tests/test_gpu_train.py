"""End-to-end training parity (gbdt_train through the C ABI) against the oracle,
plus determinism and the failure contract ("Module Design: Training Core"
s.5: Failed must not export a model; s.8: repeated training is deterministic)."""
import ctypes

import numpy as np
import pytest

from tests.gpu_util import compare_training, g, needs_gpu, oracle, torch
import synth

pytestmark = [pytest.mark.gpu, needs_gpu]


def _prepare(name, n):
    X, y = synth.make(name, n=n)
    B = synth.CONFIGS[name]["max_bins"]
    bins, _, n_bins = g.quantize(torch.from_numpy(X).cuda(), B)
    ob, _, on = oracle.quantize(X, B, n_threads=8)
    assert np.array_equal(bins[:, : X.shape[1]].cpu().numpy(), ob)
    return bins, n_bins, torch.from_numpy(y).cuda(), ob, on, y


@pytest.mark.parametrize("name,n,trees", [("tiny", None, 5), ("mid", 20_011, 8), ("covtype", 30_007, 4),
                                          ("large", 40_009, 4)])
def test_training_matches_oracle(name, n, trees):
    bins, n_bins, yd, ob, on, y = _prepare(name, n)
    params = dict(synth.CONFIGS[name])
    params["n_trees"] = trees
    out = g.train(bins, n_bins, yd, **params)
    rep = {}
    compare_training(out, ob, on, y, params, rep)
    print(name, rep)


@pytest.mark.parametrize("extra", [dict(max_depth=0), dict(max_depth=1, reg_lambda=0.0),
                                   dict(min_child_weight=50.0, gamma=0.2), dict(min_samples_leaf=400),
                                   dict(max_depth=12, min_samples_leaf=1), dict(n_trees=0)])
def test_training_parameter_corners(extra):
    bins, n_bins, yd, ob, on, y = _prepare("tiny", 3_001)
    params = dict(synth.CONFIGS["tiny"], n_trees=3)
    params.update(extra)
    out = g.train(bins, n_bins, yd, **params)
    if params["n_trees"] == 0:
        assert np.allclose(out["pred"].cpu().numpy(), np.float64(y).mean(), rtol=1e-12)
        return
    compare_training(out, ob, on, y, params)


def test_constant_labels_give_single_leaf_trees():
    bins, n_bins, _, ob, on, _ = _prepare("tiny", 1000)
    y = np.full(1000, 2.5, np.float32)
    out = g.train(bins, n_bins, torch.from_numpy(y).cuda(), **dict(synth.CONFIGS["tiny"], n_trees=2))
    assert list(out["nodes_per_tree"]) == [1, 1]
    assert np.all(out["nodes"][:, 0]["is_leaf"] == 1) and np.all(out["nodes"][:, 0]["leaf_value"] == 0.0)
    assert np.all(out["pred"].cpu().numpy() == 2.5)


def test_repeated_training_is_bit_identical():
    bins, n_bins, yd, *_ = _prepare("covtype", 20_000)
    params = dict(synth.CONFIGS["covtype"], n_trees=3)
    a = g.train(bins, n_bins, yd, **params)
    b = g.train(bins, n_bins, yd, **params)
    assert a["nodes"].tobytes() == b["nodes"].tobytes()
    assert torch.equal(a["pred"], b["pred"])


@pytest.mark.parametrize("name,n,trees,extra", [("covtype", 20_000, 6, dict(num_leaves=200)),
                                                ("large", 30_000, 5, {}), ("mid", 10_000, 4, dict(objective=1))])
def test_graph_replay_equals_tree_by_tree(name, n, trees, extra):
    """Trees 1 .. T-2 replay one captured graph (T >= 4), with or without diagnostics (whose timing events
    are nodes of the graph); a run of 3 trees launches every tree on its own.  The first trees of both
    must be the same, the runs with and without diagnostics identical (model, predictions, launch counts),
    and the graph trees' histogram timings present."""
    bins, n_bins, yd, *_ = _prepare(name, n)
    y = yd
    if extra.get("objective") == 1:
        y = torch.from_numpy(synth.binary_label(yd.cpu().numpy())).cuda()
    params = dict(synth.CONFIGS[name], n_trees=trees, **extra)
    l0 = g.kernel_launch_count()
    a = g.train(bins, n_bins, y, **params)
    torch.cuda.synchronize()
    l1 = g.kernel_launch_count()
    b = g.train(bins, n_bins, y, diagnostics=True, **params)
    torch.cuda.synchronize()
    l2 = g.kernel_launch_count()
    assert a["nodes"].tobytes() == b["nodes"].tobytes()
    assert list(a["nodes_per_tree"]) == list(b["nodes_per_tree"])
    assert torch.equal(a["pred"], b["pred"]) and a["init_pred"] == b["init_pred"]
    assert l1 - l0 == l2 - l1  # the replayed graph's kernels are counted as launches
    D = params["max_depth"]
    assert b["diag"]["hist_launches"] == trees * D and b["diag"]["hist_ms"] > 0
    c = g.train(bins, n_bins, y, **dict(params, n_trees=3))  # tree by tree
    assert a["nodes"][:3].tobytes() == c["nodes"].tobytes()
    assert list(a["nodes_per_tree"][:3]) == list(c["nodes_per_tree"])


def _raw_train(bins, n_bins, label, params, nodes, npt):
    L = g.lib()
    p = g.make_params(**params)
    N = label.shape[0]
    ws = torch.empty(L.gbdt_train_workspace_size(N, bins.shape[0], ctypes.byref(p)), dtype=torch.uint8,
                     device="cuda")
    pred = torch.empty(N, dtype=torch.float64, device="cuda")
    init = ctypes.c_double(0)
    return L.gbdt_train(ctypes.c_void_p(bins.data_ptr()), bins.shape[1], ctypes.c_void_p(n_bins.data_ptr()), N,
                        bins.shape[0], ctypes.c_void_p(label.data_ptr()), ctypes.byref(p),
                        ctypes.c_void_p(pred.data_ptr()), ctypes.byref(init), nodes.ctypes.data_as(ctypes.c_void_p),
                        npt.ctypes.data_as(ctypes.c_void_p), None, ctypes.c_void_p(ws.data_ptr()), ws.numel(),
                        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_failures_leave_no_partial_model():
    bins, n_bins, yd, *_ = _prepare("tiny", 2000)
    params = dict(synth.CONFIGS["tiny"])
    M = (1 << (params["max_depth"] + 1)) - 1
    sentinel = np.full((params["n_trees"], M), 0, g.NODE_DTYPE)
    sentinel["feature"] = 777
    # non-finite label
    bad = yd.clone()
    bad[1234] = float("nan")
    nodes, npt = sentinel.copy(), np.full(params["n_trees"], 9, np.int32)
    assert _raw_train(bins, n_bins, bad, params, nodes, npt) == g.ERR_NONFINITE
    assert np.all(nodes["feature"] == 777) and np.all(npt == 0)
    # failure injected on the host after 7 levels (inside tree 2)
    g.inject_failure(7)
    try:
        nodes, npt = sentinel.copy(), np.full(params["n_trees"], 9, np.int32)
        assert _raw_train(bins, n_bins, yd, params, nodes, npt) == g.ERR_INTERNAL
        assert np.all(nodes["feature"] == 777) and np.all(npt == 0)
        assert b"injected" in g.lib().gbdt_last_error()
    finally:
        g.inject_failure(-1)
    # the library still trains normally afterwards
    nodes, npt = sentinel.copy(), np.zeros(params["n_trees"], np.int32)
    assert _raw_train(bins, n_bins, yd, params, nodes, npt) == g.OK and np.all(npt >= 1)
    # n_bins out of range and invalid parameters are rejected
    with pytest.raises(g.GbdtError) as e:
        g.train(bins, torch.full_like(n_bins, 300), yd, **params)
    assert e.value.code == g.ERR_INVALID_ARG
    with pytest.raises(g.GbdtError) as e:
        g.train(bins, n_bins, yd, **dict(params, min_samples_leaf=0))
    assert e.value.code == g.ERR_INVALID_ARG
    with pytest.raises(g.GbdtError) as e:
        g.train(bins, n_bins, yd, ws=torch.empty(1024, dtype=torch.uint8, device="cuda"), **params)
    assert e.value.code == g.ERR_WORKSPACE


def test_diagnostics_report_histogram_work():
    bins, n_bins, yd, *_ = _prepare("mid", 50_000)
    params = dict(synth.CONFIGS["mid"], n_trees=3)
    out = g.train(bins, n_bins, yd, diagnostics=True, **params)
    d = out["diag"]
    assert d["hist_launches"] == 3 * params["max_depth"]
    assert d["hist_ms"] > 0 and d["total_ms"] >= d["hist_ms"]
    assert d["hist_rows"] <= 3 * params["max_depth"] * 50_000 and d["hist_rows"] >= 3 * 50_000
    assert d["hist_bytes"] >= d["hist_rows"] * (28 + 10)
    # the level formula counts every row of a level's nodes (every row at the root) once per level
    assert d["hist_level_bytes"] >= 3 * 50_000 * (28 + 10) and d["hist_level_bytes"] >= d["hist_bytes"]


@pytest.mark.parametrize("name,n,depth,budget,trees", [("covtype", 30_011, 10, 1023, 3), ("mid", 20_011, 6, 20, 3),
                                                       ("tiny", 3_001, 4, 2, 2), ("large", 40_009, 8, 100, 2)])
def test_leaf_budget_matches_oracle(name, n, depth, budget, trees):
    """Leaf budget: levels split while all their valid splits fit num_leaves; the level where they would not
    keeps its top candidates by (gain desc, node index asc) and is the last to split."""
    bins, n_bins, yd, ob, on, y = _prepare(name, n)
    params = dict(synth.CONFIGS[name], n_trees=trees, max_depth=depth, num_leaves=budget)
    out = g.train(bins, n_bins, yd, **params)
    for t in range(trees):
        nd = out["nodes"][t][: out["nodes_per_tree"][t]]
        assert 1 <= int(nd["is_leaf"].sum()) <= budget
    compare_training(out, ob, on, y, params)


def test_leaf_budget_of_one_is_rejected():
    assert g.validate_params(num_leaves=1) == g.ERR_INVALID_ARG
    assert g.validate_params(num_leaves=0) == g.OK and g.validate_params(num_leaves=2) == g.OK


def _mixed_cardinality(n, seed=5):
    """Columns with 2..17 distinct values in an irregular order among continuous ones."""
    rng = np.random.default_rng(seed)
    ks = [2, 3, 300, 16, 17, 5, 2, 256, 9, 16, 4, 1000, 2, 7, 15, 3, 2, 40, 11]
    X = np.empty((len(ks), n), np.float32)
    for j, k in enumerate(ks):
        X[j] = rng.integers(0, k, n) if k <= 300 else rng.standard_normal(n)
    y = (X[0] * 2 - X[3] * 0.3 + np.sin(X[11]) + 0.5 * (X[9] > 7) + rng.normal(0, 0.3, n)).astype(np.float32)
    return X, y


@pytest.mark.parametrize("case", ["covtype", "large", "mixed", "mixed_logistic"])
def test_4bit_slots_give_identical_training(case):
    """Features with <= 16 bins stored two per byte in the training copies: the same model, bit for
    bit, as one byte per feature, with fewer bytes read; and the oracle's model."""
    if case in ("covtype", "large"):
        bins, n_bins, yd, ob, on, y = _prepare(case, 30_011)
        params = dict(synth.CONFIGS[case], n_trees=3)
    else:
        X, y = _mixed_cardinality(25_013)
        if case == "mixed_logistic":
            y = synth.binary_label(y)
        bins, _, n_bins = g.quantize(torch.from_numpy(X).cuda(), 255)
        ob, _, on = oracle.quantize(X, 255)
        yd = torch.from_numpy(y).cuda()
        params = dict(n_trees=4, max_depth=7, learning_rate=0.2, reg_lambda=1.0, gamma=0.0, min_samples_leaf=3,
                      min_child_weight=0.0, objective=1 if case == "mixed_logistic" else 0)
    assert int((n_bins <= 16).sum()) >= 2
    a = g.train(bins, n_bins, yd, diagnostics=True, bin_packing=g.BIN_PACKING_4BIT, **params)
    b = g.train(bins, n_bins, yd, diagnostics=True, bin_packing=g.BIN_PACKING_OFF, **params)
    assert a["nodes"].tobytes() == b["nodes"].tobytes()
    assert torch.equal(a["pred"], b["pred"])
    assert a["diag"]["hist_bytes"] < b["diag"]["hist_bytes"] and a["diag"]["part_bytes"] < b["diag"]["part_bytes"]
    compare_training(a, ob, on, y, params)


def test_bins_beyond_n_bins_are_rejected():
    bins, n_bins, yd, *_ = _prepare("large", 5_003)
    nb = n_bins.cpu().numpy()
    for f in (int(np.argmax(nb <= 16)), 0):  # a 4-bit feature and a whole-byte one
        bad = n_bins.clone()
        bad[f] -= 1
        with pytest.raises(g.GbdtError) as e:
            g.train(bins, bad, yd, **dict(synth.CONFIGS["large"], n_trees=1, max_depth=3))
        assert e.value.code == g.ERR_INVALID_ARG and "n_bins" in str(e.value)


@pytest.mark.parametrize("case,packing,budget", [("covtype", 0, 0), ("covtype", 0, 1023), ("large", 0, 0),
                                                 ("mixed", 0, 0), ("mixed", 1, 0), ("mixed_logistic", 0, 0)])
def test_register_histograms_give_identical_training(case, packing, budget):
    """Features with at most 8 bins (two per slot when their bin counts multiply to at most 8) accumulated
    per code in registers: the same model, bit for bit, as with shared-memory atomics, across filtered
    levels, the root's reused counts (second and later trees), 4- and 8-code slots and the leaf budget;
    with the logistic objective the option changes nothing."""
    if case in ("covtype", "large"):
        bins, n_bins, yd, ob, on, y = _prepare(case, 30_011)
        params = dict(synth.CONFIGS[case], n_trees=3)
        if budget:
            params.update(num_leaves=budget)
    else:
        X, y = _mixed_cardinality(25_013)
        if case == "mixed_logistic":
            y = synth.binary_label(y)
        bins, _, n_bins = g.quantize(torch.from_numpy(X).cuda(), 255)
        ob, _, on = oracle.quantize(X, 255)
        yd = torch.from_numpy(y).cuda()
        params = dict(n_trees=4, max_depth=7, learning_rate=0.2, reg_lambda=1.0, gamma=0.0, min_samples_leaf=3,
                      min_child_weight=0.0, objective=1 if case == "mixed_logistic" else 0)
    assert int((n_bins <= 8).sum()) >= 2
    a = g.train(bins, n_bins, yd, hist_registers=g.HIST_REGISTERS_ON, bin_packing=packing, **params)
    b = g.train(bins, n_bins, yd, hist_registers=g.HIST_REGISTERS_OFF, bin_packing=packing, **params)
    assert a["nodes"].tobytes() == b["nodes"].tobytes()
    assert torch.equal(a["pred"], b["pred"])
    if case != "mixed_logistic":
        compare_training(a, ob, on, y, params)

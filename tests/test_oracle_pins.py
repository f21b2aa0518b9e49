"""Pins for the CPU oracle that do not call it back.

* Split search: brute force over every (feature, threshold) with a direct
  two-sided recount of the rows and exact rational arithmetic (no prefix
  sums, no floating point), compared under the frozen rule of "Module
  Design: Training Core" s.3.
* Gain / weight closed forms: with lambda = gamma = 0 the gain equals half the
  drop in the sum of squared errors of the residuals and the leaf weight is
  the mean residual, so a depth-1 tree with learning rate 1 from the mean is
  the exact greedy CART stump of "Gradient boosted trees (spec model)"
  (classical training, SSE), written here independently on raw feature values.
* Histograms: bincount per (slot, feature); counts exact, G within rounding.
* Quantize: ranks of distinct values, balanced-count closed form, order
  statistics, monotonicity.
* Training invariants: child counts add up, depth limit, BFS layout,
  determinism, and predictions equal init + lr * sum of tree outputs by
  an independent traversal ("Gradient boosted trees (spec model)", forward pass).
"""
from fractions import Fraction

import numpy as np
import pytest

import synth


# ----------------------------------------------------------------------------- split search
def _brute_best(bins, n_bins, g, lam, gamma, msl, mcw):
    """Exact best split at one node by enumeration; returns (f, b, gain) or None."""
    F, N = bins.shape
    gq = [Fraction(float(v)) for v in g]
    lam, gamma, mcw = Fraction(lam), Fraction(gamma), Fraction(mcw)
    GP, HP = sum(gq), Fraction(N)
    best = None
    for f in range(F):
        for b in range(int(n_bins[f]) - 1):
            left = [i for i in range(N) if bins[f, i] <= b]
            right = [i for i in range(N) if bins[f, i] > b]
            GL, HL = sum((gq[i] for i in left), Fraction(0)), Fraction(len(left))
            GR, HR = sum((gq[i] for i in right), Fraction(0)), Fraction(len(right))
            if not (len(left) >= msl and len(right) >= msl and HL >= mcw and HR >= mcw and HL > 0 and HR > 0):
                continue
            gain = Fraction(1, 2) * (GL * GL / (HL + lam) + GR * GR / (HR + lam) - GP * GP / (HP + lam)) - gamma
            if best is None or gain > best[2]:
                best = (f, b, gain)
    return best


@pytest.mark.parametrize("seed", range(12))
def test_root_split_matches_brute_force(orc, seed):
    rng = np.random.default_rng(100 + seed)
    F, N = int(rng.integers(1, 5)), int(rng.integers(5, 60))
    n_bins = rng.integers(1, 9, F).astype(np.int32)
    bins = np.stack([rng.integers(0, nb, N) for nb in n_bins]).astype(np.uint8)
    y = rng.normal(0, 1, N).astype(np.float32)
    lam = float(rng.choice([0.0, 0.5, 1.0, 3.0]))
    gamma = float(rng.choice([0.0, 0.0, 0.05]))
    msl = int(rng.choice([1, 1, 2, 4]))
    mcw = float(rng.choice([0.0, 0.0, 2.0]))
    out = orc.train(bins, n_bins, y, n_trees=1, max_depth=1, learning_rate=1.0, reg_lambda=lam, gamma=gamma,
                    min_samples_leaf=msl, min_child_weight=mcw)
    g = np.full(N, out["init_pred"]) - y.astype(np.float64)
    best = _brute_best(bins, n_bins, g, lam, gamma, msl, mcw)
    root = out["nodes"][0][0]
    info = out["info"][0][0]
    if best is None or best[2] <= 0:
        assert root["is_leaf"] == 1
        return
    if info["n_near"] > 1:  # floating point may order exactly-tied rationals either way
        assert (root["feature"], root["threshold_bin"]) in set(
            zip(info["near_feature"][: info["n_near"]], info["near_bin"][: info["n_near"]])) | {best[:2]}
        return
    assert (root["feature"], root["threshold_bin"]) == best[:2]
    assert root["gain"] == pytest.approx(float(best[2]), rel=1e-10, abs=1e-12)


def test_best_split_function_brute_force(orc):
    # orc_best_split on oracle-made histograms vs enumeration, many random nodes.
    rng = np.random.default_rng(7)
    for _ in range(25):
        F, N = 3, int(rng.integers(4, 40))
        n_bins = rng.integers(2, 7, F).astype(np.int32)
        bins = np.stack([rng.integers(0, nb, N) for nb in n_bins]).astype(np.uint8)
        g = np.round(rng.normal(0, 1, N), 3)
        h = orc.histograms(bins, g, np.zeros(N, np.int32), 1)
        s = orc.best_split(h["cnt"][0], h["G"][0], h["H"][0], n_bins, N, h["Gt"][0], h["Ht"][0], reg_lambda=1.0)
        best = _brute_best(bins, n_bins, g, 1.0, 0.0, 1, 0.0)
        if best is None:
            assert s.valid == 0
            continue
        assert s.valid == 1
        if s.n_near <= 1:
            assert (s.feature, s.bin) == best[:2]
        assert s.gain == pytest.approx(float(best[2]), rel=1e-9, abs=1e-12)


# ----------------------------------------------------------------------------- CART special case
def _cart_stump_pred(X, y):
    """Exact-greedy CART stump on raw values: thresholds are observed values, x > t goes
    right, minimise SSE_L + SSE_R, first best in (feature, threshold) ascending order;
    leaves predict the mean target."""
    F, N = X.shape
    best = None
    for f in range(F):
        for t in np.unique(X[f])[:-1]:
            right = X[f] > t
            yl, yr = y[~right], y[right]
            sse = ((yl - yl.mean()) ** 2).sum() + ((yr - yr.mean()) ** 2).sum()
            if best is None or sse < best[0] - 1e-9 * max(1.0, abs(best[0])):
                best = (sse, f, t)
    sse, f, t = best
    right = X[f] > t
    return np.where(right, y[right].mean(), y[~right].mean()), f


@pytest.mark.parametrize("seed", range(5))
def test_depth1_tree_is_cart_stump(orc, seed):
    rng = np.random.default_rng(200 + seed)
    F, N = 3, 80
    X = rng.integers(0, 12, (F, N)).astype(np.float32)  # <= 12 distinct values per feature: bins = ranks
    y = (2.0 * X[0] - X[1] + rng.normal(0, 0.5, N)).astype(np.float32)
    bins, _, n_bins = orc.quantize(X, 32)
    out = orc.train(bins, n_bins, y, n_trees=1, max_depth=1, learning_rate=1.0, reg_lambda=0.0, gamma=0.0)
    cart_pred, cart_f = _cart_stump_pred(X.astype(np.float64), y.astype(np.float64))
    np.testing.assert_allclose(out["pred"], cart_pred, rtol=0, atol=1e-9)
    root = out["nodes"][0][0]
    assert root["feature"] == cart_f
    # gain = 0.5 (SSE_P - SSE_L - SSE_R) of the residuals
    r = y.astype(np.float64) - out["init_pred"]
    left = bins[root["feature"]] <= root["threshold_bin"]
    sse = lambda v: ((v - v.mean()) ** 2).sum()
    assert root["gain"] == pytest.approx(0.5 * (sse(r) - sse(r[left]) - sse(r[~left])), rel=1e-9)
    # leaf weights are the mean residual of each side
    t = out["nodes"][0]
    assert t[root["left"]]["leaf_value"] == pytest.approx(r[left].mean(), rel=1e-12, abs=1e-12)
    assert t[root["right"]]["leaf_value"] == pytest.approx(r[~left].mean(), rel=1e-12, abs=1e-12)


def test_closed_forms(orc):
    # weight(G,H) = -G/(H+lambda); gain = 0.5 (G_L^2/(H_L+l) + G_R^2/(H_R+l) - G_P^2/(H_P+l)) - gamma
    assert orc.weight(3.0, 2.0, 1.0) == -1.0
    assert orc.weight(-6.0, 1.0, 0.5) == 4.0
    assert orc.gain(2.0, 1.0, -2.0, 3.0, 0.0, 4.0, 0.0, 0.0) == pytest.approx(8.0 / 3.0, rel=1e-15)
    assert orc.gain(3.0, 2.0, 1.0, 1.0, 4.0, 3.0, 1.0, 0.25) == pytest.approx(0.5 * (3 + 0.5 - 4) - 0.25, rel=1e-15)
    # symmetry of left/right
    assert orc.gain(1.5, 2.0, -0.5, 5.0, 1.0, 7.0, 2.0, 0.0) == orc.gain(-0.5, 5.0, 1.5, 2.0, 1.0, 7.0, 2.0, 0.0)


# ----------------------------------------------------------------------------- histograms
def test_histograms_brute_force(orc):
    rng = np.random.default_rng(11)
    F, N, S = 4, 3000, 5
    bins = rng.integers(0, 256, (F, N)).astype(np.uint8)
    bins[1] = rng.integers(0, 3, N)  # low-cardinality column
    g = rng.normal(0, 2, N)
    slot = rng.integers(-1, S + 1, N).astype(np.int32)  # -1 and S are inactive
    h = orc.histograms(bins, g, slot, S)
    for s in range(S):
        m = slot == s
        assert h["n"][s] == m.sum()
        assert h["Gt"][s] == pytest.approx(g[m].sum(), rel=1e-12, abs=1e-12)
        assert h["At"][s] == pytest.approx(np.abs(g[m]).sum(), rel=1e-12)
        for f in range(F):
            cnt = np.bincount(bins[f][m], minlength=256)
            np.testing.assert_array_equal(h["cnt"][s, f], cnt)
            np.testing.assert_array_equal(h["H"][s, f], cnt.astype(np.float64))
            Gb = np.bincount(bins[f][m], weights=g[m], minlength=256)
            Ab = np.bincount(bins[f][m], weights=np.abs(g[m]), minlength=256)
            assert np.all(np.abs(h["G"][s, f] - Gb) <= 1e-12 * (Ab + 1e-300))
            assert h["cnt"][s, f].sum() == m.sum()


def test_histogram_row_order_accumulation(orc):
    # "accumulates each bin's count/G/H in supplied row-index order": a sum
    # whose value depends on order is reproduced exactly by a left fold.
    g = np.array([1e16, 1.0, -1e16, 1.0], np.float64)
    bins = np.zeros((1, 4), np.uint8)
    h = orc.histograms(bins, g, np.zeros(4, np.int32), 1)
    acc = 0.0
    for v in g:
        acc = acc + v
    assert h["G"][0, 0, 0] == acc == 1.0


# ----------------------------------------------------------------------------- quantize
def test_quantize_few_distinct_values_are_ranks(orc):
    rng = np.random.default_rng(5)
    X = rng.choice(np.array([-3.5, -0.0, 0.0, 1.25, 7.0, 9.5], np.float32), (3, 500))
    bins, edges, n_bins = orc.quantize(X, 32)
    for f in range(3):
        canon = np.where(X[f] == 0, np.float32(0), X[f])
        u, inv = np.unique(canon, return_inverse=True)
        np.testing.assert_array_equal(bins[f], inv)
        assert n_bins[f] == len(u)
        np.testing.assert_array_equal(edges[f][: len(u) - 1], u[:-1])
        assert np.all(np.isinf(edges[f][len(u) - 1:]))
    # -0.0 and +0.0 share a bin
    z = (X == 0)
    assert len(np.unique(bins[z])) <= 3


@pytest.mark.parametrize("N,B", [(1000, 32), (1001, 255), (255, 255), (300, 2), (4097, 256)])
def test_quantize_all_distinct_balanced(orc, N, B):
    rng = np.random.default_rng(N + B)
    X = rng.permutation(np.arange(N, dtype=np.float32) * 0.5 - 17.0)[None, :]
    bins, edges, n_bins = orc.quantize(X, B)
    if N <= B:
        assert n_bins[0] == N
        return
    assert n_bins[0] == B
    cnt = np.bincount(bins[0], minlength=B)
    b = np.arange(B)
    expect = (-(-(b + 1) * N // B)) - (-(-b * N // B))  # ceil((b+1)N/B) - ceil(bN/B)
    np.testing.assert_array_equal(cnt, expect)


def test_quantize_order_statistics_and_monotone(orc):
    X, _ = synth.make_large(n=20_000)
    X = X[[0, 55, 81, 95]]  # normal, lognormal, 3-valued and 2..16-valued integer columns
    bins, edges, n_bins = orc.quantize(X, 255)
    for f in range(X.shape[0]):
        x = X[f].astype(np.float64)
        order = np.argsort(x, kind="stable")
        assert np.all(np.diff(bins[f][order].astype(int)) >= 0)  # monotone
        e = edges[f][: n_bins[f] - 1].astype(np.float64)
        assert np.all(np.diff(e) > 0) and (len(e) == 0 or e[-1] < x.max())
        assert set(e).issubset(set(x))  # edges are observed values
        np.testing.assert_array_equal(bins[f], (x[None, :] > e[:, None]).sum(0))
        N, B = x.size, 255
        if len(np.unique(x)) > B:
            v = np.sort(x)
            pk = np.array([-(-k * N // B) - 1 for k in range(1, B)])
            lt, le = np.searchsorted(v, e, "left"), np.searchsorted(v, e, "right")
            # every edge is a k/B quantile: #{x < e} <= p_k < #{x <= e} for some k
            assert all(np.any((lt[i] <= pk) & (pk < le[i])) for i in range(len(e)))
            # every k/B quantile below the maximum is an edge
            assert set(v[pk][v[pk] < v[-1]]) == set(e)


def test_quantize_constant_and_nonfinite(orc):
    bins, edges, n_bins = orc.quantize(np.full((1, 10), 3.0, np.float32), 16)
    assert n_bins[0] == 1 and np.all(bins == 0) and np.all(np.isinf(edges))
    with pytest.raises(orc.OracleError):
        orc.quantize(np.array([[0.0, np.inf]], np.float32), 16)


# ----------------------------------------------------------------------------- training invariants
def _traverse(nodes, n, bins):
    v = np.zeros(bins.shape[1], np.int64)
    for _ in range(64):
        nd = nodes[v]
        internal = nd["is_leaf"] == 0
        if not internal.any():
            break
        go_right = bins[np.where(internal, nd["feature"], 0), np.arange(bins.shape[1])] > nd["threshold_bin"]
        v = np.where(internal, np.where(go_right, nd["right"], nd["left"]), v)
    return v


@pytest.mark.parametrize("name,n,trees", [("tiny", None, 5), ("mid", 3000, 6), ("covtype", 4000, 3)])
def test_training_invariants(orc, name, n, trees):
    X, y = synth.make(name, n=n)
    cfg = dict(synth.CONFIGS[name])
    cfg["n_trees"] = trees
    bins, _, n_bins = orc.quantize(X, cfg["max_bins"])
    out = orc.train(bins, n_bins, y, **cfg)
    again = orc.train(bins, n_bins, y, **dict(cfg, n_threads=4))
    np.testing.assert_array_equal(out["pred"], again["pred"])  # deterministic, thread-count independent
    assert out["nodes"].tobytes() == again["nodes"].tobytes()
    D, lr = cfg["max_depth"], cfg["learning_rate"]
    recon = np.full(bins.shape[1], out["init_pred"])
    for t in range(trees):
        n_t = out["nodes_per_tree"][t]
        nodes, info = out["nodes"][t][:n_t], out["info"][t][:n_t]
        assert info[0]["n_rows"] == bins.shape[1]
        for i, nd in enumerate(nodes):
            assert nd["depth"] <= D
            if nd["is_leaf"]:
                assert nd["feature"] == -1 and nd["left"] == -1
                continue
            L, R = nd["left"], nd["right"]
            assert i < L and R == L + 1 < n_t  # BFS: children appended left then right
            assert info[L]["n_rows"] + info[R]["n_rows"] == info[i]["n_rows"]
            assert nodes[L]["depth"] == nd["depth"] + 1
            assert nd["gain"] > 0
            assert min(info[L]["n_rows"], info[R]["n_rows"]) >= cfg["min_samples_leaf"]
        # BFS order: depths never decrease along the array
        assert np.all(np.diff(nodes["depth"]) >= 0)
        leaf = _traverse(nodes, n_t, bins)
        recon = recon + lr * nodes["leaf_value"][leaf]
    np.testing.assert_allclose(out["pred"], recon, rtol=1e-12, atol=1e-12)


def test_leaf_values_are_node_weights(orc):
    X, y = synth.make_tiny(n=500)
    bins, _, n_bins = orc.quantize(X, 32)
    out = orc.train(bins, n_bins, y, n_trees=2, max_depth=3, learning_rate=0.3, reg_lambda=1.0)
    for t in range(2):
        n_t = out["nodes_per_tree"][t]
        nodes, info = out["nodes"][t][:n_t], out["info"][t][:n_t]
        np.testing.assert_allclose(nodes["leaf_value"], -info["G"] / (info["H"] + 1.0), rtol=1e-15)
        np.testing.assert_array_equal(info["H"], info["n_rows"].astype(np.float64))


def test_partition_is_stable_and_routes_by_threshold(orc):
    rng = np.random.default_rng(9)
    F, N = 3, 200
    bins = rng.integers(0, 10, (F, N)).astype(np.uint8)
    idx = rng.permutation(N).astype(np.int64)
    seg_start, seg_count = np.array([0, 50, 120]), np.array([50, 70, 80])
    idx[0:50].sort(), idx[50:120].sort(), idx[120:].sort()
    sf, sb = np.array([2, -1, 0]), np.array([4, -1, 7])
    out, lc = orc.partition(bins, sf, sb, seg_start, seg_count, idx)
    np.testing.assert_array_equal(out[50:120], idx[50:120])
    for s in (0, 2):
        seg = idx[seg_start[s]: seg_start[s] + seg_count[s]]
        o = out[seg_start[s]: seg_start[s] + seg_count[s]]
        left = seg[bins[sf[s], seg] <= sb[s]]
        right = seg[bins[sf[s], seg] > sb[s]]
        np.testing.assert_array_equal(o, np.concatenate([left, right]))
        assert lc[s] == len(left)

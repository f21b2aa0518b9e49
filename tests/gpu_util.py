"""Helpers for the GPU parity tests: device marshalling and the stated tolerances.

Tolerances (also in the design notes):
  * bins, counts, row partitions, tree structure: bit-exact;
  * a histogram entry's G: |G_gpu - G_orc| <= 1e-9 * A + n * 2^-(S+1), where A is
    sum |g| over the entry's rows and the second term is the documented rounding
    bound of the library's fixed point (q = round(g * 2^S) per row);
  * leaf values: the node's G bound divided by (H + lambda);
  * logistic objective: an H entry's |H_gpu - H_orc| <= 1e-9 * H + n * (2^-(S_h+1) + 2^-53),
    the rounding bound of H's own fixed point plus the rounding of g = p - 1 from which the
    library recovers h; a leaf value's bound is (G bound + |w| * H bound) / (H + lambda);
  * predictions: 1e-6 * max(|p_orc|, std(label)).
"""
import json
import math
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import histogram_gradient_boosted_gb300 as g  # noqa: E402
import oracle  # noqa: E402

needs_gpu = pytest.mark.skipif(not torch.cuda.is_available(), reason="needs a CUDA GPU")


def fixed_exponent(maxabs: float, n: int) -> int:
    """Exponent S of the library's fixed point, from its documented definition:
    S = 62 - ceil(log2 N) - E with max|g| < 2^E (0 if all g are 0)."""
    if not maxabs > 0:
        return 0
    _, E = math.frexp(maxabs)
    L = 0
    while (1 << L) < n:
        L += 1
    return max(-1000, min(1000, 62 - L - E))


def dev_bins(bins: np.ndarray):
    F, N = bins.shape
    t = torch.zeros((F, g.padded_ld(N)), dtype=torch.uint8)
    t[:, :N] = torch.from_numpy(np.ascontiguousarray(bins))
    return t.cuda()


def dev_struct(arr: np.ndarray, dtype):
    return g._dev(arr, dtype)


def host_struct(t, dtype, count):
    return np.frombuffer(t.cpu().numpy().tobytes(), dtype=dtype, count=count)


def level(node_begin: int, n_slots: int):
    return dev_struct(np.array([(node_begin, n_slots)], g.LEVEL_DTYPE), g.LEVEL_DTYPE)


def u16(a: np.ndarray):
    """uint16 node ids as a CUDA tensor (int16 storage with the same bits), 16-byte aligned."""
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint16).view(np.int16)).cuda()


def g_tolerance(A, n, S):
    return 1e-9 * np.asarray(A) + np.asarray(n, dtype=np.float64) * 2.0 ** (-(S + 1)) * (1 + 1e-12) + 1e-300


def h_tolerance(H, n, S_h):
    n = np.asarray(n, dtype=np.float64)
    return 1e-9 * np.asarray(H) + n * (2.0 ** (-(S_h + 1)) + 2.0 ** -53) * (1 + 1e-12) + 1e-300


def traverse(nodes, bins):
    v = np.zeros(bins.shape[1], np.int64)
    for _ in range(64):
        nd = nodes[v]
        internal = nd["is_leaf"] == 0
        if not internal.any():
            break
        go_right = bins[np.where(internal, nd["feature"], 0), np.arange(bins.shape[1])] > nd["threshold_bin"]
        v = np.where(internal, np.where(go_right, nd["right"], nd["left"]), v)
    return v


def compare_training(gpu, bins, n_bins, y, params, report=None):
    """Tree-by-tree lockstep comparison of a GPU model with the oracle.

    Tree t is compared with the oracle's tree grown from the GPU's own predictions before tree t (rebuilt
    here bit for bit from the GPU's trees: init + (lr * leaf value) tree by tree, the product rounded
    first), so both programs see the same gradients and only their summation differs.  The oracle takes
    the GPU's (feature, bin) at a node only where the two are tied: oracle gains within 1e-12 relative
    (kind 1, the benchmark spec's near-ties), or within the proven bound by which the gains of the same rows
    can move when the GPU sums them in its fixed point, whose per-row rounding is 2^-(S+1) for G (kind 2,
    reported separately).  Everything else must match: structure exactly, leaf values within the G
    tolerance, gains within 1e-6 relative; the GPU's final predictions must equal the rebuilt ones bit for
    bit and agree with the oracle's leaf values summed along the same trees within 1e-6 relative."""
    T, D = params["n_trees"], params["max_depth"]
    M = (1 << (D + 1)) - 1
    N = bins.shape[1]
    lam, lr = params["reg_lambda"], params["learning_rate"]
    logistic = params.get("objective", 0) == 1
    one = dict(params, n_trees=1)
    pred_g = np.full(N, gpu["init_pred"])  # the GPU's predictions before the current tree
    pred_o = None                          # the oracle's leaf values summed along the same trees
    adopted = {1: 0, 2: 0}
    near = 0
    max_gap_over_bound = 0.0
    for t in range(T):
        gt, ht = oracle.gradients(pred_g, y, 1 if logistic else 0)
        S = fixed_exponent(float(np.abs(gt).max()), N)
        qg, qh = 2.0 ** -(S + 1), 0.0
        if logistic:  # sigmoid rounding on either side; H's own fixed point with S_h taken one lower (as the
            qg += 2.0 ** -50  # H tolerance below), whose half quantum is 2^-S_h, and h recovered from g (2^-53)
            qh = 2.0 ** -fixed_exponent(float(ht.max()), N) + 2.0 ** -53
        guide = np.full((1, M, 2), -1, np.int32)
        n = gpu["nodes_per_tree"][t]
        guide[0, :n, 0] = gpu["nodes"][t][:n]["feature"]
        guide[0, :n, 1] = gpu["nodes"][t][:n]["threshold_bin"]
        ref = oracle.train(bins, n_bins, y, guide=guide, tie_quanta=np.array([[qg, qh]]), pred_in=pred_g, **one)
        if t == 0:
            assert gpu["init_pred"] == pytest.approx(ref["init_pred"], rel=1e-12)
            pred_o = np.full(N, ref["init_pred"])
        n = ref["nodes_per_tree"][0]
        info = ref["info"][0][:n]
        bad = np.nonzero(info["guide_mismatch"])[0]
        if len(bad):
            i = bad[0]
            on = ref["nodes"][0][i]
            gn = gpu["nodes"][t][i] if i < gpu["nodes_per_tree"][t] else None
            raise AssertionError(
                f"tree {t} node {i}: GPU chose "
                f"({gn['feature'] if gn is not None else '-'},{gn['threshold_bin'] if gn is not None else '-'}) "
                f"gain {gn['gain'] if gn is not None else None!r}, oracle ({on['feature']},{on['threshold_bin']}) "
                f"gain {on['gain']!r}, second {info[i]['second_gain']!r}, gap {info[i]['guide_gap']!r}, "
                f"bound {info[i]['guide_bound']!r}")
        assert gpu["nodes_per_tree"][t] == n, f"tree {t}: {gpu['nodes_per_tree'][t]} nodes vs oracle {n}"
        a, b = gpu["nodes"][t][:n], ref["nodes"][0][:n]
        for k in ("feature", "threshold_bin", "left", "right", "is_leaf"):
            assert np.array_equal(a[k].astype(np.int64), b[k].astype(np.int64)), f"tree {t}: {k} differs"
        for kind in (1, 2):
            adopted[kind] += int((info["adopted"] == kind).sum())
        ad = info["adopted"] > 0
        if ad.any():
            max_gap_over_bound = max(max_gap_over_bound, float(np.max(np.where(
                info["guide_bound"][ad] > 0, info["guide_gap"][ad] / np.maximum(info["guide_bound"][ad], 1e-300),
                0.0))))
        near += int((info["n_near"] > 1).sum())
        tol = g_tolerance(info["A"], info["n_rows"], S) / (info["H"] + lam)
        if logistic:  # S_h one lower: the library's max h may sit an ulp across a power of two
            th = h_tolerance(info["H"], info["n_rows"], fixed_exponent(float(ht.max()), N) - 1)
            tol = (g_tolerance(info["A"], info["n_rows"], S) + np.abs(b["leaf_value"]) * th) / np.maximum(
                info["H"] + lam - th, 1e-300)
        err = np.abs(a["leaf_value"] - b["leaf_value"])
        assert np.all(err <= tol), f"tree {t}: leaf value off by {err.max()} (tol {tol[err.argmax()]})"
        internal = b["is_leaf"] == 0
        np.testing.assert_allclose(a["gain"][internal], b["gain"][internal], rtol=1e-6, atol=1e-9)
        leaf = traverse(a, bins)
        pred_g = pred_g + lr * a["leaf_value"][leaf]
        pred_o = pred_o + lr * b["leaf_value"][leaf]
    p_gpu = gpu["pred"].cpu().numpy()
    if T > 0:
        assert np.array_equal(p_gpu, pred_g), "GPU predictions differ from init + sum of (lr * its leaf values)"
        scale = np.maximum(np.abs(pred_o), float(np.std(y)))
        assert np.all(np.abs(p_gpu - pred_o) <= 1e-6 * scale), "predictions differ beyond 1e-6 relative"
    if report is not None:
        report.update(trees=T, near_ties=near, adopted_near_tie=adopted[1], adopted_within_rounding=adopted[2],
                      max_adopted_gap_over_bound=max_gap_over_bound)
    return dict(pred=pred_o)


def record_parity(config: str, **fields):
    """Print a parity record (near-tie counts and the like) and, when GBDT_PARITY_RECORD names a file,
    append it there as one JSON line."""
    rec = dict(config=config, **fields)
    print("parity record:", json.dumps(rec))
    path = os.environ.get("GBDT_PARITY_RECORD")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")

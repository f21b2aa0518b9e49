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
    """Lockstep comparison of a GPU model with the oracle (near-tie rule in the design notes)."""
    T, D = params["n_trees"], params["max_depth"]
    M = (1 << (D + 1)) - 1
    guide = np.full((T, M, 2), -1, np.int32)
    for t in range(T):
        n = gpu["nodes_per_tree"][t]
        guide[t, :n, 0] = gpu["nodes"][t][:n]["feature"]
        guide[t, :n, 1] = gpu["nodes"][t][:n]["threshold_bin"]
    ref = oracle.train(bins, n_bins, y, guide=guide, **params)
    lam, lr = params["reg_lambda"], params["learning_rate"]
    logistic = params.get("objective", 0) == 1
    assert gpu["init_pred"] == pytest.approx(ref["init_pred"], rel=1e-12)
    pred = np.full(bins.shape[1], ref["init_pred"])
    adopted = near = 0
    for t in range(T):
        n = ref["nodes_per_tree"][t]
        info = ref["info"][t][:n]
        bad = np.nonzero(info["guide_mismatch"])[0]
        if len(bad):
            i = bad[0]
            on = ref["nodes"][t][i]
            gn = gpu["nodes"][t][i]
            raise AssertionError(
                f"tree {t} node {i}: GPU chose ({gn['feature']},{gn['threshold_bin']}) gain {gn['gain']!r}, "
                f"oracle ({on['feature']},{on['threshold_bin']}) gain {on['gain']!r}, second {info[i]['second_gain']!r}")
        assert gpu["nodes_per_tree"][t] == n, f"tree {t}: {gpu['nodes_per_tree'][t]} nodes vs oracle {n}"
        a, b = gpu["nodes"][t][:n], ref["nodes"][t][:n]
        for k in ("feature", "threshold_bin", "left", "right", "is_leaf"):
            assert np.array_equal(a[k].astype(np.int64), b[k].astype(np.int64)), f"tree {t}: {k} differs"
        adopted += int(info["adopted"].sum())
        near += int((info["n_near"] > 1).sum())
        gt, ht = oracle.gradients(pred, y, 1 if logistic else 0)
        S = fixed_exponent(float(np.abs(gt).max()), bins.shape[1])
        tol = g_tolerance(info["A"], info["n_rows"], S) / (info["H"] + lam)
        if logistic:  # S_h one lower: the library's max h may sit an ulp across a power of two
            th = h_tolerance(info["H"], info["n_rows"], fixed_exponent(float(ht.max()), bins.shape[1]) - 1)
            tol = (g_tolerance(info["A"], info["n_rows"], S) + np.abs(b["leaf_value"]) * th) / np.maximum(
                info["H"] + lam - th, 1e-300)
        err = np.abs(a["leaf_value"] - b["leaf_value"])
        assert np.all(err <= tol), f"tree {t}: leaf value off by {err.max()} (tol {tol[err.argmax()]})"
        internal = b["is_leaf"] == 0
        np.testing.assert_allclose(a["gain"][internal], b["gain"][internal], rtol=1e-6, atol=1e-9)
        pred = pred + lr * b["leaf_value"][traverse(b, bins)]
    p_gpu = gpu["pred"].cpu().numpy()
    scale = np.maximum(np.abs(ref["pred"]), float(np.std(y)))
    assert np.all(np.abs(p_gpu - ref["pred"]) <= 1e-6 * scale), "predictions differ beyond 1e-6 relative"
    if report is not None:
        report.update(adopted=adopted, near_ties=near, trees=T)
    return ref


def record_parity(config: str, **fields):
    """Print a parity record (near-tie counts and the like) and, when GBDT_PARITY_RECORD names a file,
    append it there as one JSON line."""
    rec = dict(config=config, **fields)
    print("parity record:", json.dumps(rec))
    path = os.environ.get("GBDT_PARITY_RECORD")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(rec) + "\n")

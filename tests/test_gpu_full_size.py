"""Parity at the workloads' stated sizes, in the configurations bench.py times.

Every training workload is checked node by node against the oracle (multithreaded over features;
near-ties under the rule of tests/gpu_util.compare_training, recorded per workload):
  * mid: 100,000 rows x 28 features, depth 6, all 100 trees;
  * covtype-shaped: 581,012 rows x 54 features, depth 10, 1,023-leaf budget, all 100 trees (the
    benchmark's covtype leg);
  * large: 10,000,000 rows x 100 features, depth 8, the first three trees (the second and third use
    the root kernel that reuses the first tree's counts), and quantize on sampled columns.
The one-level microbench (50,000,000 rows x 64 pre-binned features, 256 nodes) is checked after the
GPU's own partition: every segment holds exactly its node's rows, and every built histogram matches
the oracle's.
"""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest

from tests.gpu_util import (compare_training, dev_struct, g, g_tolerance, level, needs_gpu, oracle, record_parity,
                            torch)
import synth

pytestmark = [pytest.mark.gpu, needs_gpu]
THREADS = os.cpu_count() or 1


@pytest.fixture(scope="module")
def large():
    X, y = synth.make("large")
    Xd = torch.from_numpy(X).cuda()
    bins, edges, n_bins = g.quantize(Xd, synth.CONFIGS["large"]["max_bins"])
    return X, y, Xd, bins, edges, n_bins


def test_large_quantize_matches_oracle_on_sampled_columns(large):
    X, _, _, bins, edges, n_bins = large
    N = X.shape[1]
    sel = [0, 49, 50, 79, 80, 99]  # normal, log-normal and low-cardinality integer columns
    ob, oe, on = oracle.quantize(X[sel], synth.CONFIGS["large"]["max_bins"], n_threads=THREADS)
    assert np.array_equal(bins[sel, :N].cpu().numpy(), ob)
    assert np.array_equal(edges[sel].cpu().numpy(), oe)
    assert np.array_equal(n_bins[sel].cpu().numpy(), on)


def test_large_first_trees_match_oracle(large):
    X, y, _, bins, _, n_bins = large
    N = X.shape[1]
    params = dict(synth.CONFIGS["large"], n_trees=3, n_threads=THREADS)
    out = g.train(bins, n_bins, torch.from_numpy(y).cuda(), **params)
    ob = bins[:, :N].cpu().numpy()
    rep = {}
    compare_training(out, ob, n_bins.cpu().numpy(), y, params, rep)
    record_parity("large 10,000,000 x 100, depth 8, first 3 of 200 trees", **rep)


def _full_config(name, **extra):
    X, y = synth.make(name)
    cfg = dict(synth.CONFIGS[name], **extra)
    Xd = torch.from_numpy(X).cuda()
    bins, edges, n_bins = g.quantize(Xd, cfg["max_bins"])
    N = X.shape[1]
    ob, oe, on = oracle.quantize(X, cfg["max_bins"], n_threads=THREADS)
    assert np.array_equal(bins[:, :N].cpu().numpy(), ob), "quantize differs from the oracle"
    assert np.array_equal(edges.cpu().numpy(), oe) and np.array_equal(n_bins.cpu().numpy(), on)
    params = dict(cfg, n_threads=THREADS)
    out = g.train(bins, n_bins, torch.from_numpy(y).cuda(), **params)
    rep = {}
    compare_training(out, ob, on, y, params, rep)
    return out, rep


def test_mid_full_config_matches_oracle():
    out, rep = _full_config("mid")
    assert rep["trees"] == 100
    record_parity("mid 100,000 x 28, depth 6, 100 trees", **rep)


def test_covtype_full_config_with_leaf_budget_matches_oracle():
    out, rep = _full_config("covtype", num_leaves=1023)
    assert rep["trees"] == 100
    assert max(out["nodes_per_tree"]) <= 2 * 1023 - 1
    record_parity("covtype-shaped 581,012 x 54, depth 10, 1023 leaves, 100 trees", **rep,
                  max_leaves=int((max(out["nodes_per_tree"]) + 1) // 2))


def _oracle_histograms_parallel(bins, gv, slot_of_row, n_slots, groups=8):
    """oracle.histograms over slot groups in parallel threads (each call sees every row in row order and
    keeps its own slots; the oracle releases the interpreter while it runs).  Returns cnt, G and A, the
    sum of |g| per entry (the oracle's G of |g|)."""
    bounds = np.linspace(0, n_slots, groups + 1).astype(int)
    local = [np.where((slot_of_row >= bounds[k]) & (slot_of_row < bounds[k + 1]), slot_of_row - bounds[k],
                      -1).astype(np.int32) for k in range(groups)]
    ga = np.abs(gv)

    def one(k, weights):
        return oracle.histograms(bins, weights, local[k], bounds[k + 1] - bounds[k])

    with ThreadPoolExecutor(max_workers=min(THREADS, 2 * groups)) as ex:
        gf = [ex.submit(one, k, gv) for k in range(groups)]
        af = [ex.submit(one, k, ga) for k in range(groups)]
        parts = [f.result() for f in gf]
        aparts = [f.result() for f in af]
    cnt = np.concatenate([p["cnt"] for p in parts])
    G = np.concatenate([p["G"] for p in parts])
    A = np.concatenate([p["G"] for p in aparts])
    return cnt, G, A


def test_micro_level_all_nodes_after_partition():
    N, F, n_nodes = synth.CONFIGS["micro"]["n"], synth.CONFIGS["micro"]["f"], synth.CONFIGS["micro"]["n_nodes"]
    bins, node, gv = synth.make_micro(n=N)
    P = n_nodes // 2
    parent = node >> 1
    pc = np.bincount(parent, minlength=P)
    pseg = np.zeros(P, g.SEGMENT_DTYPE)
    pseg["start"], pseg["count"] = np.concatenate([[0], np.cumsum(pc)[:-1]]), pc
    counts = np.bincount(node, minlength=n_nodes)
    sp = np.zeros(P, g.SPLIT_DTYPE)
    sp["feature"], sp["bin"], sp["cnt_left"], sp["cnt_total"] = 0, 0, counts[0::2], pc
    Bd = torch.zeros((F, g.padded_ld(N)), dtype=torch.uint8, device="cuda")
    Bd[:, :N] = torch.from_numpy(bins).cuda()
    gd = torch.from_numpy(gv).cuda()
    orig = torch.arange(N, dtype=torch.int32, device="cuda")
    go_right = torch.from_numpy((node & 1).astype(np.uint8)).cuda()
    cb, cg, co, cseg, _ = g.partition_rows(Bd, N, gd, orig, dev_struct(sp, g.SPLIT_DTYPE), level(0, P), P,
                                           dev_struct(pseg, g.SEGMENT_DTYPE), go_right=go_right)
    flags = np.zeros(n_nodes, np.uint8)
    left_small = counts[0::2] <= counts[1::2]
    flags[0::2], flags[1::2] = left_small, ~left_small
    S = g.gradient_scale(gd)
    rb = g.to_row_blocks(cb, N)
    hc, hq = g.build_histograms_segmented(cb, N, cg, S, level(P, n_nodes), n_nodes, torch.from_numpy(flags).cuda(),
                                          P, cseg, row_blocks=rb)
    # every child's segment holds exactly its node's rows, each side in its parent's order (stable)
    co_h = co.cpu().numpy().view(np.uint32)[:N]
    seg_h = np.frombuffer(cseg.cpu().numpy().tobytes(), g.SEGMENT_DTYPE)[:n_nodes]
    by_node = np.argsort(node, kind="stable")  # rows of node 0, then node 1, ... each in row order
    want_start = np.concatenate([[0], np.cumsum(counts)[:-1]])
    assert np.array_equal(seg_h["start"], want_start) and np.array_equal(seg_h["count"], counts)
    assert np.array_equal(co_h, by_node)
    # every built histogram against the oracle's (slots in node order; the unbuilt ones come by subtraction)
    built = np.nonzero(flags)[0]
    slot_of_row = np.full(N, -1, np.int32)
    rank = np.full(n_nodes, -1, np.int32)
    rank[built] = np.arange(len(built))
    slot_of_row[:] = rank[node]
    cnt, G, A = _oracle_histograms_parallel(bins, gv.astype(np.float64), slot_of_row, len(built))
    hc_h, hq_h = hc.cpu().numpy().view(np.uint32), hq.cpu().numpy()
    s_exp = int(S.item())
    assert np.array_equal(hc_h[built], cnt)
    Gg = np.ldexp(hq_h[built].astype(np.float64), -s_exp)
    err = np.abs(Gg - G)
    tol = g_tolerance(A, cnt, s_exp)
    assert np.all(err <= tol), f"G off by {err.max()} (tol {tol.flat[err.argmax()]})"
    record_parity("micro 50,000,000 x 64, 256 nodes (row-grouped level)", built_nodes=int(len(built)),
                  segments_checked=n_nodes, max_G_err_over_tol=float((err / tol).max()))


def test_micro_level_node_id_call_all_built_nodes():
    """The 50M-row level as stated: rows in no node order, each carrying its node id; gbdt_build_histograms
    (which groups the built slots' rows inside the call) against the oracle on every built node."""
    N, F, n_nodes = synth.CONFIGS["micro"]["n"], synth.CONFIGS["micro"]["f"], synth.CONFIGS["micro"]["n_nodes"]
    bins, node, gv = synth.make_micro(n=N, grouped=False)
    P = n_nodes // 2
    counts = np.bincount(node, minlength=n_nodes)
    flags = np.zeros(n_nodes, np.uint8)
    left_small = counts[0::2] <= counts[1::2]
    flags[0::2], flags[1::2] = left_small, ~left_small
    Bd = torch.zeros((F, g.padded_ld(N)), dtype=torch.uint8, device="cuda")
    Bd[:, :N] = torch.from_numpy(bins).cuda()
    gd = torch.from_numpy(gv).cuda()
    S = g.gradient_scale(gd)
    ids = torch.from_numpy((P + node.astype(np.int32)).astype(np.uint16).view(np.int16)).cuda()
    ws = g._workspace(g.lib().gbdt_histograms_workspace_size(N, F, n_nodes))
    hc, hq = g.build_histograms(Bd, N, gd, S, ids, level(P, n_nodes), n_nodes, torch.from_numpy(flags).cuda(), P,
                                ws=ws)
    assert g.workspace_status(ws) == 0
    built = np.nonzero(flags)[0]
    rank = np.full(n_nodes, -1, np.int32)
    rank[built] = np.arange(len(built))
    cnt, G, A = _oracle_histograms_parallel(bins, gv.astype(np.float64), rank[node], len(built))
    hc_h, hq_h = hc.cpu().numpy().view(np.uint32), hq.cpu().numpy()
    s_exp = int(S.item())
    assert np.array_equal(hc_h[built], cnt)
    Gg = np.ldexp(hq_h[built].astype(np.float64), -s_exp)
    err = np.abs(Gg - G)
    tol = g_tolerance(A, cnt, s_exp)
    assert np.all(err <= tol), f"G off by {err.max()} (tol {tol.flat[err.argmax()]})"
    record_parity("micro 50,000,000 x 64, 256 nodes (rows in no node order, gbdt_build_histograms)",
                  built_nodes=int(len(built)), max_G_err_over_tol=float((err / tol).max()))

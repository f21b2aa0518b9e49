"""Parity at the benchmark's full sizes, in the configuration bench.py times.

The large workload (10,000,000 rows x 100 features, depth 8) and the one-level
microbench (50,000,000 rows x 64 pre-binned features, 256 nodes) are checked
against the oracle where the oracle finishes in seconds: quantize on sampled
columns of every kind, one whole tree node by node (the oracle multithreaded
over features), and the level's histograms on sampled nodes after the GPU's
own partition.
"""
import os

import numpy as np
import pytest

from tests.gpu_util import compare_training, dev_struct, g, g_tolerance, level, needs_gpu, oracle, torch
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


def test_large_one_tree_matches_oracle(large):
    X, y, _, bins, _, n_bins = large
    N = X.shape[1]
    params = dict(synth.CONFIGS["large"], n_trees=1, n_threads=THREADS)
    out = g.train(bins, n_bins, torch.from_numpy(y).cuda(), **params)
    ob = bins[:, :N].cpu().numpy()
    rep = {}
    compare_training(out, ob, n_bins.cpu().numpy(), y, params, rep)
    print("large, one tree:", rep)


def test_micro_level_histograms_after_partition():
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
    # the moved row ids map positions back to rows: every child's rows are exactly its node's rows
    co_h = co.cpu().numpy().view(np.uint32)[:N]
    seg_h = np.frombuffer(cseg.cpu().numpy().tobytes(), g.SEGMENT_DTYPE)[:n_nodes]
    s_exp = int(S.item())
    sample = [s for s in (0, 1, 2, 3, 100, 101, 254, 255) if flags[s]]
    slot_of_row = np.full(N, -1, np.int32)
    idx = {s: np.nonzero(node == s)[0] for s in sample}
    for s in sample:
        rows = co_h[seg_h["start"][s]: seg_h["start"][s] + seg_h["count"][s]]
        assert np.array_equal(np.sort(rows), idx[s])
        slot_of_row[idx[s]] = sample.index(s)
    ref = oracle.histograms(bins, gv.astype(np.float64), slot_of_row, len(sample))
    hc_h, hq_h = hc.cpu().numpy().view(np.uint32), hq.cpu().numpy()
    for i, s in enumerate(sample):
        assert np.array_equal(hc_h[s], ref["cnt"][i]), f"node {s}"
        w = np.abs(gv[idx[s]].astype(np.float64))
        A = np.stack([np.bincount(bins[f, idx[s]], weights=w, minlength=256) for f in range(F)])
        G = np.ldexp(hq_h[s].astype(np.float64), -s_exp)
        assert np.all(np.abs(G - ref["G"][i]) <= g_tolerance(A, ref["cnt"][i], s_exp)), f"node {s}"

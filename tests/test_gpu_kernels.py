"""Per-kernel parity of the CUDA path against the CPU oracle, through the C ABI.

Inputs are seeded and synthetic, sized so the oracle finishes in seconds while
the launches still span several CTAs and end on a ragged tail.
"""
import numpy as np
import pytest

from tests.gpu_util import (dev_bins, dev_struct, fixed_exponent, g, g_tolerance, host_struct, level, needs_gpu,
                            oracle, torch, u16)
import synth

pytestmark = [pytest.mark.gpu, needs_gpu]


# ----------------------------------------------------------------------------- quantize
@pytest.mark.parametrize("name,n", [("tiny", 2000), ("mid", 20_011), ("covtype", 30_007), ("large", 25_003)])
def test_quantize_matches_oracle(name, n):
    X, _ = synth.make(name, n=n)
    B = synth.CONFIGS[name]["max_bins"]
    bins, edges, n_bins = g.quantize(torch.from_numpy(X).cuda(), B)
    ob, oe, on = oracle.quantize(X, B, n_threads=8)
    assert np.array_equal(n_bins.cpu().numpy(), on)
    assert np.array_equal(edges.cpu().numpy(), oe)  # includes the +inf padding
    assert np.array_equal(bins[:, :n].cpu().numpy(), ob)


@pytest.mark.parametrize("case", ["constant", "two_values", "signed_zero", "n1", "n15", "n17", "all_distinct_256",
                                  "ties_at_quantiles", "huge_range", "sorted_blocks_300", "u256", "u257"])
def test_quantize_edge_cases(case):
    rng = np.random.default_rng(hash(case) % 2**32)
    if case == "constant":
        X = np.full((2, 1000), 7.5, np.float32)
    elif case == "two_values":
        X = rng.choice(np.array([0, 1], np.float32), (3, 999))
    elif case == "signed_zero":
        X = rng.choice(np.array([-0.0, 0.0, 1.0, -1.0], np.float32), (2, 5000))
    elif case == "n1":
        X = np.array([[3.0], [-2.0]], np.float32)
    elif case == "n15":
        X = rng.normal(size=(2, 15)).astype(np.float32)
    elif case == "n17":
        X = rng.normal(size=(2, 17)).astype(np.float32)
    elif case == "all_distinct_256":
        X = rng.permutation(np.arange(70_000, dtype=np.float32))[None, :]
    elif case == "ties_at_quantiles":
        X = np.round(rng.exponential(3.0, (4, 40_000))).astype(np.float32)
    elif case == "sorted_blocks_300":  # few distinct values per stretch of rows, 300 in the column
        X = np.repeat(np.arange(300, dtype=np.float32), 200)[None, :] * 0.5 - 20.0
    elif case in ("u256", "u257"):  # exactly max_bins distinct values, and one more, in random order
        U = 256 if case == "u256" else 257
        X = rng.permutation(np.tile(rng.normal(size=U).astype(np.float32), 90))[None, :]
    else:
        X = (rng.normal(size=(2, 9000)) * 10.0 ** rng.integers(-30, 30, (2, 9000))).astype(np.float32)
    for B in (2, 16, 255, 256):
        bins, edges, n_bins = g.quantize(torch.from_numpy(X).cuda(), B)
        ob, oe, on = oracle.quantize(X, B)
        N = X.shape[1]
        assert np.array_equal(n_bins.cpu().numpy(), on), (case, B)
        assert np.array_equal(edges.cpu().numpy(), oe), (case, B)
        assert np.array_equal(bins[:, :N].cpu().numpy(), ob), (case, B)


def test_quantize_rejects_nonfinite():
    X = np.zeros((2, 100), np.float32)
    X[1, 57] = np.nan
    with pytest.raises(g.GbdtError) as e:
        g.quantize(torch.from_numpy(X).cuda(), 32)
    assert e.value.code == g.ERR_NONFINITE


@pytest.mark.parametrize("pinned", [True, False])
@pytest.mark.parametrize("name,n", [("large", 25_003), ("covtype", 30_007)])
def test_quantize_from_host_equals_device_path(name, n, pinned):
    """gbdt_quantize_host (column batches copied on a stream of their own while earlier batches are binned)
    gives the oracle's bins, edges and n_bins, and leaves the device copy equal to the host features; also
    with a leading dimension above N (the copy of the last column stops at N)."""
    X, _ = synth.make(name, n=n)
    B = synth.CONFIGS[name]["max_bins"]
    ob, oe, on = oracle.quantize(X, B, n_threads=8)
    F, N = X.shape
    for ld in (N, N + 5):
        Xh = torch.zeros((F, ld), dtype=torch.float32, pin_memory=pinned)[:, :N]
        Xh.copy_(torch.from_numpy(X))
        Xd = torch.full((F, ld), -1.0, dtype=torch.float32, device="cuda")[:, :N]
        bins, edges, n_bins = g.quantize(Xh, B, x_device=Xd)
        assert np.array_equal(n_bins.cpu().numpy(), on)
        assert np.array_equal(edges.cpu().numpy(), oe)
        assert np.array_equal(bins[:, :N].cpu().numpy(), ob)
        assert torch.equal(Xd.cpu(), Xh)


def test_quantize_from_host_rejects_nonfinite():
    X = torch.zeros((20, 1000), dtype=torch.float32, pin_memory=True)
    X[17, 999] = float("inf")  # in the last batch of columns
    with pytest.raises(g.GbdtError) as e:
        g.quantize(X, 32)
    assert e.value.code == g.ERR_NONFINITE


# ----------------------------------------------------------------------------- gradients
def test_gradients_and_scale():
    rng = np.random.default_rng(1)
    N = 100_003
    pred = rng.normal(size=N)
    label = rng.normal(size=N).astype(np.float32)
    gd, S = g.compute_gradients(torch.from_numpy(pred).cuda(), torch.from_numpy(label).cuda())
    og, oh = oracle.gradients(pred, label)
    assert np.array_equal(gd.cpu().numpy(), og)  # one exact subtraction on both sides
    assert int(S.item()) == fixed_exponent(float(np.abs(og).max()), N)
    S32 = g.gradient_scale(torch.from_numpy(og.astype(np.float32)).cuda())
    assert int(S32.item()) == fixed_exponent(float(np.abs(og.astype(np.float32)).max()), N)
    assert int(g.gradient_scale(torch.zeros(10, dtype=torch.float64, device="cuda")).item()) == 0


def test_update_predictions_bit_exact():
    rng = np.random.default_rng(2)
    N, L = 77_777, 63
    pred = rng.normal(size=N)
    leaf = rng.normal(size=L)
    nodes = rng.integers(0, L, N).astype(np.uint16)
    out = g.update_predictions(torch.from_numpy(pred.copy()).cuda(), u16(nodes), torch.from_numpy(leaf).cuda(), 0.37)
    ref = oracle.update_predictions(pred, leaf, nodes.astype(np.int32), 0.37)
    assert np.array_equal(out.cpu().numpy(), ref)


# ----------------------------------------------------------------------------- histograms
def _hist_case(N, F, n_slots, node_begin, flags, gdtype, seed, n_bins_max=256):
    rng = np.random.default_rng(seed)
    bins = rng.integers(0, n_bins_max, (F, N)).astype(np.uint8)
    if F > 1:  # a Zipf-skewed column, and a binary one
        p = (np.arange(1, 257) ** -1.1)
        bins[0] = (rng.choice(256, N, p=p / p.sum()) % n_bins_max).astype(np.uint8)
        bins[F - 1] = rng.integers(0, 2, N)
    node = rng.integers(max(0, node_begin - 3), node_begin + n_slots + 3, N).astype(np.uint16)
    gv = rng.normal(0, 2, N).astype(gdtype)
    slot = node.astype(np.int32) - node_begin
    slot[(slot < 0) | (slot >= n_slots)] = -1
    return bins, node, gv, slot


@pytest.mark.parametrize("path", ["grouped", "scan"])
@pytest.mark.parametrize("N,F,n_slots,nb,gdtype", [
    (1, 1, 1, 0, np.float64), (15, 3, 1, 0, np.float64), (17, 2, 2, 3, np.float32),
    (50_003, 7, 6, 5, np.float64), (50_003, 7, 6, 5, np.float32), (120_001, 3, 40, 31, np.float64),
    (200_009, 5, 256, 255, np.float32), (33_333, 70, 2, 1, np.float64), (70_001, 130, 4, 3, np.float64)])
def test_build_histograms_matches_oracle(N, F, n_slots, nb, gdtype, path):
    """Both paths of gbdt_build_histograms: rows grouped by slot in the workspace first (the full workspace,
    two or more built slots), and the node-id scan (a workspace holding only the error word)."""
    bins, node, gv, slot = _hist_case(N, F, n_slots, nb, None, gdtype, seed=N + F + n_slots)
    rng = np.random.default_rng(N)
    flags = (rng.random(n_slots) < 0.6).astype(np.uint8)
    flags[0] = 1
    max_slots = max(n_slots, 1)
    S = g.gradient_scale(torch.from_numpy(gv).cuda())
    sentinel = 12345
    hc = torch.full((max_slots, F, 256), sentinel, dtype=torch.int32, device="cuda")
    hq = torch.full((max_slots, F, 256), sentinel, dtype=torch.int64, device="cuda")
    ws = g._workspace(256) if path == "scan" else None
    g.build_histograms(dev_bins(bins), N, torch.from_numpy(gv).cuda(), S, u16(node), level(nb, n_slots), max_slots,
                       torch.from_numpy(flags).cuda(), int(flags.sum()), hc, hq, ws=ws)
    ref = oracle.histograms(bins, gv.astype(np.float64), slot, n_slots)
    s_exp = int(S.item())
    assert s_exp == fixed_exponent(float(np.abs(gv.astype(np.float64)).max()), N)
    hc, hq = hc.cpu().numpy().view(np.uint32), hq.cpu().numpy()
    for s in range(n_slots):
        if not flags[s]:
            assert np.all(hc[s] == sentinel) and np.all(hq[s] == sentinel)  # untouched
            continue
        assert np.array_equal(hc[s], ref["cnt"][s]), f"slot {s}: counts differ"
        m = slot == s
        A = np.stack([np.bincount(bins[f][m], weights=np.abs(gv[m].astype(np.float64)), minlength=256)
                      for f in range(F)])
        G = np.ldexp(hq[s].astype(np.float64), -s_exp)
        tol = g_tolerance(A, ref["cnt"][s], s_exp)
        assert np.all(np.abs(G - ref["G"][s]) <= tol), f"slot {s}: G off by {np.abs(G - ref['G'][s]).max()}"


def test_subtraction_equals_direct_build():
    # A/B: the larger sibling by parent - smaller must equal building it directly, bit for bit.
    N, F = 90_001, 6
    rng = np.random.default_rng(5)
    bins = rng.integers(0, 256, (F, N)).astype(np.uint8)
    parent = rng.integers(0, 3, N).astype(np.uint16)  # level 0 nodes... 3 parents (slots 0..2)
    child = (2 * parent + rng.integers(0, 2, N)).astype(np.uint16)  # 6 children
    gv = rng.normal(size=N)
    S = g.gradient_scale(torch.from_numpy(gv).cuda())
    Bd, gd = dev_bins(bins), torch.from_numpy(gv).cuda()
    pc, pq = g.build_histograms(Bd, N, gd, S, u16(parent), level(0, 3), 3, torch.ones(3, dtype=torch.uint8,
                                device="cuda"), 3)
    cnt = np.bincount(child, minlength=6)
    flags = np.array([cnt[2 * k] <= cnt[2 * k + 1] for k in range(3) for _ in (0, 1)], np.uint8)
    flags[1::2] = 1 - flags[0::2]
    fd = torch.from_numpy(flags).cuda()
    hc, hq = g.build_histograms(Bd, N, gd, S, u16(child), level(0, 6), 6, fd, 3)
    pair_parent = torch.tensor([0, 1, 2], dtype=torch.int32, device="cuda")
    g.subtract_histograms(pc, pq, pair_parent, fd, level(0, 6), 6, hc, hq)
    dc, dq = g.build_histograms(Bd, N, gd, S, u16(child), level(0, 6), 6, torch.ones(6, dtype=torch.uint8,
                                device="cuda"), 6)
    assert torch.equal(hc, dc) and torch.equal(hq, dq)


# ----------------------------------------------------------------------------- split search
@pytest.mark.parametrize("seed,params", [
    (0, dict(reg_lambda=1.0, gamma=0.0, min_samples_leaf=1, min_child_weight=0.0)),
    (1, dict(reg_lambda=0.0, gamma=0.0, min_samples_leaf=20, min_child_weight=0.0)),
    (2, dict(reg_lambda=3.0, gamma=0.5, min_samples_leaf=5, min_child_weight=30.0)),
    (3, dict(reg_lambda=1.0, gamma=1e9, min_samples_leaf=1, min_child_weight=0.0)),  # nothing splits
])
def test_find_splits_matches_oracle(seed, params):
    rng = np.random.default_rng(40 + seed)
    N, F, n_slots = 60_007, 9, 12
    n_bins = rng.integers(1, 257, F).astype(np.int32)
    n_bins[0] = 256
    bins = np.stack([rng.integers(0, nb, N) for nb in n_bins]).astype(np.uint8)
    node = rng.integers(0, n_slots, N).astype(np.uint16)
    # gradients correlated with one feature per slot so that gains differ clearly
    gv = rng.normal(size=N) + 0.3 * (bins[seed % F].astype(np.float64) / n_bins[seed % F]) * (node % 3)
    S = g.gradient_scale(torch.from_numpy(gv).cuda())
    hc, hq = g.build_histograms(dev_bins(bins), N, torch.from_numpy(gv).cuda(), S, u16(node), level(0, n_slots),
                                n_slots, torch.ones(n_slots, dtype=torch.uint8, device="cuda"), n_slots)
    out = g.find_splits(hc, hq, S, torch.from_numpy(n_bins).cuda(), level(0, n_slots), n_slots, **params)
    sp = host_struct(out, g.SPLIT_DTYPE, n_slots)
    ref = oracle.histograms(bins, gv, node.astype(np.int32), n_slots)
    for s in range(n_slots):
        o = oracle.best_split(ref["cnt"][s], ref["G"][s], ref["H"][s], n_bins, ref["n"][s], ref["Gt"][s],
                              ref["Ht"][s], **params)
        assert sp["cnt_total"][s] == ref["n"][s]
        assert np.ldexp(float(sp["q_total"][s]), -int(S.item())) == pytest.approx(ref["Gt"][s], rel=1e-9, abs=1e-6)
        if not (o.valid and o.gain > 0):
            assert sp["feature"][s] == -1
            continue
        near = {(o.near_feature[i], o.near_bin[i]) for i in range(min(o.n_near, 8))}
        got = (int(sp["feature"][s]), int(sp["bin"][s]))
        assert got == (o.feature, o.bin) or (o.n_near > 1 and got in near), (s, got, (o.feature, o.bin))
        assert sp["gain"][s] == pytest.approx(o.gain, rel=1e-7)
        assert sp["cnt_left"][s] == o.cnt_left


# ----------------------------------------------------------------------------- partition
def test_partition_matches_oracle():
    rng = np.random.default_rng(8)
    N, F, n_slots, nb = 150_001, 5, 7, 11
    bins = rng.integers(0, 256, (F, N)).astype(np.uint8)
    slot = rng.integers(0, n_slots, N)
    order = np.argsort(slot, kind="stable")  # rows grouped by slot, ascending inside
    counts = np.bincount(slot, minlength=n_slots)
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    feats = np.array([0, -1, 2, 4, -1, 1, 3])
    thr = np.array([100, -1, 3, 250, -1, 0, 128])
    cnt_left = np.array([(bins[feats[s], order[starts[s]:starts[s] + counts[s]]] <= thr[s]).sum() if feats[s] >= 0
                         else 0 for s in range(n_slots)])
    sp = np.zeros(n_slots, g.SPLIT_DTYPE)
    sp["feature"], sp["bin"], sp["cnt_left"], sp["cnt_total"] = feats, thr, cnt_left, counts
    seg = np.zeros(n_slots, g.SEGMENT_DTYPE)
    seg["start"], seg["count"] = starts, counts
    node = (nb + slot).astype(np.uint16)
    node_d = u16(node)
    idx_out, seg_out, nxt = g.partition(dev_bins(bins), N, dev_struct(sp, g.SPLIT_DTYPE), level(nb, n_slots), n_slots,
                                        dev_struct(seg, g.SEGMENT_DTYPE),
                                        torch.from_numpy(order.astype(np.int32)).cuda(), node_d)
    ref_idx, ref_left = oracle.partition(bins, feats, thr, starts, counts, order)
    assert np.array_equal(idx_out.cpu().numpy().astype(np.int64), ref_idx)
    so = host_struct(seg_out, g.SEGMENT_DTYPE, 2 * n_slots)
    nl = host_struct(nxt, g.LEVEL_DTYPE, 1)[0]
    split_slots = [s for s in range(n_slots) if feats[s] >= 0]
    assert (nl["node_begin"], nl["n_slots"]) == (nb + n_slots, 2 * len(split_slots))
    new_node = node_d.cpu().numpy().view(np.uint16)
    for k, s in enumerate(split_slots):
        assert (so["start"][2 * k], so["count"][2 * k]) == (starts[s], ref_left[s])
        assert (so["start"][2 * k + 1], so["count"][2 * k + 1]) == (starts[s] + ref_left[s], counts[s] - ref_left[s])
        rows = order[starts[s]:starts[s] + counts[s]]
        go_right = bins[feats[s], rows] > thr[s]
        assert np.array_equal(new_node[rows], nb + n_slots + 2 * k + go_right)
    for s in range(n_slots):
        if feats[s] < 0:
            assert np.all(new_node[slot == s] == nb + s)


def test_find_splits_ignores_bins_at_or_above_n_bins():
    """The split search reads a feature's bins below its n_bins only (the training's histogram passes never
    write the others): garbage there changes nothing, not even the node totals' consistency check."""
    rng = np.random.default_rng(11)
    N, F, n_slots = 40_009, 7, 6
    n_bins = np.array([3, 256, 2, 17, 64, 2, 200], np.int32)
    bins = np.stack([rng.integers(0, nb, N) for nb in n_bins]).astype(np.uint8)
    node = rng.integers(0, n_slots, N).astype(np.uint16)
    gv = rng.normal(size=N) + 0.5 * (bins[3] > 8) * (node % 2)
    S = g.gradient_scale(torch.from_numpy(gv).cuda())
    hc, hq = g.build_histograms(dev_bins(bins), N, torch.from_numpy(gv).cuda(), S, u16(node), level(0, n_slots),
                                n_slots, torch.ones(n_slots, dtype=torch.uint8, device="cuda"), n_slots)
    nbd = torch.from_numpy(n_bins).cuda()
    params = dict(reg_lambda=1.0, gamma=0.0, min_samples_leaf=5, min_child_weight=0.0)
    clean = host_struct(g.find_splits(hc, hq, S, nbd, level(0, n_slots), n_slots, **params), g.SPLIT_DTYPE, n_slots)
    unused = (torch.arange(256, device="cuda")[None, None, :] >= nbd[None, :, None]).expand(n_slots, F, 256)
    hc2, hq2 = hc.clone(), hq.clone()
    hc2[unused] = torch.randint(0, 1 << 30, (int(unused.sum()),), dtype=torch.int32, device="cuda")
    hq2[unused] = torch.randint(-(1 << 60), 1 << 60, (int(unused.sum()),), dtype=torch.int64, device="cuda")
    ws = g._workspace(g.lib().gbdt_find_splits_workspace_size(F, n_slots))
    dirty = host_struct(g.find_splits(hc2, hq2, S, nbd, level(0, n_slots), n_slots, ws=ws, **params), g.SPLIT_DTYPE,
                        n_slots)
    assert g.workspace_status(ws) == 0
    assert clean.tobytes() == dirty.tobytes()
    assert (clean["feature"] >= 0).any()

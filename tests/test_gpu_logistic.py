"""The logistic objective on the GPU path against the oracle, through the C ABI.

"Gradient boosted trees (spec model)": binary cross-entropy of a sigmoid, so
g = sigmoid(pred) - y and h = p (1 - p).  H is no longer the row count: the
library accumulates it in its own fixed-point histogram (exponent S_h), and
recovers each row's h from its g as |g| (1 - |g|) (exact for 0/1 labels up to
the rounding of g), so h moves with no array of its own.
"""
import numpy as np
import pytest

from tests.gpu_util import (compare_training, dev_bins, dev_struct, fixed_exponent, g, g_tolerance, h_tolerance,
                            host_struct, level, needs_gpu, oracle, torch)
import synth

pytestmark = [pytest.mark.gpu, needs_gpu]
LOGISTIC = 1


def _recovered_h(gv):
    a = np.abs(gv)
    return a * (1.0 - a)


def test_gradients_match_oracle():
    rng = np.random.default_rng(3)
    N = 10_007
    pred = rng.normal(scale=4.0, size=N)
    pred[:6] = [0.0, 40.0, -40.0, 700.0, -745.0, 1e-300]
    y = rng.integers(0, 2, N).astype(np.float32)
    gd, S = g.compute_gradients(torch.from_numpy(pred).cuda(), torch.from_numpy(y).cuda(), objective=LOGISTIC)
    go, ho = oracle.gradients(pred, y, LOGISTIC)
    gg = gd.cpu().numpy()
    # the device and host exp agree to an ulp or two; sigmoid and the subtraction add one rounding each
    assert np.all(np.abs(gg - go) <= 1e-15)
    assert S.cpu().tolist() == [fixed_exponent(float(np.abs(gg).max()), N),
                                fixed_exponent(float(_recovered_h(gg).max()), N)]
    # h recovered from g is the oracle's p (1 - p) up to the rounding of g
    assert np.all(np.abs(_recovered_h(gg) - ho) <= 4e-16)
    # at margin 0 every row has p = 1/2: g = +-1/2, h = 1/4 exactly
    g0, S0 = g.compute_gradients(torch.zeros(N, dtype=torch.float64, device="cuda"), torch.from_numpy(y).cuda(),
                                 objective=LOGISTIC)
    assert np.array_equal(g0.cpu().numpy(), 0.5 - y.astype(np.float64))
    assert S0.cpu().tolist()[1] == fixed_exponent(0.25, N)


def _segments(rng, N, n_slots):
    w = rng.random(n_slots) + 0.05
    counts = np.floor(w / w.sum() * N).astype(np.int64)
    counts[np.argmax(w)] += N - counts.sum()
    seg = np.zeros(n_slots, g.SEGMENT_DTYPE)
    seg["start"], seg["count"] = np.concatenate([[0], np.cumsum(counts)[:-1]]), counts
    return seg, np.repeat(np.arange(n_slots), counts).astype(np.int32)


@pytest.mark.parametrize("layout", ["columns", "row_blocks"])
@pytest.mark.parametrize("N,F,n_slots,filtered", [(200_003, 7, 5, False), (150_001, 70, 9, False),
                                                  (120_003, 33, 4, True), (37, 3, 2, False)])
def test_h_histograms_match_oracle(N, F, n_slots, filtered, layout):
    rng = np.random.default_rng(5 * N + F)
    bins = rng.integers(0, 256, (F, N)).astype(np.uint8)
    bins[1 % F] = rng.integers(0, 4, N).astype(np.uint8)
    pred = rng.normal(scale=2.5, size=N)
    y = rng.integers(0, 2, N).astype(np.float32)
    gd, S = g.compute_gradients(torch.from_numpy(pred).cuda(), torch.from_numpy(y).cuda(), objective=LOGISTIC)
    gv = gd.cpu().numpy()
    _, h_orc = oracle.gradients(pred, y, LOGISTIC)
    s_exp, s_h = S.cpu().tolist()
    if filtered:  # pairs of slots that share their parent's segment, each one side of a split on feature 1
        par, _ = _segments(rng, N, n_slots // 2)
        seg = np.repeat(par, 2)
        filt = np.zeros(n_slots, g.FILTER_DTYPE)
        filt["feature"], filt["bin"], filt["side"] = 1 % F, 1, np.arange(n_slots) & 1
        flags = np.ones(n_slots, np.uint8)
    else:
        seg, slot = _segments(rng, N, n_slots)
        filt = None
        flags = (rng.random(n_slots) < 0.7).astype(np.uint8)
        flags[0] = 1
    Bd = dev_bins(bins)
    rb = g.to_row_blocks(Bd, N) if layout == "row_blocks" else None
    hc, hq, hh = g.build_histograms_segmented(
        Bd, N, gd, S, level(0, n_slots), n_slots, torch.from_numpy(flags).cuda(), int(flags.sum()),
        dev_struct(seg, g.SEGMENT_DTYPE), filters=dev_struct(filt, g.FILTER_DTYPE) if filtered else None,
        row_blocks=rb, logistic=True)
    hc_h, hq_h, hh_h = hc.cpu().numpy().view(np.uint32), hq.cpu().numpy(), hh.cpu().numpy()
    for s in range(n_slots):
        if not flags[s]:
            continue
        rows = np.arange(seg["start"][s], seg["start"][s] + seg["count"][s])
        if filtered:
            rows = rows[(bins[filt["feature"][s], rows] > filt["bin"][s]) == bool(filt["side"][s])]
        m = np.full(N, -1, np.int32)
        m[rows] = 0
        ref = oracle.histograms(bins, gv, m, 1, h=h_orc)
        assert np.array_equal(hc_h[s], ref["cnt"][0]), f"slot {s}"
        A = np.stack([np.bincount(bins[f][rows], weights=np.abs(gv[rows]), minlength=256) for f in range(F)])
        G = np.ldexp(hq_h[s].astype(np.float64), -s_exp)
        assert np.all(np.abs(G - ref["G"][0]) <= g_tolerance(A, ref["cnt"][0], s_exp)), f"slot {s}"
        H = np.ldexp(hh_h[s].astype(np.float64), -s_h)
        assert np.all(np.abs(H - ref["H"][0]) <= h_tolerance(ref["H"][0], ref["cnt"][0], s_h)), f"slot {s}"
        # every feature's H adds up to the same node total (one bin per row per feature)
        assert np.all(hh_h[s].sum(axis=1) == hh_h[s, 0].sum())


def test_h_subtraction_and_split_search():
    """Parent minus built sibling is exact for H too; the split search on H histograms picks the
    oracle's split with H from the hessians, and fills h_left/h_total."""
    rng = np.random.default_rng(21)
    N, F = 60_001, 12
    bins = rng.integers(0, 64, (F, N)).astype(np.uint8)
    pred = rng.normal(scale=1.5, size=N) + 0.8 * (bins[3] > 30)
    y = (rng.random(N) < 1 / (1 + np.exp(-pred))).astype(np.float32)
    gd, S = g.compute_gradients(torch.zeros(N, dtype=torch.float64, device="cuda"), torch.from_numpy(y).cuda(),
                                objective=LOGISTIC)
    s_exp, s_h = S.cpu().tolist()
    seg = np.zeros(1, g.SEGMENT_DTYPE)
    seg["count"] = N
    Bd = dev_bins(bins)
    one = torch.ones(1, dtype=torch.uint8, device="cuda")
    pc, pq, ph = g.build_histograms_segmented(Bd, N, gd, S, level(0, 1), 1, one, 1, dev_struct(seg, g.SEGMENT_DTYPE),
                                              logistic=True)
    n_bins = torch.full((F,), 64, dtype=torch.int32, device="cuda")
    params = dict(reg_lambda=0.5, gamma=0.0, min_samples_leaf=10, min_child_weight=1.0, objective=LOGISTIC)
    sp = host_struct(g.find_splits(pc, pq, S, n_bins, level(0, 1), 1, hist_h=ph, **params), g.SPLIT_DTYPE, 1)[0]
    gv = gd.cpu().numpy()
    _, h_orc = oracle.gradients(np.zeros(N), y, LOGISTIC)
    ref = oracle.histograms(bins, gv, np.zeros(N, np.int32), 1, h=h_orc)
    osp = oracle.best_split(ref["cnt"][0], ref["G"][0], ref["H"][0], np.full(F, 64, np.int32), N, ref["Gt"][0],
                            ref["Ht"][0], **params)
    assert (sp["feature"], sp["bin"]) == (osp.feature, osp.bin)
    assert sp["gain"] == pytest.approx(osp.gain, rel=1e-9)
    assert sp["h_total"] == ph.cpu().numpy()[0, 0].sum()
    rows_left = bins[sp["feature"]] <= sp["bin"]
    assert np.ldexp(float(sp["h_left"]), -s_h) == pytest.approx(h_orc[rows_left].sum(), rel=1e-9)
    assert sp["cnt_left"] == rows_left.sum()
    # children of the split: build the left one, subtract for the right
    kseg = np.zeros(2, g.SEGMENT_DTYPE)
    order = np.concatenate([np.nonzero(rows_left)[0], np.nonzero(~rows_left)[0]])
    kseg["start"], kseg["count"] = [0, rows_left.sum()], [rows_left.sum(), N - rows_left.sum()]
    Bk = dev_bins(bins[:, order])
    gk = torch.from_numpy(gv[order]).cuda()
    flags = torch.tensor([1, 0], dtype=torch.uint8, device="cuda")
    kc, kq, kh = g.build_histograms_segmented(Bk, N, gk, S, level(1, 2), 2, flags, 1, dev_struct(kseg, g.SEGMENT_DTYPE),
                                              logistic=True)
    g.subtract_histograms(pc, pq, torch.zeros(1, dtype=torch.int32, device="cuda"), flags, level(1, 2), 2, kc, kq,
                          prev_h=ph, hist_h=kh)
    rc, rq, rh = g.build_histograms_segmented(Bk, N, gk, S, level(1, 2), 2, torch.tensor([0, 1], dtype=torch.uint8,
                                                                                        device="cuda"), 1,
                                              dev_struct(kseg, g.SEGMENT_DTYPE), logistic=True)
    assert torch.equal(kc[1], rc[1]) and torch.equal(kq[1], rq[1]) and torch.equal(kh[1], rh[1])


def _prepare(name, n):
    X, y = synth.make_binary(name, n=n)
    B = synth.CONFIGS[name]["max_bins"]
    bins, edges, n_bins = g.quantize(torch.from_numpy(X).cuda(), B)
    ob, _, on = oracle.quantize(X, B, n_threads=8)
    assert np.array_equal(bins[:, : X.shape[1]].cpu().numpy(), ob)
    return X, bins, edges, n_bins, torch.from_numpy(y).cuda(), ob, on, y


@pytest.mark.parametrize("name,n,trees", [("tiny", None, 5), ("mid", 20_011, 6), ("covtype", 30_007, 4),
                                          ("large", 40_009, 4)])
def test_logistic_training_matches_oracle(name, n, trees):
    _, bins, _, n_bins, yd, ob, on, y = _prepare(name, n)
    params = dict(synth.CONFIGS[name], n_trees=trees, objective=LOGISTIC)
    out = g.train(bins, n_bins, yd, **params)
    assert out["init_pred"] == 0.0
    rep = {}
    compare_training(out, ob, on, y, params, rep)
    print(name, "logistic", rep)


@pytest.mark.parametrize("extra", [dict(max_depth=0), dict(max_depth=1, reg_lambda=0.0, min_child_weight=2.0),
                                   dict(num_leaves=6, max_depth=5), dict(min_child_weight=20.0, gamma=0.05),
                                   dict(n_trees=12, learning_rate=1.0, max_depth=4)])
def test_logistic_parameter_corners(extra):
    _, bins, _, n_bins, yd, ob, on, y = _prepare("tiny", 3_001)
    params = dict(synth.CONFIGS["tiny"], n_trees=3, objective=LOGISTIC)
    params.update(extra)
    out = g.train(bins, n_bins, yd, **params)
    compare_training(out, ob, on, y, params)


def test_logistic_predictions_repeat_and_match_inference():
    X, bins, edges, n_bins, yd, *_ = _prepare("covtype", 20_000)
    params = dict(synth.CONFIGS["covtype"], n_trees=3, max_depth=6, objective=LOGISTIC)
    a = g.train(bins, n_bins, yd, **params)
    b = g.train(bins, n_bins, yd, **params)
    assert a["nodes"].tobytes() == b["nodes"].tobytes() and torch.equal(a["pred"], b["pred"])
    p = g.predict(torch.from_numpy(X).cuda(), edges, a["nodes"], a["init_pred"], params["learning_rate"],
                  nodes_per_tree=a["nodes_per_tree"])
    assert torch.equal(p, a["pred"])


def test_logistic_rejects_labels_other_than_0_and_1():
    _, bins, _, n_bins, _, _, _, y = _prepare("tiny", 1_000)
    bad = y.copy()
    bad[17] = 0.5
    with pytest.raises(g.GbdtError) as e:
        g.train(bins, n_bins, torch.from_numpy(bad).cuda(), **dict(synth.CONFIGS["tiny"], objective=LOGISTIC))
    assert e.value.code == g.ERR_INVALID_ARG and "0 or 1" in str(e.value)
    # the same labels are fine for squared error
    g.train(bins, n_bins, torch.from_numpy(bad).cuda(), **dict(synth.CONFIGS["tiny"], n_trees=1))

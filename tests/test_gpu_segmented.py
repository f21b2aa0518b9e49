"""Parity of the node-contiguous level pass (gbdt_build_histograms_segmented,
gbdt_partition_rows) against the oracle, through the C ABI.

Segments start at arbitrary (unaligned) positions, span several CTA chunks or
partition tiles, and include empty and one-row segments; gradients are f32 and
f64; feature counts cross the 64-features-per-CTA boundary.
"""
import numpy as np
import pytest

from tests.gpu_util import (dev_bins, dev_struct, fixed_exponent, g, g_tolerance, host_struct, level, needs_gpu,
                            oracle, torch, u16)

pytestmark = [pytest.mark.gpu, needs_gpu]


def _segments(rng, N, n_slots, empty=()):
    """Random segment sizes summing to N (some forced empty), in slot order."""
    w = rng.random(n_slots) + 0.05
    w[list(empty)] = 0
    counts = np.floor(w / w.sum() * N).astype(np.int64)
    counts[np.argmax(w)] += N - counts.sum()
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    seg = np.zeros(n_slots, g.SEGMENT_DTYPE)
    seg["start"], seg["count"] = starts, counts
    slot = np.repeat(np.arange(n_slots), counts)
    return seg, slot


@pytest.mark.parametrize("layout", ["columns", "row_blocks"])
@pytest.mark.parametrize("N,F,n_slots,gdtype", [(200_003, 7, 5, np.float64), (150_001, 70, 9, np.float32),
                                                 (77_777, 130, 3, np.float64), (40_000, 3, 64, np.float64),
                                                 (5, 2, 4, np.float64)])
def test_segmented_histograms_match_oracle(N, F, n_slots, gdtype, layout):
    rng = np.random.default_rng(N + F)
    seg, slot = _segments(rng, N, n_slots, empty=(1,) if n_slots > 2 else ())
    bins = rng.integers(0, 256, (F, N)).astype(np.uint8)
    p = np.arange(1, 257) ** -1.1
    bins[0] = rng.choice(256, N, p=p / p.sum()).astype(np.uint8)
    gv = rng.normal(0, 3, N).astype(gdtype)
    flags = (rng.random(n_slots) < 0.7).astype(np.uint8)
    flags[0] = 1
    S = g.gradient_scale(torch.from_numpy(gv).cuda())
    s_exp = int(S.item())
    assert s_exp == fixed_exponent(float(np.abs(gv.astype(np.float64)).max()), N)
    sentinel = 777
    hc = torch.full((n_slots, F, 256), sentinel, dtype=torch.int32, device="cuda")
    hq = torch.full((n_slots, F, 256), sentinel, dtype=torch.int64, device="cuda")
    Bd, gd = dev_bins(bins), torch.from_numpy(gv).cuda()
    rb = g.to_row_blocks(Bd, N) if layout == "row_blocks" else None
    g.build_histograms_segmented(Bd, N, gd, S, level(0, n_slots), n_slots, torch.from_numpy(flags).cuda(),
                                 int(flags.sum()), dev_struct(seg, g.SEGMENT_DTYPE), hc, hq, row_blocks=rb)
    ref = oracle.histograms(bins, gv.astype(np.float64), slot.astype(np.int32), n_slots)
    # A/B against the node-id kernel on the same rows: bit-identical integers
    dc, dq = g.build_histograms(Bd, N, gd, S, u16(slot.astype(np.uint16)), level(0, n_slots), n_slots,
                                torch.from_numpy(flags).cuda(), int(flags.sum()))
    hc_h, hq_h = hc.cpu().numpy().view(np.uint32), hq.cpu().numpy()
    for s in range(n_slots):
        if not flags[s]:
            assert np.all(hc_h[s] == sentinel) and np.all(hq_h[s] == sentinel)
            continue
        assert np.array_equal(hc_h[s], ref["cnt"][s]), f"slot {s}"
        m = slot == s
        A = np.stack([np.bincount(bins[f][m], weights=np.abs(gv[m].astype(np.float64)), minlength=256)
                      for f in range(F)])
        G = np.ldexp(hq_h[s].astype(np.float64), -s_exp)
        assert np.all(np.abs(G - ref["G"][s]) <= g_tolerance(A, ref["cnt"][s], s_exp)), f"slot {s}"
        assert torch.equal(hc[s], dc[s]) and torch.equal(hq[s], dq[s])


@pytest.mark.parametrize("layout", ["columns", "row_blocks"])
@pytest.mark.parametrize("N,F,n_slots,gdtype", [(180_001, 9, 6, np.float64), (120_003, 70, 4, np.float32),
                                                 (33, 3, 2, np.float64)])
def test_filtered_histograms_match_oracle(N, F, n_slots, gdtype, layout):
    """A slot whose rows still sit inside its parent's segment: the segment is the parent's and
    the filter keeps the rows on the slot's side of the parent's split."""
    rng = np.random.default_rng(3 * N + F)
    par, par_slot = _segments(rng, N, n_slots // 2)
    bins = rng.integers(0, 256, (F, N)).astype(np.uint8)
    bins[1] = rng.integers(0, 4, N).astype(np.uint8)  # coarse column: sides of very different sizes
    gv = rng.normal(0, 2, N).astype(gdtype)
    seg = np.zeros(n_slots, g.SEGMENT_DTYPE)
    filt = np.zeros(n_slots, g.FILTER_DTYPE)
    feats = rng.integers(0, F, n_slots // 2)
    thr = rng.integers(0, 255, n_slots // 2)
    feats[0], thr[0] = 1, 1
    slot = np.full(N, -1)
    for s in range(n_slots):
        k = s // 2
        seg[s] = par[k]
        filt[s] = (feats[k], thr[k], s & 1, 0)
        if s == n_slots - 1 and n_slots > 2:
            filt[s]["feature"] = -1  # no filter: every row of the segment
    flags = np.zeros(n_slots, np.uint8)
    flags[0::2] = 1
    flags[n_slots - 1] = 1
    S = g.gradient_scale(torch.from_numpy(gv).cuda())
    s_exp = int(S.item())
    Bd = dev_bins(bins)
    rb = g.to_row_blocks(Bd, N) if layout == "row_blocks" else None
    hc, hq = g.build_histograms_segmented(Bd, N, torch.from_numpy(gv).cuda(), S, level(0, n_slots),
                                          n_slots, torch.from_numpy(flags).cuda(), int(flags.sum()),
                                          dev_struct(seg, g.SEGMENT_DTYPE), filters=dev_struct(filt, g.FILTER_DTYPE),
                                          row_blocks=rb)
    hc_h, hq_h = hc.cpu().numpy().view(np.uint32), hq.cpu().numpy()
    for s in range(n_slots):
        if not flags[s]:
            continue
        a, c = seg["start"][s], seg["count"][s]
        rows = np.arange(a, a + c)
        if filt["feature"][s] >= 0:
            right = bins[filt["feature"][s], rows] > filt["bin"][s]
            rows = rows[right == bool(filt["side"][s])]
        m = np.zeros(N, np.int32) - 1
        m[rows] = 0
        ref = oracle.histograms(bins, gv.astype(np.float64), m, 1)
        assert np.array_equal(hc_h[s], ref["cnt"][0]), f"slot {s}"
        A = np.stack([np.bincount(bins[f][rows], weights=np.abs(gv[rows].astype(np.float64)), minlength=256)
                      for f in range(F)])
        G = np.ldexp(hq_h[s].astype(np.float64), -s_exp)
        assert np.all(np.abs(G - ref["G"][0]) <= g_tolerance(A, ref["cnt"][0], s_exp)), f"slot {s}"


@pytest.mark.parametrize("N,F,n_slots,gdtype,explicit", [(300_007, 9, 6, np.float64, False),
                                                          (100_003, 35, 11, np.float32, False),
                                                          (65_536, 3, 2, np.float64, True),
                                                          (9, 2, 3, np.float64, False)])
def test_partition_rows_matches_oracle(N, F, n_slots, gdtype, explicit):
    rng = np.random.default_rng(7 * N + F)
    seg, slot = _segments(rng, N, n_slots, empty=(n_slots - 1,) if n_slots > 2 else ())
    bins = rng.integers(0, 256, (F, N)).astype(np.uint8)
    gv = rng.normal(size=N).astype(gdtype)
    orig = rng.permutation(N).astype(np.uint32)
    feats = rng.integers(0, F, n_slots)
    thr = rng.integers(0, 255, n_slots)
    feats[1] = -1  # a slot that does not split: its rows are recorded as a leaf
    thr[1] = -1
    go_right = (rng.random(N) < 0.4).astype(np.uint8) if explicit else None
    sp = np.zeros(n_slots, g.SPLIT_DTYPE)
    sp["feature"], sp["bin"], sp["cnt_total"] = feats, thr, seg["count"]
    decide = (go_right != 0) if explicit else None
    for s in range(n_slots):
        if feats[s] < 0:
            continue
        pos = np.arange(seg["start"][s], seg["start"][s] + seg["count"][s])
        right = decide[pos] if explicit else bins[feats[s], pos] > thr[s]
        sp["cnt_left"][s] = int((~right).sum())
    node_begin = 3
    leaf = torch.full((N,), -1, dtype=torch.int16, device="cuda")  # 0xffff
    Bd = dev_bins(bins)
    bo, go, oo, seg_out, nxt = g.partition_rows(
        Bd, N, torch.from_numpy(gv).cuda(), torch.from_numpy(orig.view(np.int32)).cuda(),
        dev_struct(sp, g.SPLIT_DTYPE), level(node_begin, n_slots), n_slots, dev_struct(seg, g.SEGMENT_DTYPE),
        go_right=torch.from_numpy(go_right).cuda() if explicit else None, leaf_of_row=leaf)
    bo = bo.cpu().numpy()[:, :N]
    go = go.cpu().numpy()
    oo = oo.cpu().numpy().view(np.uint32)
    # oracle: stable partition of the position lists (positions are the row indices here)
    if explicit:  # express the explicit decision as a one-column split on a 0/1 column
        dec_bins = np.vstack([bins, go_right[None, :]])
        of, ob = np.where(feats >= 0, F, -1), np.where(feats >= 0, 0, -1)
        ref_idx, ref_left = oracle.partition(dec_bins, of, ob, seg["start"], seg["count"], np.arange(N))
    else:
        ref_idx, ref_left = oracle.partition(bins, feats, thr, seg["start"], seg["count"], np.arange(N))
    so = host_struct(seg_out, g.SEGMENT_DTYPE, 2 * n_slots)
    nl = host_struct(nxt, g.LEVEL_DTYPE, 1)[0]
    splitting = [s for s in range(n_slots) if feats[s] >= 0]
    assert (nl["node_begin"], nl["n_slots"]) == (node_begin + n_slots, 2 * len(splitting))
    leaf_h = leaf.cpu().numpy().view(np.uint16)
    for k, s in enumerate(splitting):
        a, c = seg["start"][s], seg["count"][s]
        order = ref_idx[a:a + c]
        assert np.array_equal(bo[:, a:a + c], bins[:, order]), f"slot {s}: bins"
        assert np.array_equal(go[a:a + c], gv[order]), f"slot {s}: g"
        assert np.array_equal(oo[a:a + c], orig[order]), f"slot {s}: orig"
        assert (so["start"][2 * k], so["count"][2 * k]) == (a, ref_left[s])
        assert (so["start"][2 * k + 1], so["count"][2 * k + 1]) == (a + ref_left[s], c - ref_left[s])
    for s in range(n_slots):
        rows = orig[seg["start"][s]:seg["start"][s] + seg["count"][s]]
        want = node_begin + s if feats[s] < 0 else 65535
        assert np.all(leaf_h[rows] == want)

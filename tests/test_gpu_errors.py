"""Device consistency checks of the per-step calls reach the caller ("Module Design: Training Core"
s.5, the Failed state).

Each call that takes a workspace keeps its device error word in the workspace's first 4 bytes;
gbdt_workspace_status reads it back (gbdt_partition_noalloc_status for the call with built-in
scratch).  Every case gives a call an input that is inconsistent but safe on the device -- a split
record whose cnt_left is wrong (the kernels still place rows by the counts they compute, inside the
slot's segment), histograms whose features disagree on a node's totals, a built child larger than
its parent, a level larger than its bound -- and checks that the status names it, and that the
next consistent call on the same workspace reads clean.
"""
import numpy as np
import pytest

from tests.gpu_util import dev_bins, dev_struct, g, level, needs_gpu, torch, u16

pytestmark = [pytest.mark.gpu, needs_gpu]

ERR_HIST_TOTALS, ERR_PARTITION_COUNT, ERR_LEVEL_SIZE = 1, 4, 8


def _partition_case(seed, N=50_000, F=3, n_slots=6, node_begin=3, wrong_slot=None):
    rng = np.random.default_rng(seed)
    bins = rng.integers(0, 256, (F, N)).astype(np.uint8)
    slot = rng.integers(0, n_slots, N)
    order = np.argsort(slot, kind="stable")
    counts = np.bincount(slot, minlength=n_slots)
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    feats = rng.integers(0, F, n_slots)
    thr = rng.integers(0, 255, n_slots)
    cnt_left = np.array([(bins[feats[s], order[starts[s]:starts[s] + counts[s]]] <= thr[s]).sum()
                         for s in range(n_slots)])
    if wrong_slot is not None:
        cnt_left[wrong_slot] += 1  # the record disagrees with the rows by one
    sp = np.zeros(n_slots, g.SPLIT_DTYPE)
    sp["feature"], sp["bin"], sp["cnt_left"], sp["cnt_total"] = feats, thr, cnt_left, counts
    seg = np.zeros(n_slots, g.SEGMENT_DTYPE)
    seg["start"], seg["count"] = starts, counts
    return dict(bins=dev_bins(bins), N=N, splits=dev_struct(sp, g.SPLIT_DTYPE), level=level(node_begin, n_slots),
                max_slots=n_slots, seg=dev_struct(seg, g.SEGMENT_DTYPE),
                idx=torch.from_numpy(order.astype(np.int32)).cuda(), node=u16(node_begin + slot))


def _status(ws):
    try:
        return g.workspace_status(ws)
    except g.GbdtError as e:
        assert e.code == g.ERR_INTERNAL
        assert "error bits" in str(e)
        bits = int(str(e).split("error bits 0x")[1].split(":")[0], 16)
        return bits


def test_partition_reports_a_split_record_that_disagrees_with_the_rows():
    c = _partition_case(1, wrong_slot=2)
    ws = g._workspace(g.lib().gbdt_partition_workspace_size(c["N"], c["max_slots"]))
    g.partition(c["bins"], c["N"], c["splits"], c["level"], c["max_slots"], c["seg"], c["idx"], c["node"], ws=ws)
    assert _status(ws) == ERR_PARTITION_COUNT
    ok = _partition_case(1)
    g.partition(ok["bins"], ok["N"], ok["splits"], ok["level"], ok["max_slots"], ok["seg"], ok["idx"], ok["node"],
                ws=ws)
    assert _status(ws) == 0  # the call clears the word it queues with


def test_partition_rows_reports_a_split_record_that_disagrees_with_the_rows():
    c = _partition_case(2, wrong_slot=0)
    bins_pos = c["bins"][:, :]  # rows at positions: take the column layout in the slot order
    order = c["idx"].long()
    pb = torch.zeros_like(bins_pos)
    pb[:, :c["N"]] = bins_pos[:, order]
    gd = torch.randn(c["N"], dtype=torch.float64, device="cuda")
    orig = c["idx"].clone()
    ws = g._workspace(g.lib().gbdt_partition_rows_workspace_size(c["N"], c["max_slots"]))
    g.partition_rows(pb, c["N"], gd, orig, c["splits"], c["level"], c["max_slots"], c["seg"], ws=ws)
    assert _status(ws) == ERR_PARTITION_COUNT


def test_find_splits_reports_features_that_disagree_on_node_totals():
    F, slots = 3, 2
    hc = torch.zeros((slots, F, 256), dtype=torch.int32, device="cuda")
    hq = torch.zeros((slots, F, 256), dtype=torch.int64, device="cuda")
    hc[:, :, 0], hc[:, :, 1] = 10, 10
    hq[:, :, 0], hq[:, :, 1] = -(1 << 30), 1 << 30
    n_bins = torch.full((F,), 256, dtype=torch.int32, device="cuda")
    S = torch.tensor([30], dtype=torch.int32, device="cuda")
    ws = g._workspace(g.lib().gbdt_find_splits_workspace_size(F, slots))
    g.find_splits(hc, hq, S, n_bins, level(1, slots), slots, ws=ws)
    assert _status(ws) == 0
    hc[1, 2, 1] = 9  # feature 2 of slot 1 holds one row fewer than feature 0
    g.find_splits(hc, hq, S, n_bins, level(1, slots), slots, ws=ws)
    assert _status(ws) == ERR_HIST_TOTALS


def test_subtract_reports_a_built_child_larger_than_its_parent():
    F = 2
    pc = torch.full((1, F, 256), 5, dtype=torch.int32, device="cuda")
    pq = torch.zeros((1, F, 256), dtype=torch.int64, device="cuda")
    hc = torch.full((2, F, 256), 3, dtype=torch.int32, device="cuda")
    hq = torch.zeros((2, F, 256), dtype=torch.int64, device="cuda")
    flags = torch.tensor([1, 0], dtype=torch.uint8, device="cuda")
    pair_parent = torch.zeros(1, dtype=torch.int32, device="cuda")
    ws = g._workspace(g.lib().gbdt_subtract_histograms_workspace_size())
    g.subtract_histograms(pc, pq, pair_parent, flags, level(1, 2), 2, hc, hq, ws=ws)
    assert _status(ws) == 0
    assert int(hc[1, 0, 0]) == 2
    hc[0, 1, 7] = 6  # built child above its parent's 5
    g.subtract_histograms(pc, pq, pair_parent, flags, level(1, 2), 2, hc, hq, ws=ws)
    assert _status(ws) == ERR_HIST_TOTALS


def test_build_histograms_reports_a_level_larger_than_its_bound():
    rng = np.random.default_rng(3)
    N, F = 4096, 2
    bins = dev_bins(rng.integers(0, 256, (F, N)).astype(np.uint8))
    gv = torch.from_numpy(rng.normal(size=N)).cuda()
    S = g.gradient_scale(gv)
    node = u16(rng.integers(0, 8, N))
    flags = torch.ones(8, dtype=torch.uint8, device="cuda")
    ws = g._workspace(g.lib().gbdt_histograms_workspace_size(N, F, 4))
    g.build_histograms(bins, N, gv, S, node, level(0, 4), 4, flags, 4, ws=ws)
    assert _status(ws) == 0
    g.build_histograms(bins, N, gv, S, node, level(0, 8), 4, flags, 4, ws=ws)  # 8 slots, bound 4
    assert _status(ws) == ERR_LEVEL_SIZE


def test_status_of_calls_without_checks_reads_clean():
    gv = torch.randn(1000, dtype=torch.float64, device="cuda")
    ws = g._workspace(g.lib().gbdt_gradients_workspace_size(1000))
    ws.fill_(0xFF)  # whatever the workspace held, the call clears its error word
    S = torch.empty(1, dtype=torch.int32, device="cuda")
    import ctypes

    g._check(g.lib().gbdt_gradient_scale(g._ptr(gv), g.DTYPE_F64, 1000, g._ptr(S), g._ptr(ws), ws.numel(),
                                         g._stream()))
    assert g.workspace_status(ws) == 0
    assert ctypes.sizeof(ctypes.c_int32) == 4

"""gbdt_partition_noalloc: the partition for callers that cannot allocate device memory.

Some callers (code living inside another framework's fixed memory pool, plugins
without access to the host's allocator, loops where a cudaMalloc could stall the
device) cannot hand the library a workspace.  This entry point keeps its
scratch in a fixed array inside the library instead.  These tests call it
through the C ABI and check that it gives exactly what gbdt_partition (with a
caller workspace) gives, on two calls in a row -- the second call meets the
first call's leftovers in the shared array -- and that sizes beyond its limits
are refused before anything runs.  The file sorts last so that a run stopping
at the first failure has run every other test before it.
"""
import ctypes

import numpy as np
import pytest

from tests.gpu_util import dev_bins, dev_struct, g, host_struct, level, needs_gpu, oracle, torch, u16

pytestmark = [pytest.mark.gpu, needs_gpu]


def _case(seed, N, F, n_slots, node_begin, wrong_slot=None):
    rng = np.random.default_rng(seed)
    bins = rng.integers(0, 256, (F, N)).astype(np.uint8)
    slot = rng.integers(0, n_slots, N)
    order = np.argsort(slot, kind="stable")
    counts = np.bincount(slot, minlength=n_slots)
    starts = np.concatenate([[0], np.cumsum(counts)[:-1]])
    feats = rng.integers(-1, F, n_slots)  # -1: the slot does not split
    thr = rng.integers(0, 256, n_slots)
    thr[feats < 0] = -1
    cnt_left = np.array([(bins[feats[s], order[starts[s]:starts[s] + counts[s]]] <= thr[s]).sum() if feats[s] >= 0
                         else 0 for s in range(n_slots)])
    if wrong_slot is not None:
        cnt_left[wrong_slot] += 1  # a record that disagrees with its rows (safe: rows go where they are counted)
    sp = np.zeros(n_slots, g.SPLIT_DTYPE)
    sp["feature"], sp["bin"], sp["cnt_left"], sp["cnt_total"] = feats, thr, cnt_left, counts
    seg = np.zeros(n_slots, g.SEGMENT_DTYPE)
    seg["start"], seg["count"] = starts, counts
    node = (node_begin + slot).astype(np.uint16)
    return dict(bins=dev_bins(bins), N=N, splits=dev_struct(sp, g.SPLIT_DTYPE), level=level(node_begin, n_slots),
                max_slots=n_slots, seg=dev_struct(seg, g.SEGMENT_DTYPE),
                idx=torch.from_numpy(order.astype(np.int32)).cuda(), node=node,
                host=dict(bins=bins, feats=feats, thr=thr, starts=starts, counts=counts, order=order,
                          node_begin=node_begin))


def _run(fn, c):
    node_d = u16(c["node"])
    idx_out, seg_out, nxt = fn(c["bins"], c["N"], c["splits"], c["level"], c["max_slots"], c["seg"], c["idx"], node_d)
    torch.cuda.synchronize()
    return (idx_out.cpu().numpy(), host_struct(seg_out, g.SEGMENT_DTYPE, 2 * c["max_slots"]),
            host_struct(nxt, g.LEVEL_DTYPE, 1), node_d.cpu().numpy())


def test_noalloc_partition_matches_workspace_partition_twice():
    # two different cases back to back: the second runs on scratch the first one filled
    for c in (_case(1, 250_003, 6, 37, 40), _case(2, 90_001, 3, 5, 3)):
        want = _run(g.partition, c)
        got = _run(g.partition_noalloc, c)
        for a, b in zip(got, want):  # index work: bit-exact
            assert np.array_equal(a, b)


def _oracle_expectation(c):
    """The oracle's partition of the case (its own restatement of the stable partition), and from it the
    children's segments and node ids: the k-th splitting slot's children are next_begin + 2k, + 2k + 1."""
    h = c["host"]
    n_slots = len(h["counts"])
    out, left = oracle.partition(h["bins"], h["feats"], h["thr"], h["starts"], h["counts"], h["order"])
    seg = np.zeros(2 * n_slots, g.SEGMENT_DTYPE)
    node = c["node"].copy()
    next_begin = h["node_begin"] + n_slots
    k = 0
    for s in range(n_slots):
        if h["feats"][s] < 0:
            continue
        st, n, nl = h["starts"][s], h["counts"][s], left[s]
        seg[2 * k], seg[2 * k + 1] = (st, nl), (st + nl, n - nl)
        node[out[st:st + nl]] = next_begin + 2 * k
        node[out[st + nl:st + n]] = next_begin + 2 * k + 1
        k += 1
    return out.astype(np.int32), seg[:2 * k], node, np.array([(next_begin, 2 * k)], g.LEVEL_DTYPE)


def test_noalloc_partition_matches_the_oracle_twice():
    for c in (_case(4, 120_007, 5, 29, 20), _case(5, 70_001, 2, 3, 1)):
        idx, seg, nxt, node = _run(g.partition_noalloc, c)
        want_idx, want_seg, want_node, want_next = _oracle_expectation(c)
        assert np.array_equal(idx, want_idx)
        assert np.array_equal(seg[:len(want_seg)], want_seg)
        assert np.array_equal(node.view(np.uint16), want_node)
        assert np.array_equal(nxt, want_next)
        assert g.partition_noalloc_status() == 0


def test_noalloc_partition_reports_a_record_that_disagrees_with_its_rows():
    _run(g.partition_noalloc, _case(6, 40_000, 3, 9, 5, wrong_slot=4))
    with pytest.raises(g.GbdtError) as e:
        g.partition_noalloc_status()
    assert e.value.code == g.ERR_INTERNAL and "partition count" in str(e.value)
    _run(g.partition_noalloc, _case(6, 40_000, 3, 9, 5))  # the next call clears the word
    assert g.partition_noalloc_status() == 0


def test_noalloc_partition_rejects_sizes_beyond_its_scratch():
    L = g.lib()
    c = _case(3, 1000, 2, 4, 0)
    args = [ctypes.c_void_p(c["bins"].data_ptr()), c["bins"].shape[1], None, 2, ctypes.c_void_p(c["splits"].data_ptr()),
            ctypes.c_void_p(c["level"].data_ptr()), None, ctypes.c_void_p(c["seg"].data_ptr()),
            ctypes.c_void_p(c["idx"].data_ptr()), ctypes.c_void_p(u16(c["node"]).data_ptr()),
            ctypes.c_void_p(torch.zeros_like(c["idx"]).data_ptr()),
            ctypes.c_void_p(torch.zeros(4096, dtype=torch.uint8, device="cuda").data_ptr()),
            ctypes.c_void_p(torch.zeros(8, dtype=torch.uint8, device="cuda").data_ptr()), None]
    big_n = (1 << 24) + 1
    too_many_rows = list(args)
    too_many_rows[1], too_many_rows[2], too_many_rows[6] = big_n + 15, big_n, 4
    assert L.gbdt_partition_noalloc(*too_many_rows) == g.ERR_INVALID_ARG
    assert b"16777216" in L.gbdt_last_error()
    too_many_slots = list(args)
    too_many_slots[2], too_many_slots[6] = 1000, 1025
    assert L.gbdt_partition_noalloc(*too_many_slots) == g.ERR_INVALID_ARG
    assert b"1024" in L.gbdt_last_error()

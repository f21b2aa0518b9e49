"""The C-ABI library builds, loads and exports every entry point include/gbdt.h declares
(no compute calls: these run without a GPU)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    src = open(os.path.join(ROOT, "include", "gbdt.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(gbdt_[a-z_0-9]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import histogram_gradient_boosted_gb300 as g
    from histogram_gradient_boosted_gb300 import build

    build.build()
    return g.lib()


def test_header_declares_the_entry_points():
    names = _declared()
    for required in ("gbdt_quantize", "gbdt_compute_gradients", "gbdt_build_histograms", "gbdt_find_splits",
                     "gbdt_partition", "gbdt_update_predictions", "gbdt_train"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), f"{name} declared in gbdt.h but not exported"


def test_binding_covers_every_declared_symbol():
    import histogram_gradient_boosted_gb300 as g

    assert sorted(g.EXPORTED_SYMBOLS) == _declared()


def test_version_and_workspace_queries_without_gpu(lib):
    import histogram_gradient_boosted_gb300 as g

    assert b"sm_103a" in lib.gbdt_version()
    p = g.make_params(n_trees=10, max_depth=8)
    n = lib.gbdt_train_workspace_size(10_000_000, 100, ctypes.byref(p))
    # g (8 B/row) + node ids (2 B/row) + two histogram buffers of 128 slots x 100 x 256 x 12 B
    assert n >= 10_000_000 * 10 + 2 * 128 * 100 * 256 * 12
    assert lib.gbdt_quantize_workspace_size(1000, 4) >= 2 * 4 * 1000 * 4
    assert lib.gbdt_partition_workspace_size(1000, 8) > 0
    bad = g.make_params(max_depth=13)
    assert lib.gbdt_train_workspace_size(100, 1, ctypes.byref(bad)) == 0


def test_parameter_rules_on_host(lib):
    import histogram_gradient_boosted_gb300 as g

    assert g.validate_params(n_trees=1, max_depth=3) == g.OK
    for bad in (dict(min_samples_leaf=0), dict(min_child_weight=-1.0), dict(reg_lambda=-0.1), dict(gamma=-1.0),
                dict(learning_rate=float("nan")), dict(reg_lambda=float("inf")), dict(max_depth=13),
                dict(n_trees=-1), dict(objective=2), dict(objective=-1), dict(num_leaves=1),
                dict(bin_packing=2)):
        assert g.validate_params(**bad) == g.ERR_INVALID_ARG, bad
        assert lib.gbdt_last_error() != b""
    assert g.validate_params(objective=g.OBJECTIVE_LOGISTIC) == g.OK


def test_struct_layouts_match_header():
    import histogram_gradient_boosted_gb300 as g

    assert ctypes.sizeof(g.Params) == 64 and g.Params.objective.offset == 52 and g.Params.bin_packing.offset == 56
    assert g.NODE_DTYPE.itemsize == 40 and g.SPLIT_DTYPE.itemsize == 56
    assert g.SPLIT_DTYPE.fields["h_left"][1] == 40 and g.SPLIT_DTYPE.fields["h_total"][1] == 48
    assert g.LEVEL_DTYPE.itemsize == 8 and g.SEGMENT_DTYPE.itemsize == 16
    assert ctypes.sizeof(g.Diagnostics) == 80


def test_entry_points_reject_bad_arguments_before_any_launch(lib):
    # null pointers are caught on the host, so no GPU is touched
    assert lib.gbdt_quantize(None, 0, 0, 0, 0, None, 0, None, None, None, 0, None) == -1
    assert lib.gbdt_train(None, 0, None, 0, 0, None, None, None, None, None, None, None, None, 0, None) == -1
    assert lib.gbdt_build_histograms(None, 0, 0, 0, None, 0, None, None, None, 0, None, 0, None, None, None, 0,
                                     None) == -1
    assert b"null pointer" in lib.gbdt_last_error()
    assert lib.gbdt_build_histograms_segmented_h(None, 0, 0, 0, 0, None, 0, None, None, 0, None, 0, None, None, None,
                                                 None, None, None, 0, None) == -1
    assert lib.gbdt_find_splits_h(None, None, None, None, 0, None, None, 0, None, None, None, 0, None) == -1
    assert lib.gbdt_subtract_histograms_h(None, None, None, None, None, None, 0, 0, None, None, None, None, 0,
                                          None) == -1
    assert lib.gbdt_compute_gradients_objective(None, None, 0, 1, None, None, None, 0, None) == -1
    assert b"null pointer" in lib.gbdt_last_error()
    # the status query needs a workspace pointer (checked before any copy)
    assert lib.gbdt_workspace_status(None, None, None) == -1
    assert b"workspace" in lib.gbdt_last_error()


def test_noalloc_scratch_covers_its_limits(lib):
    """gbdt_partition_noalloc's built-in scratch (128 KiB) must hold the partition's carve at its documented
    limits (16,777,216 rows, 1,024 slots); the carve is the workspace gbdt_partition asks for."""
    need = lib.gbdt_partition_workspace_size(1 << 24, 1024)
    assert 0 < need <= 128 * 1024, need


def test_error_word_leads_every_asynchronous_workspace(lib):
    """Each asynchronous call's workspace starts with its 4-byte error word: the sizes leave room for it."""
    assert lib.gbdt_subtract_histograms_workspace_size() >= 4
    assert lib.gbdt_gradients_workspace_size(10) >= 256 + 16
    assert lib.gbdt_histograms_segmented_workspace_size(8) >= 256 + 8 * 12
    assert lib.gbdt_find_splits_workspace_size(4, 8) >= 256


def test_row_block_slot_plan_on_host(lib):
    """4-bit slots: features with <= 16 bins pair up in feature order (low nibble first), an unpaired
    one keeps a whole byte, the rest have slots of their own, numbered by their first feature."""
    import numpy as np

    import histogram_gradient_boosted_gb300 as g

    nb = [256, 16, 3, 17, 2, 255, 16, 2, 9]
    loc, src = g.row_block_slots(nb)
    slot, nib = loc & 0xFFFF, loc >> 16
    # slots: 0 <- f0; 1 <- f1 (low) + f2 (high); 2 <- f3; 3 <- f4 (low) + f6 (high); 4 <- f5;
    #        5 <- f7 (low) + f8 (high)
    assert list(slot) == [0, 1, 1, 2, 3, 4, 3, 5, 5] and list(nib) == [0, 1, 2, 0, 1, 0, 2, 1, 2]
    assert list(src & 0xFFFF) == [0, 1, 3, 4, 5, 7] and list(src >> 16) == [0xFFFF, 2, 0xFFFF, 6, 0xFFFF, 8]
    loc, src = g.row_block_slots([2, 2, 2])  # an odd count: the last one keeps a whole byte
    assert list(loc & 0xFFFF) == [0, 0, 1] and list(loc >> 16) == [1, 2, 0] and len(src) == 2
    loc, src = g.row_block_slots(nb, packing=g.BIN_PACKING_OFF)
    assert list(loc) == list(range(len(nb))) and list(src) == [f | 0xFFFF0000 for f in range(len(nb))]
    # every feature is stored exactly once
    rng = np.random.default_rng(0)
    for _ in range(20):
        nb = rng.choice([2, 5, 16, 17, 200, 256], size=rng.integers(1, 300))
        loc, src = g.row_block_slots(nb)
        seen = sorted([int(s & 0xFFFF) for s in src] + [int(s >> 16) for s in src if s >> 16 != 0xFFFF])
        assert seen == list(range(len(nb)))
        assert all((l >> 16) == 0 or nb[i] <= 16 for i, l in enumerate(loc))
        assert len(src) == len(nb) - sum(1 for s in src if s >> 16 != 0xFFFF)
    with pytest.raises(g.GbdtError):
        g.row_block_slots([0, 3])


def test_register_slot_plan_on_host(lib):
    """With register slots the features of at most 8 bins follow the ordinary plan, in feature order, two to a
    slot (low nibble first) when their bin counts multiply to at most 8, else one to a whole byte."""
    import numpy as np

    import histogram_gradient_boosted_gb300 as g

    nb = [2, 3, 200, 16, 17, 5, 2, 256, 9, 16, 4, 7, 3, 2]
    loc, src, rb = g.row_block_slots_ex(nb)
    slot, nib = loc & 0xFFFF, loc >> 16
    # ordinary: f2 (whole), f3 + f8 (4-bit pair: 16 and 9 bins), f4, f7, f9 (16 bins, unpaired: whole byte)
    assert rb == 5 and list(src[:rb] & 0xFFFF) == [2, 3, 4, 7, 9]
    assert list(src[1:2] >> 16) == [8] and slot[8] == 1 and nib[8] == 2 and nib[3] == 1
    # register: (f0, f1) 2 x 3 = 6; f5 alone (5 x 2 > 8); (f6, f10) 2 x 4 = 8; f11 alone (7 x 3); (f12, f13) 3 x 2
    reg = [(int(s & 0xFFFF), int(s >> 16)) for s in src[rb:]]
    assert reg == [(0, 1), (5, 0xFFFF), (6, 10), (11, 0xFFFF), (12, 13)]
    for a, b in reg:
        assert (b == 0xFFFF and nb[a] <= 8) or nb[a] * nb[b] <= 8
    # every feature exactly once; without registers the plan is gbdt_row_block_slots'
    seen = sorted([int(s & 0xFFFF) for s in src] + [int(s >> 16) for s in src if s >> 16 != 0xFFFF])
    assert seen == list(range(len(nb)))
    l0, s0, rb0 = g.row_block_slots_ex(nb, hist_registers=g.HIST_REGISTERS_OFF)
    l1, s1 = g.row_block_slots(nb)
    assert rb0 == len(s0) and np.array_equal(l0, l1) and np.array_equal(s0, s1)
    # packing off: register features keep whole bytes
    _, s2, rb2 = g.row_block_slots_ex(nb, packing=g.BIN_PACKING_OFF)
    assert all(s >> 16 == 0xFFFF for s in s2) and len(s2) == len(nb) and rb2 == 6

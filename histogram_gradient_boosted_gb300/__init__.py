"""Python binding of libgbdt.so, the GB300 (sm_103a) level-wise histogram GBDT library.

Argument marshalling only: every step runs in the library's CUDA kernels; the
functions here turn torch CUDA tensors into device pointers, allocate the
caller-side workspace the C ABI asks for, pass the current CUDA stream, and
raise ``GbdtError`` on a non-zero status.  There is no CPU path: without a
CUDA device or without the built library every call raises.

The C declarations, with their argument meaning, layout and error behaviour,
are in ``include/gbdt.h``; names here match them without the ``gbdt_`` prefix
(the raw symbols are reachable through ``lib()``).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

__all__ = ["lib", "GbdtError", "Params", "NODE_DTYPE", "SPLIT_DTYPE", "LEVEL_DTYPE", "SEGMENT_DTYPE",
           "Diagnostics", "quantize", "train", "compute_gradients", "gradient_scale", "build_histograms",
           "subtract_histograms", "find_splits", "partition", "update_predictions", "padded_ld",
           "EXPORTED_SYMBOLS"]

OK, ERR_INVALID_ARG, ERR_NONFINITE, ERR_WORKSPACE, ERR_CUDA, ERR_INTERNAL = 0, -1, -2, -3, -4, -5
DTYPE_F32, DTYPE_F64 = 0, 1
OBJECTIVE_SQUARED_ERROR, OBJECTIVE_LOGISTIC = 0, 1
BIN_PACKING_4BIT, BIN_PACKING_OFF = 0, 1
HIST_REGISTERS_OFF, HIST_REGISTERS_ON = 0, 1
LAYOUT_COLUMNS, LAYOUT_ROW_BLOCKS = 0, 1
MAX_BINS, MAX_DEPTH = 256, 12

EXPORTED_SYMBOLS = [
    "gbdt_last_error", "gbdt_version", "gbdt_validate_params", "gbdt_quantize_workspace_size", "gbdt_quantize",
    "gbdt_gradients_workspace_size", "gbdt_compute_gradients", "gbdt_gradient_scale",
    "gbdt_histograms_workspace_size", "gbdt_build_histograms", "gbdt_subtract_histograms", "gbdt_find_splits",
    "gbdt_find_splits_workspace_size",
    "gbdt_partition_workspace_size", "gbdt_partition", "gbdt_update_predictions", "gbdt_train_workspace_size",
    "gbdt_train", "gbdt_debug_inject_failure", "gbdt_kernel_launch_count", "gbdt_partition_noalloc",
    "gbdt_histograms_segmented_workspace_size", "gbdt_build_histograms_segmented", "gbdt_partition_rows_workspace_size",
    "gbdt_partition_rows", "gbdt_predict_workspace_size", "gbdt_predict", "gbdt_row_block_pitch",
    "gbdt_row_block_bytes", "gbdt_bins_to_row_blocks", "gbdt_compute_gradients_objective",
    "gbdt_subtract_histograms_h", "gbdt_build_histograms_segmented_h", "gbdt_find_splits_h", "gbdt_row_block_slots",
    "gbdt_workspace_status", "gbdt_partition_noalloc_status", "gbdt_subtract_histograms_workspace_size",
    "gbdt_row_block_slots_ex", "gbdt_quantize_host",
]


class GbdtError(RuntimeError):
    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


class Params(ctypes.Structure):
    _fields_ = [("n_trees", ctypes.c_int32), ("max_depth", ctypes.c_int32), ("learning_rate", ctypes.c_double),
                ("reg_lambda", ctypes.c_double), ("gamma", ctypes.c_double), ("min_samples_leaf", ctypes.c_int32),
                ("min_child_weight", ctypes.c_double), ("num_leaves", ctypes.c_int32), ("objective", ctypes.c_int32),
                ("bin_packing", ctypes.c_int32), ("hist_registers", ctypes.c_int32)]


class Diagnostics(ctypes.Structure):
    _fields_ = [("hist_launches", ctypes.c_int64), ("hist_ms", ctypes.c_double), ("hist_bytes", ctypes.c_double),
                ("hist_rows", ctypes.c_int64), ("part_ms", ctypes.c_double), ("part_bytes", ctypes.c_double),
                ("total_ms", ctypes.c_double), ("kernel_launches", ctypes.c_int64),
                ("trees_at_full_size", ctypes.c_int32), ("reserved", ctypes.c_int32),
                ("hist_level_bytes", ctypes.c_double)]

    def as_dict(self):
        return {k: getattr(self, k) for k, _ in self._fields_ if k != "reserved"}


NODE_DTYPE = np.dtype([("feature", np.int32), ("threshold_bin", np.int32), ("left", np.int32), ("right", np.int32),
                       ("leaf_value", np.float64), ("gain", np.float64), ("is_leaf", np.uint8),
                       ("reserved", np.uint8, (7,))])
SPLIT_DTYPE = np.dtype([("feature", np.int32), ("bin", np.int32), ("gain", np.float64), ("q_left", np.int64),
                        ("q_total", np.int64), ("cnt_left", np.uint32), ("cnt_total", np.uint32),
                        ("h_left", np.int64), ("h_total", np.int64)])
LEVEL_DTYPE = np.dtype([("node_begin", np.int32), ("n_slots", np.int32)])
SEGMENT_DTYPE = np.dtype([("start", np.int64), ("count", np.int64)])
FILTER_DTYPE = np.dtype([("feature", np.int32), ("bin", np.int32), ("side", np.int32), ("reserved", np.int32)])
assert NODE_DTYPE.itemsize == 40 and SPLIT_DTYPE.itemsize == 56

_lib = None


def lib():
    """Load (building first if needed) libgbdt.so and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB if os.path.exists(_build.LIB) else _build.build()
    L = ctypes.CDLL(path)
    P, i32, i64, sz, dbl = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t, ctypes.c_double
    sig = {
        "gbdt_last_error": ([], ctypes.c_char_p),
        "gbdt_version": ([], ctypes.c_char_p),
        "gbdt_validate_params": ([P], i32),
        "gbdt_quantize_workspace_size": ([i64, i32], sz),
        "gbdt_quantize": ([P, i64, i64, i32, i32, P, i64, P, P, P, sz, P], i32),
        "gbdt_quantize_host": ([P, i64, i64, i32, i32, P, P, i64, P, P, P, sz, P], i32),
        "gbdt_gradients_workspace_size": ([i64], sz),
        "gbdt_compute_gradients": ([P, P, i64, P, P, P, sz, P], i32),
        "gbdt_compute_gradients_objective": ([P, P, i64, i32, P, P, P, sz, P], i32),
        "gbdt_gradient_scale": ([P, i32, i64, P, P, sz, P], i32),
        "gbdt_histograms_workspace_size": ([i64, i32, i32], sz),
        "gbdt_build_histograms": ([P, i64, i64, i32, P, i32, P, P, P, i32, P, i32, P, P, P, sz, P], i32),
        "gbdt_subtract_histograms_workspace_size": ([], sz),
        "gbdt_subtract_histograms": ([P, P, P, P, P, i32, i32, P, P, P, sz, P], i32),
        "gbdt_subtract_histograms_h": ([P, P, P, P, P, P, i32, i32, P, P, P, P, sz, P], i32),
        "gbdt_workspace_status": ([P, P, P], i32),
        "gbdt_partition_noalloc_status": ([P, P], i32),
        "gbdt_find_splits_workspace_size": ([i32, i32], sz),
        "gbdt_find_splits": ([P, P, P, i32, P, P, i32, P, P, P, sz, P], i32),
        "gbdt_find_splits_h": ([P, P, P, P, i32, P, P, i32, P, P, P, sz, P], i32),
        "gbdt_partition_workspace_size": ([i64, i32], sz),
        "gbdt_partition": ([P, i64, i64, i32, P, P, i32, P, P, P, P, P, P, P, sz, P], i32),
        "gbdt_update_predictions": ([P, P, P, i32, i64, dbl, P], i32),
        "gbdt_train_workspace_size": ([i64, i32, P], sz),
        "gbdt_train": ([P, i64, P, i64, i32, P, P, P, P, P, P, P, P, sz, P], i32),
        "gbdt_debug_inject_failure": ([i32], None),
        "gbdt_kernel_launch_count": ([], i64),
        "gbdt_partition_noalloc": ([P, i64, i64, i32, P, P, i32, P, P, P, P, P, P, P], i32),
        "gbdt_histograms_segmented_workspace_size": ([i32], sz),
        "gbdt_build_histograms_segmented": ([P, i64, i32, i64, i32, P, i32, P, P, i32, P, i32, P, P, P, P, P, sz, P],
                                            i32),
        "gbdt_build_histograms_segmented_h": ([P, i64, i32, i64, i32, P, i32, P, P, i32, P, i32, P, P, P, P, P, P, sz,
                                               P], i32),
        "gbdt_row_block_pitch": ([i32], i64),
        "gbdt_row_block_slots": ([P, i32, i32, P, P], i32),
        "gbdt_row_block_slots_ex": ([P, i32, i32, i32, P, P, P], i32),
        "gbdt_row_block_bytes": ([i64, i32], sz),
        "gbdt_bins_to_row_blocks": ([P, i64, i64, i32, P, P], i32),
        "gbdt_partition_rows_workspace_size": ([i64, i32], sz),
        "gbdt_partition_rows": ([P, P, i64, i64, i32, P, P, i32, P, P, P, P, P, i32, P, P, P, P, P, sz, P], i32),
        "gbdt_predict_workspace_size": ([i32, i32], sz),
        "gbdt_predict": ([P, i64, i64, i32, P, i32, P, P, i32, i32, dbl, dbl, P, P, sz, P], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(L, name)
        fn.argtypes = args
        fn.restype = res
    _lib = L
    return _lib


# ---------------------------------------------------------------------------------------- helpers
def _torch():
    import torch

    if not torch.cuda.is_available():
        raise GbdtError(ERR_CUDA, "no CUDA device: this library has no CPU path")
    return torch


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream():
    return ctypes.c_void_p(_torch().cuda.current_stream().cuda_stream)


def _check(rc: int):
    if rc != OK:
        raise GbdtError(rc, lib().gbdt_last_error().decode())


def _workspace(nbytes: int):
    torch = _torch()
    return torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device="cuda")


def _dev(arr, dtype):
    """numpy structured array -> CUDA byte tensor with the same bytes."""
    torch = _torch()
    a = np.ascontiguousarray(arr, dtype=dtype)
    return torch.from_numpy(a.view(np.uint8).reshape(-1).copy()).cuda()


def _host(t, dtype, count):
    return np.frombuffer(t.cpu().numpy().tobytes(), dtype=dtype, count=count)


def padded_ld(n: int) -> int:
    """Column stride for binned features: n rounded up to a multiple of 16."""
    return (int(n) + 15) // 16 * 16


def make_params(n_trees=1, max_depth=6, learning_rate=0.1, reg_lambda=1.0, gamma=0.0, min_samples_leaf=1,
                min_child_weight=0.0, num_leaves=0, objective=OBJECTIVE_SQUARED_ERROR, bin_packing=BIN_PACKING_4BIT,
                hist_registers=HIST_REGISTERS_OFF, **_ignored) -> Params:
    return Params(int(n_trees), int(max_depth), float(learning_rate), float(reg_lambda), float(gamma),
                  int(min_samples_leaf), float(min_child_weight), int(num_leaves), int(objective), int(bin_packing),
                  int(hist_registers))


def version() -> str:
    return lib().gbdt_version().decode()


def validate_params(**kw) -> int:
    p = make_params(**kw)
    return lib().gbdt_validate_params(ctypes.byref(p))


# ---------------------------------------------------------------------------------------- entry points
def quantize(X, max_bins: int, ldb: int | None = None, x_device=None):
    """X: (F, N) float32 tensor -> bins (F, ldb) uint8, edges (F, max_bins-1) f32, n_bins (F,) i32 (CUDA).

    X on the GPU: gbdt_quantize.  X in host memory (pinned for overlap): gbdt_quantize_host, which copies X
    into x_device (a (F, N) float32 CUDA tensor with X's strides; allocated if None) column batch by column
    batch while the earlier batches are binned."""
    torch = _torch()
    assert X.dtype == torch.float32 and X.dim() == 2 and X.stride(1) == 1
    F, N = X.shape
    ldb = padded_ld(N) if ldb is None else ldb
    bins = torch.empty((F, ldb), dtype=torch.uint8, device="cuda")
    edges = torch.empty((F, max_bins - 1), dtype=torch.float32, device="cuda")
    n_bins = torch.empty(F, dtype=torch.int32, device="cuda")
    ws = _workspace(lib().gbdt_quantize_workspace_size(N, F))
    ldx = X.stride(0) if F > 1 else N  # a size-1 leading dim may carry any stride
    if X.is_cuda:
        _check(lib().gbdt_quantize(_ptr(X), ldx, N, F, max_bins, _ptr(bins), ldb, _ptr(edges), _ptr(n_bins),
                                   _ptr(ws), ws.numel(), _stream()))
        return bins, edges, n_bins
    if x_device is None:
        x_device = torch.empty_strided((F, N), (ldx, 1), dtype=torch.float32, device="cuda")
    assert x_device.is_cuda and x_device.dtype == torch.float32 and x_device.shape == X.shape
    assert F == 1 or x_device.stride(0) == ldx, "x_device needs X's leading dimension"
    _check(lib().gbdt_quantize_host(_ptr(X), ldx, N, F, max_bins, _ptr(x_device), _ptr(bins), ldb, _ptr(edges),
                                    _ptr(n_bins), _ptr(ws), ws.numel(), _stream()))
    return bins, edges, n_bins


def compute_gradients(pred, label, objective=OBJECTIVE_SQUARED_ERROR):
    """g (N,) f64 and the fixed-point exponents: S (1,) for squared error, (S, S_h) (2,) for logistic."""
    torch = _torch()
    N = pred.shape[0]
    g = torch.empty(N, dtype=torch.float64, device="cuda")
    S = torch.zeros(2 if objective == OBJECTIVE_LOGISTIC else 1, dtype=torch.int32, device="cuda")
    ws = _workspace(lib().gbdt_gradients_workspace_size(N))
    if objective == OBJECTIVE_SQUARED_ERROR:
        _check(lib().gbdt_compute_gradients(_ptr(pred), _ptr(label), N, _ptr(g), _ptr(S), _ptr(ws), ws.numel(),
                                            _stream()))
    else:
        _check(lib().gbdt_compute_gradients_objective(_ptr(pred), _ptr(label), N, int(objective), _ptr(g), _ptr(S),
                                                      _ptr(ws), ws.numel(), _stream()))
    return g, S


def gradient_scale(g):
    torch = _torch()
    S = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = _workspace(lib().gbdt_gradients_workspace_size(g.shape[0]))
    dt = DTYPE_F32 if g.dtype == torch.float32 else DTYPE_F64
    _check(lib().gbdt_gradient_scale(_ptr(g), dt, g.shape[0], _ptr(S), _ptr(ws), ws.numel(), _stream()))
    return S


def build_histograms(bins, N, g, fixed_exp, node_of_row, level, max_slots, build_flag, max_build, hist_cnt=None,
                     hist_q=None, ws=None):
    """bins (F, ldb) uint8; g f32/f64 (N,); node_of_row uint16-valued int16 tensor or uint16 (N,);
    level: CUDA tensor of LEVEL_DTYPE bytes; build_flag uint8 (max_slots,).  Returns (hist_cnt, hist_q)."""
    torch = _torch()
    F, ldb = bins.shape
    if hist_cnt is None:
        hist_cnt = torch.zeros((max_slots, F, 256), dtype=torch.int32, device="cuda")
        hist_q = torch.zeros((max_slots, F, 256), dtype=torch.int64, device="cuda")
    if ws is None:
        ws = _workspace(lib().gbdt_histograms_workspace_size(N, F, max_slots))
    dt = DTYPE_F32 if g.dtype == torch.float32 else DTYPE_F64
    _check(lib().gbdt_build_histograms(_ptr(bins), ldb, N, F, _ptr(g), dt, _ptr(fixed_exp), _ptr(node_of_row),
                                       _ptr(level), max_slots, _ptr(build_flag), max_build, _ptr(hist_cnt),
                                       _ptr(hist_q), _ptr(ws), ws.numel(), _stream()))
    return hist_cnt, hist_q


def row_block_slots(n_bins, packing=BIN_PACKING_4BIT):
    """Host-side slot plan of gbdt_train's row-block copies: (loc (F,) uint32, src (S,) uint32)."""
    nb = np.ascontiguousarray(n_bins, dtype=np.int32)
    F = nb.shape[0]
    loc = np.zeros(F, np.uint32)
    src = np.zeros(F, np.uint32)
    S = lib().gbdt_row_block_slots(nb.ctypes.data_as(ctypes.c_void_p), F, int(packing),
                                   loc.ctypes.data_as(ctypes.c_void_p), src.ctypes.data_as(ctypes.c_void_p))
    _check(0 if S > 0 else S)
    return loc, src[:S]


def row_block_slots_ex(n_bins, packing=BIN_PACKING_4BIT, hist_registers=HIST_REGISTERS_ON):
    """Host-side slot plan with register slots: (loc (F,) uint32, src (S,) uint32, reg_begin)."""
    nb = np.ascontiguousarray(n_bins, dtype=np.int32)
    F = nb.shape[0]
    loc = np.zeros(F, np.uint32)
    src = np.zeros(F, np.uint32)
    rb = ctypes.c_int32(0)
    S = lib().gbdt_row_block_slots_ex(nb.ctypes.data_as(ctypes.c_void_p), F, int(packing), int(hist_registers),
                                      loc.ctypes.data_as(ctypes.c_void_p), src.ctypes.data_as(ctypes.c_void_p),
                                      ctypes.byref(rb))
    _check(0 if S > 0 else S)
    return loc, src[:S], rb.value


def to_row_blocks(bins, N: int):
    """Column-major bins (F, ldb) CUDA uint8 -> the row-block layout (a flat CUDA uint8 tensor) and its pitch."""
    torch = _torch()
    F, ldb = bins.shape
    out = torch.empty(lib().gbdt_row_block_bytes(N, F) + 256, dtype=torch.uint8, device="cuda")
    off = (-out.data_ptr()) % 256  # 256-byte aligned view
    out = out[off: off + lib().gbdt_row_block_bytes(N, F)]
    _check(lib().gbdt_bins_to_row_blocks(_ptr(bins), ldb, N, F, _ptr(out), _stream()))
    return out, lib().gbdt_row_block_pitch(F)


def build_histograms_segmented(bins, N, g, fixed_exp, level, max_slots, build_flag, max_build, segments,
                               hist_cnt=None, hist_q=None, ws=None, filters=None, row_blocks=None, hist_h=None,
                               logistic=False):
    """Histograms of flagged slots whose rows are contiguous segments (SEGMENT_DTYPE bytes, device),
    optionally narrowed per slot by FILTER_DTYPE records (device bytes).  bins: column-major (F, ldb)
    CUDA uint8; with row_blocks = (buffer, pitch) from to_row_blocks the kernel reads that layout instead
    (bins then only gives F).  logistic: also the H histograms of h = |g| (1 - |g|) with exponent
    fixed_exp[1]; returns (hist_cnt, hist_q, hist_h) then, else (hist_cnt, hist_q)."""
    torch = _torch()
    F, ldb = bins.shape
    if hist_cnt is None:
        hist_cnt = torch.zeros((max_slots, F, 256), dtype=torch.int32, device="cuda")
        hist_q = torch.zeros((max_slots, F, 256), dtype=torch.int64, device="cuda")
    if logistic and hist_h is None:
        hist_h = torch.zeros((max_slots, F, 256), dtype=torch.int64, device="cuda")
    if ws is None:
        ws = _workspace(lib().gbdt_histograms_segmented_workspace_size(max_slots))
    dt = DTYPE_F32 if g.dtype == torch.float32 else DTYPE_F64
    src, ld, layout = (bins, ldb, LAYOUT_COLUMNS) if row_blocks is None else (row_blocks[0], row_blocks[1],
                                                                              LAYOUT_ROW_BLOCKS)
    args = (_ptr(src), ld, layout, N, F, _ptr(g), dt, _ptr(fixed_exp), _ptr(level), max_slots, _ptr(build_flag),
            max_build, _ptr(segments), _ptr(filters) if filters is not None else None, _ptr(hist_cnt), _ptr(hist_q))
    if logistic:
        _check(lib().gbdt_build_histograms_segmented_h(*args, _ptr(hist_h), _ptr(ws), ws.numel(), _stream()))
        return hist_cnt, hist_q, hist_h
    _check(lib().gbdt_build_histograms_segmented(*args, _ptr(ws), ws.numel(), _stream()))
    return hist_cnt, hist_q


def partition_rows(bins_in, N, g_in, orig_in, splits, level, max_slots, seg_in, go_right=None, leaf_of_row=None,
                   out=None, ws=None):
    """Stable partition of the per-position data.  Returns (bins_out, g_out, orig_out, seg_out, next_level)."""
    torch = _torch()
    F, ldb = bins_in.shape
    if out is None:
        out = (torch.empty_like(bins_in), torch.empty_like(g_in), torch.empty_like(orig_in))
    bins_out, g_out, orig_out = out
    seg_out = torch.zeros(2 * max_slots * SEGMENT_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    next_level = torch.zeros(LEVEL_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    if ws is None:
        ws = _workspace(lib().gbdt_partition_rows_workspace_size(N, max_slots))
    dt = DTYPE_F32 if g_in.dtype == torch.float32 else DTYPE_F64
    _check(lib().gbdt_partition_rows(_ptr(bins_in), _ptr(bins_out), ldb, N, F, _ptr(g_in), _ptr(g_out), dt,
                                     _ptr(orig_in), _ptr(orig_out), _ptr(go_right), _ptr(splits), _ptr(level),
                                     max_slots, _ptr(seg_in), _ptr(seg_out), _ptr(next_level), _ptr(leaf_of_row),
                                     _ptr(ws), ws.numel(), _stream()))
    return bins_out, g_out, orig_out, seg_out, next_level


def subtract_histograms(prev_cnt, prev_q, pair_parent, build_flag, level, max_slots, hist_cnt, hist_q, prev_h=None,
                        hist_h=None, ws=None):
    """Sibling subtraction; ws (optional, a workspace of gbdt_subtract_histograms_workspace_size bytes) receives
    the call's error word (see workspace_status)."""
    F = hist_cnt.shape[1]
    wp, wn = (_ptr(ws), ws.numel()) if ws is not None else (None, 0)
    if prev_h is None and hist_h is None:
        _check(lib().gbdt_subtract_histograms(_ptr(prev_cnt), _ptr(prev_q), _ptr(pair_parent), _ptr(build_flag),
                                              _ptr(level), max_slots, F, _ptr(hist_cnt), _ptr(hist_q), wp, wn,
                                              _stream()))
        return hist_cnt, hist_q
    _check(lib().gbdt_subtract_histograms_h(_ptr(prev_cnt), _ptr(prev_q), _ptr(prev_h), _ptr(pair_parent),
                                            _ptr(build_flag), _ptr(level), max_slots, F, _ptr(hist_cnt),
                                            _ptr(hist_q), _ptr(hist_h), wp, wn, _stream()))
    return hist_cnt, hist_q, hist_h


def workspace_status(ws) -> int:
    """Error word of the last call queued with workspace ws (synchronises the stream): 0, else GbdtError."""
    bits = ctypes.c_int32(0)
    _check(lib().gbdt_workspace_status(_ptr(ws), ctypes.byref(bits), _stream()))
    return bits.value


def partition_noalloc_status() -> int:
    """Error word of the last gbdt_partition_noalloc call on this device: 0, else GbdtError."""
    bits = ctypes.c_int32(0)
    _check(lib().gbdt_partition_noalloc_status(ctypes.byref(bits), _stream()))
    return bits.value


def find_splits(hist_cnt, hist_q, fixed_exp, n_bins, level, max_slots, out=None, hist_h=None, ws=None, **params):
    """Best split per slot (SPLIT_DTYPE bytes, device); hist_h: H from that histogram (exponent fixed_exp[1])."""
    torch = _torch()
    F = hist_cnt.shape[1]
    p = make_params(**params)
    if out is None:
        out = torch.empty(max_slots * SPLIT_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    if ws is None:
        ws = _workspace(lib().gbdt_find_splits_workspace_size(F, max_slots))
    if hist_h is None:
        _check(lib().gbdt_find_splits(_ptr(hist_cnt), _ptr(hist_q), _ptr(fixed_exp), F, _ptr(n_bins), _ptr(level),
                                      max_slots, ctypes.byref(p), _ptr(out), _ptr(ws), ws.numel(), _stream()))
    else:
        _check(lib().gbdt_find_splits_h(_ptr(hist_cnt), _ptr(hist_q), _ptr(hist_h), _ptr(fixed_exp), F,
                                        _ptr(n_bins), _ptr(level), max_slots, ctypes.byref(p), _ptr(out), _ptr(ws),
                                        ws.numel(), _stream()))
    return out


def partition(bins, N, splits, level, max_slots, seg_in, idx_in, node_of_row, idx_out=None, ws=None):
    torch = _torch()
    F, ldb = bins.shape
    if idx_out is None:
        idx_out = torch.zeros_like(idx_in)
    seg_out = torch.zeros(2 * max_slots * SEGMENT_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    next_level = torch.zeros(LEVEL_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    if ws is None:
        ws = _workspace(lib().gbdt_partition_workspace_size(N, max_slots))
    _check(lib().gbdt_partition(_ptr(bins), ldb, N, F, _ptr(splits), _ptr(level), max_slots, _ptr(seg_in),
                                _ptr(idx_in), _ptr(node_of_row), _ptr(idx_out), _ptr(seg_out), _ptr(next_level),
                                _ptr(ws), ws.numel(), _stream()))
    return idx_out, seg_out, next_level


def partition_noalloc(bins, N, splits, level, max_slots, seg_in, idx_in, node_of_row, idx_out=None):
    """gbdt_partition with the library's built-in scratch instead of a workspace."""
    torch = _torch()
    F, ldb = bins.shape
    if idx_out is None:
        idx_out = torch.zeros_like(idx_in)
    seg_out = torch.zeros(2 * max_slots * SEGMENT_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    next_level = torch.zeros(LEVEL_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    _check(lib().gbdt_partition_noalloc(_ptr(bins), ldb, N, F, _ptr(splits), _ptr(level), max_slots, _ptr(seg_in),
                                        _ptr(idx_in), _ptr(node_of_row), _ptr(idx_out), _ptr(seg_out),
                                        _ptr(next_level), _stream()))
    return idx_out, seg_out, next_level


def update_predictions(pred, leaf_of_row, leaf_value, lr):
    _check(lib().gbdt_update_predictions(_ptr(pred), _ptr(leaf_of_row), _ptr(leaf_value), leaf_value.shape[0],
                                         pred.shape[0], float(lr), _stream()))
    return pred


def train_workspace_size(N: int, F: int, **params) -> int:
    p = make_params(**params)
    return lib().gbdt_train_workspace_size(N, F, ctypes.byref(p))


def train(bins, n_bins, label, N: int | None = None, diagnostics: bool = False, ws=None, pred=None, **params):
    """Train on binned features.  bins (F, ldb) uint8 CUDA, n_bins (F,) int32 CUDA, label (N,) float32 CUDA.
    Returns dict(nodes (T, M) NODE_DTYPE, nodes_per_tree, init_pred, pred (CUDA f64), diag)."""
    torch = _torch()
    F, ldb = bins.shape
    N = label.shape[0] if N is None else N
    p = make_params(**params)
    T, M = p.n_trees, (1 << (p.max_depth + 1)) - 1
    if pred is None:
        pred = torch.empty(N, dtype=torch.float64, device="cuda")
    if ws is None:
        ws = _workspace(lib().gbdt_train_workspace_size(N, F, ctypes.byref(p)))
    nodes = np.zeros((max(T, 1), M), NODE_DTYPE)
    npt = np.zeros(max(T, 1), np.int32)
    init = ctypes.c_double(0.0)
    diag = Diagnostics() if diagnostics else None
    rc = lib().gbdt_train(_ptr(bins), ldb, _ptr(n_bins), N, F, _ptr(label), ctypes.byref(p), _ptr(pred),
                          ctypes.byref(init), nodes.ctypes.data_as(ctypes.c_void_p),
                          npt.ctypes.data_as(ctypes.c_void_p), ctypes.byref(diag) if diag is not None else None,
                          _ptr(ws), ws.numel(), _stream())
    _check(rc)
    return dict(nodes=nodes[:T], nodes_per_tree=npt[:T], init_pred=init.value, pred=pred,
                diag=diag.as_dict() if diag is not None else None)


def kernel_launch_count() -> int:
    """Kernels the library has launched in this process so far."""
    return int(lib().gbdt_kernel_launch_count())


def inject_failure(after_levels: int):
    """Testing hook: make the next gbdt_train calls fail on the host after that many levels (-1 disables)."""
    lib().gbdt_debug_inject_failure(int(after_levels))


def predict(X, edges, nodes, init_pred, learning_rate, nodes_per_tree=None, out=None, ws=None):
    """Predictions on raw fp32 features X (F, ldx) CUDA of a model: nodes (T, M) NODE_DTYPE (host numpy, as
    train returns them) with nodes_per_tree (T,) (None: every slot is a node), edges (F, max_bins - 1) CUDA."""
    torch = _torch()
    F, ldx = X.shape
    N = ldx if out is None else out.shape[0]
    max_bins = edges.shape[1] + 1
    if not isinstance(nodes, np.ndarray):
        raise TypeError("nodes: a (T, M) NODE_DTYPE numpy array")
    T, M = (nodes.shape[0], nodes.shape[1]) if nodes.ndim == 2 else (0, 1)
    nodes_d = torch.from_numpy(np.ascontiguousarray(nodes).view(np.uint8).reshape(-1).copy()).cuda() if T else None
    npt_d = (torch.from_numpy(np.ascontiguousarray(nodes_per_tree, np.int32)).cuda()
             if nodes_per_tree is not None and T else None)
    if out is None:
        out = torch.empty(N, dtype=torch.float64, device="cuda")
    if ws is None:
        ws = _workspace(lib().gbdt_predict_workspace_size(T, max(M, 1)))
    _check(lib().gbdt_predict(_ptr(X), ldx, N, F, _ptr(edges), max_bins, _ptr(nodes_d), _ptr(npt_d), T, max(M, 1),
                              float(init_pred), float(learning_rate), _ptr(out), _ptr(ws), ws.numel(), _stream()))
    return out

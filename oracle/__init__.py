"""CPU oracle for level-wise histogram GBDT (squared error) -- TEST INFRASTRUCTURE.

Only the test suite, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``gbdt_oracle.c`` (plain FP64
C, built here with gcc) through ctypes and shares no code with the CUDA
library in ``histogram_gradient_boosted_gb300``.

The C source cites the passages each function follows ("Module Design:
Training Core", sections 2, 3, 6 and 7; "Gradient boosted trees (spec
model)", forward pass and tree representation).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gbdt_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, EINVAL, ENONFINITE, ENOMEM = 0, -1, -2, -3
NBINS = 256
NEAR_MAX = 8


class Params(ctypes.Structure):
    _fields_ = [("n_trees", ctypes.c_int32), ("max_depth", ctypes.c_int32),
                ("learning_rate", ctypes.c_double), ("reg_lambda", ctypes.c_double),
                ("gamma", ctypes.c_double), ("min_samples_leaf", ctypes.c_int32),
                ("min_child_weight", ctypes.c_double), ("num_leaves", ctypes.c_int32), ("objective", ctypes.c_int32),
                ("n_threads", ctypes.c_int32)]


class Split(ctypes.Structure):
    _fields_ = [("valid", ctypes.c_int32), ("feature", ctypes.c_int32), ("bin", ctypes.c_int32),
                ("gain", ctypes.c_double), ("cnt_left", ctypes.c_int64), ("G_left", ctypes.c_double),
                ("H_left", ctypes.c_double), ("second_gain", ctypes.c_double), ("n_near", ctypes.c_int32),
                ("near_feature", ctypes.c_int32 * NEAR_MAX), ("near_bin", ctypes.c_int32 * NEAR_MAX)]


NODE_DTYPE = np.dtype([("feature", np.int32), ("threshold_bin", np.int32), ("left", np.int32),
                       ("right", np.int32), ("leaf_value", np.float64), ("gain", np.float64),
                       ("is_leaf", np.int32), ("depth", np.int32)], align=True)
INFO_DTYPE = np.dtype([("n_rows", np.int64), ("G", np.float64), ("H", np.float64), ("A", np.float64),
                       ("best_gain", np.float64), ("second_gain", np.float64), ("n_near", np.int32),
                       ("near_feature", np.int32, (NEAR_MAX,)), ("near_bin", np.int32, (NEAR_MAX,)),
                       ("adopted", np.int32), ("guide_mismatch", np.int32), ("guide_gap", np.float64),
                       ("guide_bound", np.float64)], align=True)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP if available).  Returns the .so path."""
    with _lock:
        if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
            return _LIB
        os.makedirs(_BUILD, exist_ok=True)
        base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
        tmp = _LIB + f".tmp{os.getpid()}"
        for extra in (["-fopenmp"], []):
            r = subprocess.run(base + extra + ["-o", tmp, _SRC, "-lm"], capture_output=True, text=True)
            if r.returncode == 0:
                os.replace(tmp, _LIB)
                return _LIB
        raise RuntimeError("oracle build failed:\n" + r.stderr)


def lib():
    global _lib
    if _lib is None:
        path = build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        i64, i32, dbl = ctypes.c_int64, ctypes.c_int32, ctypes.c_double
        L.orc_quantize.argtypes = [P, i64, i32, i32, i32, P, P, P]
        L.orc_gradients.argtypes = [P, P, i64, P, P]
        L.orc_histograms.argtypes = [P, i64, i32, P, P, P, i32, P, P, P, P, P, P, P]
        L.orc_best_split.argtypes = [P, P, P, i32, P, i64, dbl, dbl, ctypes.POINTER(Params),
                                     ctypes.POINTER(Split)]
        L.orc_train.argtypes = [P, P, i64, i32, P, ctypes.POINTER(Params), P, P, P, P, P, P, P, P, P]
        L.orc_partition.argtypes = [P, i64, i32, P, P, P, P, P, P, P]
        L.orc_update_predictions.argtypes = [P, P, P, i64, dbl]
        L.orc_predict.argtypes = [P, i64, i32, P, i32, P, i32, i32, dbl, dbl, P]
        L.orc_gradients_objective.argtypes = [P, P, i64, i32, P, P]
        L.orc_weight.argtypes = [dbl, dbl, dbl]
        L.orc_weight.restype = dbl
        L.orc_gain.argtypes = [dbl] * 8
        L.orc_gain.restype = dbl
        L.orc_validate_params.argtypes = [ctypes.POINTER(Params)]
        _lib = L
    return _lib


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None else None


def _check(rc: int, what: str):
    if rc != OK:
        raise OracleError(rc, what)


class OracleError(RuntimeError):
    def __init__(self, code: int, what: str):
        super().__init__(f"{what} failed with oracle status {code}")
        self.code = code


def make_params(n_trees=1, max_depth=3, learning_rate=0.1, reg_lambda=1.0, gamma=0.0, min_samples_leaf=1,
                min_child_weight=0.0, num_leaves=0, objective=0, n_threads=1, **_ignored) -> Params:
    return Params(int(n_trees), int(max_depth), float(learning_rate), float(reg_lambda), float(gamma),
                  int(min_samples_leaf), float(min_child_weight), int(num_leaves), int(objective), int(n_threads))


def weight(G: float, H: float, reg_lambda: float) -> float:
    return lib().orc_weight(G, H, reg_lambda)


def gain(GL, HL, GR, HR, GP, HP, reg_lambda, gamma) -> float:
    return lib().orc_gain(GL, HL, GR, HR, GP, HP, reg_lambda, gamma)


def validate_params(**kw) -> int:
    p = make_params(**kw)
    return lib().orc_validate_params(ctypes.byref(p))


def quantize(X: np.ndarray, max_bins: int, n_threads: int = 1):
    """X: (F, N) float32 -> bins (F, N) uint8, edges (F, max_bins-1) float32, n_bins (F,) int32."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    F, N = X.shape
    bins = np.empty((F, N), dtype=np.uint8)
    edges = np.empty((F, max_bins - 1), dtype=np.float32)
    n_bins = np.empty(F, dtype=np.int32)
    _check(lib().orc_quantize(_p(X), N, F, max_bins, n_threads, _p(bins), _p(edges), _p(n_bins)), "quantize")
    return bins, edges, n_bins


def gradients(pred: np.ndarray, label: np.ndarray, objective: int = 0):
    pred = np.ascontiguousarray(pred, dtype=np.float64)
    label = np.ascontiguousarray(label, dtype=np.float32)
    g = np.empty(pred.shape[0], dtype=np.float64)
    h = np.empty(pred.shape[0], dtype=np.float64)
    _check(lib().orc_gradients_objective(_p(pred), _p(label), pred.shape[0], int(objective), _p(g), _p(h)),
           "gradients")
    return g, h


def histograms(bins: np.ndarray, g: np.ndarray, slot_of_row: np.ndarray, n_slots: int, h: np.ndarray | None = None):
    """Row-order FP64 histograms of every slot (h: per-row hessians, None for h = 1).  Returns dict of arrays:
    cnt (S,F,256) uint32, G/H (S,F,256) float64, n (S,) int64, Gt/Ht/At (S,) float64."""
    bins = np.ascontiguousarray(bins, dtype=np.uint8)
    F, N = bins.shape
    g = np.ascontiguousarray(g, dtype=np.float64)
    h = None if h is None else np.ascontiguousarray(h, dtype=np.float64)
    slot = np.ascontiguousarray(slot_of_row, dtype=np.int32)
    out = dict(cnt=np.empty((n_slots, F, NBINS), np.uint32), G=np.empty((n_slots, F, NBINS), np.float64),
               H=np.empty((n_slots, F, NBINS), np.float64), n=np.empty(n_slots, np.int64),
               Gt=np.empty(n_slots, np.float64), Ht=np.empty(n_slots, np.float64), At=np.empty(n_slots, np.float64))
    _check(lib().orc_histograms(_p(bins), N, F, _p(g), _p(h) if h is not None else None, _p(slot), n_slots,
                                _p(out["cnt"]), _p(out["G"]),
                                _p(out["H"]), _p(out["n"]), _p(out["Gt"]), _p(out["Ht"]), _p(out["At"])),
           "histograms")
    return out


def best_split(cnt, G, H, n_bins, n_P, G_P, H_P, **params) -> Split:
    cnt = np.ascontiguousarray(cnt, dtype=np.uint32)
    G = np.ascontiguousarray(G, dtype=np.float64)
    H = np.ascontiguousarray(H, dtype=np.float64)
    n_bins = np.ascontiguousarray(n_bins, dtype=np.int32)
    p = make_params(**params)
    s = Split()
    _check(lib().orc_best_split(_p(cnt), _p(G), _p(H), cnt.shape[0], _p(n_bins), int(n_P), float(G_P),
                                float(H_P), ctypes.byref(p), ctypes.byref(s)), "best_split")
    return s


def max_nodes(max_depth: int) -> int:
    return (1 << (max_depth + 1)) - 1


def train(bins: np.ndarray, n_bins: np.ndarray, label: np.ndarray, guide: np.ndarray | None = None,
          want_info: bool = True, want_leaf_of_row: bool = False, tie_quanta: np.ndarray | None = None,
          pred_in: np.ndarray | None = None, **params):
    """Train; returns dict(pred, init_pred, nodes (T, M) NODE_DTYPE, nodes_per_tree, info, leaf_of_row).

    Parity-harness options: guide (T, M, 2) the other program's (feature, bin) per node, tie_quanta (T, 2)
    its per-row rounding bounds of g and h (see orc_train), pred_in (N,) predictions to start from."""
    bins = np.ascontiguousarray(bins, dtype=np.uint8)
    F, N = bins.shape
    n_bins = np.ascontiguousarray(n_bins, dtype=np.int32)
    label = np.ascontiguousarray(label, dtype=np.float32)
    p = make_params(**params)
    T, M = p.n_trees, max_nodes(p.max_depth)
    pred = np.empty(N, np.float64)
    init = np.zeros(1, np.float64)
    nodes = np.zeros((T, M), NODE_DTYPE)
    npt = np.zeros(T, np.int32)
    info = np.zeros((T, M), INFO_DTYPE) if want_info else None
    lor = np.empty(N, np.int32) if want_leaf_of_row else None
    if guide is not None:
        guide = np.ascontiguousarray(guide, dtype=np.int32)
        assert guide.shape == (T, M, 2)
    if tie_quanta is not None:
        tie_quanta = np.ascontiguousarray(tie_quanta, dtype=np.float64)
        assert tie_quanta.shape == (T, 2)
    if pred_in is not None:
        pred_in = np.ascontiguousarray(pred_in, dtype=np.float64)
        assert pred_in.shape == (N,)
    _check(lib().orc_train(_p(bins), _p(n_bins), N, F, _p(label), ctypes.byref(p), _p(guide), _p(tie_quanta),
                           _p(pred_in), _p(pred), _p(init), _p(nodes), _p(npt), _p(info), _p(lor)), "train")
    return dict(pred=pred, init_pred=float(init[0]), nodes=nodes, nodes_per_tree=npt, info=info,
                leaf_of_row=lor)


def partition(bins, split_feature, split_bin, seg_start, seg_count, idx_in):
    bins = np.ascontiguousarray(bins, dtype=np.uint8)
    F, N = bins.shape
    sf = np.ascontiguousarray(split_feature, np.int32)
    sb = np.ascontiguousarray(split_bin, np.int32)
    ss = np.ascontiguousarray(seg_start, np.int64)
    sc = np.ascontiguousarray(seg_count, np.int64)
    ii = np.ascontiguousarray(idx_in, np.int64)
    out = np.empty_like(ii)
    lc = np.empty(sf.shape[0], np.int64)
    _check(lib().orc_partition(_p(bins), N, sf.shape[0], _p(sf), _p(sb), _p(ss), _p(sc), _p(ii), _p(out),
                               _p(lc)), "partition")
    return out, lc


def update_predictions(pred, leaf_value, node_of_row, lr):
    pred = np.array(pred, dtype=np.float64, copy=True)
    lv = np.ascontiguousarray(leaf_value, np.float64)
    nr = np.ascontiguousarray(node_of_row, np.int32)
    _check(lib().orc_update_predictions(_p(pred), _p(lv), _p(nr), pred.shape[0], float(lr)), "update")
    return pred


def predict(X, edges, nodes, init_pred, learning_rate):
    """Predictions on raw fp32 features [F][N] of trees nodes (T, M) NODE_DTYPE with quantize edges."""
    X = np.ascontiguousarray(X, dtype=np.float32)
    F, N = X.shape
    edges = np.ascontiguousarray(edges, dtype=np.float32)
    nodes = np.ascontiguousarray(nodes, dtype=NODE_DTYPE)
    T, M = (nodes.shape if nodes.ndim == 2 else (0, 1))
    out = np.empty(N, np.float64)
    _check(lib().orc_predict(_p(X), N, F, _p(edges), edges.shape[1] + 1, _p(nodes) if T else None, T, M,
                             float(init_pred), float(learning_rate), _p(out)), "predict")
    return out

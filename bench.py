#!/usr/bin/env python3
"""Benchmark: GBDT training throughput (rows*features*trees/s) on one GB300,
with the level-histogram kernel's HBM roofline.

Default workload: the large heavy-tailed configuration (10,000,000 rows x 100
fp32 features, 255 bins, depth 8, 200 trees, lr 0.05, lambda 1, gamma 0.1,
min_samples_leaf 20), seeded synthetic data.  One step is one pass of the whole
hot path over that matrix: quantile binning (gbdt_quantize) followed by a full
training run (gbdt_train: gradients, level histograms, subtraction, split
search, partition, leaves, prediction updates) -- features already resident
in HBM.  Inputs (4 GB fp32 features, 1 GB bins) are larger than L2.

Also reported on the same line:
  e2e                  the same metric through the public API with host inputs:
                       pinned host -> device copy of X and labels, quantize,
                       train, device -> host read of the model and predictions;
  roofline             algorithmic bytes / CUDA-event time of the histogram
                       launches inside the timed steps, against measured HBM;
  histogram_microbench one tree level at 50,000,000 rows x 64 pre-binned
                       features, 256 nodes: build (smaller siblings),
                       subtraction and split search, each timed with events;
  cpu_baseline         the CPU oracle (test infrastructure) on a bounded sample.

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
For N > 1 (torchrun), each rank trains an independent replica; value is the
sum of the ranks' units over the slowest rank's time ("replicas only").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "GBDT train rows·features·trees/sec on 1 GB300; histogram HBM GB/s vs peak"
UNIT = "rows*features*trees/s"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------------------------ helpers
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 0, 1, None
    import torch.distributed as dist

    dist.init_process_group("gloo")  # host-side barrier and timing exchange only
    return dist.get_rank(), int(os.environ.get("LOCAL_RANK", "0")), ws, dist


def _max_over_ranks(x: float, dist):
    if dist is None:
        return x
    import torch

    t = torch.tensor([x], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _barrier(dist):
    if dist is not None:
        dist.barrier()


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


class ClockSampler:
    """nvidia-smi sampled every 200 ms while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.out.close()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            for line in open(self.path):
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None

        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows),
                "power_w_max": max((num(r[2]) for r in rows if num(r[2]) is not None), default=None)}


# the histogram kernel, its launch plan (CTA shares per column group) and its launcher all live in
# segments.cu; the training loop only passes each level's sizes to them
HIST_SOURCES = [os.path.join("histogram_gradient_boosted_gb300", "csrc", "segments.cu")]


def _code_only(text: str) -> str:
    """C++/CUDA source without its comments and blank lines (string literals here hold no comment
    markers), so that a comment edit does not count as a change of the kernel."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln.strip())


def hist_source_sha256() -> str:
    """Hash of the code that defines the level-histogram launches (the kernel and its launch plan)."""
    h = hashlib.sha256()
    for rel in HIST_SOURCES:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(_code_only(f.read()).encode())
    return h.hexdigest()


def _traffic_record():
    """ncu DRAM bytes per histogram launch, if recorded for the current sources (else None)."""
    p = os.path.join(ROOT, "profiles", "histogram_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        rec = json.load(f)
    return rec if rec.get("kernel_source_sha256") == hist_source_sha256() else None


def _scaled_traffic(rec, read_bytes_per_launch):
    """DRAM bytes per launch of this workload from a smaller capture: the captured bytes scaled by this
    run's read bytes over the captured run's (rows scanned and built histograms both counted)."""
    if not rec:
        return None
    if "read_bytes_per_launch_captured" not in rec:
        return rec.get("dram_bytes_per_launch")
    return rec["dram_bytes_per_launch_captured"] * read_bytes_per_launch / rec["read_bytes_per_launch_captured"]


# ------------------------------------------------------------------------------------ reference arm
def cpu_baseline_sample(X, y, cfg, n_rows, n_trees, threads, repeats=1):
    """The oracle as it stands on the first n_rows rows: quantize (untimed), train (timed)."""
    import oracle

    oracle.build()
    Xs = np.ascontiguousarray(X[:, :n_rows])
    ys = np.ascontiguousarray(y[:n_rows])
    bins, _, n_bins = oracle.quantize(Xs, cfg["max_bins"], n_threads=threads)
    params = dict(cfg, n_trees=n_trees, n_threads=threads)
    times = []
    for _ in range(repeats):
        t0 = time.perf_counter()
        oracle.train(bins, n_bins, ys, want_info=False, **params)
        times.append(time.perf_counter() - t0)
    units = n_rows * X.shape[0] * n_trees
    return units, times


def parity_sample(g, torch, X, y, cfg, n_rows, n_trees):
    """The CUDA path against the oracle on a sample of the benchmark's matrix: every tree node by node, grown
    from the same predictions (tests/gpu_util.compare_training), near-ties counted as the tests count them."""
    import oracle
    from tests.gpu_util import compare_training

    Xs = np.ascontiguousarray(X[:, :n_rows])
    ys = np.ascontiguousarray(y[:n_rows])
    params = dict(cfg, n_trees=n_trees, n_threads=os.cpu_count() or 1)
    bins, _, n_bins = g.quantize(torch.from_numpy(Xs).cuda(), cfg["max_bins"])
    out = g.train(bins, n_bins, torch.from_numpy(ys).cuda(), **params)
    ob, _, on = oracle.quantize(Xs, cfg["max_bins"], n_threads=params["n_threads"])
    same_bins = bool(np.array_equal(bins[:, :n_rows].cpu().numpy(), ob))
    rep = {}
    compare_training(out, ob, on, ys, params, rep)
    rep.pop("trees", None)
    return dict(rows=n_rows, features=int(X.shape[0]), trees=n_trees, bins_identical=same_bins,
                trees_identical=True, **rep,
                rule="structure identical node by node; near_ties: nodes whose top two oracle gains differ by less "
                     "than 1e-12 relative; adopted_*: nodes where the GPU's equally good choice was taken (within "
                     "1e-12, or within the proven bound of its fixed-point rounding)")


def baseline_table(g, torch, args):
    """The results table of every configuration: the CUDA path (quantize + train, CUDA events; for the 50M-row
    level, build + subtract + find) and the oracle on the machine's host cores, one thread and all threads, on
    bounded samples of the same workload (rows x features x trees per second; the level: rows x features per
    second).  Parity is what tests/ checks; this table times."""
    import oracle

    threads = os.cpu_count() or 1
    stream = torch.cuda.current_stream()
    peak = _peaks()[0]
    out = {"cores": threads, "peak_gbs": peak, "configs": {}}
    # (name, extra params, oracle sample for all threads (rows, trees), for one thread (rows, trees))
    plan = [("tiny", {}, (None, None), (None, None)), ("mid", {}, (None, None), (None, 20)),
            ("covtype", {"num_leaves": 1023}, (None, 10), (None, 2)), ("large", {}, (1_000_000, 8), (1_000_000, 1))]
    for name, extra, s_all, s_one in plan:
        cfg = dict(synth.CONFIGS[name], **extra)
        X, y = synth.make(name)
        F, N = X.shape
        T = cfg["n_trees"]
        Xd, yd = torch.from_numpy(X).cuda(), torch.from_numpy(y).cuda()
        wsp = g._workspace(g.train_workspace_size(N, F, **cfg))
        pred = torch.empty(N, dtype=torch.float64, device="cuda")

        def run(diag=False):
            bins, _, n_bins = g.quantize(Xd, cfg["max_bins"])
            return g.train(bins, n_bins, yd, diagnostics=diag, ws=wsp, pred=pred, **cfg)

        run()
        torch.cuda.synchronize()
        steps = 3 if name != "large" else 1
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            run()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / steps
        diags = [run(diag=True)["diag"]]  # the histogram launches' event times (timing nodes in the tree graph)
        hist_ms = sum(d["hist_ms"] for d in diags)
        frac = sum(d["hist_level_bytes"] for d in diags) / (hist_ms * 1e-3) / 1e9 / peak if hist_ms else None
        frac_read = sum(d["hist_bytes"] for d in diags) / (hist_ms * 1e-3) / 1e9 / peak if hist_ms else None
        row = {"rows": N, "features": F, "trees": T, "gpu_ms": ms, "gpu_value": N * F * T / (ms * 1e-3),
               "hist_frac": frac, "hist_frac_read": frac_read}
        for key, (rows_s, trees_s), th in (("oracle_all", s_all, threads), ("oracle_1", s_one, 1)):
            n_s = min(N, rows_s or N)
            t_s = trees_s or T
            units, times = cpu_baseline_sample(X, y, cfg, n_s, t_s, th)
            row[key] = {"value": units / times[0], "seconds": times[0], "rows": n_s, "trees": t_s, "threads": th}
        out["configs"][name] = row
        del Xd, yd, wsp, pred
    # the 50M-row level: the CUDA path's build + subtract + find; the oracle's histograms of every node of the
    # level (it builds each node directly) and the split search of each, on a row sample
    mb = microbench(g, torch, args, peak)
    cfgm = synth.CONFIGS["micro"]
    N, F, n_nodes = args.micro_rows, cfgm["f"], cfgm["n_nodes"]
    out["configs"]["micro"] = {"rows": N, "features": F, "gpu_ms": mb["level_ms"],
                               "gpu_value": N * F / (mb["level_ms"] * 1e-3), "hist_frac": mb["build_frac"],
                               "hist_frac_moved": mb["build_moved_frac"], "unit": "rows*features/s (one level)"}
    n_s = min(N, 5_000_000)
    bins, node, gv = synth.make_micro(n=n_s, grouped=False)
    g64 = gv.astype(np.float64)
    params = dict(reg_lambda=1.0, gamma=0.0, min_samples_leaf=1, min_child_weight=0.0)
    for key, th in (("oracle_all", threads), ("oracle_1", 1)):
        groups = th if th > 1 else 1
        bounds = np.linspace(0, n_nodes, groups + 1).astype(int)
        t0 = time.perf_counter()
        if groups > 1:
            from concurrent.futures import ThreadPoolExecutor

            def one(k):
                lo, hi = bounds[k], bounds[k + 1]
                loc = np.where((node >= lo) & (node < hi), node.astype(np.int32) - lo, -1).astype(np.int32)
                h = oracle.histograms(bins, g64, loc, hi - lo)
                return [oracle.best_split(h["cnt"][i], h["G"][i], h["H"][i], np.full(F, 256, np.int32), int(h["n"][i]),
                                          float(h["Gt"][i]), float(h["Ht"][i]), **params) for i in range(hi - lo)]

            with ThreadPoolExecutor(max_workers=groups) as ex:
                list(ex.map(one, range(groups)))
        else:
            h = oracle.histograms(bins, g64, node.astype(np.int32), n_nodes)
            for i in range(n_nodes):
                oracle.best_split(h["cnt"][i], h["G"][i], h["H"][i], np.full(F, 256, np.int32), int(h["n"][i]),
                                  float(h["Gt"][i]), float(h["Ht"][i]), **params)
        sec = time.perf_counter() - t0
        out["configs"]["micro"][key] = {"value": n_s * F / sec, "seconds": sec, "rows": n_s, "threads": th}
    return out


def run_reference(args, rank, ws, dist):
    if rank != 0:
        return 0
    name = args.config
    cfg = dict(synth.CONFIGS[name])
    n_rows = min(cfg["n"], args.cpu_rows)
    X, y = synth.make(name, n=n_rows)
    threads = os.cpu_count() or 1
    units, times = cpu_baseline_sample(X, y, cfg, n_rows, args.cpu_trees, threads, repeats=args.warmup + args.steps)
    timed = times[args.warmup:]
    t = sum(timed)
    value = units * len(timed) / t
    sample = f"{n_rows:,} rows x {X.shape[0]} features x {args.cpu_trees} trees of the '{name}' workload per step"
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * t / len(timed), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": name, "rows": n_rows, "features": int(X.shape[0]), "trees": args.cpu_trees,
                       "max_depth": cfg["max_depth"], "what": "CPU oracle (plain C, FP64, row-order)"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------------------------ our arm
def microbench(g, torch, args, peak):
    """One tree level at 50M rows x 64 pre-binned features, 256 nodes (128 sibling pairs), the stated input
    and calls: each row's node is uniform over the 256 nodes and the rows are in no node order (they carry
    node ids, as a per-level node-id pass leaves them).  Timed, each with CUDA events: gbdt_build_histograms
    of the smaller child of every pair (the call groups those rows by node inside itself, then builds),
    sibling subtraction, and split search.  The parents' histograms are built untimed by the same call.
    Also timed: the same call with a workspace that only holds its error word (the node-id scan, which
    reads every row once per group of nodes) for comparison.
    """
    cfg = synth.CONFIGS["micro"]
    N, F, n_nodes = args.micro_rows, cfg["f"], cfg["n_nodes"]
    P = n_nodes // 2
    bins_h, node_h, g_h = synth.make_micro(n=N, f=F, n_nodes=n_nodes, grouped=False)
    ld = g.padded_ld(N)
    bins = torch.zeros((F, ld), dtype=torch.uint8, device="cuda")
    bins[:, :N] = torch.from_numpy(bins_h).cuda()
    del bins_h
    gd = torch.from_numpy(g_h).cuda()
    counts = np.bincount(node_h, minlength=n_nodes).astype(np.int64)
    left_small = counts[0::2] <= counts[1::2]
    flags = np.empty(n_nodes, np.uint8)
    flags[0::2], flags[1::2] = left_small, ~left_small
    fd = torch.from_numpy(flags).cuda()
    # node ids: parents 0..P-1 (the level above), children P .. P + n_nodes - 1
    child_id = torch.from_numpy((P + node_h.astype(np.int32)).astype(np.uint16).view(np.int16)).cuda()
    parent_id = torch.from_numpy((node_h >> 1).astype(np.uint16).view(np.int16)).cuda()
    dev = g._dev
    plvl = dev(np.array([(0, P)], g.LEVEL_DTYPE), g.LEVEL_DTYPE)
    lvl = dev(np.array([(P, n_nodes)], g.LEVEL_DTYPE), g.LEVEL_DTYPE)
    S = g.gradient_scale(gd)
    n_bins = torch.full((F,), 256, dtype=torch.int32, device="cuda")
    hws = g._workspace(g.lib().gbdt_histograms_workspace_size(N, F, n_nodes))
    ph_c, ph_q = g.build_histograms(bins, N, gd, S, parent_id, plvl, P, torch.ones(P, dtype=torch.uint8,
                                    device="cuda"), P, ws=hws)
    hc = torch.zeros((n_nodes, F, 256), dtype=torch.int32, device="cuda")
    hq = torch.zeros((n_nodes, F, 256), dtype=torch.int64, device="cuda")
    pair_parent = torch.arange(P, dtype=torch.int32, device="cuda")
    split_out = torch.empty(n_nodes * g.SPLIT_DTYPE.itemsize, dtype=torch.uint8, device="cuda")
    sws = g._workspace(g.lib().gbdt_subtract_histograms_workspace_size())
    stream = torch.cuda.current_stream()
    times = {"build": [], "subtract": [], "find": []}
    for it in range(args.warmup + args.steps):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record(stream)
        g.build_histograms(bins, N, gd, S, child_id, lvl, n_nodes, fd, P, hc, hq, ws=hws)
        ev[1].record(stream)
        g.subtract_histograms(ph_c, ph_q, pair_parent, fd, lvl, n_nodes, hc, hq, ws=sws)
        ev[2].record(stream)
        g.find_splits(hc, hq, S, n_bins, lvl, n_nodes, out=split_out, reg_lambda=1.0, gamma=0.0,
                      min_samples_leaf=1, min_child_weight=0.0)
        ev[3].record(stream)
        torch.cuda.synchronize()
        if it >= args.warmup:
            for k, name in enumerate(times):
                times[name].append(ev[k].elapsed_time(ev[k + 1]))
    statuses = {"build": g.workspace_status(hws), "subtract": g.workspace_status(sws)}
    ms = {k: statistics.mean(v) for k, v in times.items()}
    n_small = int(np.minimum(counts[0::2], counts[1::2]).sum())
    hist_out = P * F * 256 * 12
    formula_bytes = N * (F + 4 + 1) + hist_out  # the level formula: every row of the level read once
    # what the call moves: node ids twice (count, scatter), every row's bins and g once, the smaller children's
    # rows written grouped and read back by the histogram kernel, the built histograms written
    moved_bytes = N * (2 + 2 + F + 4) + 2 * n_small * (F + 4) + hist_out
    level_ms = ms["build"] + ms["subtract"] + ms["find"]
    res = {"workload": f"one level: {N:,} rows x {F} pre-binned uint8 features (Zipf 1.1), {n_nodes} nodes "
                       f"(each row's node uniform, rows in no node order), fp32 g",
           "call": "gbdt_build_histograms (rows grouped by node inside the call, then the node-contiguous "
                   "histogram kernel) on the smaller child of each of the 128 pairs",
           "build_ms": ms["build"], "subtract_ms": ms["subtract"], "find_splits_ms": ms["find"],
           "level_ms": level_ms,
           "build_algorithmic_bytes": formula_bytes,
           "build_gbs": formula_bytes / (ms["build"] * 1e-3) / 1e9,
           "build_frac": formula_bytes / (ms["build"] * 1e-3) / 1e9 / peak,
           "build_accounting": "level formula: N x (F + 4 B g + 1 B node id) + 128 built histograms x F x 256 x 12 B",
           "build_moved_bytes": moved_bytes,
           "build_moved_gbs": moved_bytes / (ms["build"] * 1e-3) / 1e9,
           "build_moved_frac": moved_bytes / (ms["build"] * 1e-3) / 1e9 / peak,
           "build_moved_accounting": "every byte the call reads or writes: node ids (count and scatter passes), "
                                     "all bins and g, the grouped copy of the smaller children written and read, "
                                     "the histograms",
           "level_effective_gbs": formula_bytes / (level_ms * 1e-3) / 1e9,
           "level_effective_frac": formula_bytes / (level_ms * 1e-3) / 1e9 / peak,
           "device_status": statuses, "peak_gbs": peak, "target_frac": 0.5,
           "note": "build_ms, build_gbs, build_frac and build_moved_* all time the same call; level_effective_* "
                   "divides the level formula's bytes by build + subtract + find"}
    # the node-id scan: the same call with a workspace holding only its error word
    small = g._workspace(256)
    rt = []
    for it in range(2):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        g.build_histograms(bins, N, gd, S, child_id, lvl, n_nodes, fd, P, hc, hq, ws=small)
        e1.record(stream)
        torch.cuda.synchronize()
        rt.append(e0.elapsed_time(e1))
    res["node_id_scan_build_ms"] = rt[-1]
    return res


def logistic_leg(g, torch, args, cfg, N, F, Xd, y, pred, peak, peak_kind, stream):
    """The logistic objective on the same matrix (0/1 labels: above the median): whole training runs
    timed with CUDA events, and the level histograms (count, G and H) against the HBM roofline."""
    params = dict(cfg, objective=1)
    T = params["n_trees"]
    yb = torch.from_numpy(synth.binary_label(y)).cuda()
    lws = g._workspace(g.train_workspace_size(N, F, **params))

    def run(diag=False):
        bins, _, n_bins = g.quantize(Xd, params["max_bins"])
        return g.train(bins, n_bins, yb, diagnostics=diag, ws=lws, pred=pred, **params)

    for _ in range(max(1, min(args.warmup, 2))):
        run()
    torch.cuda.synchronize()
    steps = max(1, min(args.steps, 2))
    diags = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = g.kernel_launch_count()
    e0.record(stream)
    for _ in range(steps):
        diags.append(run(diag=True)["diag"])
    e1.record(stream)
    torch.cuda.synchronize()
    n_launch = g.kernel_launch_count() - l0
    ms = e0.elapsed_time(e1) / steps
    hist_ms = sum(d["hist_ms"] for d in diags)
    hist_bytes = sum(d["hist_bytes"] for d in diags)
    level_bytes = sum(d["hist_level_bytes"] for d in diags)
    launches = sum(d["hist_launches"] for d in diags)
    part_ms = sum(d["part_ms"] for d in diags)
    part_bytes = sum(d["part_bytes"] for d in diags)
    achieved = level_bytes / (hist_ms * 1e-3) / 1e9
    achieved_read = hist_bytes / (hist_ms * 1e-3) / 1e9
    return {"metric": METRIC, "value": N * F * T / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "objective": "logistic (binary cross-entropy of a sigmoid); labels 1 where the regression label "
                         "exceeds its median",
            "step": "gbdt_quantize + gbdt_train, same matrix and parameters as the main line",
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                         "frac": achieved / peak, "traffic": None, "peak_kind": peak_kind,
                         "kernel": "seg_hist_kernel with H (count, G and H per entry; 32 features per CTA)",
                         "launches": launches, "avg_launch_ms": hist_ms / launches,
                         "algorithmic_bytes_per_launch": level_bytes / launches,
                         "accounting": "level formula (as the main line; 20 B per histogram entry with H)",
                         "read_bytes_per_launch": hist_bytes / launches, "achieved_read": achieved_read,
                         "frac_read": achieved_read / peak, "share_of_step": hist_ms / (ms * steps)},
            "partition": {"achieved_gbs": part_bytes / (part_ms * 1e-3) / 1e9,
                          "frac": part_bytes / (part_ms * 1e-3) / 1e9 / peak, "share_of_step": part_ms / (ms * steps)},
            "trees_at_full_size": diags[-1]["trees_at_full_size"]}


def covtype_leg(g, torch, args, peak, peak_kind, stream):
    """The covtype-shaped workload in the pages' configuration (581,012 x 54, 255 bins, depth 10,
    1023 leaves, 100 trees): whole quantize + training runs timed with CUDA events."""
    cfg = dict(synth.CONFIGS["covtype"], num_leaves=1023, hist_registers=args.hist_registers)
    if args.covtype_trees is not None:
        cfg["n_trees"] = args.covtype_trees
    X, y = synth.make("covtype")
    F, N = X.shape
    T = cfg["n_trees"]
    Xd, yd = torch.from_numpy(X).cuda(), torch.from_numpy(y).cuda()
    cws = g._workspace(g.train_workspace_size(N, F, **cfg))
    cpred = torch.empty(N, dtype=torch.float64, device="cuda")

    def run(diag=False):
        bins, _, n_bins = g.quantize(Xd, cfg["max_bins"])
        return g.train(bins, n_bins, yd, diagnostics=diag, ws=cws, pred=cpred, **cfg)

    for _ in range(2):
        run()
    torch.cuda.synchronize()
    steps = 3
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    l0 = g.kernel_launch_count()
    e0.record(stream)
    for _ in range(steps):
        run()
    e1.record(stream)
    torch.cuda.synchronize()
    n_launch = g.kernel_launch_count() - l0
    ms = e0.elapsed_time(e1) / steps
    # the histogram launches' own times: the same runs with diagnostics (timing events around every
    # level's launches, recorded as nodes of the replayed tree graph; they add gaps, so these runs are
    # not the timed ones)
    diags = [run(diag=True)["diag"] for _ in range(2)]
    torch.cuda.synchronize()
    ms_diag = sum(d["total_ms"] for d in diags) / len(diags)
    hist_ms = sum(d["hist_ms"] for d in diags)
    hist_bytes = sum(d["hist_bytes"] for d in diags)
    level_bytes = sum(d["hist_level_bytes"] for d in diags)
    launches = sum(d["hist_launches"] for d in diags)
    achieved = level_bytes / (hist_ms * 1e-3) / 1e9
    achieved_read = hist_bytes / (hist_ms * 1e-3) / 1e9
    return {"metric": METRIC, "value": N * F * T / (ms * 1e-3), "unit": UNIT, "ms_per_step": ms, "steps": steps,
            "workload": f"covtype-shaped: {N:,} rows x {F} features (10 integer, 44 one-hot binary), 255 bins, "
                        f"depth 10, 1023 leaves, {T} trees",
            "step": "gbdt_quantize + gbdt_train",
            "launches_per_step": n_launch / steps,
            "launches_per_tree": n_launch / (steps * T),
            "train_ms_with_diagnostics": ms_diag,
            "timing": "ms_per_step: runs without diagnostics (trees 1 .. T-2 replay one captured graph); hist: "
                      "two more runs with diagnostics (the same graph with timing events around each level's "
                      "launches)",
            "hist": {"achieved_gbs": achieved, "frac": achieved / peak, "accounting": "level formula",
                     "achieved_read_gbs": achieved_read, "frac_read": achieved_read / peak, "peak_kind": peak_kind,
                     "avg_launch_ms": hist_ms / launches, "share_of_step": hist_ms / (ms * len(diags))},
            "part_share_of_step": sum(d["part_ms"] for d in diags) / (ms * len(diags)),
            "page_context": {"train_s": 4.5, "hardware": "RTX 5090", "semantics": "leaf-wise, real covtype data",
                             "value": 581012 * 54 * 100 / 4.5,
                             "note": "the pages' own figure, other hardware and semantics: context, not a target"}}


def run_ours(args, rank, local_rank, ws, dist):
    import torch

    import histogram_gradient_boosted_gb300 as g
    from histogram_gradient_boosted_gb300 import build as gb

    torch.cuda.set_device(local_rank)
    gb.build()
    g.lib()
    if args.only_micro:
        print(json.dumps({"histogram_microbench": microbench(g, torch, args, _peaks()[0])}), flush=True)
        return 0
    if args.baseline_table:
        print(json.dumps({"baseline_table": baseline_table(g, torch, args)}), flush=True)
        return 0
    if args.only_covtype:
        peak, peak_kind = _peaks()
        print(json.dumps({"covtype": covtype_leg(g, torch, args, peak, peak_kind, torch.cuda.current_stream())}),
              flush=True)
        return 0
    name = args.config
    cfg = dict(synth.CONFIGS[name], hist_registers=args.hist_registers)
    if args.trees is not None:
        cfg["n_trees"] = args.trees
    X, y = synth.make(name, n=args.rows)
    F, N = X.shape
    T = cfg["n_trees"]
    Xd = torch.from_numpy(X).cuda()
    yd = torch.from_numpy(y).cuda()
    peak, peak_kind = _peaks()
    stream = torch.cuda.current_stream()
    train_ws = g._workspace(g.train_workspace_size(N, F, **cfg))
    pred = torch.empty(N, dtype=torch.float64, device="cuda")

    def step(diag=False):
        bins, _, n_bins = g.quantize(Xd, cfg["max_bins"])
        return g.train(bins, n_bins, yd, diagnostics=diag, ws=train_ws, pred=pred, **cfg)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # ---- timed region: K steps, device time by CUDA events ----
    diags = []
    _barrier(dist)
    torch.cuda.synchronize()
    l0 = g.kernel_launch_count()
    with ClockSampler(local_rank) as clk:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            out = step(diag=True)
            diags.append(out["diag"])
        e1.record(stream)
        torch.cuda.synchronize()
    launches = g.kernel_launch_count() - l0
    _barrier(dist)
    ms_total = _max_over_ranks(e0.elapsed_time(e1), dist)
    units = N * F * T * args.steps * ws
    value = units / (ms_total * 1e-3)
    clocks = clk.summary()

    # train-only (bins already binned), from the library's own device time of the call
    train_ms = statistics.mean(d["total_ms"] for d in diags)
    hist_ms = sum(d["hist_ms"] for d in diags)
    hist_bytes = sum(d["hist_bytes"] for d in diags)
    level_bytes = sum(d["hist_level_bytes"] for d in diags)
    hist_launches = sum(d["hist_launches"] for d in diags)
    achieved = level_bytes / (hist_ms * 1e-3) / 1e9
    achieved_read = hist_bytes / (hist_ms * 1e-3) / 1e9
    trec = _traffic_record()
    part_ms = sum(d["part_ms"] for d in diags)
    part_bytes = sum(d["part_bytes"] for d in diags)
    roofline = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s", "frac": achieved / peak,
                "traffic": _scaled_traffic(trec, hist_bytes / hist_launches),
                "traffic_source": (f"ncu DRAM bytes of one tree's level histograms at {trec.get('captured_rows', N):,} "
                                   "rows, scaled to this workload's launches by the bytes they read "
                                   "(profiles/histogram_traffic.json)" if trec else "not recorded for this kernel"),
                "kernel": "seg_hist_kernel (level histograms inside gbdt_train; smaller children, node-contiguous)",
                "launches": hist_launches, "avg_launch_ms": hist_ms / hist_launches,
                "algorithmic_bytes_per_launch": level_bytes / hist_launches,
                "accounting": "level formula: rows of the level's nodes x (F + 8 B g + 2 B node id) + built "
                              "histograms x F x 256 x 12 B",
                "read_bytes_per_launch": hist_bytes / hist_launches, "achieved_read": achieved_read,
                "frac_read": achieved_read / peak,
                "read_accounting": "what this kernel reads: rows scanned (smaller children after a move, the "
                                   "parents' rows at a filtered level) x (slots + 8 B g (+1 B decision)) + the "
                                   "built histograms; traffic (ncu DRAM bytes) compares with this",
                "peak_kind": peak_kind, "share_of_step": hist_ms / ms_total if ms_total else None}

    # ---- e2e: public API with host inputs ----
    Xp = torch.empty((F, N), dtype=torch.float32, pin_memory=True)
    Xp.copy_(torch.from_numpy(X))
    yp = torch.empty(N, dtype=torch.float32, pin_memory=True)
    yp.copy_(torch.from_numpy(y))
    pred_h = torch.empty(N, dtype=torch.float64, pin_memory=True)
    e2e_steps = max(1, min(args.steps, 2))

    def e2e_step():
        # the public API on host features: gbdt_quantize_host copies X into Xd column batch by column batch
        # while the batches already copied are binned; labels copied before; predictions read back
        c0, c1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        c0.record(stream)
        yd.copy_(yp, non_blocking=True)
        bins_e, _, n_bins_e = g.quantize(Xp, cfg["max_bins"], x_device=Xd)
        c1.record(stream)
        out = g.train(bins_e, n_bins_e, yd, ws=train_ws, pred=pred, **cfg)
        pred_h.copy_(out["pred"], non_blocking=True)
        torch.cuda.synchronize()
        return c0.elapsed_time(c1)

    # one untimed step first, as for the device-resident steps: the first host-input call allocates its
    # outputs and workspace (the caching allocator may have no block of that size yet)
    e2e_step()
    # this machine's host link: one plain copy of the pinned features (boxes differ several-fold here)
    torch.cuda.synchronize()
    k0, k1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    k0.record(stream)
    Xd.copy_(Xp, non_blocking=True)
    k1.record(stream)
    torch.cuda.synchronize()
    host_copy_gbs = Xp.numel() * 4 / (k0.elapsed_time(k1) * 1e-3) / 1e9
    _barrier(dist)
    torch.cuda.synchronize()
    h2d_each = []
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        h2d_each.append(e2e_step())
    e2e_s = _max_over_ranks(time.perf_counter() - t0, dist)
    h2d_ms = sum(h2d_each)
    M = (1 << (cfg["max_depth"] + 1)) - 1
    h2d = Xp.numel() * 4 + yp.numel() * 4
    d2h = T * M * 40 + T * 4 + N * 8
    e2e = {"value": N * F * T * e2e_steps * ws / e2e_s, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": 1e3 * e2e_s / e2e_steps,
           "h2d_and_quantize_ms_per_step": h2d_ms / e2e_steps, "h2d_and_quantize_ms_each": h2d_each,
           "warmup": 1, "host_copy_gbs": host_copy_gbs,
           "path": "gbdt_quantize_host (pinned host features, copies overlapped with binning) + gbdt_train; "
                   "labels copied before, predictions and model read back"}

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": ms_total / args.steps, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "int64 fixed-point histograms, f64 gradients/gains", "data": "synthetic (seeded numpy)",
            "config": {"workload": f"{name}: {N:,} rows x {F} features, {cfg['max_bins']} bins, depth "
                                   f"{cfg['max_depth']}, {T} trees", "rows": N, "features": F, "trees": T,
                       "max_depth": cfg["max_depth"], "step": "gbdt_quantize + gbdt_train (all hot-path steps)",
                       "l2": "inputs larger than L2 (4 GB fp32 features, 1 GB bins)",
                       "parallelism": "replicas" if ws > 1 else "single GPU"},
            "e2e": e2e, "gpu_launches": launches, "gpu_launches_per_step": launches / args.steps,
            "roofline": roofline, "clocks": clocks,
            "partition": {"ms_per_step": part_ms / args.steps, "achieved_gbs": part_bytes / (part_ms * 1e-3) / 1e9,
                          "frac": part_bytes / (part_ms * 1e-3) / 1e9 / peak,
                          "share_of_step": part_ms / ms_total if ms_total else None},
            "train_only": {"ms_per_run": train_ms, "value": N * F * T / (train_ms * 1e-3)},
            "trees_at_full_size": diags[-1]["trees_at_full_size"]}
    # ---- batched prediction of the training rows with the trained model (raw fp32 features) ----
    bins_i, edges_i, n_bins_i = g.quantize(Xd, cfg["max_bins"])
    model = g.train(bins_i, n_bins_i, yd, ws=train_ws, pred=pred, **cfg)
    del bins_i
    pout = torch.empty(N, dtype=torch.float64, device="cuda")
    pws = g._workspace(g.lib().gbdt_predict_workspace_size(T, M))
    for _ in range(2):
        g.predict(Xd, edges_i, model["nodes"], model["init_pred"], cfg["learning_rate"], model["nodes_per_tree"],
                  out=pout, ws=pws)
    torch.cuda.synchronize()
    p_steps = 3
    e0.record(stream)
    for _ in range(p_steps):
        g.predict(Xd, edges_i, model["nodes"], model["init_pred"], cfg["learning_rate"], model["nodes_per_tree"],
                  out=pout, ws=pws)
    e1.record(stream)
    torch.cuda.synchronize()
    p_ms = e0.elapsed_time(e1) / p_steps
    line["inference"] = {"metric": "rows x trees predicted per second (raw fp32 features)",
                         "value": N * T / (p_ms * 1e-3), "ms": p_ms, "rows": N, "trees": T,
                         "equals_training_predictions": bool(torch.equal(pout, model["pred"])),
                         "note": "gbdt_predict on the training rows, inputs resident; the call includes its node "
                                 "preparation pass and one stream synchronisation"}
    del pout, pws
    if not args.no_logistic:
        line["logistic"] = logistic_leg(g, torch, args, cfg, N, F, Xd, y, pred, peak, peak_kind, stream)
    if not args.no_covtype:
        line["covtype"] = covtype_leg(g, torch, args, peak, peak_kind, stream)
    if rank == 0 and not args.no_micro:
        line["histogram_microbench"] = microbench(g, torch, args, peak)
    if rank == 0 and not args.no_cpu:
        threads = os.cpu_count() or 1
        n_rows = min(N, args.cpu_rows)
        units_c, times_c = cpu_baseline_sample(X, y, cfg, n_rows, args.cpu_trees, threads)
        line["cpu_baseline"] = {"value": units_c / times_c[0], "unit": UNIT, "cores": threads, "kind": "oracle",
                                "sample": f"first {n_rows:,} rows x {F} features x {args.cpu_trees} trees of the "
                                          f"same matrix (oracle quantize untimed)", "seconds": times_c[0]}
        n1 = min(N, args.cpu_rows_single)
        units_1, times_1 = cpu_baseline_sample(X, y, cfg, n1, args.cpu_trees_single, 1)
        line["cpu_baseline"]["single_thread"] = {
            "value": units_1 / times_1[0], "unit": UNIT, "cores": 1, "seconds": times_1[0],
            "sample": f"first {n1:,} rows x {F} features x {args.cpu_trees_single} trees of the same matrix"}
        if not args.no_parity_sample:
            line["parity_sample"] = parity_sample(g, torch, X, y, cfg, min(N, args.parity_rows), args.parity_trees)
    if rank == 0:
        print(json.dumps(line), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default="large", choices=["tiny", "mid", "covtype", "large"])
    ap.add_argument("--rows", type=int, default=None, help="override the workload's row count")
    ap.add_argument("--trees", type=int, default=None, help="override the workload's tree count (profiling runs)")
    ap.add_argument("--micro-rows", type=int, default=synth.CONFIGS["micro"]["n"])
    ap.add_argument("--cpu-rows", type=int, default=1_000_000)
    ap.add_argument("--cpu-trees", type=int, default=32, help="trees of the oracle sample (about 10 s on 16 cores)")
    ap.add_argument("--cpu-rows-single", type=int, default=1_000_000)
    ap.add_argument("--cpu-trees-single", type=int, default=2, help="trees of the single-thread oracle sample")
    ap.add_argument("--parity-rows", type=int, default=1_000_000)
    ap.add_argument("--parity-trees", type=int, default=8, help="trees of the node-by-node parity sample")
    ap.add_argument("--no-parity-sample", action="store_true")
    ap.add_argument("--no-micro", action="store_true")
    ap.add_argument("--no-cpu", action="store_true")
    ap.add_argument("--no-logistic", action="store_true", help="skip the logistic-objective leg")
    ap.add_argument("--no-covtype", action="store_true", help="skip the covtype-shaped leg")
    ap.add_argument("--only-micro", action="store_true", help="run only the level microbench (profiling)")
    ap.add_argument("--only-covtype", action="store_true", help="run only the covtype-shaped leg (profiling)")
    ap.add_argument("--hist-registers", type=int, default=0, choices=[0, 1],
                    help="accumulate features of at most 8 bins in registers (gbdt_params.hist_registers)")
    ap.add_argument("--baseline-table", action="store_true",
                    help="time every configuration on the GPU and the oracle (one thread, all threads)")
    ap.add_argument("--covtype-trees", type=int, default=None, help="trees of the covtype-shaped leg (profiling)")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        print("note: fewer than 3 warm-up steps", file=sys.stderr)
    rank, local_rank, ws, dist = _dist()
    try:
        if args.impl == "reference":
            return run_reference(args, rank, ws, dist)
        return run_ours(args, rank, local_rank, ws, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


if __name__ == "__main__":
    sys.exit(main())

#!/usr/bin/env python3
"""Benchmark: one k-means Lloyd iteration (assign + mean update) per step.

Workload (default ``sample_heavy``, the largest of the five shapes): n =
131072 samples, k = 8192 centroids, d = 8192 features, float32 planted
Gaussian blobs (8192 centers ~ N(0, 1), noise sigma 0.5), initial centroids =
seeded random rows of X.  Each step is one Lloyd iteration whose output
centroids feed the next step.  ``--workload`` selects another shape (probe,
lloyd10, centroid_heavy, feature_heavy).

Printed JSON line (rank 0):
* ``value``: whole-job throughput in TFLOP/s, 2 n k d per Lloyd iteration
  over the device time of the K timed iterations (inputs resident in HBM);
* ``ms_per_step``: the Lloyd iteration time;
* ``assign``: the assignment call alone (2 n k d over its time) and its
  fraction of the fp32-accurate tensor roofline; ``roofline`` describes it;
* ``e2e``: the same metric through the public API with the step's inputs
  copied from pinned host memory and its results copied back, every step;
* ``cpu_baseline``: the CPU oracle on a bounded sample of the same workload;
* ``parity``: the GPU assignment and update against the oracle outputs of
  that same leg (sampled rows; the update on every row), and the k-means++
  indices against the stored oracle indices.

``--impl reference`` times the CPU oracle alone (the reference arm).
Under torchrun every rank runs its own replica of the workload (the update
needs every sample's label, so one problem does not shard without an
all-reduce; replicas only).
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

MEASURED_PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "assign_tc_kernel_traffic.json")
KMEANSPP_GOLDEN = os.path.join(ROOT, "tests", "golden", "kmeanspp_workload_indices.txt")
KERNEL_SOURCE = os.path.join(ROOT, "distance_argmin_gb300", "csrc", "assign_tc.cu")
METRIC = "Lloyd iter time & assign TFLOP/s (2nkd/t) at 1 GB300, % of fp32-accurate roofline"
SPLIT_PRODUCTS = 3  # bf16x3: hi*hi + hi*lo + lo*hi per fp32 product
TF32_NOMINAL_TFLOPS = 1100.0  # dense, per GPU (context; no measured TF32 peak)


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--workload", default="sample_heavy")
    ap.add_argument("--rows", type=int, default=0,
                    help="keep only the workload's first ROWS samples (a smaller case of the same shape for "
                         "profiler captures; the JSON line names it)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-kmeanspp", action="store_true")
    ap.add_argument("--e2e-slices", type=int, default=16,
                    help="row slices of kmeans_lloyd_iter_host in the end-to-end leg")
    return ap.parse_args()


def load_peaks():
    if os.path.exists(MEASURED_PEAKS):
        with open(MEASURED_PEAKS) as f:
            p = json.load(f)
        return p, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def code_sha256(path):
    """sha256 of a C++ source with its comments and blank lines removed, so
    that a comment edit does not count as a kernel change."""
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = [re.sub(r"//.*$", "", l).rstrip() for l in text.splitlines()]
    return hashlib.sha256("\n".join(l for l in lines if l.strip()).encode()).hexdigest()


def recorded_traffic(workload):
    """Per-launch DRAM bytes (read + write) of the assign kernel on this
    workload, from the committed ncu record, if it was taken on the current
    kernel code; else None."""
    if not os.path.exists(TRAFFIC_RECORD):
        return None
    with open(TRAFFIC_RECORD) as f:
        rec = json.load(f).get("records", {}).get(workload)
    if not rec or rec.get("code_sha256") != code_sha256(KERNEL_SOURCE):
        return None
    return float(rec["dram_bytes_per_launch"])


def gib(nbytes):
    return f"{nbytes / 2**30:.3g} GiB" if nbytes >= 2**30 else f"{nbytes / 2**20:.3g} MiB"


def launches_per_lloyd_step(k: int) -> int:
    """Kernels one kmeans_lloyd_iter call launches (the library's own)."""
    assign = 3  # prep_split, assign_tc, finalize
    if k <= 32768:
        # finalize also counts the members per tile; then col_prefix (with
        # the offsets scan), tile_scatter, segmented_mean, fixup
        return assign + 4
    bits = 0
    while (1 << bits) < k:
        bits += 1
    passes = max(1, (bits + 7) // 8)
    return assign + 1 + 3 * passes + 3  # clear, passes x (hist, scan, scatter), scan, mean, fixup


# ---------------------------------------------------------------- clocks
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: str):
        self.gpu_index = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_index, f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), float(parts[3]), parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        pmax = max(r[2] for r in rows)
        loaded = [r for r in rows if r[2] >= 0.5 * pmax] or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in loaded for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in loaded), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(loaded), "power_w_max": pmax}


# ---------------------------------------------------------------- helpers
def env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(values, world, device="cpu"):
    """Element-wise maximum of this rank's timings over all ranks (the
    slowest rank sets every time); a plain copy when world == 1."""
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    if world > 1:
        import torch.distributed as dist
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(v) for v in t.cpu()]


def whole_job_tflops(flop_per_rank, world, seconds):
    """Whole-job throughput: every rank's work over the slowest rank's time."""
    return world * flop_per_rank / seconds / 1e12


def oracle_sample_step(oracle, X, C, rows):
    """One bounded-sample Lloyd step of the oracle: assign the sampled rows,
    then the mean update over those rows.  Returns (seconds, the assignment's
    (labels, best, second))."""
    t0 = time.perf_counter()
    o_l, o_b, o_s, _ = oracle.assign(X[rows], C)
    oracle.update(X[rows], o_l, C)
    return time.perf_counter() - t0, (o_l, o_b, o_s)


DIST_RTOL = 1e-4      # best distance, relative to ||x||^2 + ||c_best||^2
CENTROID_RTOL = 1e-5  # centroid row, relative to the row's largest magnitude


def sq_norms(A):
    import numpy as np
    A64 = A.astype(np.float64)
    return np.einsum("ij,ij->i", A64, A64)


def assign_parity(X, C, rows, labels, best, o_l, o_b, o_s):
    """The GPU's labels and best distances on ``rows`` against the oracle's:
    the worst relative distance error, label mismatches where the oracle's
    winner is clear (must be 0) and near-tie flips (allowed, counted)."""
    import numpy as np
    lab = labels[rows]
    scale = sq_norms(X[rows]) + sq_norms(C)[o_l]
    rel = np.abs(best[rows].astype(np.float64) - o_b) / scale
    clear = (o_s - o_b) > DIST_RTOL * scale
    return {"rows_checked": int(len(rows)), "worst_rel_distance_error": float(rel.max()),
            "distances_within_tolerance": bool((rel <= DIST_RTOL).all()),
            "clear_label_mismatches": int((clear & (lab != o_l)).sum()),
            "near_tie_flips": int((~clear & (lab != o_l)).sum()),
            "near_ties": int((~clear).sum())}


def centroid_parity(C_gpu, counts_gpu, o_C, o_counts):
    """Per centroid row: max |gpu - oracle| over max |oracle row|."""
    import numpy as np
    got = C_gpu.astype(np.float64)
    want = o_C.astype(np.float64)
    row_scale = np.maximum(np.abs(want).max(axis=1), np.finfo(np.float32).tiny)
    rel = np.abs(got - want).max(axis=1) / row_scale
    return {"worst_centroid_row_error": float(rel.max()),
            "centroids_within_tolerance": bool((rel <= CENTROID_RTOL).all()),
            "counts_equal": bool(np.array_equal(counts_gpu.astype(np.int64), o_counts))}


def cpu_baseline(oracle, w, X, C0, gpu=None, budget_s=20.0):
    """Time the oracle (as it stands, all host cores) on seeded row samples
    of the workload; TFLOP/s = 2 * rows * k * d / time (the per-row cost of
    the full iteration is the same for every row).

    ``gpu`` (labels, best, C_new, counts of the GPU's assignment of every row
    to C0 and its update on those labels) is compared, after the timing, with
    the oracle outputs of the timed sample and with the oracle's update of
    every row on the GPU's labels (so near-tie flips do not cascade)."""
    import numpy as np
    rng = np.random.default_rng(7)
    rows = np.sort(rng.choice(w.n, size=min(w.n, 256), replace=False))
    t, _ = oracle_sample_step(oracle, X, C0, rows)  # calibrate
    m = int(min(w.n, max(256, 256 * budget_s / max(t, 1e-3) * 0.8)))
    rows = np.sort(rng.choice(w.n, size=m, replace=False))
    t, (o_l, o_b, o_s) = oracle_sample_step(oracle, X, C0, rows)
    base = {"value": 2.0 * m * w.k * w.d / t / 1e12, "unit": "TFLOP/s", "cores": oracle.max_threads(),
            "kind": "oracle", "sample": f"{m} of {w.n} seeded rows: binary64 brute-force assign of the rows "
                                        f"against all {w.k} centroids + mean update of those rows; {t:.1f} s"}
    parity = None
    if gpu is not None:
        labels, best, C_new, counts = gpu
        parity = assign_parity(X, C0, rows, labels, best, o_l, o_b, o_s)
        parity["rows"] = "the cpu_baseline leg's seeded sample, assigned to the initial centroids"
        o_C, o_cnt = oracle.update(X, labels, C0)
        parity.update(centroid_parity(C_new, counts, o_C, o_cnt))
        parity["update"] = "every row, on the GPU's labels"
    return base, parity


# ------------------------------------------------------------ reference arm
def run_reference(args):
    rank, world, _ = env_rank()
    if rank != 0:
        return 0
    import numpy as np
    import oracle
    import synth
    oracle.build()
    w = synth.WORKLOADS[args.workload]
    X, C0, _ = synth.workload_inputs(w)
    rng = np.random.default_rng(11)
    rows_per_step = 256
    samples = [np.sort(rng.choice(w.n, size=rows_per_step, replace=False)) for _ in range(args.warmup + args.steps)]
    for i in range(args.warmup):
        oracle_sample_step(oracle, X, C0, samples[i])
    t = 0.0
    for i in range(args.steps):
        t += oracle_sample_step(oracle, X, C0, samples[args.warmup + i])[0]
    ms_per_step = 1e3 * t / args.steps
    value = 2.0 * rows_per_step * w.k * w.d / (t / args.steps) / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "n": w.n, "k": w.k, "d": w.d, "blobs": w.blobs,
                   "step": f"oracle Lloyd step on {rows_per_step} seeded rows"},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": f"{rows_per_step} seeded rows of {w.n} per step"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# -------------------------------------------------------------- GB300 arm
def kmeanspp_matches_stored_oracle(X, w, T, got):
    """The seeding's indices against the oracle's, stored with the SHA-256 of
    the samples it saw: True/False, or None when this host's generator gave
    other samples (the stored answer then does not apply)."""
    import numpy as np
    if not os.path.exists(KMEANSPP_GOLDEN):
        return None
    meta, want = {}, []
    for line in open(KMEANSPP_GOLDEN):
        if line.startswith("#"):
            meta.update(tok.split("=", 1) for tok in line[1:].split() if "=" in tok)
        elif line.strip():
            want.append(int(line))
    if ((int(meta.get("n", -1)), int(meta.get("d", -1)), int(meta.get("k", -1)), int(meta.get("seed", -1)),
         int(meta.get("trials", -1))) != (w.n, w.d, w.k, w.init_seed, T)
            or hashlib.sha256(X.tobytes()).hexdigest() != meta.get("x_sha256")):
        return None
    return bool(np.array_equal(np.asarray(got), np.asarray(want, dtype=np.int64)))


def time_kmeanspp(km, synth, dev, stream, barrier):
    """Greedy k-means++ on its own workload (65536 x 8192, 1024 centers,
    8 trials): one timed call after a short warm-up call."""
    import torch
    w = synth.KMEANSPP
    X, _, _ = synth.planted_blobs(w.n, w.d, w.blobs, w.data_seed)
    Xd = torch.from_numpy(X).to(dev)
    T = km.n_trials_for(w.k)
    ws = km.workspace(km.OP_KMEANSPP, w.n, w.k, w.d, dev)
    idx = torch.empty(w.k, dtype=torch.int64, device=dev)
    cen = torch.empty((w.k, w.d), dtype=torch.float32, device=dev)
    km.kmeanspp_init(Xd, 8, w.init_seed, n_trials=T, ws=ws, stream=stream)
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def seed_once(trace):
        # event records between the chained launches hold each launch back
        # until its predecessor has drained, so the call is timed without
        # them and then once more with them for the distance pass alone
        if trace:
            km.kmeans_trace_start(2 * w.k + 8)
        e0.record(stream)
        km.kmeanspp_init(Xd, w.k, w.init_seed, n_trials=T, centers=cen, indices=idx, ws=ws, stream=stream)
        e1.record(stream)
        barrier()
        return e0.elapsed_time(e1) / 1e3

    t = seed_once(False)
    first = idx.clone()
    rows = km.kmeanspp_rows_read(ws, stream)
    match = kmeanspp_matches_stored_oracle(X, w, T, first.cpu().numpy())
    t_traced = seed_once(True)
    dist_ms, dist_timed, dist_seen = km.kmeans_trace_read(km.KERNEL_KMEANSPP_DIST)
    km.kmeans_trace_stop()
    assert torch.equal(first, idx)
    # one distance pass over every row: X once, plus its (slice, trial,
    # sample) float2 partial sums; rows that every trial provably leaves at
    # their D^2 are skipped, so the passes read `rows` rows in all
    passes = w.k * ((T + 7) // 8)
    if rows <= 0:
        rows = w.n * passes  # no pruning: every pass reads every row
    slices = (w.d + km.KPP_SLICE_FEATURES - 1) // km.KPP_SLICE_FEATURES
    row_bytes = 4.0 * w.d + 8.0 * slices * T
    full_pass = row_bytes * w.n
    read = row_bytes * rows  # over the whole seeding
    t_pass = dist_ms / 1e3 / max(dist_timed, 1)
    return {"workload": f"n={w.n} d={w.d} k={w.k} trials={T}", "ms": 1e3 * t, "gbs": read / t / 1e9,
            "ms_per_center": 1e3 * t / w.k, "indices_match_oracle": match,
            "rows_read_fraction": rows / (w.n * passes),
            "unpruned_hbm_floor_ms": 1e3 * full_pass * passes / (load_peaks()[0]["hbm_gbs"] * 1e9),
            "distance_pass": {"kernel": "kpp_dist_part_kernel", "launches": dist_seen, "us": 1e6 * t_pass,
                              "bytes_per_launch": read / passes, "gbs": read / passes / t_pass / 1e9,
                              "bytes_per_launch_unpruned": full_pass,
                              "share_of_call": dist_ms / 1e3 / t_traced,
                              "timed": "a second seeding with CUDA events around each distance pass "
                                       f"({1e3 * t_traced:.1f} ms with them)"},
            "pruning": "each round reads only the rows some trial can bring below their D^2 (triangle "
                       "inequality through the nearest chosen center); gbs and frac_of_hbm count the bytes read"}


def run_gb300(args):
    import numpy as np
    import torch
    import torch.distributed as dist

    import distance_argmin_gb300 as km
    import synth

    rank, world, local = env_rank()
    if world > 1:
        dist.init_process_group("nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    from distance_argmin_gb300 import build as kb
    kb.build()
    km.load()

    w = synth.WORKLOADS[args.workload]
    X, C0, _ = synth.workload_inputs(w)
    if 0 < args.rows < w.n:
        if args.rows < w.k:
            raise SystemExit(f"--rows {args.rows} is below k = {w.k}")
        X = np.ascontiguousarray(X[:args.rows])
        w = synth.Workload(f"{w.name}_rows{args.rows}", args.rows, w.k, w.d, w.blobs, w.iters, w.data_seed,
                           w.init_seed, w.note + f"; first {args.rows} samples only")
    n, k, d = w.n, w.k, w.d
    flop = 2.0 * n * k * d
    Xd = torch.from_numpy(X).to(dev)
    C0d = torch.from_numpy(C0).to(dev)
    Cbuf = [C0d.clone(), torch.empty_like(C0d)]
    labels = torch.empty(n, dtype=torch.int64, device=dev)
    best = torch.empty(n, dtype=torch.float32, device=dev)
    counts = torch.empty(k, dtype=torch.int32, device=dev)
    steps, warm = args.steps, args.warmup
    inertia = torch.zeros(max(steps, warm, 1), dtype=torch.float64, device=dev)
    ws = km.workspace(km.OP_LLOYD, n, k, d, dev)
    stream = torch.cuda.current_stream(dev)

    def lloyd(i, slot):
        src, dst = Cbuf[i % 2], Cbuf[(i + 1) % 2]
        km.kmeans_lloyd_iter(Xd, src, dst, labels, best, inertia[slot:slot + 1], counts, ws=ws, stream=stream)

    def barrier():
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize(dev)

    gpu_index = os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[local if world > 1 else 0]
    sampler = ClockSampler(gpu_index)

    # warm-up Lloyd iterations from C0, then restart from C0 for the timed run
    for i in range(warm):
        lloyd(i, i)
    Cbuf[0].copy_(C0d)
    barrier()
    sampler.start()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        lloyd(i, i)
    ev1.record(stream)
    barrier()
    t_lloyd = ev0.elapsed_time(ev1) / 1e3 / steps
    inertia_hist = inertia[:steps].cpu().numpy()
    final_C = Cbuf[steps % 2].clone()

    # The same run again with the library's CUDA events around its two
    # dominant kernels, on this stream, for their own durations.  An event
    # record between two chained launches holds the second back until the
    # first has drained, which costs the step about 4% here, so the run
    # above, without them, gives the step time.
    Cbuf[0].copy_(C0d)
    km.kmeans_trace_start(steps + 8)
    barrier()
    ev0.record(stream)
    for i in range(steps):
        lloyd(i, i)
    ev1.record(stream)
    barrier()
    t_lloyd_traced = ev0.elapsed_time(ev1) / 1e3 / steps
    tc_ms, tc_timed, tc_seen = km.kmeans_trace_read(km.KERNEL_ASSIGN_TC)
    mean_ms, mean_timed, _ = km.kmeans_trace_read(km.KERNEL_UPDATE_MEAN)
    km.kmeans_trace_stop()
    assert tc_timed == steps and tc_seen == steps and mean_timed == steps
    t_tc = tc_ms / 1e3 / tc_timed
    t_mean = mean_ms / 1e3 / mean_timed
    # both runs start from C0 and are deterministic
    assert torch.equal(final_C, Cbuf[steps % 2])

    # the assignment alone (prep + tensor-core kernel + finalize), same stream
    ws_a = km.workspace(km.OP_ASSIGN, n, k, d, dev)
    inertia_a = torch.empty(1, dtype=torch.float64, device=dev)
    for _ in range(warm):
        km.kmeans_assign(Xd, C0d, labels, best, inertia_a, ws=ws_a, stream=stream)
    barrier()
    ev0.record(stream)
    for _ in range(steps):
        km.kmeans_assign(Xd, C0d, labels, best, inertia_a, ws=ws_a, stream=stream)
    ev1.record(stream)
    barrier()
    t_assign = ev0.elapsed_time(ev1) / 1e3 / steps

    # the update alone (labels from the assignment above)
    C_upd = torch.empty_like(C0d)
    ws_u = km.workspace(km.OP_UPDATE, n, k, d, dev)
    for _ in range(warm):
        km.kmeans_update(Xd, labels, C0d, C_upd, counts, ws=ws_u, stream=stream)
    barrier()
    ev0.record(stream)
    for _ in range(steps):
        km.kmeans_update(Xd, labels, C0d, C_upd, counts, ws=ws_u, stream=stream)
    ev1.record(stream)
    barrier()
    t_update = ev0.elapsed_time(ev1) / 1e3 / steps
    # the assignment of every row to C0 and the update on those labels, kept
    # for the parity check against the oracle (after all timed regions)
    gpu_c0 = (labels.cpu().numpy(), best.cpu().numpy(), C_upd.cpu().numpy(), counts.cpu().numpy())

    # the FFMA comparator on the same workload (fewer calls: it is ~10x slower)
    ws_f = km.workspace(km.OP_ASSIGN_FFMA, n, k, d, dev)
    f_steps = max(1, min(steps, 20, int(4e13 / flop)))  # about 10x the tensor path's time
    km.kmeans_assign_ffma(Xd, C0d, labels, best, inertia_a, ws=ws_f, stream=stream)
    barrier()
    ev0.record(stream)
    for _ in range(f_steps):
        km.kmeans_assign_ffma(Xd, C0d, labels, best, inertia_a, ws=ws_f, stream=stream)
    ev1.record(stream)
    barrier()
    t_ffma = ev0.elapsed_time(ev1) / 1e3 / f_steps
    del ws_f

    # the Lloyd iteration with the update fused into the assignment (float
    # atomics, not bitwise reproducible), against the sorted pass above
    t_fused = None
    if d <= 4096:
        ws_fu = km.workspace(km.OP_LLOYD_FUSED, n, k, d, dev)
        C_fu = torch.empty_like(C0d)
        for _ in range(3):
            km.kmeans_lloyd_iter_fused(Xd, C0d, C_fu, labels, best, inertia_a, counts, ws=ws_fu, stream=stream)
        barrier()
        ev0.record(stream)
        for _ in range(steps):
            km.kmeans_lloyd_iter_fused(Xd, C0d, C_fu, labels, best, inertia_a, counts, ws=ws_fu, stream=stream)
        ev1.record(stream)
        barrier()
        t_fused = ev0.elapsed_time(ev1) / 1e3 / steps
        del ws_fu

    # the 3xTF32 comparator of the operand split: the same kernel with
    # kind::tf32 MMAs (TF32 runs at half the bf16 rate)
    ws_t = km.workspace(km.OP_ASSIGN_3XTF32, n, k, d, dev)
    t_steps = max(1, min(steps, 50))
    for _ in range(2):
        km.kmeans_assign_3xtf32(Xd, C0d, labels, best, inertia_a, ws=ws_t, stream=stream)
    barrier()
    ev0.record(stream)
    for _ in range(t_steps):
        km.kmeans_assign_3xtf32(Xd, C0d, labels, best, inertia_a, ws=ws_t, stream=stream)
    ev1.record(stream)
    barrier()
    t_tf32 = ev0.elapsed_time(ev1) / 1e3 / t_steps
    del ws_t

    # empty-cluster relocation, the opt-in step of kmeans_fit: on this
    # workload's labels (no cluster is empty: one counting pass) and with
    # every odd cluster emptied (k / 2 clusters relocated); each step first
    # restores the labels with a device copy of n int64, included in the time
    ws_r = km.workspace(km.OP_RELOCATE, n, k, 1, dev)
    r_steps = max(1, min(steps, 50))
    lab_work = torch.empty_like(labels)
    lab_src = {"none_empty": labels.clone(), "half_empty": (labels // 2) * 2}
    t_reloc = {}
    for case, src in lab_src.items():
        for _ in range(2):
            lab_work.copy_(src)
            km.kmeans_relocate_empty(lab_work, best, k, ws=ws_r, stream=stream)
        barrier()
        ev0.record(stream)
        for _ in range(r_steps):
            lab_work.copy_(src)
            km.kmeans_relocate_empty(lab_work, best, k, ws=ws_r, stream=stream)
        ev1.record(stream)
        barrier()
        t_reloc[case] = ev0.elapsed_time(ev1) / 1e3 / r_steps
    moved = int((lab_work != lab_src["half_empty"]).sum().item())
    del ws_r, lab_work, lab_src
    clocks = sampler.stop()

    kpp = None
    if not args.no_kmeanspp:
        kpp = time_kmeanspp(km, synth, dev, stream, barrier)

    # end to end: pinned host inputs in, results out, every step
    e2e = None
    if not args.no_e2e:
        Xh = torch.from_numpy(X).pin_memory()
        Ch = torch.from_numpy(C0).pin_memory()
        C_out_h = [torch.empty((k, d), dtype=torch.float32).pin_memory() for _ in range(2)]
        lab_h = [torch.empty(n, dtype=torch.int64).pin_memory() for _ in range(2)]
        in_h = [torch.empty(1, dtype=torch.float64).pin_memory() for _ in range(2)]
        # two sets of device buffers (inputs and outputs) and two copy
        # streams, alternated: a step's copies in overlap the previous step's
        # assignment, and its read-back (on its copy stream) the next step's
        Xe = [torch.empty_like(Xd), torch.empty_like(Xd)]
        Ce = [torch.empty_like(C0d), torch.empty_like(C0d)]
        Cn = [torch.empty_like(C0d), torch.empty_like(C0d)]
        labels_e = [torch.empty_like(labels), torch.empty_like(labels)]
        inertia_e = [torch.empty(1, dtype=torch.float64, device=dev) for _ in range(2)]
        e2e_steps = max(1, min(steps, 50))

        slices = args.e2e_slices  # lloyd10, per step: 2 -> 3.00 ms, 4 -> 2.91, 8 -> 2.86, 16 -> 2.84 (no overlap)
        copy_streams = [torch.cuda.Stream(dev), torch.cuda.Stream(dev)]

        def e2e_step(j):
            # a set is reused only by the copies of the step after next, which
            # its copy stream orders after that set's read-back, itself after
            # the step's update
            slot = j % 2
            km.kmeans_lloyd_iter_host(Xh, Ch, Xe[slot], Ce[slot], Cn[slot], labels_e[slot], best, counts,
                                      C_out_h[slot], lab_h[slot], in_h[slot], slices=slices, ws=ws,
                                      inertia=inertia_e[slot],
                                      copy_stream=copy_streams[slot], stream=stream, overlap_previous=True,
                                      readback_on_copy_stream=True)

        for j in range(min(warm, 3)):
            e2e_step(j)
        for cs in copy_streams:
            stream.wait_stream(cs)
        barrier()
        ev0.record(stream)
        for cs in copy_streams:
            cs.wait_event(ev0)  # the first timed steps' copies start inside the timed region
        for j in range(e2e_steps):
            e2e_step(j)
        for cs in copy_streams:
            stream.wait_stream(cs)  # the last read-backs end inside it
        ev1.record(stream)
        barrier()
        # the host link's rate for one whole copy of X, after the timed
        # region: what the copies in could take at most (the link is shared
        # with the rest of the machine, so it differs from run to run)
        h0, h1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        h0.record(copy_streams[0])
        with torch.cuda.stream(copy_streams[0]):
            Xe[0].copy_(Xh, non_blocking=True)
        h1.record(copy_streams[0])
        h1.synchronize()
        link_gbs = Xh.numel() * 4 / (h0.elapsed_time(h1) / 1e3) / 1e9
        t_e2e = ev0.elapsed_time(ev1) / 1e3 / e2e_steps
        e2e = {"value": flop / t_e2e / 1e12, "unit": "TFLOP/s", "ms_per_step": 1e3 * t_e2e,
               "steps": e2e_steps, "pipeline": f"kmeans_lloyd_iter_host: {slices} row slices copied on a copy "
                                               "stream, each assigned as it lands; finalize and update; C_new, "
                                               "labels and inertia copied back on the copy stream; two device "
                                               "buffer sets and two copy streams alternate, so each step's copies "
                                               "in and out overlap the neighbouring steps' compute",
               "h2d_bytes_per_step": int(Xh.numel() * 4 + Ch.numel() * 4),
               "host_link_gbs": round(link_gbs, 1),
               "d2h_bytes_per_step": int(C_out_h[0].numel() * 4 + lab_h[0].numel() * 8 + in_h[0].numel() * 8)}

    # max over ranks
    t_lloyd, t_assign, t_update, t_e2e_max = max_over_ranks(
        [t_lloyd, t_assign, t_update, e2e["ms_per_step"] / 1e3 if e2e else 0.0], world, dev)
    if e2e and world > 1:
        e2e["value"] = whole_job_tflops(flop, world, t_e2e_max)

    peaks, peaks_src = load_peaks()
    r_peak = peaks["bf16_tflops"] / SPLIT_PRODUCTS
    r_sustained = peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]) / SPLIT_PRODUCTS
    assign_tflops = flop / t_assign / 1e12
    tc_tflops = flop / t_tc / 1e12
    upd_bytes = 4.0 * n * d + 8.0 * n + 4.0 * k * d
    # segmented mean: X once through the member list, the list itself, C_new
    mean_bytes = 4.0 * n * d + 8.0 * n + 4.0 * k * d
    line = {
        "metric": METRIC,
        "value": whole_job_tflops(flop, world, t_lloyd),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": steps,
        "warmup": warm,
        "ms_per_step": 1e3 * t_lloyd,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "n": n, "k": k, "d": d, "blobs": w.blobs,
                   "init": "seeded random rows of X", "l2": f"inputs larger than L2 (X {gib(X.nbytes)})",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "assign": {"ms": 1e3 * t_assign, "tflops": assign_tflops, "frac_of_R": assign_tflops / r_peak,
                   "R_tflops": r_peak, "R": f"fp32-accurate roofline = bf16 dense peak ({peaks_src}, burst) / 3 "
                                             "(bf16x3 split: 3 MMAs per fp32 product)"},
        "update": {"ms": 1e3 * t_update, "gbs": upd_bytes / t_update / 1e9,
                   "frac_of_hbm": upd_bytes / t_update / 1e9 / peaks["hbm_gbs"],
                   "segmented_mean_kernel": {"us": 1e6 * t_mean, "gbs": mean_bytes / t_mean / 1e9,
                                             "frac_of_hbm": mean_bytes / t_mean / 1e9 / peaks["hbm_gbs"],
                                             "timed": "in the traced Lloyd run"}},
        "assign_ffma": {"ms": 1e3 * t_ffma, "tflops": flop / t_ffma / 1e12,
                        "speedup_of_tensor_path": t_ffma / t_assign},
        "lloyd_fused": None if t_fused is None else {
            "ms": 1e3 * t_fused, "tflops": flop / t_fused / 1e12, "speedup_over_sorted_update": t_lloyd / t_fused,
            "note": "kmeans_lloyd_iter_fused from the same centroids every step: the update fused into the "
                    "assignment epilogue with float atomics (C_new not bitwise reproducible)"},
        "assign_3xtf32": {"ms": 1e3 * t_tf32, "tflops": flop / t_tf32 / 1e12,
                          "frac_of_tf32_R": flop / t_tf32 / 1e12 / (TF32_NOMINAL_TFLOPS / SPLIT_PRODUCTS),
                          "speedup_of_bf16x3": t_tf32 / t_assign,
                          "note": "whole kmeans_assign_3xtf32 call against the nominal dense TF32 rate "
                                  f"{TF32_NOMINAL_TFLOPS} TFLOP/s / 3 (no measured TF32 peak)"},
        "relocate_empty": {"us_none_empty": 1e6 * t_reloc["none_empty"],
                           "us_half_empty": 1e6 * t_reloc["half_empty"], "moved_half_empty": moved,
                           "share_of_lloyd_none_empty": t_reloc["none_empty"] / t_lloyd,
                           "note": "kmeans_relocate_empty on this workload's labels and distances; each step "
                                   "restores the labels first (a device copy of n int64, in the time)"},
        "lloyd_frac_of_roofline": (flop / (r_peak * 1e12) + upd_bytes / (peaks["hbm_gbs"] * 1e9)) / t_lloyd,
        "roofline": {"bound": "tensor", "achieved": tc_tflops, "peak": r_peak, "unit": "TFLOP/s",
                     "frac": tc_tflops / r_peak, "traffic": recorded_traffic(w.name),
                     "peak_sustained": r_sustained, "frac_sustained": tc_tflops / r_sustained,
                     "kernel": "assign_tc_kernel",
                     "kernel_us": 1e6 * t_tc, "kernel_share_of_step": t_tc / t_lloyd_traced,
                     "timing": "CUDA events the library records around each launch on the launch stream, in "
                               f"a second timed Lloyd run of {steps} steps from the same centroids "
                               f"({1e3 * t_lloyd_traced:.4f} ms per step with the events, "
                               f"{1e3 * t_lloyd:.4f} without: each record holds the next chained launch back "
                               "until the kernel has drained, so the kernel time includes its own ramp-up)",
                     "algorithmic": "2 n k d flops per launch",
                     "peak_source": f"{peaks_src} bf16 burst {peaks['bf16_tflops']} / 3; peak_sustained: "
                                    f"{peaks_src} sustained {peaks.get('bf16_tflops_sustained')} / 3",
                     "algorithmic_bytes": 4.0 * n * d + 4.0 * k * d + 12.0 * n,
                     "traffic_source": "profiles/assign_tc_kernel_traffic.json (ncu dram__bytes_read.sum + "
                                       "dram__bytes_write.sum, one launch on this workload)"},
        "inertia_first10": [float(v) for v in inertia_hist[:10]],
        "gpu_launches": steps * launches_per_lloyd_step(k),
        "clocks": clocks,
    }
    if e2e:
        line["e2e"] = e2e
    if kpp:
        kpp["frac_of_hbm"] = kpp["gbs"] / peaks["hbm_gbs"]
        line["kmeanspp"] = kpp
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        import oracle
        oracle.build()
        line["cpu_baseline"], line["parity"] = cpu_baseline(oracle, w, X, C0, gpu=gpu_c0)
        if kpp:
            line["parity"]["kmeanspp_indices_match"] = kpp["indices_match_oracle"]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_gb300(args)


if __name__ == "__main__":
    sys.exit(main())

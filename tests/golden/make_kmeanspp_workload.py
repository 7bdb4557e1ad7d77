"""Writes kmeanspp_workload_indices.txt: the oracle's greedy D^2 seeding of the
full k-means++ workload, for the GPU test that checks every chosen index.

The workload is the k-means++ set of the tile-tradeoff page ("004 — tile
sizes, a Cython Lloyd step, and k-means++", section "k-means++"): n = 65536
samples of 1024 planted blobs, d = 8192 float32 features, 1024 centers with
2 + floor(ln 1024) = 8 candidate trials each, seed 42.  The indices come from
the CPU oracle alone (no GPU code is loaded); the file also records a SHA-256
of the sample matrix, so a test on another machine can tell whether the input
generator gave it the same bytes, and the draw margins (how far each draw's
target lay from the nearest running-sum boundary, over the total).

numpy's float32 normal draws are not bit-identical across CPU architectures
(x86-64 and aarch64 gave different matrices), so the file is written on the
architecture the GPU tests run on, and it names that architecture.

Run from the repository root (about 7 minutes on 8 to 16 cores):

    python tests/golden/make_kmeanspp_workload.py
"""
from __future__ import annotations

import hashlib
import os
import platform
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "kmeanspp_workload_indices.txt")


def main() -> None:
    w = synth.KMEANSPP
    X, _, _ = synth.planted_blobs(w.n, w.d, w.blobs, w.data_seed)
    digest = hashlib.sha256(X.tobytes()).hexdigest()
    T = oracle.n_trials_for(w.k)
    t0 = time.time()
    idx, margins, _ = oracle.kmeanspp(X, w.k, w.init_seed, n_trials=T)
    secs = time.time() - t0
    below = int((margins < 1e-7).sum())
    lines = [
        "# Greedy D^2 (k-means++) seeding of the k-means++ workload, by the CPU oracle.",
        "# Source of the workload: \"004 - tile sizes, a Cython Lloyd step, and k-means++\",",
        "# section \"k-means++\" (n = 65536, d = 8192, 1024 centers, 2 + floor(ln k) trials).",
        "# Written by tests/golden/make_kmeanspp_workload.py (oracle only).",
        f"# n={w.n} d={w.d} k={w.k} trials={T} blobs={w.blobs} data_seed={w.data_seed} seed={w.init_seed}",
        f"# x_sha256={digest}",
        f"# draws={margins.size} smallest_margin={margins.min():.3e} draws_below_1e-7={below}",
        f"# oracle_seconds={secs:.0f} threads={oracle.max_threads()} machine={platform.machine()} numpy={np.__version__}",
        "# one chosen sample index per line, in the order the centers were chosen",
    ]
    lines += [str(int(v)) for v in idx]
    with open(OUT, "w") as f:
        f.write("\n".join(lines) + "\n")
    print(f"wrote {OUT}: {w.k} indices, {secs:.0f} s, smallest margin {margins.min():.3e}, {below} below 1e-7")


if __name__ == "__main__":
    main()

"""Writes assign_<workload>.npz: the oracle's assignment of every sample of the
three large workloads to their initial centroids, for the GPU test that
compares every row.

The workloads are the sample-, centroid- and feature-heavy shapes of "Three
shapes that fit an eager Gram assignment" (section "Shapes"): 131072 x 8192
x 8192, 65536 x 16384 x 8192 and 65536 x 4096 x 16384 float32 planted blobs,
initial centroids = seeded random rows of X.  The brute-force argmin over all
centroids is the expensive part (2 n k d binary64 operations, minutes on a
many-core host), so it is stored; a pair's distance is cheap and the test
recomputes it.  Per workload the file holds:

* ``labels`` (uint16, n): the oracle's nearest centroid (lowest index on
  ties);
* ``near_rows`` (int64): the samples whose runner-up lies within
  ``NEAR_RTOL`` * (||x||^2 + ||c_best||^2) of the best, with ``near_best``
  and ``near_second`` (float64), the two distances: a test decides near ties
  with its own tolerance (at most NEAR_RTOL) from these;
* ``inertia`` (float64): the sum of the winning distances;
* ``meta`` (JSON): the shape, the seeds, the SHA-256 of X and of the initial
  centroids, and the host the oracle ran on.

The numbers come from the CPU oracle alone (no GPU code is loaded).  numpy's
float32 normal draws differ between x86-64 and aarch64, so the files are
written on the architecture the GPU tests run on, and they name it; the test
checks the hashes before it compares.

Run from the repository root (about 7 minutes on 16 cores for all three):

    python tests/golden/make_large_assign.py [workload ...]
"""
from __future__ import annotations

import hashlib
import json
import os
import platform
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

HERE = os.path.dirname(os.path.abspath(__file__))
NAMES = ("sample_heavy", "centroid_heavy", "feature_heavy")
NEAR_RTOL = 1e-3


def path_for(name: str) -> str:
    return os.path.join(HERE, f"assign_{name}.npz")


def write(name: str) -> None:
    w = synth.WORKLOADS[name]
    X, C0, init_idx = synth.workload_inputs(w)
    t0 = time.time()
    labels, best, second, inertia = oracle.assign(X, C0)
    secs = time.time() - t0
    xn = np.einsum("ij,ij->i", X.astype(np.float64), X.astype(np.float64))
    cn = np.einsum("ij,ij->i", C0.astype(np.float64), C0.astype(np.float64))
    near = np.flatnonzero((second - best) <= NEAR_RTOL * (xn + cn[labels]))
    assert w.k <= 65535
    meta = {"workload": name, "n": w.n, "k": w.k, "d": w.d, "blobs": w.blobs, "data_seed": w.data_seed,
            "init_seed": w.init_seed, "near_rtol": NEAR_RTOL,
            "x_sha256": hashlib.sha256(X.tobytes()).hexdigest(),
            "c_sha256": hashlib.sha256(C0.tobytes()).hexdigest(),
            "writer": "tests/golden/make_large_assign.py (oracle only)",
            "oracle_seconds": round(secs, 1), "threads": oracle.max_threads(),
            "machine": platform.machine(), "numpy": np.__version__}
    np.savez_compressed(path_for(name), labels=labels.astype(np.uint16), near_rows=near.astype(np.int64),
                        near_best=best[near], near_second=second[near], inertia=np.float64(inertia),
                        meta=np.array(json.dumps(meta)))
    print(f"wrote {path_for(name)}: {w.n} labels, {near.size} near ties, {secs:.0f} s", flush=True)


def load(name: str):
    """``(labels int64, near_rows, near_best, near_second, inertia, meta)``."""
    z = np.load(path_for(name))
    return (z["labels"].astype(np.int64), z["near_rows"], z["near_best"], z["near_second"],
            float(z["inertia"]), json.loads(str(z["meta"])))


if __name__ == "__main__":
    for name in sys.argv[1:] or NAMES:
        write(name)

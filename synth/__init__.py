"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module only draws random numbers; it holds none of the k-means arithmetic,
so both the CPU oracle and the GPU library can be fed from it without sharing
any of the method's code.

Workloads follow the journal pages' shapes ("Three shapes that fit an eager
Gram assignment", section "Shapes"; "Fusion probe", section "Probe shape";
"004 — tile sizes, a Cython Lloyd step, and k-means++", sections "Same arrays
as the Cython iteration" and "k-means++").  The pages used no public dataset;
the data here are planted isotropic Gaussian blobs:

* ``m`` blob centers, each coordinate ~ N(0, 1);
* sample ``i`` belongs to blob ``i mod m`` (equal sizes);
* sample = its blob center + N(0, sigma^2) noise per coordinate, sigma = 0.5.

Generation is chunked by rows with one independent PCG64 stream per chunk
(``SeedSequence.spawn``), so the bytes depend only on the seed and the shape,
never on the thread count.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

_CHUNK = 2048


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    k: int
    d: int
    blobs: int
    iters: int
    data_seed: int
    init_seed: int
    note: str


# The five workloads (n samples, k centroids, d features; float32).
WORKLOADS = {
    "probe": Workload("probe", 4096, 256, 512, 256, 1, 1000, 2000,
                      "probe shape of the fusion-probe page; one Lloyd iteration"),
    "lloyd10": Workload("lloyd10", 65536, 1024, 2048, 1024, 10, 1001, 2001,
                        "the shape sized against the 4-thread Cython Lloyd step; "
                        "10 Lloyd iterations with per-iteration inertia"),
    "sample_heavy": Workload("sample_heavy", 131072, 8192, 8192, 8192, 1, 1002, 2002,
                             "sample-heavy shape; assignment + mean update"),
    "centroid_heavy": Workload("centroid_heavy", 65536, 16384, 8192, 16384, 1, 1003, 2003,
                               "centroid-heavy shape; one Lloyd iteration"),
    "feature_heavy": Workload("feature_heavy", 65536, 4096, 16384, 4096, 1, 1004, 2004,
                              "feature-heavy shape; one Lloyd iteration"),
}

# k-means++ seeding set of the tile-tradeoff page: 65536 x 8192, 1024 centers.
KMEANSPP = Workload("kmeanspp", 65536, 1024, 8192, 1024, 1, 1005, 42,
                    "k-means++ seeding, 2 + floor(ln k) = 8 trials per center")


def _threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def blob_centers(m: int, d: int, seed: int) -> np.ndarray:
    """The ``m`` planted centers, each coordinate ~ N(0, 1), float32 (m, d)."""
    ss = np.random.SeedSequence([seed, 0xC3])
    return np.random.default_rng(ss).standard_normal((m, d), dtype=np.float32)


def planted_blobs(n: int, d: int, m: int, seed: int, sigma: float = 0.5,
                  out: np.ndarray | None = None, threads: int | None = None):
    """Samples of ``m`` planted Gaussian blobs.

    Returns ``(X float32 (n, d), centers float32 (m, d), blob int64 (n,))`` with
    ``blob[i] = i % m``.
    """
    centers = blob_centers(m, d, seed)
    X = out if out is not None else np.empty((n, d), dtype=np.float32)
    assert X.shape == (n, d) and X.dtype == np.float32 and X.flags.c_contiguous
    nchunks = (n + _CHUNK - 1) // _CHUNK
    streams = np.random.SeedSequence([seed, 0x5A]).spawn(nchunks)
    s32 = np.float32(sigma)

    def fill(c: int) -> None:
        r0, r1 = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        rows = X[r0:r1]
        np.random.default_rng(streams[c]).standard_normal(out=rows, dtype=np.float32)
        rows *= s32
        rows += centers[np.arange(r0, r1) % m]

    with ThreadPoolExecutor(max_workers=threads or _threads()) as pool:
        list(pool.map(fill, range(nchunks)))
    blob = np.arange(n, dtype=np.int64) % m
    return X, centers, blob


def init_rows(n: int, k: int, seed: int) -> np.ndarray:
    """``k`` distinct sample indices from a seeded permutation of ``0..n-1``."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x1D]))
    return rng.permutation(n)[:k].astype(np.int64)


def workload_inputs(w: Workload, threads: int | None = None):
    """``(X, C0)`` for a workload: its blobs and its seeded initial centroids."""
    X, _, _ = planted_blobs(w.n, w.d, w.blobs, w.data_seed, threads=threads)
    idx = init_rows(w.n, w.k, w.init_seed)
    return X, np.ascontiguousarray(X[idx]), idx


def gaussian(shape, seed: int, scale: float = 1.0, dtype=np.float32) -> np.ndarray:
    """Plain seeded N(0, scale^2) array (for small unstructured test cases)."""
    rng = np.random.default_rng(np.random.SeedSequence([seed, 0x77]))
    return (rng.standard_normal(shape, dtype=np.float64) * scale).astype(dtype)

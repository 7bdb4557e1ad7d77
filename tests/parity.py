"""Comparison rules between the CUDA library and the CPU oracle.

Tolerances (fixed by the target specification of this library):
* best distance: |gpu - oracle| <= 1e-4 * (||x||^2 + ||c_best||^2);
* labels: identical wherever the oracle's runner-up exceeds its best by more
  than 1e-4 * (||x||^2 + ||c_best||^2); elsewhere (near ties) the GPU's choice
  must itself be within that tolerance of the best, and the flips are counted;
* centroids: per row, max |gpu - oracle| <= 1e-5 * max |oracle row|;
* k-means++ indices: identical.
"""
from __future__ import annotations

import numpy as np

import oracle

DIST_RTOL = 1e-4
CENTROID_RTOL = 1e-5


def sq_norms(A: np.ndarray) -> np.ndarray:
    A64 = A.astype(np.float64)
    return np.einsum("ij,ij->i", A64, A64)


def check_assign(X, C, labels, best, o_labels, o_best, o_second, rows=None, what=""):
    """Compare a GPU assignment (labels, best) on ``rows`` with the oracle's.

    ``X`` holds the sample rows the oracle saw (already subset when ``rows``
    is given); ``labels``/``best`` are the GPU's full outputs.  Returns the
    number of near-tie label flips and the worst relative distance error.
    """
    labels = np.asarray(labels)
    best = np.asarray(best, dtype=np.float64)
    if rows is not None:
        labels = labels[rows]
        best = best[rows]
    xn = sq_norms(X)
    cn = sq_norms(C)
    scale = xn + cn[o_labels]
    err = np.abs(best - o_best)
    bad = err > DIST_RTOL * scale
    assert not bad.any(), (f"{what}: {bad.sum()} distances outside tolerance; worst rel "
                           f"{(err / scale).max():.3e}")
    clear = (o_second - o_best) > DIST_RTOL * scale
    mism = clear & (labels != o_labels)
    assert not mism.any(), f"{what}: {mism.sum()} labels differ where the oracle winner is clear"
    flips = np.nonzero(~clear & (labels != o_labels))[0]
    for i in flips:  # a flip must be a valid near-tie choice
        dj = oracle.sqdist(X[i], C[labels[i]])
        assert dj - o_best[i] <= DIST_RTOL * scale[i], f"{what}: flip at {i} is not a near tie"
    assert labels.min() >= 0 and labels.max() < C.shape[0]
    return int(len(flips)), float((err / scale).max())


def check_centroids(got, want, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    row_scale = np.abs(want).max(axis=1)
    err = np.abs(got - want).max(axis=1)
    bad = err > CENTROID_RTOL * np.maximum(row_scale, np.finfo(np.float32).tiny)
    assert not bad.any(), (f"{what}: {bad.sum()} centroid rows outside 1e-5; worst "
                           f"{(err / np.maximum(row_scale, 1e-30)).max():.3e}")


def check_assign_every_row(X, C, labels, best, o_labels, near_rows, near_best, near_second, what=""):
    """Compare a GPU assignment of every row with stored oracle results.

    ``o_labels`` is the oracle's label of every row; ``near_rows`` the rows
    whose oracle runner-up lies close to the best (a superset of the near
    ties at DIST_RTOL), with the oracle's two distances.  The oracle's best
    distance of every other row is its squared distance to ``o_labels``,
    recomputed here in binary64 by definition.  Returns ``(near-tie flips,
    worst relative distance error, near ties)``."""
    labels = np.asarray(labels)
    best = np.asarray(best, dtype=np.float64)
    n = X.shape[0]
    o_best = np.empty(n, dtype=np.float64)
    for r0 in range(0, n, 2048):
        r1 = min(n, r0 + 2048)
        diff = X[r0:r1].astype(np.float64) - C[o_labels[r0:r1]].astype(np.float64)
        o_best[r0:r1] = np.einsum("ij,ij->i", diff, diff)
    # the stored distances belong to these rows and labels
    np.testing.assert_allclose(o_best[near_rows], near_best, rtol=1e-9, atol=0)
    scale = sq_norms(X) + sq_norms(C)[o_labels]
    rel = np.abs(best - o_best) / scale
    bad = rel > DIST_RTOL
    assert not bad.any(), f"{what}: {bad.sum()} distances outside tolerance; worst rel {rel.max():.3e}"
    near = np.zeros(n, dtype=bool)
    near[near_rows] = (near_second - near_best) <= DIST_RTOL * scale[near_rows]
    mism = ~near & (labels != o_labels)
    assert not mism.any(), f"{what}: {mism.sum()} labels differ where the oracle winner is clear"
    assert labels.min() >= 0 and labels.max() < C.shape[0]
    flips = np.nonzero(near & (labels != o_labels))[0]
    for i in flips:  # a flip must be a valid near-tie choice
        dj = oracle.sqdist(X[i], C[labels[i]])
        assert dj - o_best[i] <= DIST_RTOL * scale[i], f"{what}: flip at {i} is not a near tie"
    return int(len(flips)), float(rel.max()), int(near.sum())

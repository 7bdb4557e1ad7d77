"""Empty-cluster relocation on the GPU against the oracle.

The relocation is pure selection on (labels, best distances): both sides get
the same inputs (the GPU's own assignment output, or synthetic arrays) and
must agree bit for bit.  The fits with relocation are compared on planted
blobs with some centroids moved far away, on inputs whose oracle trajectory
takes no decision near a tie (the test asserts it first)."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from parity import check_centroids

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _relocate_both(km, labels, best, k):
    got = km.kmeans_relocate_empty(_dev(labels), _dev(best), k).cpu().numpy()
    want, moved = oracle.relocate_empty(labels, best, k)
    return got, want, moved


@pytest.mark.parametrize("n,k,used,values,seed", [
    (1, 1, 1, None, 1),               # a single sample: nothing can be empty
    (37, 37, 5, None, 2),             # k = n, most clusters empty
    (4099, 1500, 700, None, 3),       # ragged per-thread ranges, 800 empties
    (4099, 1500, 700, "ties", 4),     # distances from five values, -0.0 among them
    (300000, 70000, 9000, "ties", 5),  # 61000 empties, long tie runs
    (300000, 70000, 9000, None, 6),
    (65536, 1024, 1024, None, 7),     # every cluster occupied: nothing moves
])
def test_relocation_matches_the_oracle(gpu_lib, n, k, used, values, seed):
    rng = np.random.default_rng(seed)
    clusters = rng.choice(k, size=used, replace=False)
    labels = rng.choice(clusters, size=n).astype(np.int64)
    labels[:used] = clusters  # every chosen cluster has a member
    if values == "ties":
        best = rng.choice(np.array([0.0, -0.0, 3.0, 3.0, 11.5], np.float32), size=n)
    else:
        best = (rng.random(n) * 1e3).astype(np.float32)
    got, want, moved = _relocate_both(gpu_lib, labels, best, k)
    np.testing.assert_array_equal(got, want)
    assert len(moved) == k - used
    if used == k:
        np.testing.assert_array_equal(got, labels)


def test_relocation_of_the_assignments_own_output(gpu_lib):
    # most centroids far from every sample: their clusters are empty after
    # the assignment, and the relocation must pick the same samples from the
    # GPU's distances as the oracle does
    X = synth.gaussian((6000, 64), seed=11)
    C = synth.gaussian((900, 64), seed=12) * np.float32(8.0)
    labels, best, _ = gpu_lib.kmeans_assign(_dev(X), _dev(C))
    lab, bst = labels.cpu().numpy(), best.cpu().numpy()
    assert (np.bincount(lab, minlength=900) == 0).sum() > 100
    got, want, _ = _relocate_both(gpu_lib, lab, bst, 900)
    np.testing.assert_array_equal(got, want)
    assert (np.bincount(got, minlength=900) > 0).all()


def test_relocation_leaves_labels_alone_on_a_bad_label(gpu_lib):
    labels = np.zeros(5000, np.int64)
    labels[4321] = 7  # k = 7: out of range
    best = np.arange(5000, dtype=np.float32)
    ws = gpu_lib.workspace(gpu_lib.OP_RELOCATE, 5000, 7, 1)
    d_labels = _dev(labels)
    gpu_lib.kmeans_relocate_empty(d_labels, _dev(best), 7, ws=ws)
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_ERR_DEVICE_LABEL
    np.testing.assert_array_equal(d_labels.cpu().numpy(), labels)
    # the next call clears the status word
    labels[4321] = 6
    d_labels = _dev(labels)
    gpu_lib.kmeans_relocate_empty(d_labels, _dev(best), 7, ws=ws)
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_OK
    np.testing.assert_array_equal(d_labels.cpu().numpy(), oracle.relocate_empty(labels, best, 7)[0])


def _far_centroid_case(n, d, m, moved, seed):
    X, centers, blob = synth.planted_blobs(n, d, m, seed=seed)
    C0 = centers.copy()
    for r, j in enumerate(moved):
        C0[j] += np.float32(1e3 * (r + 1))
    return X, C0, blob


def _smallest_gap_on_the_way(X, C0, k, max_iter=100):
    """The oracle's relocating fit from C0, returning the smallest relative
    margin of any decision along it: a sample's runner-up over its winner,
    (second - best) / (||x||^2 + ||c||^2), and each relocation's cut between
    the m-th and (m+1)-th largest distance.  Orphaned blobs sit far from
    every remaining center, so such near ties are common; the trajectories
    can only be compared where none is below the distance tolerance."""
    C = np.ascontiguousarray(C0, np.float32)
    hist, gap = [], np.inf
    Xn = (X.astype(np.float64) ** 2).sum(1)
    for it in range(max_iter):
        labels, best, second, inertia = oracle.assign(X, C)
        norm = Xn + (C.astype(np.float64)[labels] ** 2).sum(1)
        gap = min(gap, ((second - best) / norm).min())
        relocated, moved = oracle.relocate_empty(labels, best, k)
        if len(moved):
            s = np.sort(best)[::-1]
            gap = min(gap, (s[len(moved) - 1] - s[len(moved)]) / s[len(moved) - 1])
        C, _ = oracle.update(X, relocated, C)
        hist.append(inertia)
        if it > 0 and inertia >= hist[-2]:
            break
    return gap


@pytest.mark.parametrize("n,d,m,moved,seed", [
    (2048, 32, 16, [3], 44),
    (4096, 64, 32, [2, 7, 11], 45),
])
def test_fit_with_relocation_matches_the_oracle(gpu_lib, n, d, m, moved, seed):
    X, C0, blob = _far_centroid_case(n, d, m, moved, seed)
    assert _smallest_gap_on_the_way(X, C0, m) > 2e-4  # the inputs hold no near tie
    C, labels, best, counts, hist, n_iter = gpu_lib.kmeans_fit(_dev(X), C=_dev(C0), init="given", max_iter=100,
                                                                tol=0.0, relocate_empty=True)
    o_C, o_labels, _, o_hist, o_n = oracle.fit(X, C0, max_iter=100, tol=0.0, relocate=True)
    assert n_iter == o_n
    np.testing.assert_array_equal(labels.cpu().numpy(), o_labels)
    check_centroids(C.cpu().numpy(), o_C, what="fit with relocation")
    np.testing.assert_allclose(hist, o_hist, rtol=1e-4)
    np.testing.assert_array_equal(counts.cpu().numpy(), np.bincount(o_labels, minlength=m))
    assert (counts.cpu().numpy() > 0).all()


def test_fit_relocation_changes_nothing_without_empty_clusters(gpu_lib):
    # the relocation path (plain finalize, relocation, update with its own
    # count) must give the same bits as the default path when no cluster
    # ever empties
    X, _, _ = synth.planted_blobs(6000, 64, 24, seed=61)
    C0 = np.ascontiguousarray(X[synth.init_rows(6000, 24, seed=62)])
    a = gpu_lib.kmeans_fit(_dev(X), C=_dev(C0), init="given", max_iter=100, tol=0.0)
    b = gpu_lib.kmeans_fit(_dev(X), C=_dev(C0), init="given", max_iter=100, tol=0.0, relocate_empty=True)
    assert a[5] == b[5]
    for u, v in zip(a[:4], b[:4]):
        assert u.cpu().numpy().tobytes() == v.cpu().numpy().tobytes()
    np.testing.assert_array_equal(a[4], b[4])


def test_fit_rejects_unknown_option_bits(gpu_lib):
    lib = gpu_lib.load()
    fake = ctypes.c_void_p(0x10000)
    it = ctypes.c_int(0)
    for init in (0x200, 0x101 | 0x400, 2 | gpu_lib.FIT_RELOCATE_EMPTY):
        assert lib.kmeans_fit(fake, fake, fake, fake, None, 1024, 16, 32, init, 0, 10, 0.0, ctypes.byref(it), None,
                              fake, 1 << 30, None) == gpu_lib.KMEANS_ERR_INVALID_ARG

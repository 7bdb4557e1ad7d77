"""kmeans_fit: Lloyd iterations to a tolerance, against the oracle's fit.

On well-separated planted blobs no sample sits near a tie, so the GPU and the
oracle follow the same trajectory: the same iteration count, labels equal
and centroids within the update tolerance.  The seeding is the library's
k-means++, whose indices match the oracle's exactly."""
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


@pytest.mark.parametrize("tol", [0.0, 1e-3])
def test_fit_from_given_centroids_matches_the_oracle(gpu_lib, tol):
    X, _, _ = synth.planted_blobs(6000, 64, 24, seed=61)
    C0 = np.ascontiguousarray(X[synth.init_rows(6000, 24, seed=62)])
    C, labels, best, counts, hist, n_iter = gpu_lib.kmeans_fit(_dev(X), C=_dev(C0), init="given", max_iter=100,
                                                                tol=tol)
    o_C, o_labels, o_best, o_hist, o_n = oracle.fit(X, C0, max_iter=100, tol=tol)
    assert n_iter == o_n
    np.testing.assert_array_equal(labels.cpu().numpy(), o_labels)
    check_centroids(C.cpu().numpy(), o_C, what=f"fit tol={tol}")
    np.testing.assert_allclose(hist, o_hist, rtol=1e-4)
    assert np.all(np.diff(hist) <= 1e-6 * hist[:-1])


def test_fit_with_kmeanspp_seeding_matches_the_oracle(gpu_lib):
    X, _, _ = synth.planted_blobs(5000, 48, 20, seed=71)
    k, seed = 20, 5
    C, labels, best, counts, hist, n_iter = gpu_lib.kmeans_fit(_dev(X), k=k, init="kmeans++", seed=seed,
                                                                max_iter=100, tol=0.0)
    idx, _, _ = oracle.kmeanspp(X, k, seed)
    o_C, o_labels, _, o_hist, o_n = oracle.fit(X, X[idx], max_iter=100, tol=0.0)
    assert n_iter == o_n
    np.testing.assert_array_equal(labels.cpu().numpy(), o_labels)
    check_centroids(C.cpu().numpy(), o_C, what="fit after k-means++")
    np.testing.assert_array_equal(counts.cpu().numpy(), np.bincount(o_labels, minlength=k))


def test_fit_honours_max_iter_and_rejects_bad_arguments(gpu_lib):
    X, _, _ = synth.planted_blobs(3000, 32, 12, seed=81)
    C0 = np.ascontiguousarray(X[synth.init_rows(3000, 12, seed=82)])
    _, _, _, _, hist, n_iter = gpu_lib.kmeans_fit(_dev(X), C=_dev(C0), init="given", max_iter=2, tol=0.0)
    assert n_iter == 2 and len(hist) == 2
    lib = gpu_lib.load()
    fake = ctypes.c_void_p(0x10000)  # validation fails before any pointer is used
    it = ctypes.c_int(0)
    args = lambda init, max_iter, tol: (fake, fake, fake, fake, None, 1024, 16, 32, init, 0, max_iter, tol,
                                        ctypes.byref(it), None, fake, 1 << 30, None)
    assert lib.kmeans_fit(*args(2, 10, 0.0)) == gpu_lib.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_fit(*args(0, 0, 0.0)) == gpu_lib.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_fit(*args(0, 10, -1.0)) == gpu_lib.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_fit(*args(0, 10, float("nan"))) == gpu_lib.KMEANS_ERR_INVALID_ARG


def test_fit_on_a_shape_whose_assignment_splits_its_last_round(gpu_lib):
    # 20480 samples x 256 centroids: 80 tiles of 256 x 256 over a GB300's 76
    # CTA pairs, so every assignment of the fit runs its last round as K
    # halves.  Starting from the planted centers moved by N(0, 0.3^2) keeps
    # every decision on the way clear of a tie (smallest margin 0.27 of
    # ||x||^2 + ||c||^2), so both fits take the same path.
    X, centers, _ = synth.planted_blobs(20480, 64, 256, seed=91)
    C0 = np.ascontiguousarray(centers + synth.gaussian(centers.shape, seed=93) * np.float32(0.3), dtype=np.float32)
    C, labels, best, counts, hist, n_iter = gpu_lib.kmeans_fit(_dev(X), C=_dev(C0), init="given", max_iter=50,
                                                                tol=0.0)
    o_C, o_labels, _, o_hist, o_n = oracle.fit(X, C0, max_iter=50, tol=0.0)
    assert n_iter == o_n
    np.testing.assert_array_equal(labels.cpu().numpy(), o_labels)
    check_centroids(C.cpu().numpy(), o_C, what="fit with split assignment rounds")
    np.testing.assert_allclose(hist, o_hist, rtol=1e-4)

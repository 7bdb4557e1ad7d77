"""Degenerate and boundary shapes through every entry point, against the
oracle: one sample and one centroid at the smallest d, k = n, and a Lloyd
iteration whose update takes the radix-sort path (k > 32768)."""
import numpy as np
import pytest

import oracle
import synth
from parity import check_assign, check_centroids

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _host(t):
    return t.cpu().numpy()


def test_one_sample_one_centroid_through_every_entry_point(gpu_lib):
    X = np.array([[1.0, -2.0, 3.0, 0.5]], dtype=np.float32)
    C = np.array([[0.0, 0.0, 1.0, 1.0]], dtype=np.float32)
    exact = float(((X[0].astype(np.float64) - C[0]) ** 2).sum())
    for fn in (gpu_lib.kmeans_assign, gpu_lib.kmeans_assign_ffma, gpu_lib.kmeans_assign_3xtf32):
        labels, best, inertia = fn(_dev(X), _dev(C))
        assert int(_host(labels)[0]) == 0
        assert abs(float(_host(best)[0]) - exact) <= 1e-4 * (14.25 + 2.0)
    for fn in (gpu_lib.kmeans_lloyd_iter, gpu_lib.kmeans_lloyd_iter_fused):
        C1, labels, _, _, counts = fn(_dev(X), _dev(C))
        assert _host(C1).tobytes() == X.tobytes()  # the mean of one sample is the sample
        assert int(_host(counts)[0]) == 1
    C_fit, labels, _, counts, hist, n_iter = gpu_lib.kmeans_fit(_dev(X), C=_dev(C), init="given", max_iter=5, tol=0.0)
    assert _host(C_fit).tobytes() == X.tobytes() and n_iter <= 5
    idx, centers = gpu_lib.kmeanspp_init(_dev(X), 1, seed=3)
    assert int(_host(idx)[0]) == 0


def test_every_sample_its_own_centroid(gpu_lib):
    # k = n: each sample is a centroid, so every distance is 0 and every
    # cluster keeps exactly its sample
    X = synth.gaussian((300, 36), seed=12)
    C1, labels, best, inertia, counts = gpu_lib.kmeans_lloyd_iter(_dev(X), _dev(X))
    o_l, o_b, o_s, _ = oracle.assign(X, X)
    check_assign(X, X, _host(labels), _host(best), o_l, o_b, o_s, what="k = n")
    np.testing.assert_array_equal(_host(counts), np.ones(300, dtype=np.int32))
    assert _host(C1).tobytes() == X.tobytes()


def test_lloyd_iteration_on_the_radix_update_path(gpu_lib):
    n, k, d = 40000, 33000, 8
    X = synth.gaussian((n, d), seed=21)
    C0 = np.ascontiguousarray(X[synth.init_rows(n, k, seed=22)])
    C1, labels, best, inertia, counts = gpu_lib.kmeans_lloyd_iter(_dev(X), _dev(C0))
    lab = _host(labels)
    rows = np.sort(np.random.default_rng(23).choice(n, 512, replace=False))
    o_l, o_b, o_s, _ = oracle.assign(X[rows], C0)
    check_assign(X[rows], C0, lab, _host(best), o_l, o_b, o_s, rows=rows, what="radix Lloyd")
    o_C1, o_cnt = oracle.update(X, lab, C0)
    check_centroids(_host(C1), o_C1, what="radix Lloyd update")
    np.testing.assert_array_equal(_host(counts).astype(np.int64), o_cnt)

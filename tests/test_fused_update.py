"""kmeans_lloyd_iter_fused: the update fused into the assignment's epilogue.

The assignment half is the same kernel, so labels, distances and inertia must
equal kmeans_lloyd_iter's bit for bit while no tile is split (no more tiles
than CTA pairs); kmeans_lloyd_iter may run a partly filled last round as two
K halves per tile, whose sum carries a different float32 accumulation error
(within the distance tolerance), and the fused kernel never does.  The counts are exact; the centroids are float32
sums in a varying order, checked against the oracle's mean of the same labels
within the centroid tolerance, with empty clusters bit for bit."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from parity import DIST_RTOL, check_centroids

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _host(t):
    return t.cpu().numpy()


@pytest.mark.parametrize("shape", [(1000, 300, 100), (2000, 513, 132), (260, 257, 4), (4096, 256, 512),
                                   (20000, 700, 4096)], ids=lambda s: "x".join(map(str, s)))
def test_fused_iteration_matches_the_sorted_one_and_the_oracle(gpu_lib, shape):
    n, k, d = shape
    X, _, _ = synth.planted_blobs(n, d, k, seed=n + d)
    C0 = np.ascontiguousarray(X[synth.init_rows(n, k, seed=k)])
    Xd, Cd = _dev(X), _dev(C0)
    ref = gpu_lib.kmeans_lloyd_iter(Xd, Cd)
    got = gpu_lib.kmeans_lloyd_iter_fused(Xd, Cd)
    labels = _host(got[1])
    np.testing.assert_array_equal(labels, _host(ref[1]))  # planted blobs: no near ties
    tiles = ((n + 255) // 256) * ((k + 255) // 256)
    if tiles <= 76:  # no more tiles than a GB300 has CTA pairs: nothing splits
        assert _host(got[2]).tobytes() == _host(ref[2]).tobytes()
        assert float(got[3].item()) == float(ref[3].item())
    else:
        scale = (X.astype(np.float64) ** 2).sum(1) + (C0.astype(np.float64) ** 2).sum(1)[labels]
        diff = np.abs(_host(got[2]).astype(np.float64) - _host(ref[2]).astype(np.float64))
        assert (diff <= DIST_RTOL * scale).all()
        assert abs(float(got[3].item()) - float(ref[3].item())) <= DIST_RTOL * scale.sum()
    np.testing.assert_array_equal(_host(got[4]), _host(ref[4]))
    o_C, o_cnt = oracle.update(X, labels, C0)
    check_centroids(_host(got[0]), o_C, what=f"fused {shape}")
    np.testing.assert_array_equal(_host(got[4]).astype(np.int64), o_cnt)


def test_fused_iteration_keeps_empty_clusters_bit_for_bit(gpu_lib):
    X, _, _ = synth.planted_blobs(3000, 64, 20, seed=3)
    C0 = np.ascontiguousarray(X[synth.init_rows(3000, 20, seed=4)])
    C0[7] += 1e3  # far away: no member
    C_new, labels, _, _, counts = gpu_lib.kmeans_lloyd_iter_fused(_dev(X), _dev(C0))
    assert _host(counts)[7] == 0
    assert _host(C_new)[7].tobytes() == C0[7].tobytes()


@pytest.mark.slow
def test_fused_iteration_on_the_lloyd10_workload(gpu_lib):
    w = synth.WORKLOADS["lloyd10"]
    X, C0, _ = synth.workload_inputs(w)
    Xd, Cd = _dev(X), _dev(C0)
    ref = gpu_lib.kmeans_lloyd_iter(Xd, Cd)
    got = gpu_lib.kmeans_lloyd_iter_fused(Xd, Cd)
    np.testing.assert_array_equal(_host(got[1]), _host(ref[1]))
    o_C, o_cnt = oracle.update(X, _host(got[1]), C0)
    check_centroids(_host(got[0]), o_C, what="fused lloyd10")
    np.testing.assert_array_equal(_host(got[4]).astype(np.int64), o_cnt)


def test_fused_iteration_rejects_what_it_does_not_support(gpu_lib):
    lib = gpu_lib.load()
    fake = ctypes.c_void_p(0x10000)  # validation fails before any pointer is used
    other = ctypes.c_void_p(0x20000)
    args = lambda c_new, d: (fake, fake, c_new, fake, fake, None, None, 1024, 16, d, fake, 1 << 30, 0, None)
    assert lib.kmeans_lloyd_iter_fused(*args(other, 4100)) == gpu_lib.KMEANS_ERR_UNSUPPORTED
    assert lib.kmeans_lloyd_iter_fused(*args(fake, 64)) == gpu_lib.KMEANS_ERR_INVALID_ARG  # C_new aliases C_old

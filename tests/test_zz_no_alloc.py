"""The assignment entry point that allocates nothing: kmeans_assign_noalloc.

It serves callers that cannot allocate device memory at the moment they need
an assignment: code running under an allocator that refuses new device
allocations, a plugin that is handed only its input and output buffers, or a
real-time loop where an allocation (and the synchronisation it can bring) is
not allowed.  Instead of a caller-provided workspace it uses a fixed-size
array built into the library, so it must give exactly what kmeans_assign
gives with a workspace.  Two calls in a row on different problems check that
the shared built-in scratch carries nothing over from the previous call.

This file is collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest

import synth
from parity import DIST_RTOL, sq_norms

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _outputs(n):
    return (torch.empty(n, dtype=torch.int64, device="cuda"), torch.empty(n, dtype=torch.float32, device="cuda"),
            torch.empty(1, dtype=torch.float64, device="cuda"))


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _assign_noalloc(lib, X, C, labels, best, inertia):
    n, d = X.shape
    return lib.kmeans_assign_noalloc(X.data_ptr(), C.data_ptr(), n, C.shape[0], d, labels.data_ptr(),
                                     best.data_ptr(), inertia.data_ptr(), 0, _stream())


def _assign_with_workspace(km, lib, X, C, labels, best, inertia):
    n, d = X.shape
    k = C.shape[0]
    ws = km.workspace(km.OP_ASSIGN, n, k, d)
    return lib.kmeans_assign(X.data_ptr(), C.data_ptr(), n, k, d, labels.data_ptr(), best.data_ptr(),
                             inertia.data_ptr(), ws.data_ptr(), ws.numel(), 0, _stream())


def test_noalloc_matches_the_workspace_entry_point_on_two_calls(gpu_lib):
    lib = gpu_lib.load()
    # two different problems back to back: ragged tiles first, then the probe workload
    X1, _, _ = synth.planted_blobs(20000, 132, 600, seed=71)
    C1 = np.ascontiguousarray(X1[synth.init_rows(20000, 600, seed=72)])
    X2, C2, _ = synth.workload_inputs(synth.WORKLOADS["probe"])
    for X, C in ((X1, C1), (X2, C2)):
        Xd, Cd = _dev(X), _dev(C)
        n = X.shape[0]
        got, ref = _outputs(n), _outputs(n)
        assert _assign_noalloc(lib, Xd, Cd, *got) == gpu_lib.KMEANS_OK
        assert _assign_with_workspace(gpu_lib, lib, Xd, Cd, *ref) == gpu_lib.KMEANS_OK
        torch.cuda.synchronize()
        g_lab, g_best, g_in = (t.cpu().numpy() for t in got)
        r_lab, r_best, r_in = (t.cpu().numpy() for t in ref)
        np.testing.assert_array_equal(g_lab, r_lab)
        scale = sq_norms(X) + sq_norms(C)[r_lab]
        assert np.all(np.abs(g_best.astype(np.float64) - r_best) <= DIST_RTOL * scale)
        assert abs(float(g_in[0]) - float(r_in[0])) <= DIST_RTOL * scale.sum()


def test_noalloc_rejects_problems_beyond_its_scratch(gpu_lib):
    lib = gpu_lib.load()
    n, k, d = 65536, 4096, 2048  # the centroid copies alone need 32 MiB
    fake = ctypes.c_void_p(0x10000)  # validation fails before any pointer is used
    st = lib.kmeans_assign_noalloc(fake, fake, n, k, d, fake, fake, None, 0, None)
    assert st == gpu_lib.KMEANS_ERR_SCRATCH_LIMIT
    assert "built-in scratch" in gpu_lib.kmeans_status_string(st)


def test_noalloc_leaves_device_memory_untouched(gpu_lib):
    lib = gpu_lib.load()
    X, C, _ = synth.workload_inputs(synth.WORKLOADS["probe"])
    Xd, Cd = _dev(X), _dev(C)
    outs = _outputs(X.shape[0])
    assert _assign_noalloc(lib, Xd, Cd, *outs) == gpu_lib.KMEANS_OK  # per-device set-up happens here
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        assert _assign_noalloc(lib, Xd, Cd, *outs) == gpu_lib.KMEANS_OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0


# With n and k multiples of 256 and d = 64, the scratch is exactly 12 n + 4 k
# + 4 k * 64 bytes plus 9 KiB (a 1 KiB header region and the 8 KiB of inertia
# block sums): (1386240, 512, 64) needs exactly 16 MiB, (1391872, 256, 64)
# exactly 16 MiB + 1 KiB.
AT_LIMIT = (1386240, 512, 64)
ONE_KIB_OVER = (1391872, 256, 64)


def test_noalloc_scratch_limit_boundary(gpu_lib):
    lib = gpu_lib.load()
    fake = ctypes.c_void_p(0x10000)  # validation fails before any pointer is used
    n, k, d = ONE_KIB_OVER
    assert lib.kmeans_assign_noalloc(fake, fake, n, k, d, fake, fake, None, 0, None) == \
        gpu_lib.KMEANS_ERR_SCRATCH_LIMIT
    # the problem that fills the scratch exactly runs, and gives kmeans_assign's answer
    n, k, d = AT_LIMIT
    X, _, _ = synth.planted_blobs(n, d, k, seed=81)
    C = np.ascontiguousarray(X[synth.init_rows(n, k, seed=82)])
    Xd, Cd = _dev(X), _dev(C)
    got, ref = _outputs(n), _outputs(n)
    assert _assign_noalloc(lib, Xd, Cd, *got) == gpu_lib.KMEANS_OK
    assert _assign_with_workspace(gpu_lib, lib, Xd, Cd, *ref) == gpu_lib.KMEANS_OK
    torch.cuda.synchronize()
    # with a workspace this many tiles split their last round along K (the
    # built-in scratch never does): distances agree within the tolerance, and
    # a label may differ only where its own distance is that close too
    g_lab, r_lab = got[0].cpu().numpy(), ref[0].cpu().numpy()
    g_best, r_best = got[1].cpu().numpy().astype(np.float64), ref[1].cpu().numpy().astype(np.float64)
    scale = sq_norms(X) + sq_norms(C)[r_lab]
    assert np.all(np.abs(g_best - r_best) <= DIST_RTOL * scale)
    for i in np.flatnonzero(g_lab != r_lab):
        diff = X[i].astype(np.float64) - C[g_lab[i]].astype(np.float64)
        assert abs(float(diff @ diff) - r_best[i]) <= DIST_RTOL * scale[i]


def test_noalloc_timeout_leaves_minus_one_then_recovers(gpu_lib, monkeypatch):
    # The bounded pipeline waits of the built-in scratch's call run out when
    # the producer is starved on purpose (a host-side switch; no fault): the
    # call returns, its labels hold -1, and the next call resets the shared
    # scratch's status word and gives kmeans_assign's answer again.
    lib = gpu_lib.load()
    X, C, _ = synth.workload_inputs(synth.WORKLOADS["probe"])
    Xd, Cd = _dev(X), _dev(C)
    n = X.shape[0]
    outs = _outputs(n)
    monkeypatch.setenv("KMEANS_GB300_TEST_STARVE_PIPELINE", "1")
    assert _assign_noalloc(lib, Xd, Cd, *outs) == gpu_lib.KMEANS_OK
    torch.cuda.synchronize()
    assert (outs[0].cpu().numpy() == -1).all()
    monkeypatch.delenv("KMEANS_GB300_TEST_STARVE_PIPELINE")
    ref = _outputs(n)
    assert _assign_noalloc(lib, Xd, Cd, *outs) == gpu_lib.KMEANS_OK
    assert _assign_with_workspace(gpu_lib, lib, Xd, Cd, *ref) == gpu_lib.KMEANS_OK
    torch.cuda.synchronize()
    np.testing.assert_array_equal(outs[0].cpu().numpy(), ref[0].cpu().numpy())
    assert outs[1].cpu().numpy().tobytes() == ref[1].cpu().numpy().tobytes()

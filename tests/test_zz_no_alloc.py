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

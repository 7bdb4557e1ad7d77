"""Kernel timing for measurement tools: kmeans_trace_start / _read / _stop.

The host-side checks (argument validation, reading with tracing off) run
without a GPU; the GPU checks make sure each call brackets exactly its
dominant kernel, that launches beyond the capacity are counted but not
timed, and that the traced durations fit inside the calls' own time."""
import numpy as np
import pytest

import synth


@pytest.fixture(scope="module")
def km():
    from distance_argmin_gb300 import build as b
    b.build()
    import distance_argmin_gb300 as km
    km.load()
    return km


def test_trace_rejects_bad_arguments_without_a_gpu(km):
    lib = km.load()
    assert lib.kmeans_trace_start(0) == km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_trace_start(km.TRACE_MAX_CAPACITY + 1) == km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_trace_read(3, None, None, None) == km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_trace_read(-1, None, None, None) == km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_trace_read(0, None, None, None) == km.KMEANS_ERR_INVALID_ARG  # no output pointer


def test_trace_read_while_off_reports_nothing(km):
    assert km.load().kmeans_trace_stop() == km.KMEANS_OK
    for kernel in (km.KERNEL_ASSIGN_TC, km.KERNEL_UPDATE_MEAN, km.KERNEL_KMEANSPP_DIST):
        assert km.kmeans_trace_read(kernel) == (0.0, 0, 0)


@pytest.mark.gpu
def test_trace_counts_each_dominant_kernel_once_per_call(gpu_lib):
    import torch
    X, C, _ = synth.workload_inputs(synth.WORKLOADS["probe"])
    Xd, Cd = torch.from_numpy(X).cuda(), torch.from_numpy(C).cuda()
    ws = gpu_lib.workspace(gpu_lib.OP_LLOYD, X.shape[0], C.shape[0], X.shape[1])
    gpu_lib.kmeans_lloyd_iter(Xd, Cd, ws=ws)  # per-device set-up outside the traced region
    torch.cuda.synchronize()
    gpu_lib.kmeans_trace_start(16)
    try:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(3):
            gpu_lib.kmeans_lloyd_iter(Xd, Cd, ws=ws)
        gpu_lib.kmeans_assign(Xd, Cd, ws=ws)
        e1.record()
        torch.cuda.synchronize()
        wall_ms = e0.elapsed_time(e1)
        tc_ms, tc_timed, tc_seen = gpu_lib.kmeans_trace_read(gpu_lib.KERNEL_ASSIGN_TC)
        mean_ms, mean_timed, mean_seen = gpu_lib.kmeans_trace_read(gpu_lib.KERNEL_UPDATE_MEAN)
        assert (tc_timed, tc_seen) == (4, 4)
        assert (mean_timed, mean_seen) == (3, 3)
        assert gpu_lib.kmeans_trace_read(gpu_lib.KERNEL_KMEANSPP_DIST) == (0.0, 0, 0)
        assert 0.0 < tc_ms and 0.0 < mean_ms and tc_ms + mean_ms < wall_ms
    finally:
        gpu_lib.kmeans_trace_stop()
    assert gpu_lib.kmeans_trace_read(gpu_lib.KERNEL_ASSIGN_TC) == (0.0, 0, 0)


@pytest.mark.gpu
def test_trace_counts_launches_beyond_its_capacity(gpu_lib):
    import torch
    X, _, _ = synth.planted_blobs(3000, 64, 8, seed=5)
    Xd = torch.from_numpy(X).cuda()
    k = 6
    T = gpu_lib.n_trials_for(k)
    gpu_lib.kmeans_trace_start(2)
    try:
        gpu_lib.kmeanspp_init(Xd, k, 9, n_trials=T)
        torch.cuda.synchronize()
        ms, timed, seen = gpu_lib.kmeans_trace_read(gpu_lib.KERNEL_KMEANSPP_DIST)
        assert timed == 2 and seen > 2 and ms > 0.0
    finally:
        gpu_lib.kmeans_trace_stop()
    # tracing off: calls leave no records
    gpu_lib.kmeanspp_init(Xd, k, 9, n_trials=T)
    torch.cuda.synchronize()
    assert gpu_lib.kmeans_trace_read(gpu_lib.KERNEL_KMEANSPP_DIST) == (0.0, 0, 0)

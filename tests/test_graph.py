"""The entry points under CUDA graph capture.

Every entry point but kmeans_fit (which synchronises to read the inertia)
only enqueues work on the caller's stream, so a captured call replays as a
graph.  The chained launches become programmatic dependencies, and each
call's prologue resets the K-split tickets and tags, so a replay of a
captured assignment whose last round splits gives the eager call's bits."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


def test_captured_lloyd_iteration_replays_the_eager_bits(gpu_lib):
    n, k, d = 5000, 1000, 260  # 80 tiles: on a GB300 the last round splits along K
    X, _, _ = synth.planted_blobs(n, d, k, seed=7)
    C0 = np.ascontiguousarray(X[synth.init_rows(n, k, seed=8)])
    Xd = torch.from_numpy(X).cuda()
    Cd = torch.from_numpy(C0).cuda()
    ws = gpu_lib.workspace(gpu_lib.OP_LLOYD, n, k, d)
    outs = dict(C_new=torch.empty_like(Cd), labels=torch.empty(n, dtype=torch.int64, device="cuda"),
                best_dist=torch.empty(n, device="cuda"), inertia=torch.empty(1, dtype=torch.float64, device="cuda"),
                counts=torch.empty(k, dtype=torch.int32, device="cuda"))
    eager = [t.clone() for t in gpu_lib.kmeans_lloyd_iter(Xd, Cd, ws=ws, **outs)]  # also the per-device set-up
    torch.cuda.synchronize()
    for t in outs.values():
        t.zero_()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gpu_lib.kmeans_lloyd_iter(Xd, Cd, ws=ws, **outs)
    for _ in range(3):
        for t in outs.values():
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        got = [outs[key] for key in ("C_new", "labels", "best_dist", "inertia", "counts")]
        for a, b in zip(got, eager):
            assert a.cpu().numpy().tobytes() == b.cpu().numpy().tobytes()
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_OK


def test_captured_assignment_on_a_graph_stream(gpu_lib):
    # the assignment alone, several replays of one graph in a row with no
    # synchronisation in between
    n, k, d = 25600, 200, 256  # 100 tiles: splits on a GB300
    X, _, _ = synth.planted_blobs(n, d, k, seed=9)
    C = np.ascontiguousarray(X[synth.init_rows(n, k, seed=10)])
    Xd, Cd = torch.from_numpy(X).cuda(), torch.from_numpy(C).cuda()
    ws = gpu_lib.workspace(gpu_lib.OP_ASSIGN, n, k, d)
    labels = torch.empty(n, dtype=torch.int64, device="cuda")
    best = torch.empty(n, device="cuda")
    inertia = torch.empty(1, dtype=torch.float64, device="cuda")
    gpu_lib.kmeans_assign(Xd, Cd, labels, best, inertia, ws=ws)
    torch.cuda.synchronize()
    ref = (labels.clone(), best.clone(), inertia.clone())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        gpu_lib.kmeans_assign(Xd, Cd, labels, best, inertia, ws=ws)
    best.zero_()
    for _ in range(5):
        g.replay()
    torch.cuda.synchronize()
    for a, b in zip((labels, best, inertia), ref):
        assert a.cpu().numpy().tobytes() == b.cpu().numpy().tobytes()

"""Out-of-bounds writes and uninitialised reads, caught without a sanitizer.

Every workspace and output buffer here sits between two 64 KiB guard regions
filled with a canary byte; outputs start poisoned (NaN, or -7 for integers)
and the workspace starts as 0xFF bytes rather than zeros.  After each call
the guards must be intact, every output element must have been written, and
the results must equal, bit for bit, those of a call on fresh buffers: a
write past a buffer, a skipped output or a read of scratch the call did not
initialise shows up as a failure.  The shape has more tiles than a GB300 has
CTA pairs, so the assignment's last round splits along K.

A fit also resumes exactly from centroids saved to and loaded from a file:
the Lloyd state is the centroids alone."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

GUARD = 64 * 1024  # bytes on each side
CANARY = 0xA5
N, K, D = 5000, 1000, 260  # 80 tiles of 256 x 256: the last round splits along K


class Guarded:
    """A device buffer between two canary-filled guard regions."""

    def __init__(self, shape, dtype, fill):
        nbytes = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
        self.raw = torch.full((2 * GUARD + nbytes,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + nbytes].view(dtype).view(shape)
        self.t.fill_(fill)

    def intact(self):
        torch.cuda.synchronize()
        return bool((self.raw[:GUARD] == CANARY).all()) and bool((self.raw[-GUARD:] == CANARY).all())


def _inputs():
    X, _, _ = synth.planted_blobs(N, D, K, seed=N + K + D)
    C = np.ascontiguousarray(X[synth.init_rows(N, K, seed=D + 1)])
    return torch.from_numpy(X).cuda(), torch.from_numpy(C).cuda()


def _ws(km, op):
    return Guarded((km.kmeans_workspace_bytes(op, N, K, D),), torch.uint8, 0xFF)


def _outputs():
    return {"labels": Guarded((N,), torch.int64, -7), "best": Guarded((N,), torch.float32, float("nan")),
            "inertia": Guarded((1,), torch.float64, float("nan")), "counts": Guarded((K,), torch.int32, -7),
            "C_new": Guarded((K, D), torch.float32, float("nan"))}


def _same(a, b):
    return a.cpu().numpy().tobytes() == b.cpu().numpy().tobytes()


def _all_intact(*bufs):
    return all(b.intact() for b in bufs)


def _clean(km, *workspaces):
    # no bounded device wait ran out and no label was out of range
    return all(km.kmeans_device_status(w) == km.KMEANS_OK for w in workspaces)


@pytest.mark.parametrize("name,op", [("kmeans_assign", "OP_ASSIGN"), ("kmeans_assign_3xtf32", "OP_ASSIGN_3XTF32"),
                                     ("kmeans_assign_ffma", "OP_ASSIGN_FFMA")])
def test_assignment_stays_inside_its_buffers(gpu_lib, name, op):
    X, C = _inputs()
    fn = getattr(gpu_lib, name)
    wsr = gpu_lib.workspace(getattr(gpu_lib, op), N, K, D)
    ref = fn(X, C, ws=wsr)
    ws, out = _ws(gpu_lib, getattr(gpu_lib, op)), _outputs()
    got = fn(X, C, labels=out["labels"].t, best_dist=out["best"].t, inertia=out["inertia"].t, ws=ws.t)
    assert _clean(gpu_lib, wsr, ws.t)
    assert _all_intact(ws, out["labels"], out["best"], out["inertia"])
    assert not torch.isnan(out["best"].t).any() and not torch.isnan(out["inertia"].t).any()
    for a, b in zip(got, ref):
        assert _same(a, b)


def test_update_stays_inside_its_buffers(gpu_lib):
    X, C = _inputs()
    wsa = gpu_lib.workspace(gpu_lib.OP_ASSIGN, N, K, D)
    labels, _, _ = gpu_lib.kmeans_assign(X, C, ws=wsa)
    assert _clean(gpu_lib, wsa)
    labels[labels == 3] = 4  # cluster 3 empty: its row comes from C_old
    wsr = gpu_lib.workspace(gpu_lib.OP_UPDATE, N, K, D)
    ref = gpu_lib.kmeans_update(X, labels, C, ws=wsr)
    ws, out = _ws(gpu_lib, gpu_lib.OP_UPDATE), _outputs()
    got = gpu_lib.kmeans_update(X, labels, C, C_new=out["C_new"].t, counts=out["counts"].t, ws=ws.t)
    assert _clean(gpu_lib, wsr, ws.t)
    assert _all_intact(ws, out["C_new"], out["counts"])
    assert not torch.isnan(out["C_new"].t).any() and int(out["counts"].t.sum()) == N
    for a, b in zip(got, ref):
        assert _same(a, b)


@pytest.mark.parametrize("name,op", [("kmeans_lloyd_iter", "OP_LLOYD"), ("kmeans_lloyd_iter_fused", "OP_LLOYD_FUSED")])
def test_lloyd_iteration_stays_inside_its_buffers(gpu_lib, name, op):
    X, C = _inputs()
    fn = getattr(gpu_lib, name)
    wsr = gpu_lib.workspace(getattr(gpu_lib, op), N, K, D)
    ref = fn(X, C, ws=wsr)
    ws, out = _ws(gpu_lib, getattr(gpu_lib, op)), _outputs()
    got = fn(X, C, C_new=out["C_new"].t, labels=out["labels"].t, best_dist=out["best"].t,
             inertia=out["inertia"].t, counts=out["counts"].t, ws=ws.t)
    assert _clean(gpu_lib, wsr, ws.t)
    assert _all_intact(ws, *out.values())
    assert not torch.isnan(out["C_new"].t).any() and not torch.isnan(out["best"].t).any()
    assert int(out["counts"].t.sum()) == N
    if name == "kmeans_lloyd_iter":
        for a, b in zip(got, ref):
            assert _same(a, b)
    else:
        # float atomics in the fused update: its labels and counts are exact
        assert _same(got[1], ref[1]) and _same(got[4], ref[4])


def test_kmeanspp_stays_inside_its_buffers(gpu_lib):
    X, _ = _inputs()
    wsr = gpu_lib.workspace(gpu_lib.OP_KMEANSPP, N, K, D)
    ref_idx, ref_cen = gpu_lib.kmeanspp_init(X, K, 17, ws=wsr)
    ws = _ws(gpu_lib, gpu_lib.OP_KMEANSPP)
    idx, cen = Guarded((K,), torch.int64, -7), Guarded((K, D), torch.float32, float("nan"))
    gpu_lib.kmeanspp_init(X, K, 17, centers=cen.t, indices=idx.t, ws=ws.t)
    assert _clean(gpu_lib, wsr, ws.t)
    assert _all_intact(ws, idx, cen)
    assert _same(idx.t, ref_idx) and _same(cen.t, ref_cen)


def test_relocation_stays_inside_its_buffers(gpu_lib):
    X, C = _inputs()
    wsa = gpu_lib.workspace(gpu_lib.OP_ASSIGN, N, K, D)
    labels, best, _ = gpu_lib.kmeans_assign(X, C, ws=wsa)
    assert _clean(gpu_lib, wsa)
    labels[labels % 2 == 1] = 0  # every odd cluster empty
    wsr = gpu_lib.workspace(gpu_lib.OP_RELOCATE, N, K, 1)
    ref = gpu_lib.kmeans_relocate_empty(labels.clone(), best, K, ws=wsr)
    ws = Guarded((gpu_lib.kmeans_workspace_bytes(gpu_lib.OP_RELOCATE, N, K, 1),), torch.uint8, 0xFF)
    lab = Guarded((N,), torch.int64, 0)
    lab.t.copy_(labels)
    gpu_lib.kmeans_relocate_empty(lab.t, best, K, ws=ws.t)
    assert _clean(gpu_lib, wsr, ws.t)
    assert _all_intact(ws, lab)
    assert _same(lab.t, ref)


def test_fit_stays_inside_its_buffers(gpu_lib):
    X, C0 = _inputs()
    ref = gpu_lib.kmeans_fit(X, C=C0.clone(), init="given", max_iter=3, tol=0.0)
    ws, out = _ws(gpu_lib, gpu_lib.OP_FIT), _outputs()
    C = Guarded((K, D), torch.float32, 0.0)
    C.t.copy_(C0)
    got = gpu_lib.kmeans_fit(X, C=C.t, init="given", max_iter=3, tol=0.0, labels=out["labels"].t,
                             best_dist=out["best"].t, counts=out["counts"].t, ws=ws.t)
    assert _all_intact(ws, C, out["labels"], out["best"], out["counts"])
    for a, b in zip(got[:4], ref[:4]):
        assert _same(a, b)
    assert got[5] == ref[5] and np.array_equal(got[4], ref[4])


def test_fit_resumes_from_saved_centroids(gpu_lib, tmp_path):
    # unstructured data converges slowly, so five iterations run in full
    X = torch.from_numpy(synth.gaussian((20000, 16), seed=71)).cuda()
    C0 = X[torch.from_numpy(synth.init_rows(20000, 300, seed=72)).cuda()].contiguous()
    C5, lab5, best5, cnt5, hist5, n5 = gpu_lib.kmeans_fit(X, C=C0.clone(), init="given", max_iter=5, tol=0.0)
    assert n5 == 5
    C2, _, _, _, hist2, n2 = gpu_lib.kmeans_fit(X, C=C0.clone(), init="given", max_iter=2, tol=0.0)
    assert n2 == 2
    path = tmp_path / "centroids.npy"
    np.save(path, C2.cpu().numpy())
    C = torch.from_numpy(np.load(path)).cuda()
    C, lab, best, cnt, hist3, n3 = gpu_lib.kmeans_fit(X, C=C, init="given", max_iter=3, tol=0.0)
    assert n3 == 3
    assert _same(C, C5) and _same(lab, lab5) and _same(best, best5) and _same(cnt, cnt5)
    assert np.array_equal(np.concatenate([hist2, hist3]), hist5)

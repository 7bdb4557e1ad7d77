"""The tensor-core assignment's K split of a partly filled last round.

The assignment runs a persistent schedule of 256 x 256 tiles over the GPU's
CTA pairs (76 on a GB300).  When its last round is at most half full, those
tiles run as two K halves on two pairs each; the half that finishes first
parks its raw accumulator, the other adds it before the argmin, and both add
their part of ||x||^2 for tiles of the first centroid block.  These shapes
have more tiles than a GB300 has pairs, and their last rounds split."""
import numpy as np
import pytest

import oracle
import synth
from parity import check_assign, check_centroids, sq_norms

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")

SPLIT = [
    # (n, k, d) -> tiles = ceil(n / 256) * ceil(k / 256)
    (25600, 200, 256),  # 100 tiles in one centroid block: every split tile also reports ||x||^2
    (5000, 1000, 260),  # 80 tiles; ragged n, k and K halves (4 and 5 k-blocks)
    (40000, 600, 128),  # 471 tiles: a last round of 15 after six full ones
]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _inputs(n, k, d):
    X, _, _ = synth.planted_blobs(n, d, k, seed=n + k + d)
    C = np.ascontiguousarray(X[synth.init_rows(n, k, seed=d + 1)])
    return X, C


@pytest.mark.parametrize("shape", SPLIT, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("impl", ["kmeans_assign", "kmeans_assign_3xtf32"])
def test_split_tiles_match_the_oracle_and_repeat_bit_for_bit(gpu_lib, shape, impl):
    n, k, d = shape
    X, C = _inputs(n, k, d)
    fn = getattr(gpu_lib, impl)
    Xd, Cd = _dev(X), _dev(C)
    labels, best, inertia = fn(Xd, Cd)
    o_l, o_b, o_s, o_in = oracle.assign(X, C)
    check_assign(X, C, labels.cpu().numpy(), best.cpu().numpy(), o_l, o_b, o_s, what=f"{impl} {shape}")
    scale = (sq_norms(X) + sq_norms(C)[o_l]).sum()
    assert abs(float(inertia.item()) - o_in) <= 1e-4 * scale
    # which half parks is a race; the sum is not
    labels2, best2, inertia2 = fn(Xd, Cd)
    assert labels2.cpu().numpy().tobytes() == labels.cpu().numpy().tobytes()
    assert best2.cpu().numpy().tobytes() == best.cpu().numpy().tobytes()
    assert float(inertia2.item()) == float(inertia.item())


@pytest.mark.parametrize("shape,impl", [
    ((25600, 200, 4), "kmeans_assign"),            # one k-block: nothing to split
    ((20480, 200, 2052), "kmeans_assign_3xtf32"),  # 3xTF32 past its single-accumulator limit: never split
], ids=["one_kblock", "tf32_separate_accumulators"])
def test_many_tiles_without_a_split(gpu_lib, shape, impl):
    n, k, d = shape
    X, C = _inputs(n, k, d)
    labels, best, inertia = getattr(gpu_lib, impl)(_dev(X), _dev(C))
    o_l, o_b, o_s, o_in = oracle.assign(X, C)
    check_assign(X, C, labels.cpu().numpy(), best.cpu().numpy(), o_l, o_b, o_s, what=f"{impl} {shape}")
    scale = (sq_norms(X) + sq_norms(C)[o_l]).sum()
    assert abs(float(inertia.item()) - o_in) <= 1e-4 * scale


def test_the_split_runs_on_a_gb300(gpu_lib):
    # the built-in scratch of kmeans_assign_noalloc has no parking area, so
    # it never splits: on a GB300 the split tiles' sums round differently
    # (the K halves add at the end), while the labels agree
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the split schedule is sized for 152 SMs")
    n, k, d = SPLIT[0]
    X, C = _inputs(n, k, d)
    Xd, Cd = _dev(X), _dev(C)
    l_split, b_split, _ = gpu_lib.kmeans_assign(Xd, Cd)
    l_whole = torch.empty(n, dtype=torch.int64, device="cuda")
    b_whole = torch.empty(n, dtype=torch.float32, device="cuda")
    gpu_lib.kmeans_assign_noalloc(Xd, Cd, l_whole, b_whole)
    assert np.array_equal(l_split.cpu().numpy(), l_whole.cpu().numpy())
    differ = b_split.cpu().numpy() != b_whole.cpu().numpy()
    assert differ.any()
    # 100 tiles over 76 pairs: the last 24 tiles (rows 76 * 256 onwards) split
    assert not differ[:76 * 256].any()


def test_lloyd_iteration_with_split_tiles(gpu_lib):
    n, k, d = SPLIT[1]
    X, C = _inputs(n, k, d)
    C1, labels, best, inertia, counts = gpu_lib.kmeans_lloyd_iter(_dev(X), _dev(C))
    o_l, o_b, o_s, _ = oracle.assign(X, C)
    lab = labels.cpu().numpy()
    check_assign(X, C, lab, best.cpu().numpy(), o_l, o_b, o_s, what="lloyd with split tiles")
    o_C, o_cnt = oracle.update(X, lab, C)
    check_centroids(C1.cpu().numpy(), o_C, what="lloyd with split tiles")
    assert np.array_equal(counts.cpu().numpy().astype(np.int64), o_cnt)


def test_a_withheld_ready_tag_times_out_and_reports(gpu_lib, monkeypatch):
    # Fault injection on the host side: with the test switch set, the first
    # K half of every split tile parks its accumulator but never tags it.
    # Every second half's bounded wait (2 s) runs out, the kernel winds down,
    # the status word says so, and the next call on the same workspace is
    # correct again.  No trap, no fault, no unbounded spin.
    if torch.cuda.get_device_properties(0).multi_processor_count != 152:
        pytest.skip("the split schedule is sized for 152 SMs")
    n, k, d = SPLIT[0]
    X, C = _inputs(n, k, d)
    Xd, Cd = _dev(X), _dev(C)
    ws = gpu_lib.workspace(gpu_lib.OP_ASSIGN, n, k, d)
    monkeypatch.setenv("KMEANS_GB300_TEST_HOLD_KSPLIT_TAG", "1")
    gpu_lib.kmeans_assign(Xd, Cd, ws=ws)
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_ERR_DEVICE_TIMEOUT
    monkeypatch.delenv("KMEANS_GB300_TEST_HOLD_KSPLIT_TAG")
    labels, best, _ = gpu_lib.kmeans_assign(Xd, Cd, ws=ws)
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_OK
    o_l, o_b, o_s, _ = oracle.assign(X, C)
    check_assign(X, C, labels.cpu().numpy(), best.cpu().numpy(), o_l, o_b, o_s, what="after a withheld tag")


def test_host_iteration_whose_slices_each_split(gpu_lib):
    # kmeans_lloyd_iter_host with two slices launches the tensor-core pass
    # twice in one call, and on a GB300 each launch splits its last round
    # (320 tiles each: a last round of 16).  The second launch reuses the
    # tickets and tags without a prologue in between: its distinct epoch and
    # the reset by each first launch's second halves must keep it correct.
    n, k, d = 40960, 1024, 128
    X, C = _inputs(n, k, d)
    ref = gpu_lib.kmeans_lloyd_iter(_dev(X), _dev(C))
    Xh = torch.from_numpy(X).pin_memory()
    Ch = torch.from_numpy(C).pin_memory()
    Xd, Cd = torch.empty_like(Xh, device="cuda"), torch.empty_like(Ch, device="cuda")
    C_new = torch.empty_like(Cd)
    labels = torch.empty(n, dtype=torch.int64, device="cuda")
    best = torch.empty(n, device="cuda")
    counts = torch.empty(k, dtype=torch.int32, device="cuda")
    C_out_h = torch.empty((k, d), dtype=torch.float32).pin_memory()
    lab_h = torch.empty(n, dtype=torch.int64).pin_memory()
    in_h = torch.empty(1, dtype=torch.float64).pin_memory()
    ws = gpu_lib.workspace(gpu_lib.OP_LLOYD, n, k, d)
    for _ in range(2):  # twice on one workspace: the tickets left by the first call are clean
        done = gpu_lib.kmeans_lloyd_iter_host(Xh, Ch, Xd, Cd, C_new, labels, best, counts, C_out_h, lab_h, in_h,
                                              slices=2, ws=ws)
        done.synchronize()
        assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_OK
        lab = labels.cpu().numpy()
        np.testing.assert_array_equal(lab, ref[1].cpu().numpy())
        assert C_new.cpu().numpy().tobytes() == ref[0].cpu().numpy().tobytes()
        scale = sq_norms(X) + sq_norms(C)[lab]
        assert (np.abs(best.cpu().numpy().astype(np.float64) - ref[2].cpu().numpy()) <= 1e-4 * scale).all()
    rows = np.sort(np.random.default_rng(5).choice(n, 2048, replace=False))
    o_l, o_b, o_s, _ = oracle.assign(X[rows], C)
    check_assign(X[rows], C, lab, best.cpu().numpy(), o_l, o_b, o_s, rows=rows, what="two splitting slices")

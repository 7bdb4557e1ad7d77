"""GPU parity: the CUDA library (through its C ABI) against the CPU oracle on
the same seeded inputs.  Small shapes are compared on every row.  The three
large workloads' assignments are compared on every row with stored oracle
results, lloyd10's first iteration with the oracle run live, and its ten
iterations on a seeded sample of rows; updates on every row, with the GPU's
own labels so near-tie flips do not cascade."""
import ctypes
import hashlib
import os
import sys

import numpy as np
import pytest

import oracle
import synth
from parity import DIST_RTOL, check_assign, check_assign_every_row, check_centroids, sq_norms

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")


def dev_tensor(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy()


SMALL = [
    # (n, k, d): the fusion-probe page's separate check shape first, then
    # tails in every tile dimension (128 samples, 256 centroids, 32 features)
    (512, 17, 64),
    (1000, 300, 100),
    (777, 1, 36),
    (300, 300, 8),
    (2000, 513, 132),
    (260, 257, 4),
    (4096, 256, 512),
]


ASSIGN_IMPLS = {"tc": "kmeans_assign", "tf32": "kmeans_assign_3xtf32", "ffma": "kmeans_assign_ffma"}


@pytest.mark.parametrize("shape", SMALL, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("impl", list(ASSIGN_IMPLS))
@pytest.mark.parametrize("data", ["blobs", "gauss"])
def test_assign_matches_oracle(gpu_lib, shape, impl, data):
    n, k, d = shape
    if data == "blobs":
        X, _, _ = synth.planted_blobs(n, d, max(1, k), seed=n + k + d)
        C = np.ascontiguousarray(X[synth.init_rows(n, k, seed=d)])
    else:
        X = synth.gaussian((n, d), seed=n * 3 + 1, scale=2.0)
        C = synth.gaussian((k, d), seed=k * 7 + 2, scale=2.0)
    fn = getattr(gpu_lib, ASSIGN_IMPLS[impl])
    labels, best, inertia = fn(dev_tensor(X), dev_tensor(C))
    o_l, o_b, o_s, o_in = oracle.assign(X, C)
    check_assign(X, C, host(labels), host(best), o_l, o_b, o_s, what=f"{impl} {shape}")
    # the inertia tolerance is the sum of the per-sample distance tolerances
    scale = (sq_norms(X) + sq_norms(C)[o_l]).sum()
    assert abs(float(inertia.item()) - o_in) <= 1e-4 * scale


@pytest.mark.parametrize("impl", list(ASSIGN_IMPLS))
def test_duplicate_centroids_resolve_to_lowest_index(gpu_lib, impl):
    X = synth.gaussian((1500, 96), seed=5)
    C = synth.gaussian((600, 96), seed=6)
    C[517] = C[3]      # across centroid tiles
    C[40] = C[39]      # inside one tile
    C[299] = C[260]
    fn = getattr(gpu_lib, ASSIGN_IMPLS[impl])
    labels, best, _ = fn(dev_tensor(X), dev_tensor(C))
    lab = host(labels)
    assert not np.isin(lab, [517, 40, 299]).any()
    o_l, o_b, o_s, _ = oracle.assign(X, C)
    check_assign(X, C, lab, host(best), o_l, o_b, o_s, what=impl)


def test_planted_centers_are_recovered_exactly(gpu_lib):
    X, centers, blob = synth.planted_blobs(8192, 256, 300, seed=9)
    labels, _, _ = gpu_lib.kmeans_assign(dev_tensor(X), dev_tensor(centers))
    assert np.array_equal(host(labels), blob)


def test_single_sample_single_centroid(gpu_lib):
    X = synth.gaussian((1, 12), seed=1)
    labels, best, inertia = gpu_lib.kmeans_assign(dev_tensor(X), dev_tensor(X))
    assert host(labels).tolist() == [0]
    # x == c: the Gram form leaves only cancellation error, within tolerance
    assert 0.0 <= float(host(best)[0]) <= 1e-4 * 2 * sq_norms(X)[0]


@pytest.mark.parametrize("shape", [(512, 17, 64), (2000, 513, 132), (5000, 40, 7), (4096, 256, 512),
                                   (70000, 3, 20), (100000, 20000, 12), (40000, 33000, 8)],
                         ids=lambda s: "x".join(map(str, s)))
def test_update_matches_oracle(gpu_lib, shape):
    n, k, d = shape
    X = synth.gaussian((n, d), seed=n + 5, scale=1.5)
    C_old = synth.gaussian((k, d), seed=k + 6)
    labels = np.random.default_rng(n).integers(0, k, size=n).astype(np.int64)
    if k > 2:
        labels[labels == 1] = 0  # cluster 1 empty: keeps its row bit for bit
    C_new, counts = gpu_lib.kmeans_update(dev_tensor(X), dev_tensor(labels), dev_tensor(C_old))
    o_C, o_cnt = oracle.update(X, labels, C_old)
    assert np.array_equal(host(counts).astype(np.int64), o_cnt)
    got = host(C_new)
    check_centroids(got, o_C, what=str(shape))
    empty = o_cnt == 0
    assert got[empty].tobytes() == C_old[empty].tobytes()


def test_update_single_cluster_and_skewed_sizes(gpu_lib):
    # one huge cluster spanning many chunks plus tiny ones
    n, k, d = 100000, 9, 36
    X = synth.gaussian((n, d), seed=3)
    labels = np.zeros(n, np.int64)
    labels[::1000] = np.arange(100) % 8 + 1
    C_old = synth.gaussian((k, d), seed=4)
    C_new, counts = gpu_lib.kmeans_update(dev_tensor(X), dev_tensor(labels), dev_tensor(C_old))
    o_C, o_cnt = oracle.update(X, labels, C_old)
    assert np.array_equal(host(counts).astype(np.int64), o_cnt)
    check_centroids(host(C_new), o_C, what="skewed")


def test_update_one_cluster_across_many_small_chunks(gpu_lib):
    # small n, large d: the member list is cut into chunks of a few dozen
    # members (one wave of 512-column slices), so cluster 0's ~4050 members
    # cross some 85 chunk boundaries and are finished by the chunk fix-up
    n, k, d = 4096, 4, 8192
    X = synth.gaussian((n, d), seed=44, scale=1.5)
    labels = np.zeros(n, np.int64)
    labels[::97] = np.arange(len(labels[::97])) % 3 + 1
    C_old = synth.gaussian((k, d), seed=45)
    C_new, counts = gpu_lib.kmeans_update(dev_tensor(X), dev_tensor(labels), dev_tensor(C_old))
    o_C, o_cnt = oracle.update(X, labels, C_old)
    assert np.array_equal(host(counts).astype(np.int64), o_cnt)
    check_centroids(host(C_new), o_C, what="one cluster over many chunks")


@pytest.mark.parametrize("shape", [(1, 1, 4), (5, 3, 8), (100, 7, 9), (255, 40, 516)],
                         ids=lambda s: "x".join(map(str, s)))
def test_update_fewer_samples_than_count_tiles(gpu_lib, shape):
    # n below the 256 counting tiles: some tiles hold no sample, and their
    # blocks only scan the totals and write their share of the counts and
    # empty rows; the last cluster is left empty
    n, k, d = shape
    X = synth.gaussian((n, d), seed=n + 11, scale=1.5)
    C_old = synth.gaussian((k, d), seed=k + 12)
    labels = (np.arange(n) % max(1, k - 1)).astype(np.int64)
    C_new, counts = gpu_lib.kmeans_update(dev_tensor(X), dev_tensor(labels), dev_tensor(C_old))
    o_C, o_cnt = oracle.update(X, labels, C_old)
    assert np.array_equal(host(counts).astype(np.int64), o_cnt)
    got = host(C_new)
    check_centroids(got, o_C, what=str(shape))
    empty = o_cnt == 0
    assert got[empty].tobytes() == C_old[empty].tobytes()


def test_update_counting_limit_with_one_block_all_empty(gpu_lib):
    # k = 32768, the largest count table: 256 scatter blocks own 128 clusters
    # each (cluster j belongs to block j mod 256).  No label is a multiple of
    # 256, so every cluster block 0 owns is empty: its list of empty rows is
    # full.
    n, k, d = 40000, 32768, 8
    X = synth.gaussian((n, d), seed=21, scale=1.5)
    C_old = synth.gaussian((k, d), seed=22)
    labels = np.random.default_rng(23).integers(0, k, size=n).astype(np.int64)
    labels[labels % 256 == 0] += 1
    C_new, counts = gpu_lib.kmeans_update(dev_tensor(X), dev_tensor(labels), dev_tensor(C_old))
    o_C, o_cnt = oracle.update(X, labels, C_old)
    assert np.array_equal(host(counts).astype(np.int64), o_cnt)
    got = host(C_new)
    check_centroids(got, o_C, what="k = 32768")
    empty = o_cnt == 0
    assert empty[::256].all()
    assert got[empty].tobytes() == C_old[empty].tobytes()


def test_update_in_place(gpu_lib):
    n, k, d = 3000, 50, 64
    X = synth.gaussian((n, d), seed=8)
    C = synth.gaussian((k, d), seed=9)
    labels = np.random.default_rng(1).integers(0, k - 1, size=n).astype(np.int64)  # k-1 empty
    Cd = dev_tensor(C)
    gpu_lib.kmeans_update(dev_tensor(X), dev_tensor(labels), Cd, C_new=Cd)
    o_C, _ = oracle.update(X, labels, C)
    check_centroids(host(Cd), o_C, what="in place")


def test_lloyd_probe_workload(gpu_lib):
    w = synth.WORKLOADS["probe"]
    X, C0, _ = synth.workload_inputs(w)
    C1, labels, best, inertia, counts = gpu_lib.kmeans_lloyd_iter(dev_tensor(X), dev_tensor(C0))
    o_l, o_b, o_s, o_in = oracle.assign(X, C0)
    lab = host(labels)
    check_assign(X, C0, lab, host(best), o_l, o_b, o_s, what="probe")
    o_C1, o_cnt = oracle.update(X, lab, C0)
    check_centroids(host(C1), o_C1, what="probe update")
    assert np.array_equal(host(counts).astype(np.int64), o_cnt)
    assert (o_cnt > 0).all()  # random-row initialisation never empties a cluster at step 1


def test_bitwise_reproducible(gpu_lib):
    X, C0, _ = synth.workload_inputs(synth.Workload("t", 20000, 700, 200, 700, 1, 31, 32, ""))
    Xd, Cd = dev_tensor(X), dev_tensor(C0)
    a = [host(t) for t in gpu_lib.kmeans_lloyd_iter(Xd, Cd)]
    b = [host(t) for t in gpu_lib.kmeans_lloyd_iter(Xd, Cd)]
    for u, v in zip(a, b):
        assert u.tobytes() == v.tobytes()


def test_library_allocates_no_device_memory(gpu_lib):
    X, C0, _ = synth.workload_inputs(synth.Workload("t", 16384, 512, 256, 512, 1, 41, 42, ""))
    Xd, Cd = dev_tensor(X), dev_tensor(C0)
    outs = [torch.empty_like(Cd), torch.empty(16384, dtype=torch.int64, device="cuda"),
            torch.empty(16384, device="cuda"), torch.empty(1, dtype=torch.float64, device="cuda"),
            torch.empty(512, dtype=torch.int32, device="cuda")]
    ws = gpu_lib.workspace(gpu_lib.OP_LLOYD, 16384, 512, 256)
    gpu_lib.kmeans_lloyd_iter(Xd, Cd, *outs, ws=ws)  # first call loads the kernels
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        gpu_lib.kmeans_lloyd_iter(Xd, Cd, *outs, ws=ws)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    assert ws.numel() < 16384 * 512 * 4  # smaller than the (n, k) matrix it replaces


def test_bad_label_is_reported_not_faulted(gpu_lib):
    n, k, d = 5000, 20, 16
    X = synth.gaussian((n, d), seed=2)
    C = synth.gaussian((k, d), seed=3)
    labels = np.random.default_rng(0).integers(0, k, size=n).astype(np.int64)
    labels[1234] = k + 7
    ws = gpu_lib.workspace(gpu_lib.OP_UPDATE, n, k, d)
    gpu_lib.kmeans_update(dev_tensor(X), dev_tensor(labels), dev_tensor(C), ws=ws)
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_ERR_DEVICE_LABEL
    labels[1234] = 0
    gpu_lib.kmeans_update(dev_tensor(X), dev_tensor(labels), dev_tensor(C), ws=ws)
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_OK


def test_status_ok_after_assign(gpu_lib):
    X = synth.gaussian((3000, 64), seed=2)
    C = synth.gaussian((100, 64), seed=3)
    ws = gpu_lib.workspace(gpu_lib.OP_ASSIGN, 3000, 100, 64)
    gpu_lib.kmeans_assign(dev_tensor(X), dev_tensor(C), ws=ws)
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_OK


# ------------------------------------------------------------- k-means++
def _record_margins(record_property, margins):
    # how close each D^2 draw came to a running-sum boundary (fraction of
    # the total): the closer, the more exactly the distances must agree
    record_property("draws", int(len(margins)))
    record_property("min_margin", float(margins.min()))
    record_property("draws_below_1e-7", int((margins < 1e-7).sum()))


@pytest.mark.parametrize("case", [(3000, 64, 40, 0, 42), (3000, 64, 40, 1, 7), (500, 33, 60, 3, 123),
                                  (2048, 128, 32, 8, 2024), (1000, 4, 1000, 2, 5),
                                  # several 256-feature steps (the register prefetch), ragged last step
                                  (1500, 700, 12, 4, 11),
                                  # two feature slices, the second ragged
                                  (1200, 4100, 6, 3, 12),
                                  # odd d: scalar loads, several steps
                                  (900, 1027, 8, 2, 13)],
                         ids=lambda c: "n%d_d%d_k%d_T%d_s%d" % c)
def test_kmeanspp_indices_match_oracle(gpu_lib, case, record_property):
    n, d, k, T, seed = case
    X, _, _ = synth.planted_blobs(n, d, max(1, k // 2), seed=n + d)
    idx, centers = gpu_lib.kmeanspp_init(dev_tensor(X), k, seed, n_trials=T)
    o_idx, margins, _ = oracle.kmeanspp(X, k, seed, n_trials=T)
    _record_margins(record_property, margins)
    got = host(idx)
    assert np.array_equal(got, o_idx), f"first mismatch at {np.argmax(got != o_idx)}"
    assert host(centers).tobytes() == np.ascontiguousarray(X[o_idx]).tobytes()


@pytest.mark.parametrize("T,aligned", [(8, True), (12, True), (8, False)], ids=["T8", "T12-two-passes", "unaligned"])
def test_kmeanspp_row_pruning_keeps_the_oracle_indices(gpu_lib, T, aligned):
    # well-separated blobs (the planted ones: center spread 1, within 0.5),
    # more centers than blobs: once a blob has a center its rows can no
    # longer change and are skipped, so the passes read fewer rows than
    # n per pass; the picks stay the oracle's.  Rows that are not 16-byte
    # groups (X offset by one float) are never pruned.
    n, d, k, seed = 6000, 512, 96, 77
    X, _, _ = synth.planted_blobs(n, d, 48, seed=n + d)
    Xd = dev_tensor(X)
    if not aligned:
        buf = torch.empty(n * d + 1, dtype=torch.float32, device="cuda")
        buf[1:].copy_(Xd.reshape(-1))
        Xd = buf[1:].view(n, d)
    ws = gpu_lib.workspace(gpu_lib.OP_KMEANSPP, n, k, d)
    idx, _ = gpu_lib.kmeanspp_init(Xd, k, seed, n_trials=T, ws=ws)
    rows = gpu_lib.kmeanspp_rows_read(ws)
    o_idx, _, _ = oracle.kmeanspp(X, k, seed, n_trials=T)
    assert np.array_equal(host(idx), o_idx), f"first mismatch at {np.argmax(host(idx) != o_idx)}"
    passes = k * ((T + 7) // 8)
    if aligned:
        assert n <= rows < 0.9 * n * passes, rows
    else:
        assert rows == 0


def test_kmeanspp_identical_points(gpu_lib):
    X = np.ones((100, 8), np.float32)
    idx, _ = gpu_lib.kmeanspp_init(dev_tensor(X), 5, 3, n_trials=2)
    o_idx, _, _ = oracle.kmeanspp(X, 5, 3, n_trials=2)
    assert np.array_equal(host(idx), o_idx)


# ------------------------------------------------------ full-size workloads
def _sample_rows(n, m, seed):
    return np.sort(np.random.default_rng(seed).choice(n, size=min(n, m), replace=False))


@pytest.mark.slow
def test_lloyd10_workload_ten_iterations(gpu_lib, record_property):
    # ten Lloyd iterations, each checked on every row: iteration t's
    # assignment against the oracle's assignment to the same C_t (the GPU's),
    # its update against the oracle's mean of the GPU's labels, and the
    # inertia never rising (2.7e11 binary64 multiply-adds per iteration for
    # the oracle: seconds on a many-core host)
    w = synth.WORKLOADS["lloyd10"]
    X, C0, _ = synth.workload_inputs(w)
    Xd = dev_tensor(X)
    C = C0
    prev = np.inf
    ws = gpu_lib.workspace(gpu_lib.OP_LLOYD, w.n, w.k, w.d)
    flips, worst = 0, 0.0
    for it in range(w.iters):
        Cd = dev_tensor(C)
        C1, labels, best, inertia, counts = gpu_lib.kmeans_lloyd_iter(Xd, Cd, ws=ws)
        lab = host(labels)
        o_l, o_b, o_s, o_in = oracle.assign(X, C)
        f, wr = check_assign(X, C, lab, host(best), o_l, o_b, o_s, what=f"iter {it}")
        flips += f
        worst = max(worst, wr)
        scale = (sq_norms(X) + sq_norms(C)[o_l]).sum()
        assert abs(float(inertia.item()) - o_in) <= DIST_RTOL * scale
        o_C1, o_cnt = oracle.update(X, lab, C)
        check_centroids(host(C1), o_C1, what=f"iter {it} update")
        assert np.array_equal(host(counts).astype(np.int64), o_cnt)
        val = float(inertia.item())
        assert val <= prev * (1 + 1e-6), f"inertia rose at iteration {it}"
        prev = val
        C = host(C1)
    record_property("near_tie_flips", flips)
    record_property("worst_rel_distance_error", worst)
    print(f"lloyd10, 10 iterations x {w.n} rows: worst relative distance error {worst:.3e}, near-tie flips {flips}")


@pytest.mark.slow
def test_lloyd10_first_iteration_every_row(gpu_lib, record_property):
    # the assignment of all 65536 samples against the 1024 initial centroids,
    # row by row against the oracle (2.7e11 float64 multiply-adds: seconds on
    # a many-core host), then the update on the GPU's labels
    w = synth.WORKLOADS["lloyd10"]
    X, C0, _ = synth.workload_inputs(w)
    C1, labels, best, inertia, counts = gpu_lib.kmeans_lloyd_iter(dev_tensor(X), dev_tensor(C0))
    lab = host(labels)
    o_l, o_b, o_s, o_in = oracle.assign(X, C0)
    flips, worst = check_assign(X, C0, lab, host(best), o_l, o_b, o_s, what="lloyd10 every row")
    record_property("near_tie_flips", flips)
    record_property("worst_rel_distance_error", worst)
    print(f"lloyd10 iteration 1, all {w.n} rows: worst relative distance error {worst:.3e}, near-tie flips {flips}")
    scale = (sq_norms(X) + sq_norms(C0)[o_l]).sum()
    assert abs(float(inertia.item()) - o_in) <= 1e-4 * scale
    o_C1, o_cnt = oracle.update(X, lab, C0)
    check_centroids(host(C1), o_C1, what="lloyd10 iteration 1 update")
    assert np.array_equal(host(counts).astype(np.int64), o_cnt)


def _large_golden(name):
    sys.path.insert(0, os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden"))
    import make_large_assign
    return make_large_assign.load(name)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["sample_heavy", "centroid_heavy", "feature_heavy"])
def test_large_workload_one_iteration(gpu_lib, name, record_property):
    # Every row of the assignment against the oracle's, which
    # tests/golden/make_large_assign.py stored ahead of time (the brute-force
    # argmin takes the oracle minutes per workload).  The stored SHA-256 of the
    # samples and centroids makes sure the input generator gave this machine
    # the bytes the oracle saw.  Then the update on the GPU's labels, every
    # row, against the oracle run live.
    w = synth.WORKLOADS[name]
    o_l, near_rows, near_best, near_second, o_inertia, meta = _large_golden(name)
    assert (meta["n"], meta["k"], meta["d"]) == (w.n, w.k, w.d)
    X, C0, _ = synth.workload_inputs(w)
    assert hashlib.sha256(X.tobytes()).hexdigest() == meta["x_sha256"], \
        f"the input generator gave different samples here than on the {meta['machine']} host the oracle ran on"
    assert hashlib.sha256(C0.tobytes()).hexdigest() == meta["c_sha256"]
    Xd, Cd = dev_tensor(X), dev_tensor(C0)
    C1, labels, best, inertia, counts = gpu_lib.kmeans_lloyd_iter(Xd, Cd)
    lab, bd = host(labels), host(best)
    del Xd
    torch.cuda.empty_cache()
    flips, worst, near = check_assign_every_row(X, C0, lab, bd, o_l, near_rows, near_best, near_second, what=name)
    record_property("rows", w.n)
    record_property("near_ties", near)
    record_property("near_tie_flips", flips)
    record_property("worst_rel_distance_error", worst)
    print(f"{name}, all {w.n} rows: worst relative distance error {worst:.3e}, {near} near ties, {flips} flips")
    scale = (sq_norms(X) + sq_norms(C0)[o_l]).sum()
    assert abs(float(inertia.item()) - o_inertia) <= DIST_RTOL * scale
    o_C1, o_cnt = oracle.update(X, lab, C0)
    check_centroids(host(C1), o_C1, what=name + " update")
    assert np.array_equal(host(counts).astype(np.int64), o_cnt)
    assert np.isfinite(bd).all() and (bd >= 0).all()


@pytest.mark.parametrize("shape", [(3000, 300, 2048), (5000, 700, 4100), (2600, 257, 8192), (9000, 1100, 2052),
                                   (2600, 300, 8196), (3000, 700, 16384), (700, 300, 24576)],
                         ids=lambda s: "x".join(map(str, s)))
def test_wide_units_with_ragged_centroid_columns(gpu_lib, shape):
    # wide units (two 256-column tiles per CTA pair) where the second tile
    # is partly or, in the last unit column, entirely past k; ragged rows.
    # Above 8192 features the units run K in chunks (8196: two uneven
    # chunks, 16384: two, 24576: three) with a running sum per CTA.
    n, k, d = shape
    X, _, _ = synth.planted_blobs(n, d, max(1, k // 3), seed=n + d)
    C = np.ascontiguousarray(X[synth.init_rows(n, k, seed=k)])
    C1, labels, best, inertia, counts = gpu_lib.kmeans_lloyd_iter(dev_tensor(X), dev_tensor(C))
    o_l, o_b, o_s, o_in = oracle.assign(X, C)
    check_assign(X, C, host(labels), host(best), o_l, o_b, o_s, what=f"wide {shape}")
    scale = (sq_norms(X) + sq_norms(C)[o_l]).sum()
    assert abs(float(inertia.item()) - o_in) <= DIST_RTOL * scale
    o_C1, o_cnt = oracle.update(X, host(labels), C)
    check_centroids(host(C1), o_C1, what=f"wide {shape} update")
    assert np.array_equal(host(counts).astype(np.int64), o_cnt)


def test_wide_units_in_step_over_many_rounds(gpu_lib):
    # 1256 wide units over 76 CTA pairs: 17 rounds, so the producers hold
    # each other at the round starts (a soft barrier, a last round of 40
    # units); sampled rows against the oracle, and a second call on the same
    # workspace gives the same bits
    n, k, d = 40000, 4000, 2048
    X, _, _ = synth.planted_blobs(n, d, 500, seed=95)
    C = np.ascontiguousarray(X[synth.init_rows(n, k, seed=96)])
    Xd, Cd = dev_tensor(X), dev_tensor(C)
    ws = gpu_lib.workspace(gpu_lib.OP_ASSIGN, n, k, d)
    labels, best, inertia = gpu_lib.kmeans_assign(Xd, Cd, ws=ws)
    rows = _sample_rows(n, 512, 97)
    o_l, o_b, o_s, _ = oracle.assign(X[rows], C)
    check_assign(X[rows], C, host(labels), host(best), o_l, o_b, o_s, rows=rows, what="many rounds")
    labels2, best2, _ = gpu_lib.kmeans_assign(Xd, Cd, ws=ws)
    assert torch.equal(labels, labels2) and torch.equal(best, best2)


def test_two_long_assignments_at_once_on_two_streams(gpu_lib):
    # two launches of 17 rounds each on two streams: while one holds the SMs
    # the other's CTAs are not all resident, so its round barrier runs out of
    # its short wait; both must finish cleanly with the bits of a call alone
    n, k, d = 40000, 4000, 2048
    X, _, _ = synth.planted_blobs(n, d, 500, seed=98)
    C = np.ascontiguousarray(X[synth.init_rows(n, k, seed=99)])
    Xd, Cd = dev_tensor(X), dev_tensor(C)
    ref = gpu_lib.kmeans_assign(Xd, Cd)
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream(), torch.cuda.Stream()]
    wss = [gpu_lib.workspace(gpu_lib.OP_ASSIGN, n, k, d) for _ in range(2)]
    torch.cuda.synchronize()
    outs = [gpu_lib.kmeans_assign(Xd, Cd, ws=wss[i], stream=streams[i]) for i in range(2)]
    torch.cuda.synchronize()
    for i in range(2):
        assert gpu_lib.kmeans_device_status(wss[i], streams[i]) == gpu_lib.KMEANS_OK
        assert torch.equal(outs[i][0], ref[0]) and torch.equal(outs[i][1], ref[1])


@pytest.mark.parametrize("impl,d,k", [("tc", 4096, 250), ("tc", 4100, 250), ("tc", 8192, 700), ("tc", 8196, 700),
                                     ("tf32", 2048, 700), ("tf32", 2052, 700), ("tf32", 8192, 700)])
def test_accumulator_modes_either_side_of_their_feature_limit(gpu_lib, d, k, impl):
    # bf16x3 with one centroid tile (k <= 256): one double-buffered
    # accumulator per tile up to 4096 features, separate accumulators for the
    # corrections above.  bf16x3 with more (k > 256): wide units, one
    # accumulator per tile, over K chunks above 8192 features.  3xTF32: one
    # double-buffered accumulator up to 2048, separate ones above.  Several
    # tiles per CTA pair, ragged sample and centroid tiles.
    n = 20000
    X, _, _ = synth.planted_blobs(n, d, 64, seed=91)
    C = np.ascontiguousarray(X[synth.init_rows(n, k, seed=92)])
    labels, best, inertia = getattr(gpu_lib, ASSIGN_IMPLS[impl])(dev_tensor(X), dev_tensor(C))
    rows = _sample_rows(n, 512, 93)
    o_l, o_b, o_s, _ = oracle.assign(X[rows], C)
    flips, worst = check_assign(X[rows], C, host(labels), host(best), o_l, o_b, o_s, rows=rows,
                                what=f"{impl} d={d}")
    print(f"{impl} d={d} k={k}: worst relative distance error {worst:.3e}, near-tie flips {flips} of {len(rows)}")


@pytest.mark.slow
def test_kmeanspp_workload_prefix(gpu_lib, record_property):
    w = synth.KMEANSPP
    X, _, _ = synth.planted_blobs(w.n, w.d, w.blobs, w.data_seed)
    T = oracle.n_trials_for(w.k)
    idx, _ = gpu_lib.kmeanspp_init(dev_tensor(X), w.k, w.init_seed, n_trials=T)
    got = host(idx)
    assert len(np.unique(got)) == w.k  # D^2 sampling never repeats a chosen sample
    o_idx, margins, _ = oracle.kmeanspp(X, 12, w.init_seed, n_trials=T)
    _record_margins(record_property, margins)
    assert np.array_equal(got[:12], o_idx), f"first mismatch at {np.argmax(got[:12] != o_idx)}"


def _read_kmeanspp_golden():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kmeanspp_workload_indices.txt")
    meta, idx = {}, []
    with open(path) as f:
        for line in f:
            if line.startswith("#"):
                for tok in line[1:].split():
                    if "=" in tok:
                        key, val = tok.split("=", 1)
                        meta[key] = val
            elif line.strip():
                idx.append(int(line))
    return meta, np.array(idx, dtype=np.int64)


@pytest.mark.slow
def test_kmeanspp_workload_every_center(gpu_lib, record_property):
    # All 1024 centers of the full seeding against the oracle's, written ahead
    # of time by tests/golden/make_kmeanspp_workload.py (the oracle needs
    # about 8 minutes for them).  The stored SHA-256 of the samples makes sure
    # the input generator gave this machine the bytes the oracle saw.
    w = synth.KMEANSPP
    meta, o_idx = _read_kmeanspp_golden()
    assert (int(meta["n"]), int(meta["d"]), int(meta["k"]), int(meta["seed"])) == (w.n, w.d, w.k, w.init_seed)
    X, _, _ = synth.planted_blobs(w.n, w.d, w.blobs, w.data_seed)
    assert hashlib.sha256(X.tobytes()).hexdigest() == meta["x_sha256"], \
        f"the input generator gave different samples here than on the {meta.get('machine')} host the oracle ran on"
    T = int(meta["trials"])
    assert T == oracle.n_trials_for(w.k) and len(o_idx) == w.k
    idx, centers = gpu_lib.kmeanspp_init(dev_tensor(X), w.k, w.init_seed, n_trials=T)
    got = host(idx)
    record_property("draws", int(meta["draws"]))
    record_property("min_margin", float(meta["smallest_margin"]))
    assert np.array_equal(got, o_idx), f"first mismatch at center {np.argmax(got != o_idx)}"
    assert host(centers).tobytes() == np.ascontiguousarray(X[o_idx]).tobytes()


def test_starved_pipeline_times_out_and_reports(gpu_lib, monkeypatch):
    # Fault injection on the host side: the producer issues no loads, every
    # bounded pipeline wait runs out (2 s), the kernel winds down and the
    # status word says so; the context stays usable for the next call.
    X = synth.gaussian((1000, 64), seed=1)
    C = synth.gaussian((50, 64), seed=2)
    Xd, Cd = dev_tensor(X), dev_tensor(C)
    ws = gpu_lib.workspace(gpu_lib.OP_ASSIGN, 1000, 50, 64)
    monkeypatch.setenv("KMEANS_GB300_TEST_STARVE_PIPELINE", "1")
    labels, best, _ = gpu_lib.kmeans_assign(Xd, Cd, ws=ws)
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_ERR_DEVICE_TIMEOUT
    assert (host(labels) == -1).all()
    monkeypatch.delenv("KMEANS_GB300_TEST_STARVE_PIPELINE")
    labels, best, _ = gpu_lib.kmeans_assign(Xd, Cd, ws=ws)
    assert gpu_lib.kmeans_device_status(ws) == gpu_lib.KMEANS_OK
    o_l, o_b, o_s, _ = oracle.assign(X, C)
    check_assign(X, C, host(labels), host(best), o_l, o_b, o_s, what="after timeout")


def _same_distances(best, ref_best, X, C, labels):
    # each slice runs its own tensor-core pass, whose schedule may split a
    # partly filled last round into K halves differently from the single
    # call: a different float32 accumulation error, within the tolerance
    scale = sq_norms(X) + sq_norms(C)[labels]
    diff = np.abs(np.asarray(best, np.float64) - np.asarray(ref_best, np.float64))
    assert (diff <= DIST_RTOL * scale).all()
    return scale.sum()


def test_lloyd_iteration_from_host_buffers_matches_device_call(gpu_lib):
    # the host-input iteration (row slices assigned as they land) gives the
    # device-resident call's labels, centroids and counts bit for bit, and its
    # distances and inertia bit for bit in one slice, within the tolerance in
    # several; 5 slices of 6144 rows over 30000 samples leave a ragged last
    # slice
    w = synth.Workload("t", 30000, 300, 132, 300, 1, 51, 52, "")
    X, C0, _ = synth.workload_inputs(w)
    n, k, d = w.n, w.k, w.d
    ref = gpu_lib.kmeans_lloyd_iter(dev_tensor(X), dev_tensor(C0))
    Xh = torch.from_numpy(X).pin_memory()
    Ch = torch.from_numpy(C0).pin_memory()
    Xd, Cd = torch.empty_like(Xh, device="cuda"), torch.empty_like(Ch, device="cuda")
    C_new = torch.empty_like(Cd)
    labels = torch.empty(n, dtype=torch.int64, device="cuda")
    best = torch.empty(n, device="cuda")
    counts = torch.empty(k, dtype=torch.int32, device="cuda")
    C_out_h = torch.empty((k, d), dtype=torch.float32).pin_memory()
    lab_h = torch.empty(n, dtype=torch.int64).pin_memory()
    in_h = torch.empty(1, dtype=torch.float64).pin_memory()
    for slices in (5, 1):
        done = gpu_lib.kmeans_lloyd_iter_host(Xh, Ch, Xd, Cd, C_new, labels, best, counts, C_out_h, lab_h, in_h,
                                              slices=slices)
        done.synchronize()
        np.testing.assert_array_equal(lab_h.numpy(), host(ref[1]))
        assert C_out_h.numpy().tobytes() == host(ref[0]).tobytes()
        np.testing.assert_array_equal(host(counts), host(ref[4]))
        if slices == 1:
            assert host(best).tobytes() == host(ref[2]).tobytes()
            assert float(in_h[0]) == float(ref[3].item())
        else:
            total = _same_distances(host(best), host(ref[2]), X, C0, host(ref[1]))
            assert abs(float(in_h[0]) - float(ref[3].item())) <= DIST_RTOL * total
        assert Xd.cpu().numpy().tobytes() == X.tobytes()


def test_back_to_back_host_iterations_overlapping_their_copies(gpu_lib):
    # two alternating device buffer sets with the overlap flag: each call's
    # copies may run beside the previous call's update; every call must still
    # give the device call's results (the inertia within the tolerance)
    w = synth.Workload("t", 20000, 200, 64, 200, 1, 53, 54, "")
    X, C0, _ = synth.workload_inputs(w)
    n, k, d = w.n, w.k, w.d
    ref = gpu_lib.kmeans_lloyd_iter(dev_tensor(X), dev_tensor(C0))
    Xh, Ch = torch.from_numpy(X).pin_memory(), torch.from_numpy(C0).pin_memory()
    Xd = [torch.empty((n, d), device="cuda") for _ in range(2)]
    Cd = [torch.empty((k, d), device="cuda") for _ in range(2)]
    C_new = torch.empty((k, d), device="cuda")
    labels = torch.empty(n, dtype=torch.int64, device="cuda")
    best = torch.empty(n, device="cuda")
    counts = torch.empty(k, dtype=torch.int32, device="cuda")
    outs = [(torch.empty((k, d)).pin_memory(), torch.empty(n, dtype=torch.int64).pin_memory(),
             torch.empty(1, dtype=torch.float64).pin_memory()) for _ in range(4)]
    cs = torch.cuda.Stream()
    done = [None, None]
    for j in range(4):
        slot = j % 2
        if done[slot] is not None:
            cs.wait_event(done[slot])
        C_h, lab_h, in_h = outs[j]
        done[slot] = gpu_lib.kmeans_lloyd_iter_host(Xh, Ch, Xd[slot], Cd[slot], C_new, labels, best, counts, C_h,
                                                    lab_h, in_h, slices=4, copy_stream=cs, overlap_previous=True)
    torch.cuda.synchronize()
    total = (sq_norms(X) + sq_norms(C0)[host(ref[1])]).sum()
    for C_h, lab_h, in_h in outs:
        np.testing.assert_array_equal(lab_h.numpy(), host(ref[1]))
        assert C_h.numpy().tobytes() == host(ref[0]).tobytes()
        assert abs(float(in_h[0]) - float(ref[3].item())) <= DIST_RTOL * total  # four slices: see above


def test_host_iterations_reading_back_on_alternating_copy_streams(gpu_lib):
    # the read-backs on the copy stream: two alternating sets of device
    # buffers (inputs and outputs) and two copy streams, so each call's
    # read-back runs beside the next call's assignment; every call must give
    # the device call's results, visible once its copy stream is done
    w = synth.Workload("t", 20000, 300, 64, 300, 1, 55, 56, "")
    X, C0, _ = synth.workload_inputs(w)
    n, k, d = w.n, w.k, w.d
    ref = gpu_lib.kmeans_lloyd_iter(dev_tensor(X), dev_tensor(C0))
    Xh, Ch = torch.from_numpy(X).pin_memory(), torch.from_numpy(C0).pin_memory()
    Xd = [torch.empty((n, d), device="cuda") for _ in range(2)]
    Cd = [torch.empty((k, d), device="cuda") for _ in range(2)]
    C_new = [torch.empty((k, d), device="cuda") for _ in range(2)]
    labels = [torch.empty(n, dtype=torch.int64, device="cuda") for _ in range(2)]
    inertia = [torch.empty(1, dtype=torch.float64, device="cuda") for _ in range(2)]
    best = torch.empty(n, device="cuda")
    counts = torch.empty(k, dtype=torch.int32, device="cuda")
    outs = [(torch.empty((k, d)).pin_memory(), torch.empty(n, dtype=torch.int64).pin_memory(),
             torch.empty(1, dtype=torch.float64).pin_memory()) for _ in range(5)]
    cs = [torch.cuda.Stream(), torch.cuda.Stream()]
    done = []
    for j in range(5):
        slot = j % 2
        C_h, lab_h, in_h = outs[j]
        done.append(gpu_lib.kmeans_lloyd_iter_host(Xh, Ch, Xd[slot], Cd[slot], C_new[slot], labels[slot], best,
                                                   counts, C_h, lab_h, in_h, slices=1, inertia=inertia[slot],
                                                   copy_stream=cs[slot], overlap_previous=True,
                                                   readback_on_copy_stream=True))
    for (C_h, lab_h, in_h), ev in zip(outs, done):
        ev.synchronize()
        np.testing.assert_array_equal(lab_h.numpy(), host(ref[1]))
        assert C_h.numpy().tobytes() == host(ref[0]).tobytes()
        assert float(in_h[0]) == float(ref[3].item())  # one slice: bit for bit


def test_lloyd_iteration_from_host_buffers_rejects_bad_arguments(gpu_lib):
    lib = gpu_lib.load()
    fake = ctypes.c_void_p(0x10000)  # validation fails before any pointer is used
    s = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = lambda slices, cs, flags=0: (fake, fake, fake, fake, fake, fake, fake, None, None, None, None, None, 1024,
                                        16, 32, slices, flags, fake, 1 << 30, s, cs)
    assert lib.kmeans_lloyd_iter_host(*args(0, None)) == gpu_lib.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_lloyd_iter_host(*args(gpu_lib.HOST_MAX_SLICES + 1, None)) == gpu_lib.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_lloyd_iter_host(*args(4, s)) == gpu_lib.KMEANS_ERR_INVALID_ARG  # copy stream == stream
    assert lib.kmeans_lloyd_iter_host(*args(4, None, 4)) == gpu_lib.KMEANS_ERR_INVALID_ARG  # unknown flag


def test_first_kernel_waits_for_the_callers_kernel(gpu_lib):
    # Each call's first kernel is launched so that it may be scheduled while
    # the kernel before it on the stream drains.  Here that kernel is the
    # caller's own (a torch multiply writing X and C, then the labels, right
    # before the call, with no synchronisation): the library must read what
    # it wrote, not the zeros underneath.
    n, k, d = 65536, 256, 512
    X = synth.gaussian((n, d), seed=71)
    Xs = dev_tensor(X)
    Cs = dev_tensor(X[:: n // k][:k])
    ref_lab, ref_best, ref_in = gpu_lib.kmeans_assign(Xs, Cs)
    ref_C, ref_cnt = gpu_lib.kmeans_update(Xs, ref_lab, Cs)
    ref_l = gpu_lib.kmeans_lloyd_iter(Xs, Cs)
    torch.cuda.synchronize()
    Xd, Cd = torch.empty_like(Xs), torch.empty_like(Cs)
    lab, best, inertia = torch.empty_like(ref_lab), torch.empty_like(ref_best), torch.empty_like(ref_in)
    labd = torch.empty_like(ref_lab)
    C_new, counts = torch.empty_like(Cs), torch.empty_like(ref_cnt)
    ws_a = gpu_lib.workspace(gpu_lib.OP_ASSIGN, n, k, d)
    ws_u = gpu_lib.workspace(gpu_lib.OP_UPDATE, n, k, d)
    ws_l = gpu_lib.workspace(gpu_lib.OP_LLOYD, n, k, d)
    for _ in range(3):
        Xd.zero_()
        Cd.zero_()
        labd.zero_()
        torch.cuda.synchronize()
        torch.mul(Xs, 1.0, out=Xd)
        torch.mul(Cs, 1.0, out=Cd)
        gpu_lib.kmeans_assign(Xd, Cd, lab, best, inertia, ws=ws_a)
        torch.mul(ref_lab, 1, out=labd)
        gpu_lib.kmeans_update(Xd, labd, Cd, C_new, counts, ws=ws_u)
        torch.cuda.synchronize()
        assert torch.equal(lab, ref_lab) and torch.equal(best, ref_best) and torch.equal(inertia, ref_in)
        assert torch.equal(C_new, ref_C) and torch.equal(counts, ref_cnt)
        Xd.zero_()
        Cd.zero_()
        torch.cuda.synchronize()
        torch.mul(Xs, 1.0, out=Xd)
        torch.mul(Cs, 1.0, out=Cd)
        got = gpu_lib.kmeans_lloyd_iter(Xd, Cd, ws=ws_l)
        torch.cuda.synchronize()
        for a, b in zip(got, ref_l):
            assert torch.equal(a, b)

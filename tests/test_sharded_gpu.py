"""The sample-sharded path on the GPU, through the C ABI.

* One rank: kmeans_lloyd_iter_partial + kmeans_reduce_partials give
  kmeans_lloyd_iter's bits, and the shard steps of k-means++ give
  kmeanspp_init's indices (the sums across ranks start from the first rank's
  value as it is, so one rank adds nothing).
* The partial sums against binary64 sums of the members; the rank-order
  reduction against the same float64 arithmetic written out in numpy.
* Two ranks as two processes that share this GPU over gloo (their kernels
  never wait on each other: every exchange goes through host memory): the
  sharded iteration against the single-GPU call (counts exact, centroids
  within the centroid tolerance) and the oracle, and the sharded seeding
  against the oracle's indices."""
import os
import socket
import sys

import numpy as np
import pytest

import oracle
import synth
from parity import check_assign, check_centroids

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def dev_tensor(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy()


class OneRank:
    """The exchange of a single rank: every collective returns its input."""
    rank, world = 0, 1

    @staticmethod
    def all_gather(t):
        return t.contiguous().view((1,) + tuple(t.shape)).clone()

    @staticmethod
    def all_to_all_rows(t, send_rows, recv_rows):
        assert list(send_rows) == [recv_rows] == [t.shape[0]]
        return t.contiguous().clone()


@pytest.mark.parametrize("shape", [(5000, 300, 132), (20000, 700, 256), (4096, 256, 512), (40000, 33000, 8)],
                         ids=lambda s: "x".join(map(str, s)))
def test_one_rank_partial_then_reduce_is_the_lloyd_iteration(gpu_lib, shape):
    from distance_argmin_gb300 import sharded
    n, k, d = shape
    X, C0, _ = synth.workload_inputs(synth.Workload("t", n, k, d, k, 1, n + 1, k + 2, ""))
    Xd, Cd = dev_tensor(X), dev_tensor(C0)
    ref = [host(t) for t in gpu_lib.kmeans_lloyd_iter(Xd, Cd)]
    C_new, counts, labels, best, inertia = sharded.lloyd_iter_sharded(Xd, Cd, OneRank())
    assert host(C_new).tobytes() == ref[0].tobytes()
    np.testing.assert_array_equal(host(labels), ref[1])
    assert host(best).tobytes() == ref[2].tobytes()
    assert float(inertia.item()) == float(ref[3][0])
    np.testing.assert_array_equal(host(counts), ref[4])
    # on a stream of its own (the library's kernels and the collectives all
    # run on it), the same bits
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    C2, counts2, _, _, inertia2 = sharded.lloyd_iter_sharded(Xd, Cd, OneRank(), stream=side)
    side.synchronize()
    assert host(C2).tobytes() == ref[0].tobytes() and float(inertia2.item()) == float(ref[3][0])


@pytest.mark.parametrize("shape", [(3000, 50, 64), (2000, 513, 132), (300, 700, 36), (100000, 20, 12),
                                   (40000, 33000, 8)], ids=lambda s: "x".join(map(str, s)))
def test_update_partial_sums_and_counts(gpu_lib, shape):
    # k may exceed the shard's samples (300 x 700); every cluster with no
    # member here gets a zero row
    n, k, d = shape
    X = synth.gaussian((n, d), seed=n + 3, scale=1.5)
    labels = np.random.default_rng(n).integers(0, k, size=n).astype(np.int64)
    labels[labels == 1] = 0
    sums, counts = gpu_lib.kmeans_update_partial(dev_tensor(X), dev_tensor(labels), k)
    want = np.zeros((k, d), np.float64)
    np.add.at(want, labels, X.astype(np.float64))
    cnt = np.bincount(labels, minlength=k)
    np.testing.assert_array_equal(host(counts), cnt)
    got = host(sums).astype(np.float64)
    assert not got[cnt == 0].any()
    # compensated float32 sums: a few units in the last place of the row's
    # largest partial magnitude
    mag = np.zeros((k, d), np.float64)
    np.add.at(mag, labels, np.abs(X.astype(np.float64)))
    assert (np.abs(got - want) <= 4 * 2.0 ** -24 * mag.max(axis=1, keepdims=True) + 1e-30).all()


def test_reduce_partials_is_the_rank_order_float64_sum(gpu_lib):
    world, rows, d = 3, 257, 36
    rng = np.random.default_rng(5)
    parts = rng.standard_normal((world, rows, d)).astype(np.float32) * 100
    pc = rng.integers(0, 5, size=(world, rows)).astype(np.int32)
    pc[:, 7] = 0  # an empty cluster keeps its old row
    C_old = rng.standard_normal((rows, d)).astype(np.float32)
    pin = rng.random(world) * 1e6
    C_new, counts, inertia = gpu_lib.kmeans_reduce_partials(dev_tensor(parts), dev_tensor(pc), dev_tensor(C_old),
                                                            part_inertia=dev_tensor(pin))
    acc = parts[0].astype(np.float64)
    for r in range(1, world):
        acc = acc + parts[r].astype(np.float64)
    cnt = pc.astype(np.int64).sum(axis=0)
    want = np.where(cnt[:, None] > 0, acc / np.maximum(cnt, 1)[:, None], C_old.astype(np.float64)).astype(np.float32)
    want[cnt == 0] = C_old[cnt == 0]
    assert host(C_new).tobytes() == want.tobytes()
    np.testing.assert_array_equal(host(counts), cnt)
    assert float(inertia.item()) == (pin[0] + pin[1]) + pin[2]
    # odd d: the scalar path
    C_new2, _, _ = gpu_lib.kmeans_reduce_partials(dev_tensor(parts[:, :, :35].copy()), dev_tensor(pc),
                                                  dev_tensor(C_old[:, :35].copy()))
    assert host(C_new2).tobytes() == np.ascontiguousarray(want[:, :35]).tobytes()


@pytest.mark.parametrize("case", [(3000, 64, 40, 0, 42), (1200, 4100, 6, 3, 12), (900, 1027, 8, 2, 13)],
                         ids=lambda c: "n%d_d%d_k%d_T%d_s%d" % c)
def test_one_rank_seeding_steps_are_kmeanspp_init(gpu_lib, case):
    from distance_argmin_gb300 import sharded
    n, d, k, T, seed = case
    X, _, _ = synth.planted_blobs(n, d, max(1, k // 2), seed=n + d)
    Xd = dev_tensor(X)
    ref_idx, ref_cen = gpu_lib.kmeanspp_init(Xd, k, seed, n_trials=T)
    idx, cen = sharded.kmeanspp_init_sharded(Xd, k, seed, OneRank(), n_trials=T)
    np.testing.assert_array_equal(host(idx), host(ref_idx))
    assert host(cen).tobytes() == host(ref_cen).tobytes()


def test_one_rank_sharded_fit_is_kmeans_fit(gpu_lib):
    # the same iterations, so the same bits, history and stopping point
    from distance_argmin_gb300 import sharded
    X, C0, _ = synth.workload_inputs(synth.Workload("t", 6000, 40, 36, 40, 1, 81, 82, ""))
    Xd = dev_tensor(X)
    C_ref = dev_tensor(C0)
    C_ref, lab_ref, best_ref, cnt_ref, hist_ref, it_ref = gpu_lib.kmeans_fit(Xd, C=C_ref, init="given", max_iter=30,
                                                                             tol=0.0)
    C, labels, best, counts, hist, n_iter = sharded.fit_sharded(Xd, dev_tensor(C0), OneRank(), max_iter=30, tol=0.0)
    assert n_iter == it_ref and n_iter > 2
    np.testing.assert_array_equal(hist, hist_ref)
    assert host(C).tobytes() == host(C_ref).tobytes()
    np.testing.assert_array_equal(host(labels), host(lab_ref))
    np.testing.assert_array_equal(host(counts), host(cnt_ref))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, case, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import synth as sy
    import distance_argmin_gb300 as km
    from distance_argmin_gb300 import sharded
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        km.load()
        ex = sharded.Exchange()
        n, k, d, splits, kpp = case
        X, C0, _ = sy.workload_inputs(sy.Workload("t", n, k, d, k, 1, 71, 72, ""))
        b = np.cumsum([0] + list(splits))
        Xl = torch.from_numpy(np.ascontiguousarray(X[b[rank]:b[rank + 1]])).cuda()
        C_new, counts, labels, best, inertia = sharded.lloyd_iter_sharded(Xl, torch.from_numpy(C0).cuda(), ex)
        kk, T, seed = kpp
        idx, cen = sharded.kmeanspp_init_sharded(Xl, kk, seed, ex, n_trials=T)
        torch.cuda.synchronize()
        q.put((rank, host(C_new), host(counts), host(labels), host(best), float(inertia.item()), host(idx),
               host(cen)))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [
    (6000, 300, 132, (3000, 3000), (30, 4, 7)),
    (1000, 700, 64, (400, 600), (20, 3, 9)),   # more centroids than either shard has samples
    (20000, 1024, 256, (9000, 11000), (64, 0, 11)),
    (3000, 1, 64, (1000, 2000), (1, 2, 3)),   # one centroid: rank 1 reduces no row
], ids=["k300", "k700_more_than_a_shard", "k1024", "k1"])
def test_two_ranks_sharing_this_gpu(gpu_lib, case):
    import torch.multiprocessing as mp
    n, k, d, splits, (kk, T, seed) = case
    world = len(splits)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, case, q)) for r in range(world)]
    for p in procs:
        p.start()
    try:
        got = dict((res[0], res[1:]) for res in (q.get(timeout=600) for _ in procs))
    finally:
        for p in procs:
            p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    X, C0, _ = synth.workload_inputs(synth.Workload("t", n, k, d, k, 1, 71, 72, ""))
    ref = [host(t) for t in gpu_lib.kmeans_lloyd_iter(dev_tensor(X), dev_tensor(C0))]
    b = np.cumsum([0] + list(splits))
    labels = np.concatenate([got[r][2] for r in range(world)])
    best = np.concatenate([got[r][3] for r in range(world)])
    # each shard's assignment is a tensor-core pass of its own (its tiles may
    # split along K differently from the single call's): checked against the
    # oracle with the usual rules, and against the single call where the
    # labels agree
    o_l, o_b, o_s, _ = oracle.assign(X, C0)
    check_assign(X, C0, labels, best, o_l, o_b, o_s, what="sharded")
    scale = (X.astype(np.float64) ** 2).sum(1) + (C0.astype(np.float64) ** 2).sum(1)[o_l]
    same = np.array_equal(labels, ref[1])
    o_C, o_cnt = oracle.update(X, labels, C0)
    T = T or oracle.n_trials_for(kk)
    o_idx, _, _ = oracle.kmeanspp(X, kk, seed, n_trials=T)
    for r in range(world):
        C_new, counts, _, _, inertia, idx, cen = got[r]
        np.testing.assert_array_equal(counts, o_cnt)
        check_centroids(C_new, o_C, what=f"rank {r} vs oracle")
        if same:
            np.testing.assert_array_equal(counts, ref[4])
            check_centroids(C_new, ref[0], what=f"rank {r} vs single GPU")
        assert abs(inertia - float(ref[3][0])) <= 1e-4 * scale.sum()
        np.testing.assert_array_equal(idx, o_idx)
        assert cen.tobytes() == np.ascontiguousarray(X[o_idx]).tobytes()
        assert C_new.tobytes() == got[0][0].tobytes()

"""The exchange logic of the sample-sharded path on CPU ranks (gloo, world
size 2 and 3), with no GPU: ``distance_argmin_gb300.sharded`` drives a
stand-in for the library's shard entry points written here in numpy from the
header's definitions (binary64 sums, so the stand-in agrees with the oracle).
What is under test is the host side: the row offsets, the all-to-all of
centroid-row slices, the rank-order gathers, the order of the steps and the
exchange blocks.  The sharded results must equal the oracle's on all the
samples: the Lloyd iteration's counts exactly and its centroids within the
centroid tolerance, the k-means++ indices exactly."""
import math
import os
import socket
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class FakeOps:
    """numpy stand-in for the shard entry points (CPU torch tensors)."""
    OP_LLOYD_PARTIAL = 10
    OP_KMEANSPP_SHARD = 9

    def __init__(self):
        import oracle
        self.oracle = oracle

    @staticmethod
    def workspace(op, n, k, d, dev):
        return {"op": op}

    # ---- Lloyd
    def kmeans_lloyd_iter_partial(self, X, C, ws=None, stream=None):
        import torch
        Xn, Cn = X.numpy(), C.numpy()
        lab, best, _, inertia = self.oracle.assign(Xn, Cn)
        k, d = Cn.shape
        sums = np.zeros((k, d), np.float64)
        np.add.at(sums, lab, Xn.astype(np.float64))
        counts = np.bincount(lab, minlength=k).astype(np.int32)
        return (torch.from_numpy(sums.astype(np.float32)), torch.from_numpy(counts), torch.from_numpy(lab),
                torch.from_numpy(best.astype(np.float32)), torch.tensor([inertia], dtype=torch.float64))

    @staticmethod
    def kmeans_reduce_partials(parts, part_counts, C_old, C_new, counts, part_inertia, inertia, stream=None):
        P, PC = parts.numpy().astype(np.float64), part_counts.numpy().astype(np.int64)
        cnt = PC.sum(axis=0)
        acc = P[0].copy()
        for r in range(1, P.shape[0]):
            acc += P[r]
        out = np.where(cnt[:, None] > 0, acc / np.maximum(cnt, 1)[:, None], C_old.numpy().astype(np.float64))
        C_new.copy_(__import__("torch").from_numpy(out.astype(np.float32)))
        counts.copy_(__import__("torch").from_numpy(cnt.astype(np.int32)))
        pi = part_inertia.numpy()
        tot = pi[0]
        for r in range(1, len(pi)):
            tot += pi[r]
        inertia[0] = tot

    # ---- k-means++ (exchange block: T int64 indices, then T rows of d float32)
    @staticmethod
    def kmeanspp_shard_exchange_bytes(T, d):
        return (8 * T + 15) // 16 * 16 + ((4 * T * d + 15) // 16) * 16

    @staticmethod
    def _block(buf, T, d):
        a = buf.numpy()
        ib = (8 * T + 15) // 16 * 16
        return a[:8 * T].view(np.int64), a[ib:ib + 4 * T * d].view(np.float32).reshape(T, d)

    def kmeanspp_shard_first(self, X, row_offset, n_global, T, seed, send, ws, stream=None):
        idx, rows = self._block(send, T, X.shape[1])
        g = min(int(math.floor(self.oracle.uniform(seed, 0) * n_global)), n_global - 1)
        idx[:] = -1
        if row_offset <= g < row_offset + X.shape[0]:
            idx[0] = g
            rows[0] = X.numpy()[g - row_offset]
        ws["T"] = T

    def kmeanspp_shard_pick(self, X, row_offset, T, seed, c, totals, rank, send, ws, stream=None):
        idx, rows = self._block(send, T, X.shape[1])
        tot = totals.numpy()
        S = tot[0]
        for r in range(1, len(tot)):
            S += tot[r]
        for t in range(T):
            target = self.oracle.uniform(seed, 1 + (c - 1) * T + t) * S
            owner, base, run, clip = len(tot) - 1, 0.0, 0.0, True
            for r in range(len(tot)):
                nxt = tot[0] if r == 0 else run + tot[r]
                if nxt > target:
                    owner, base, clip = r, run, False
                    break
                run = nxt
            if owner != rank:
                idx[t] = -1
                continue
            pick = X.shape[0] - 1
            if not clip:
                acc = base
                for i, v in enumerate(ws["D2"]):
                    acc += v
                    if acc > target:
                        pick = i
                        break
            idx[t] = row_offset + pick
            rows[t] = X.numpy()[pick]

    def kmeanspp_shard_dist(self, X, T, first, recv, world, pot, ws, stream=None):
        d = X.shape[1]
        Tn = 1 if first else T
        blocks = [self._block(recv[r], T, d) for r in range(world)]
        cg, cr = [], []
        for t in range(Tn):
            owner = next(r for r in range(world) if blocks[r][0][t] >= 0)
            cg.append(int(blocks[owner][0][t]))
            cr.append(blocks[owner][1][t].copy())
        Xn = X.numpy().astype(np.float64)
        dist = np.stack([((Xn - c.astype(np.float64)) ** 2).sum(1) for c in cr])
        ws.update(cglob=cg, crow=cr, dist=dist)
        if not first:
            for t in range(T):
                pot[t] = float(np.minimum(ws["D2"], dist[t]).sum())

    @staticmethod
    def kmeanspp_shard_commit(n, d, T, first, pots, world, c, indices, centers, total, ws, stream=None):
        best = 0
        if not first:
            p = pots.numpy().reshape(world, T)
            tot = p[0].copy()
            for r in range(1, world):
                tot += p[r]
            best = int(np.argmin(tot))  # first minimum: the lowest trial on ties
        indices[c] = ws["cglob"][best]
        centers[c] = __import__("torch").from_numpy(ws["crow"][best])
        ws["D2"] = ws["dist"][best].copy() if first else np.minimum(ws["D2"], ws["dist"][best])
        if total is not None:
            total[0] = float(ws["D2"].sum())


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, case, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import synth
    from distance_argmin_gb300 import sharded
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ex = sharded.Exchange()
        ops = FakeOps()
        n, k, d, splits = case
        X, C0, _ = synth.workload_inputs(synth.Workload("t", n, k, d, k, 1, 61, 62, ""))
        b = np.cumsum([0] + list(splits))
        Xl = torch.from_numpy(np.ascontiguousarray(X[b[rank]:b[rank + 1]]))
        C_new, counts, labels, best, inertia = sharded.lloyd_iter_sharded(Xl, torch.from_numpy(C0), ex, ops=ops)
        idx, cen = sharded.kmeanspp_init_sharded(Xl, min(k, 12), 5, ex, n_trials=3, ops=ops)
        q.put((rank, C_new.numpy().copy(), counts.numpy().copy(), labels.numpy().copy(), float(inertia[0]),
               idx.numpy().copy(), cen.numpy().copy()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("case", [
    (600, 7, 12, (300, 300)),      # k not a multiple of the world size
    (500, 5, 6, (120, 200, 180)),  # three ranks, unequal shards; the last rank reduces one row
    (240, 3, 4, (100, 140)),       # fewer centroids than ranks x 2
    (90, 40, 5, (30, 30, 30)),     # more centroids than any shard has samples
    (60, 2, 3, (20, 25, 15)),      # fewer centroids than ranks: the last rank reduces no row
], ids=["k7_w2", "k5_w3", "k3_w2", "k40_w3", "k2_w3"])
def test_sharded_iteration_and_seeding_match_the_oracle(case):
    import torch.multiprocessing as mp
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    n, k, d, splits = case
    world = len(splits)
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, case, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict((res[0], res[1:]) for res in (q.get(timeout=300) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    X, C0, _ = synth.workload_inputs(synth.Workload("t", n, k, d, k, 1, 61, 62, ""))
    o_C, o_lab, _, _, o_inertia, o_cnt = oracle.lloyd_iter(X, C0)
    o_idx, _, _ = oracle.kmeanspp(X, min(k, 12), 5, n_trials=3)
    b = np.cumsum([0] + list(splits))
    for r in range(world):
        C_new, counts, labels, inertia, idx, cen = got[r]
        np.testing.assert_array_equal(counts, o_cnt)
        scale = np.abs(o_C).max(axis=1, keepdims=True)
        assert (np.abs(C_new - o_C) <= 1e-5 * scale).all()
        np.testing.assert_array_equal(labels, o_lab[b[r]:b[r + 1]])
        assert abs(inertia - o_inertia) <= 1e-12 * o_inertia
        np.testing.assert_array_equal(idx, o_idx)
        assert cen.tobytes() == np.ascontiguousarray(X[o_idx]).tobytes()
        # every rank holds the same global results
        assert C_new.tobytes() == got[0][0].tobytes() and idx.tobytes() == got[0][4].tobytes()


def test_slices_cover_every_centroid_row_once():
    sys.path.insert(0, ROOT)
    from distance_argmin_gb300.sharded import slice_rows
    for k in range(1, 40):
        for world in range(1, 9):
            m, rows = slice_rows(k, world)
            assert sum(rows) == k and all(0 <= r <= m for r in rows)
            # only the last slices are short: the concatenated slices' first k rows are rows 0..k-1
            full = [q * m + i for q in range(world) for i in range(m)]
            kept = [q * m + i for q in range(world) for i in range(rows[q])]
            assert kept == full[:k]


def _fit_rank_main(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import synth
    from distance_argmin_gb300 import sharded
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        X, C0, _ = synth.workload_inputs(synth.Workload("t", 900, 9, 6, 9, 1, 63, 64, ""))
        b = [0, 250, 600, 900]
        Xl = torch.from_numpy(np.ascontiguousarray(X[b[rank]:b[rank + 1]]))
        C, labels, best, counts, hist, n_iter = sharded.fit_sharded(Xl, torch.from_numpy(C0), sharded.Exchange(),
                                                                    max_iter=50, tol=0.0, ops=FakeOps())
        q.put((rank, C.numpy().copy(), labels.numpy().copy(), hist, n_iter))
    finally:
        dist.destroy_process_group()


def test_sharded_fit_stops_where_the_oracle_fit_stops():
    import torch.multiprocessing as mp
    sys.path.insert(0, ROOT)
    import oracle
    import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_fit_rank_main, args=(r, 3, port, q)) for r in range(3)]
    for p in procs:
        p.start()
    got = dict((res[0], res[1:]) for res in (q.get(timeout=300) for _ in procs))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    X, C0, _ = synth.workload_inputs(synth.Workload("t", 900, 9, 6, 9, 1, 63, 64, ""))
    o_C, o_lab, _, o_hist, o_iter = oracle.fit(X, C0, 50, 0.0)
    b = [0, 250, 600, 900]
    for r in range(3):
        C, labels, hist, n_iter = got[r]
        assert n_iter == o_iter and n_iter > 2
        # the partial sums are float32, so later centroids (and inertias) carry ~1e-8 relative rounding
        np.testing.assert_allclose(hist, o_hist, rtol=1e-6)
        np.testing.assert_array_equal(labels, o_lab[b[r]:b[r + 1]])
        assert (np.abs(C - o_C) <= 1e-5 * np.abs(o_C).max(axis=1, keepdims=True)).all()


class FailingOps(FakeOps):
    """The stand-in, except that this rank's shard step raises (a rank that
    fails before the exchange)."""

    def kmeans_lloyd_iter_partial(self, X, C, ws=None, stream=None):
        raise RuntimeError("planted failure of this rank's shard step")


def _failing_rank_main(rank, world, port, q):
    import datetime
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import synth
    from distance_argmin_gb300 import sharded
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world, timeout=datetime.timedelta(seconds=10))
    X, C0, _ = synth.workload_inputs(synth.Workload("t", 400, 5, 8, 5, 1, 65, 66, ""))
    Xl = torch.from_numpy(np.ascontiguousarray(X[rank * 200:(rank + 1) * 200]))
    ops = FailingOps() if rank == 1 else FakeOps()
    try:
        sharded.lloyd_iter_sharded(Xl, torch.from_numpy(C0), sharded.Exchange(), ops=ops)
        q.put((rank, "finished"))
    except Exception as e:  # the failing rank's own error, or the survivor's collective error
        q.put((rank, type(e).__name__ + ": " + str(e)[:200]))
    # no destroy_process_group: the peer is gone


def test_a_failing_rank_ends_the_others_collective_with_an_error():
    # Rank 1 raises before its first collective and leaves; rank 0's
    # all-to-all must end with an error (the peer closed, or the process
    # group's 10 s timeout), not hang.
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_failing_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        if p.is_alive():
            p.kill()
    assert "planted failure" in got[1]
    assert got[0] != "finished", got[0]

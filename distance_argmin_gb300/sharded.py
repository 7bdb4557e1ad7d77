"""Samples split by rows across processes, one GPU each.

The update of a Lloyd iteration needs every member of a cluster ("Three
shapes that fit an eager Gram assignment", section "Full Lloyd step": each
centroid is the mean of its members), so a rank that holds only some samples
cannot finish it alone.  This module drives the library's shard entry points
and the collectives between them:

* ``lloyd_iter_sharded``: each rank assigns its rows and forms its clusters'
  sums and counts (``kmeans_lloyd_iter_partial``); an all-to-all gives rank q
  every rank's sums of centroid rows [q m, q m + m) (m = ceil(k / world));
  ``kmeans_reduce_partials`` adds them in rank order and divides (empty
  clusters keep their old row); an all-gather rebuilds C on every rank.
* ``kmeanspp_init_sharded``: greedy k-means++ ("004 — tile sizes, a Cython
  Lloyd step, and k-means++", section "k-means++") over the concatenated
  shards, three all-gathers per center: the candidate blocks, the trials'
  potentials and the shards' totals of D^2.

The collectives only move bytes; every sum across ranks is taken by the
library in rank order, so results do not depend on how a collective is
scheduled.  This module holds no arithmetic of the method: it sizes buffers,
calls the C ABI through the binding and calls torch.distributed.

``ops`` (default: the binding) is the object whose functions are called; the
host-side tests pass a stand-in with the same functions to run the exchange
logic on CPU ranks.  ``stream`` (optional, every entry): the CUDA stream the
whole sequence runs on; it is made the current stream for the duration, so the
collectives and the kernels between them stay in order.
"""
from __future__ import annotations

import contextlib
import functools
import math


def _torch():
    import torch
    return torch


def _default_ops():
    import distance_argmin_gb300 as km
    return km


def _on_stream(fn):
    """Run ``fn`` with its ``stream`` argument as the current CUDA stream, so
    that the library's kernels and the torch.distributed collectives between
    them are ordered on one stream; the library calls inside then take the
    current stream."""
    @functools.wraps(fn)
    def wrapped(*args, stream=None, **kwargs):
        ctx = contextlib.nullcontext()
        if stream is not None:
            torch = _torch()
            ctx = torch.cuda.stream(stream if isinstance(stream, torch.cuda.Stream)
                                    else torch.cuda.ExternalStream(int(stream)))
        with ctx:
            return fn(*args, **kwargs)
    return wrapped


class Exchange:
    """The collectives of the sharded path on a torch.distributed group.

    NCCL moves device tensors directly; any other backend (gloo) gets host
    copies, which synchronise the stream."""

    def __init__(self, group=None):
        import torch.distributed as dist
        self.dist = dist
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.via_host = dist.get_backend(group) != "nccl"

    def all_gather(self, t):
        """(world, *t.shape): every rank's ``t`` in rank order."""
        torch = _torch()
        t = t.contiguous()
        shape = (self.world,) + tuple(t.shape)
        if self.via_host and t.device.type != "cpu":
            out = torch.empty(self.world * t.numel(), dtype=t.dtype)
            self.dist.all_gather_into_tensor(out, t.cpu().view(-1), group=self.group)
            return out.view(shape).to(t.device)
        out = torch.empty(self.world * t.numel(), dtype=t.dtype, device=t.device)
        self.dist.all_gather_into_tensor(out, t.view(-1), group=self.group)
        return out.view(shape)

    def all_to_all_rows(self, t, send_rows, recv_rows):
        """Rows [sum(send_rows[:q]), + send_rows[q]) of ``t`` go to rank q;
        returns the (world * recv_rows, *t.shape[1:]) rows received, rank
        order."""
        torch = _torch()
        t = t.contiguous()
        tail = tuple(t.shape[1:])
        dev = t.device
        src = t.cpu() if (self.via_host and dev.type != "cpu") else t
        out = torch.empty((self.world * recv_rows,) + tail, dtype=t.dtype, device=src.device)
        self.dist.all_to_all_single(out, src, output_split_sizes=[recv_rows] * self.world,
                                    input_split_sizes=list(send_rows), group=self.group)
        return out.to(dev) if out.device != dev else out


def slice_rows(k: int, world: int):
    """Centroid rows each rank reduces: m = ceil(k / world) per rank, the
    last ranks fewer (possibly none)."""
    m = (k + world - 1) // world
    return m, [max(0, min(m, k - q * m)) for q in range(world)]


@_on_stream
def lloyd_iter_sharded(X, C_old, ex: Exchange, ws=None, ops=None):
    """One Lloyd iteration over samples split by rows across the ranks of
    ``ex``.  X: this rank's (n_local, d) rows; C_old: the (k, d) centroids,
    the same on every rank.  Returns ``(C_new (k, d), counts (k,), labels,
    best_dist, inertia)``: C_new, counts and the inertia (one float64, the
    ranks' inertias summed in rank order) are global and the same on every
    rank; labels and best_dist are this rank's rows."""
    torch = _torch()
    km = ops or _default_ops()
    n, d = X.shape
    k = C_old.shape[0]
    dev = X.device
    world, rank = ex.world, ex.rank
    if ws is None:
        ws = km.workspace(km.OP_LLOYD_PARTIAL, n, k, d, dev)
    sums, counts, labels, best, inertia = km.kmeans_lloyd_iter_partial(X, C_old, ws=ws)
    m, rows = slice_rows(k, world)
    mine = rows[rank]
    # every rank's sums and counts of this rank's centroid rows, rank-major
    parts = ex.all_to_all_rows(sums, rows, mine).view(world, mine, d)
    part_counts = ex.all_to_all_rows(counts, rows, mine).view(world, mine)
    part_inertia = ex.all_gather(inertia).view(world)
    lo = rank * m
    C_slice = torch.zeros((m, d), dtype=torch.float32, device=dev)
    cnt_slice = torch.zeros(m, dtype=torch.int32, device=dev)
    total = torch.empty(1, dtype=torch.float64, device=dev)
    km.kmeans_reduce_partials(parts, part_counts, C_old[lo:lo + mine], C_new=C_slice[:mine],
                              counts=cnt_slice[:mine], part_inertia=part_inertia, inertia=total)
    # rank q's slice holds rows [q m, q m + rows[q]); only the last slices
    # are short, so the gathered slices' first k rows are C_new in order
    C_new = ex.all_gather(C_slice).view(world * m, d)[:k]
    counts_all = ex.all_gather(cnt_slice).view(world * m)[:k]
    return C_new, counts_all, labels, best, total


def shard_offsets(n_local: int, ex: Exchange, device):
    """(row_offset, n_global) of this rank's rows among the shards in rank
    order."""
    torch = _torch()
    sizes = ex.all_gather(torch.tensor([int(n_local)], dtype=torch.int64, device=device)).view(-1).cpu().tolist()
    return int(sum(sizes[:ex.rank])), int(sum(sizes))


@_on_stream
def kmeanspp_init_sharded(X, k: int, seed: int, ex: Exchange, n_trials: int = 0, ws=None, ops=None):
    """Greedy k-means++ seeding of k centers over the samples split by rows
    across the ranks of ``ex`` (rank order = sample order).  Returns
    ``(indices (k,) global sample indices, centers (k, d))``, the same on
    every rank; with one rank they are kmeanspp_init's."""
    torch = _torch()
    km = ops or _default_ops()
    n, d = X.shape
    dev = X.device
    world, rank = ex.world, ex.rank
    T = int(n_trials) if n_trials and n_trials > 0 else 2 + int(math.floor(math.log(k)))
    row_offset, n_global = shard_offsets(n, ex, dev)
    if not 1 <= k <= n_global:
        raise ValueError(f"k = {k} must lie in [1, {n_global}]")
    if ws is None:
        ws = km.workspace(km.OP_KMEANSPP_SHARD, n, k, d, dev)
    send = torch.empty(km.kmeanspp_shard_exchange_bytes(T, d), dtype=torch.uint8, device=dev)
    pot = torch.empty(T, dtype=torch.float64, device=dev)
    total = torch.empty(1, dtype=torch.float64, device=dev)
    indices = torch.empty(k, dtype=torch.int64, device=dev)
    centers = torch.empty((k, d), dtype=torch.float32, device=dev)

    km.kmeanspp_shard_first(X, row_offset, n_global, T, seed, send, ws)
    recv = ex.all_gather(send)
    km.kmeanspp_shard_dist(X, T, True, recv, world, None, ws)
    km.kmeanspp_shard_commit(n, d, T, True, None, world, 0, indices, centers, total, ws)
    for c in range(1, k):
        totals = ex.all_gather(total).view(world)
        km.kmeanspp_shard_pick(X, row_offset, T, seed, c, totals, rank, send, ws)
        recv = ex.all_gather(send)
        km.kmeanspp_shard_dist(X, T, False, recv, world, pot, ws)
        pots = ex.all_gather(pot).view(world * T)
        last = c == k - 1
        km.kmeanspp_shard_commit(n, d, T, False, pots, world, c, indices, centers, None if last else total, ws)
    return indices, centers


@_on_stream
def fit_sharded(X, C0, ex: Exchange, max_iter: int = 300, tol: float = 1e-4, ws=None, ops=None):
    """Lloyd iterations over samples split by rows across the ranks of
    ``ex``, from the centroids C0 (the same on every rank), with the stopping
    rule of kmeans_fit: stop after iteration t when inertia_t >=
    (1 - tol) * inertia_{t-1}, or after max_iter iterations.  Every rank reads
    the same global inertia, so every rank stops at the same iteration.
    Returns ``(C (k, d), labels, best_dist, counts, inertia_history,
    n_iter)``: C, counts and the history global, labels and best_dist this
    rank's rows of the last iteration."""
    import numpy as np
    km = ops or _default_ops()
    n, d = X.shape
    k = C0.shape[0]
    if ws is None:
        ws = km.workspace(km.OP_LLOYD_PARTIAL, n, k, d, X.device)
    C = C0
    hist = []
    labels = best = counts = None
    for it in range(int(max_iter)):
        C, counts, labels, best, inertia = lloyd_iter_sharded(X, C, ex, ws=ws, ops=ops)
        hist.append(float(inertia.reshape(-1)[0].item()))
        if it > 0 and hist[-1] >= hist[-2] * (1.0 - tol):
            break
    return C, labels, best, counts, np.array(hist), len(hist)

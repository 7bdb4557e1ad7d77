"""Python binding of the GB300 k-means library (``include/kmeans_gb300.h``).

Argument marshalling only: every function checks tensor types, shapes and
devices, passes raw device pointers, sizes and the current CUDA stream to the
C ABI of ``libkmeans_gb300.so``, and raises ``KMeansError`` on a non-zero
status.  All arithmetic runs in the library's CUDA kernels.  PyTorch supplies
device memory (outputs and the workspace when the caller passes none) and
streams.  There is no CPU path: without the built library every call fails.

Names follow the C ABI: ``kmeans_assign``, ``kmeans_assign_ffma``,
``kmeans_update``, ``kmeans_lloyd_iter``, ``kmeanspp_init``,
``kmeans_workspace_bytes``, ``kmeans_device_status``, ``kmeans_status_string``,
and the shard entry points (``kmeans_lloyd_iter_partial``,
``kmeans_reduce_partials``, ``kmeanspp_shard_*``) that ``sharded.py`` drives
across processes.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkmeans_gb300.so")

KMEANS_OK = 0
KMEANS_ERR_INVALID_ARG = 1
KMEANS_ERR_UNSUPPORTED = 2
KMEANS_ERR_WORKSPACE = 3
KMEANS_ERR_CUDA = 4
KMEANS_ERR_DEVICE_TIMEOUT = 5
KMEANS_ERR_DEVICE_LABEL = 6
KMEANS_ERR_SCRATCH_LIMIT = 7
KMEANS_ERR_DEVICE_EXCHANGE = 8
NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

OP_ASSIGN = 0
OP_ASSIGN_FFMA = 1
OP_UPDATE = 2
OP_LLOYD = 3
OP_KMEANSPP = 4
OP_FIT = 5
OP_ASSIGN_3XTF32 = 6
OP_LLOYD_FUSED = 7
OP_RELOCATE = 8
OP_KMEANSPP_SHARD = 9
OP_LLOYD_PARTIAL = 10
OP_UPDATE_PARTIAL = 11

INIT_GIVEN = 0
INIT_KMEANSPP = 1
FIT_RELOCATE_EMPTY = 0x100

KERNEL_ASSIGN_TC = 0
KERNEL_UPDATE_MEAN = 1
KERNEL_KMEANSPP_DIST = 2
TRACE_MAX_CAPACITY = 65536
HOST_MAX_SLICES = 64
HOST_OVERLAP_PREVIOUS = 1
HOST_READBACK_ON_COPY_STREAM = 2
# Features per slice of the k-means++ distance pass: each pass writes one
# float2 partial sum per (slice, trial, sample), ceil(d / 4096) slices.
KPP_SLICE_FEATURES = 4096

# Every symbol the header declares (the ABI test checks the library exports them).
EXPORTS = (
    "kmeans_workspace_bytes", "kmeans_assign", "kmeans_assign_ffma", "kmeans_update",
    "kmeans_lloyd_iter", "kmeanspp_init", "kmeans_device_status", "kmeans_status_string",
    "kmeans_build_info", "kmeans_assign_noalloc", "kmeans_trace_start", "kmeans_trace_read",
    "kmeans_trace_stop", "kmeans_lloyd_iter_host", "kmeans_fit", "kmeans_assign_3xtf32",
    "kmeans_lloyd_iter_fused", "kmeans_relocate_empty", "kmeans_update_partial", "kmeans_lloyd_iter_partial",
    "kmeans_reduce_partials", "kmeanspp_shard_exchange_bytes", "kmeanspp_shard_first", "kmeanspp_shard_pick",
    "kmeanspp_shard_dist", "kmeanspp_shard_commit", "kmeanspp_rows_read",
)

_lock = threading.Lock()
_lib = None


class KMeansError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {kmeans_status_string(status)} (status {status})")


def load(path: str | None = None):
    """Load the library once; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"{p} is missing: build it with `python -m distance_argmin_gb300.build`"
                               " (the library has no CPU fallback)")
        lib = ctypes.CDLL(p)
        P, I64, U64, SZ, INT = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t,
                                ctypes.c_int)
        lib.kmeans_workspace_bytes.argtypes = [INT, I64, I64, I64]
        lib.kmeans_workspace_bytes.restype = SZ
        assign_sig = [P, P, I64, I64, I64, P, P, P, P, SZ, U64, P]
        lib.kmeans_assign.argtypes = assign_sig
        lib.kmeans_assign.restype = INT
        lib.kmeans_assign_3xtf32.argtypes = assign_sig
        lib.kmeans_assign_3xtf32.restype = INT
        lib.kmeans_assign_ffma.argtypes = assign_sig
        lib.kmeans_assign_ffma.restype = INT
        lib.kmeans_assign_noalloc.argtypes = [P, P, I64, I64, I64, P, P, P, U64, P]
        lib.kmeans_assign_noalloc.restype = INT
        lib.kmeans_update.argtypes = [P, P, P, P, P, I64, I64, I64, P, SZ, U64, P]
        lib.kmeans_update.restype = INT
        lib.kmeans_lloyd_iter.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, P, SZ, U64, P]
        lib.kmeans_lloyd_iter_fused.argtypes = lib.kmeans_lloyd_iter.argtypes
        lib.kmeans_lloyd_iter_fused.restype = INT
        lib.kmeans_lloyd_iter.restype = INT
        lib.kmeanspp_init.argtypes = [P, I64, I64, I64, INT, U64, P, P, P, SZ, P]
        lib.kmeanspp_init.restype = INT
        lib.kmeans_device_status.argtypes = [P, P]
        lib.kmeans_device_status.restype = INT
        lib.kmeanspp_rows_read.argtypes = [P, P, ctypes.POINTER(I64)]
        lib.kmeanspp_rows_read.restype = INT
        lib.kmeans_status_string.argtypes = [INT]
        lib.kmeans_status_string.restype = ctypes.c_char_p
        lib.kmeans_build_info.argtypes = []
        lib.kmeans_build_info.restype = ctypes.c_char_p
        lib.kmeans_trace_start.argtypes = [INT]
        lib.kmeans_trace_start.restype = INT
        lib.kmeans_trace_read.argtypes = [INT, P, P, P]
        lib.kmeans_trace_read.restype = INT
        lib.kmeans_lloyd_iter_host.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, I64, I64, I64, INT, INT, P, SZ, P,
                                               P]
        lib.kmeans_lloyd_iter_host.restype = INT
        lib.kmeans_fit.argtypes = [P, P, P, P, P, I64, I64, I64, INT, U64, INT, ctypes.c_double, P, P, P, SZ, P]
        lib.kmeans_fit.restype = INT
        lib.kmeans_relocate_empty.argtypes = [P, P, I64, I64, P, SZ, P]
        lib.kmeans_relocate_empty.restype = INT
        lib.kmeans_trace_stop.argtypes = []
        lib.kmeans_trace_stop.restype = INT
        lib.kmeans_update_partial.argtypes = [P, P, I64, I64, I64, P, P, P, SZ, U64, P]
        lib.kmeans_update_partial.restype = INT
        lib.kmeans_lloyd_iter_partial.argtypes = [P, P, P, P, P, P, P, I64, I64, I64, P, SZ, U64, P]
        lib.kmeans_lloyd_iter_partial.restype = INT
        lib.kmeans_reduce_partials.argtypes = [P, P, P, INT, I64, I64, P, P, P, P, P]
        lib.kmeans_reduce_partials.restype = INT
        lib.kmeanspp_shard_exchange_bytes.argtypes = [INT, I64]
        lib.kmeanspp_shard_exchange_bytes.restype = SZ
        lib.kmeanspp_shard_first.argtypes = [P, I64, I64, I64, I64, INT, U64, P, P, SZ, P]
        lib.kmeanspp_shard_first.restype = INT
        lib.kmeanspp_shard_pick.argtypes = [P, I64, I64, I64, INT, U64, I64, P, INT, INT, P, P, SZ, P]
        lib.kmeanspp_shard_pick.restype = INT
        lib.kmeanspp_shard_dist.argtypes = [P, I64, I64, INT, INT, P, INT, P, P, SZ, P]
        lib.kmeanspp_shard_dist.restype = INT
        lib.kmeanspp_shard_commit.argtypes = [I64, I64, INT, INT, P, INT, I64, P, P, P, P, SZ, P]
        lib.kmeanspp_shard_commit.restype = INT
        _lib = lib
        return lib


def kmeans_status_string(status: int) -> str:
    return load().kmeans_status_string(int(status)).decode()


def kmeans_build_info() -> str:
    return load().kmeans_build_info().decode()


def kmeans_workspace_bytes(op: int, n: int, k: int, d: int) -> int:
    return int(load().kmeans_workspace_bytes(op, n, k, d))


def n_trials_for(k: int) -> int:
    """2 + floor(ln k): the default k-means++ trial count."""
    return 2 + int(math.floor(math.log(k)))


# ----------------------------------------------------------------- helpers
def _torch():
    import torch
    return torch


def _ptr(t) -> ctypes.c_void_p:
    return ctypes.c_void_p(0 if t is None else t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    torch = _torch()
    if stream is None:
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check(t, name, dtype, shape=None, device=None):
    torch = _torch()
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be on a CUDA device (the library has no CPU path)")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def workspace(op: int, n: int, k: int, d: int, device=None):
    """A device workspace big enough for ``op`` on these sizes (uint8 tensor)."""
    torch = _torch()
    nbytes = kmeans_workspace_bytes(op, n, k, d)
    if nbytes == 0:
        raise KMeansError(KMEANS_ERR_INVALID_ARG, "kmeans_workspace_bytes")
    return torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")


def _ws(ws, op, n, k, d, device):
    if ws is None:
        return workspace(op, n, k, d, device)
    _check(ws, "ws", _torch().uint8, device=device)
    return ws


def _raise(status, what):
    if status != KMEANS_OK:
        raise KMeansError(status, what)


# ------------------------------------------------------------- entry points
def _assign(fn_name, op, X, C, labels, best_dist, inertia, ws, seed, stream):
    torch = _torch()
    _check(X, "X", torch.float32)
    n, d = X.shape
    _check(C, "C", torch.float32, device=X.device)
    k = C.shape[0]
    if C.dim() != 2 or C.shape[1] != d:
        raise ValueError("C must be (k, d) with the same d as X")
    if labels is None:
        labels = torch.empty(n, dtype=torch.int64, device=X.device)
    if best_dist is None:
        best_dist = torch.empty(n, dtype=torch.float32, device=X.device)
    if inertia is None:
        inertia = torch.empty(1, dtype=torch.float64, device=X.device)
    _check(labels, "labels", torch.int64, (n,), X.device)
    _check(best_dist, "best_dist", torch.float32, (n,), X.device)
    _check(inertia, "inertia", torch.float64, (1,), X.device)
    ws = _ws(ws, op, n, k, d, X.device)
    st = getattr(load(), fn_name)(_ptr(X), _ptr(C), n, k, d, _ptr(labels), _ptr(best_dist), _ptr(inertia),
                                  _ptr(ws), ws.numel(), seed & (2**64 - 1), _stream_handle(stream))
    _raise(st, fn_name)
    return labels, best_dist, inertia


def kmeans_assign(X, C, labels=None, best_dist=None, inertia=None, ws=None, seed=0, stream=None):
    """Nearest centroid on the tensor cores -> ``(labels, best_dist, inertia)``."""
    return _assign("kmeans_assign", OP_ASSIGN, X, C, labels, best_dist, inertia, ws, seed, stream)


def kmeans_assign_ffma(X, C, labels=None, best_dist=None, inertia=None, ws=None, seed=0, stream=None):
    """The same assignment with float32 FMA on the CUDA cores (comparator)."""
    return _assign("kmeans_assign_ffma", OP_ASSIGN_FFMA, X, C, labels, best_dist, inertia, ws, seed, stream)


def kmeans_assign_3xtf32(X, C, labels=None, best_dist=None, inertia=None, ws=None, seed=0, stream=None):
    """The tensor-core assignment with the 3xTF32 split (comparator of bf16x3)."""
    return _assign("kmeans_assign_3xtf32", OP_ASSIGN_3XTF32, X, C, labels, best_dist, inertia, ws, seed, stream)


def kmeans_assign_noalloc(X, C, labels, best_dist, inertia=None, seed=0, stream=None):
    """``kmeans_assign`` for callers that cannot allocate device memory: the
    library's built-in scratch replaces the workspace, and the caller passes
    the outputs.  Problems needing more than NOALLOC_SCRATCH_BYTES of scratch
    raise KMeansError(KMEANS_ERR_SCRATCH_LIMIT)."""
    torch = _torch()
    _check(X, "X", torch.float32)
    n, d = X.shape
    _check(C, "C", torch.float32, device=X.device)
    k = C.shape[0]
    _check(labels, "labels", torch.int64, (n,), X.device)
    _check(best_dist, "best_dist", torch.float32, (n,), X.device)
    if inertia is not None:
        _check(inertia, "inertia", torch.float64, (1,), X.device)
    st = load().kmeans_assign_noalloc(_ptr(X), _ptr(C), n, k, d, _ptr(labels), _ptr(best_dist), _ptr(inertia),
                                      seed & (2**64 - 1), _stream_handle(stream))
    _raise(st, "kmeans_assign_noalloc")
    return labels, best_dist, inertia


def kmeans_update(X, labels, C_old, C_new=None, counts=None, ws=None, seed=0, stream=None):
    """Mean of members, empty clusters keep ``C_old`` -> ``(C_new, counts)``."""
    torch = _torch()
    _check(X, "X", torch.float32)
    n, d = X.shape
    _check(labels, "labels", torch.int64, (n,), X.device)
    _check(C_old, "C_old", torch.float32, device=X.device)
    k = C_old.shape[0]
    if C_new is None:
        C_new = torch.empty_like(C_old)
    if counts is None:
        counts = torch.empty(k, dtype=torch.int32, device=X.device)
    _check(C_new, "C_new", torch.float32, (k, d), X.device)
    _check(counts, "counts", torch.int32, (k,), X.device)
    ws = _ws(ws, OP_UPDATE, n, k, d, X.device)
    st = load().kmeans_update(_ptr(X), _ptr(labels), _ptr(C_old), _ptr(C_new), _ptr(counts), n, k, d,
                              _ptr(ws), ws.numel(), seed & (2**64 - 1), _stream_handle(stream))
    _raise(st, "kmeans_update")
    return C_new, counts


def _lloyd(fn_name, op, X, C_old, C_new, labels, best_dist, inertia, counts, ws, seed, stream):
    torch = _torch()
    _check(X, "X", torch.float32)
    n, d = X.shape
    _check(C_old, "C_old", torch.float32, device=X.device)
    k = C_old.shape[0]
    if C_new is None:
        C_new = torch.empty_like(C_old)
    if labels is None:
        labels = torch.empty(n, dtype=torch.int64, device=X.device)
    if best_dist is None:
        best_dist = torch.empty(n, dtype=torch.float32, device=X.device)
    if inertia is None:
        inertia = torch.empty(1, dtype=torch.float64, device=X.device)
    if counts is None:
        counts = torch.empty(k, dtype=torch.int32, device=X.device)
    _check(C_new, "C_new", torch.float32, (k, d), X.device)
    _check(labels, "labels", torch.int64, (n,), X.device)
    _check(best_dist, "best_dist", torch.float32, (n,), X.device)
    _check(inertia, "inertia", torch.float64, (1,), X.device)
    _check(counts, "counts", torch.int32, (k,), X.device)
    ws = _ws(ws, op, n, k, d, X.device)
    st = getattr(load(), fn_name)(_ptr(X), _ptr(C_old), _ptr(C_new), _ptr(labels), _ptr(best_dist),
                                  _ptr(inertia), _ptr(counts), n, k, d, _ptr(ws), ws.numel(),
                                  seed & (2**64 - 1), _stream_handle(stream))
    _raise(st, fn_name)
    return C_new, labels, best_dist, inertia, counts


def kmeans_lloyd_iter(X, C_old, C_new=None, labels=None, best_dist=None, inertia=None, counts=None, ws=None,
                      seed=0, stream=None):
    """One Lloyd iteration -> ``(C_new, labels, best_dist, inertia, counts)``."""
    return _lloyd("kmeans_lloyd_iter", OP_LLOYD, X, C_old, C_new, labels, best_dist, inertia, counts, ws, seed,
                  stream)


def kmeans_lloyd_iter_fused(X, C_old, C_new=None, labels=None, best_dist=None, inertia=None, counts=None, ws=None,
                            seed=0, stream=None):
    """One Lloyd iteration with the update fused into the assignment (float
    atomics: C_new is not bitwise reproducible) -> as kmeans_lloyd_iter."""
    return _lloyd("kmeans_lloyd_iter_fused", OP_LLOYD_FUSED, X, C_old, C_new, labels, best_dist, inertia, counts,
                  ws, seed, stream)


def kmeanspp_init(X, k: int, seed: int, n_trials: int = 0, centers=None, indices=None, ws=None, stream=None):
    """Greedy D^2 seeding -> ``(indices, centers)``."""
    torch = _torch()
    _check(X, "X", torch.float32)
    n, d = X.shape
    if indices is None:
        indices = torch.empty(k, dtype=torch.int64, device=X.device)
    if centers is None:
        centers = torch.empty((k, d), dtype=torch.float32, device=X.device)
    _check(indices, "indices", torch.int64, (k,), X.device)
    _check(centers, "centers", torch.float32, (k, d), X.device)
    ws = _ws(ws, OP_KMEANSPP, n, k, d, X.device)
    st = load().kmeanspp_init(_ptr(X), n, d, k, int(n_trials), seed & (2**64 - 1), _ptr(centers), _ptr(indices),
                              _ptr(ws), ws.numel(), _stream_handle(stream))
    _raise(st, "kmeanspp_init")
    return indices, centers


def kmeanspp_rows_read(ws, stream=None) -> int:
    """Rows of X the last seeding on ``ws`` read over its distance passes
    (0: it read every row); synchronises the stream."""
    v = ctypes.c_int64(0)
    _raise(load().kmeanspp_rows_read(_ptr(ws), _stream_handle(stream), ctypes.byref(v)), "kmeanspp_rows_read")
    return int(v.value)


def kmeans_device_status(ws, stream=None) -> int:
    """Synchronise the stream; status of the last call that used ``ws``."""
    return int(load().kmeans_device_status(_ptr(ws), _stream_handle(stream)))


def kmeans_relocate_empty(labels, best_dist, k: int, ws=None, stream=None):
    """Move the samples farthest from their centroids into the empty
    clusters (labels rewritten in place) -> ``labels``."""
    torch = _torch()
    _check(labels, "labels", torch.int64)
    n = labels.shape[0]
    _check(best_dist, "best_dist", torch.float32, (n,), labels.device)
    ws = _ws(ws, OP_RELOCATE, n, k, 1, labels.device)
    st = load().kmeans_relocate_empty(_ptr(labels), _ptr(best_dist), n, int(k), _ptr(ws), ws.numel(),
                                      _stream_handle(stream))
    _raise(st, "kmeans_relocate_empty")
    return labels


def kmeans_fit(X, k: int = None, C=None, init: str = "kmeans++", seed: int = 0, max_iter: int = 300,
               tol: float = 1e-4, labels=None, best_dist=None, counts=None, ws=None, stream=None,
               relocate_empty: bool = False):
    """Lloyd iterations until the relative inertia improvement is at most
    ``tol`` (or ``max_iter``) -> ``(C, labels, best_dist, counts,
    inertia_history, n_iter)``.  ``init="kmeans++"`` seeds ``k`` centroids
    with ``seed``; ``init="given"`` starts from ``C`` (updated in place).
    ``relocate_empty`` passes each iteration's labels through
    kmeans_relocate_empty before the update.
    Synchronises the stream once per iteration."""
    import numpy as np
    torch = _torch()
    _check(X, "X", torch.float32)
    n, d = X.shape
    if init == "kmeans++":
        if k is None:
            raise ValueError("init='kmeans++' needs k")
        if C is None:
            C = torch.empty((int(k), d), dtype=torch.float32, device=X.device)
        code = INIT_KMEANSPP
    elif init == "given":
        if C is None:
            raise ValueError("init='given' needs C")
        code = INIT_GIVEN
    else:
        raise ValueError(f"unknown init {init!r}")
    _check(C, "C", torch.float32, device=X.device)
    k = C.shape[0]
    if labels is None:
        labels = torch.empty(n, dtype=torch.int64, device=X.device)
    if best_dist is None:
        best_dist = torch.empty(n, dtype=torch.float32, device=X.device)
    if counts is None:
        counts = torch.empty(k, dtype=torch.int32, device=X.device)
    if ws is None:
        ws = workspace(OP_FIT, n, k, d, X.device)
    hist = np.zeros(int(max_iter), dtype=np.float64)
    n_iter = ctypes.c_int(0)
    if relocate_empty:
        code |= FIT_RELOCATE_EMPTY
    st = load().kmeans_fit(_ptr(X), _ptr(C), _ptr(labels), _ptr(best_dist), _ptr(counts), n, k, d, code,
                           int(seed) & (2**64 - 1), int(max_iter), float(tol), ctypes.byref(n_iter),
                           hist.ctypes.data_as(ctypes.c_void_p), _ptr(ws), ws.numel(), _stream_handle(stream))
    _raise(st, "kmeans_fit")
    return C, labels, best_dist, counts, hist[:n_iter.value].copy(), n_iter.value


def kmeans_trace_start(capacity: int = 1024) -> None:
    """Time each call's dominant kernel with CUDA events (up to ``capacity``
    launches per kernel kind) until kmeans_trace_stop."""
    _raise(load().kmeans_trace_start(int(capacity)), "kmeans_trace_start")


def kmeans_trace_read(kernel: int):
    """``(ms_total, timed_launches, launches)`` of one traced kernel kind
    (KERNEL_ASSIGN_TC, KERNEL_UPDATE_MEAN, KERNEL_KMEANSPP_DIST); waits for
    the recorded events."""
    ms = ctypes.c_double(0.0)
    timed, seen = ctypes.c_int64(0), ctypes.c_int64(0)
    _raise(load().kmeans_trace_read(int(kernel), ctypes.byref(ms), ctypes.byref(timed), ctypes.byref(seen)),
           "kmeans_trace_read")
    return ms.value, timed.value, seen.value


def kmeans_trace_stop() -> None:
    """Turn tracing off and release its events."""
    _raise(load().kmeans_trace_stop(), "kmeans_trace_stop")


def kmeans_lloyd_iter_host(Xh, Ch, Xd, Cd, C_new, labels, best_dist, counts, C_out_h, labels_h, inertia_h,
                           slices: int = 16, ws=None, inertia=None, copy_stream=None, stream=None,
                           overlap_previous: bool = False, readback_on_copy_stream: bool = False):
    """One Lloyd iteration on inputs that live in pinned host memory.

    The library copies the samples to ``Xd`` in ``slices`` row slices on
    ``copy_stream`` and assigns each slice on ``stream`` as soon as it has
    landed; the update follows, and C_new, the labels and the inertia come
    back to ``C_out_h``, ``labels_h`` and ``inertia_h`` (one float64).  The
    device outputs are kmeans_lloyd_iter's: bit for bit with one slice; with
    more, the distances and inertia within the distance tolerance (each
    slice's pass may split other tiles along K).  Returns an event
    recorded after the last copy.  ``overlap_previous``: the copies may
    overlap earlier work on ``stream`` (the caller guarantees that ``Xd`` and
    ``Cd`` are not in use, e.g. by alternating two sets).
    ``readback_on_copy_stream``: the copies back to the host run on
    ``copy_stream`` after the update (the event is recorded there), so that
    ``stream`` can start the next iteration; the caller leaves ``C_new``,
    ``labels`` and ``inertia`` unchanged until the event.
    Xh, Ch, C_out_h, labels_h, inertia_h: pinned host tensors.
    Xd, Cd, C_new, labels, best_dist, counts: device tensors (preallocated).
    """
    torch = _torch()
    n, d = Xh.shape
    k = Ch.shape[0]
    _check(Xd, "Xd", torch.float32, (n, d))
    _check(Cd, "Cd", torch.float32, (k, d), Xd.device)
    _check(C_new, "C_new", torch.float32, (k, d), Xd.device)
    _check(labels, "labels", torch.int64, (n,), Xd.device)
    _check(best_dist, "best_dist", torch.float32, (n,), Xd.device)
    if counts is not None:
        _check(counts, "counts", torch.int32, (k,), Xd.device)
    for t, name, dt, shape in ((Xh, "Xh", torch.float32, (n, d)), (Ch, "Ch", torch.float32, (k, d)),
                               (C_out_h, "C_out_h", torch.float32, (k, d)), (labels_h, "labels_h", torch.int64, (n,)),
                               (inertia_h, "inertia_h", torch.float64, (1,))):
        if t.is_cuda or t.dtype != dt or tuple(t.shape) != shape or not t.is_contiguous():
            raise ValueError(f"{name}: expected a contiguous host tensor {dt} {shape}")
    stream = stream or torch.cuda.current_stream()
    copy_stream = copy_stream or torch.cuda.Stream()
    if inertia is None:
        inertia = torch.empty(1, dtype=torch.float64, device=Xd.device)
    if ws is None:
        ws = workspace(OP_LLOYD, n, k, d, Xd.device)
    st = load().kmeans_lloyd_iter_host(Xh.data_ptr(), Ch.data_ptr(), _ptr(Xd), _ptr(Cd), _ptr(C_new), _ptr(labels),
                                       _ptr(best_dist), _ptr(inertia), _ptr(counts), C_out_h.data_ptr(),
                                       labels_h.data_ptr(), inertia_h.data_ptr(), n, k, d, int(slices),
                                       (HOST_OVERLAP_PREVIOUS if overlap_previous else 0) |
                                       (HOST_READBACK_ON_COPY_STREAM if readback_on_copy_stream else 0), _ptr(ws),
                                       ws.numel(), _stream_handle(stream), _stream_handle(copy_stream))
    _raise(st, "kmeans_lloyd_iter_host")
    done = torch.cuda.Event()
    done.record(copy_stream if readback_on_copy_stream else stream)
    return done


# ------------------------------------------------- samples split across GPUs
def kmeans_update_partial(X, labels, k: int, sums=None, counts=None, ws=None, seed=0, stream=None):
    """One shard's cluster sums (zeros for an empty cluster) and counts ->
    ``(sums (k, d), counts (k,))``."""
    torch = _torch()
    _check(X, "X", torch.float32)
    n, d = X.shape
    _check(labels, "labels", torch.int64, (n,), X.device)
    k = int(k)
    if sums is None:
        sums = torch.empty((k, d), dtype=torch.float32, device=X.device)
    if counts is None:
        counts = torch.empty(k, dtype=torch.int32, device=X.device)
    _check(sums, "sums", torch.float32, (k, d), X.device)
    _check(counts, "counts", torch.int32, (k,), X.device)
    ws = _ws(ws, OP_UPDATE_PARTIAL, n, k, d, X.device)
    st = load().kmeans_update_partial(_ptr(X), _ptr(labels), n, k, d, _ptr(sums), _ptr(counts), _ptr(ws), ws.numel(),
                                      seed & (2**64 - 1), _stream_handle(stream))
    _raise(st, "kmeans_update_partial")
    return sums, counts


def kmeans_lloyd_iter_partial(X, C, labels=None, best_dist=None, inertia=None, sums=None, counts=None, ws=None,
                              seed=0, stream=None):
    """One shard's part of a Lloyd iteration -> ``(sums, counts, labels,
    best_dist, inertia)`` (the shard's assignment and its cluster sums)."""
    torch = _torch()
    _check(X, "X", torch.float32)
    n, d = X.shape
    _check(C, "C", torch.float32, device=X.device)
    k = C.shape[0]
    if C.dim() != 2 or C.shape[1] != d:
        raise ValueError("C must be (k, d) with the same d as X")
    labels = torch.empty(n, dtype=torch.int64, device=X.device) if labels is None else labels
    best_dist = torch.empty(n, dtype=torch.float32, device=X.device) if best_dist is None else best_dist
    inertia = torch.empty(1, dtype=torch.float64, device=X.device) if inertia is None else inertia
    sums = torch.empty((k, d), dtype=torch.float32, device=X.device) if sums is None else sums
    counts = torch.empty(k, dtype=torch.int32, device=X.device) if counts is None else counts
    _check(labels, "labels", torch.int64, (n,), X.device)
    _check(best_dist, "best_dist", torch.float32, (n,), X.device)
    _check(inertia, "inertia", torch.float64, (1,), X.device)
    _check(sums, "sums", torch.float32, (k, d), X.device)
    _check(counts, "counts", torch.int32, (k,), X.device)
    ws = _ws(ws, OP_LLOYD_PARTIAL, n, k, d, X.device)
    st = load().kmeans_lloyd_iter_partial(_ptr(X), _ptr(C), _ptr(labels), _ptr(best_dist), _ptr(inertia), _ptr(sums),
                                          _ptr(counts), n, k, d, _ptr(ws), ws.numel(), seed & (2**64 - 1),
                                          _stream_handle(stream))
    _raise(st, "kmeans_lloyd_iter_partial")
    return sums, counts, labels, best_dist, inertia


def kmeans_reduce_partials(parts, part_counts, C_old, C_new=None, counts=None, part_inertia=None, inertia=None,
                           stream=None):
    """Rank-order sum of ``parts`` (world, rows, d) over the summed
    ``part_counts`` (world, rows); C_old's row where no rank has a member ->
    ``(C_new, counts, inertia)``."""
    torch = _torch()
    _check(parts, "parts", torch.float32)
    world, rows, d = parts.shape
    dev = parts.device
    _check(part_counts, "part_counts", torch.int32, (world, rows), dev)
    _check(C_old, "C_old", torch.float32, (rows, d), dev)
    C_new = torch.empty_like(C_old) if C_new is None else C_new
    counts = torch.empty(rows, dtype=torch.int32, device=dev) if counts is None else counts
    _check(C_new, "C_new", torch.float32, (rows, d), dev)
    _check(counts, "counts", torch.int32, (rows,), dev)
    if part_inertia is not None:
        _check(part_inertia, "part_inertia", torch.float64, (world,), dev)
        inertia = torch.empty(1, dtype=torch.float64, device=dev) if inertia is None else inertia
        _check(inertia, "inertia", torch.float64, (1,), dev)
    st = load().kmeans_reduce_partials(_ptr(parts), _ptr(part_counts), _ptr(part_inertia), world, rows, d,
                                       _ptr(C_old), _ptr(C_new), _ptr(counts),
                                       _ptr(inertia if part_inertia is not None else None), _stream_handle(stream))
    _raise(st, "kmeans_reduce_partials")
    return C_new, counts, inertia


def kmeanspp_shard_exchange_bytes(n_trials: int, d: int) -> int:
    return int(load().kmeanspp_shard_exchange_bytes(int(n_trials), int(d)))


def kmeanspp_shard_first(X, row_offset: int, n_global: int, n_trials: int, seed: int, send, ws, stream=None):
    st = load().kmeanspp_shard_first(_ptr(X), X.shape[0], X.shape[1], int(row_offset), int(n_global), int(n_trials),
                                     int(seed) & (2**64 - 1), _ptr(send), _ptr(ws), ws.numel(), _stream_handle(stream))
    _raise(st, "kmeanspp_shard_first")


def kmeanspp_shard_pick(X, row_offset: int, n_trials: int, seed: int, c: int, totals, rank: int, send, ws,
                        stream=None):
    st = load().kmeanspp_shard_pick(_ptr(X), X.shape[0], X.shape[1], int(row_offset), int(n_trials),
                                    int(seed) & (2**64 - 1), int(c), _ptr(totals), totals.numel(), int(rank),
                                    _ptr(send), _ptr(ws), ws.numel(), _stream_handle(stream))
    _raise(st, "kmeanspp_shard_pick")


def kmeanspp_shard_dist(X, n_trials: int, first: bool, recv, world: int, pot, ws, stream=None):
    st = load().kmeanspp_shard_dist(_ptr(X), X.shape[0], X.shape[1], int(n_trials), 1 if first else 0, _ptr(recv),
                                    int(world), _ptr(pot), _ptr(ws), ws.numel(), _stream_handle(stream))
    _raise(st, "kmeanspp_shard_dist")


def kmeanspp_shard_commit(n: int, d: int, n_trials: int, first: bool, pots, world: int, c: int, indices, centers,
                          total, ws, stream=None):
    st = load().kmeanspp_shard_commit(int(n), int(d), int(n_trials), 1 if first else 0, _ptr(pots), int(world), int(c),
                                      _ptr(indices), _ptr(centers), _ptr(total), _ptr(ws), ws.numel(),
                                      _stream_handle(stream))
    _raise(st, "kmeanspp_shard_commit")

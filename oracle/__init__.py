"""CPU oracle for the k-means Lloyd iteration and k-means++ seeding.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The product library
(``distance_argmin_gb300``) never imports it, and this package never imports
the product: the two share no code.

The arithmetic lives in ``kmeans_oracle.c`` (plain C + OpenMP, binary64); this
module only compiles it with gcc and marshals numpy arrays through ctypes.
Every function states the page section it follows:

* ``assign``  -- "Three shapes that fit an eager Gram assignment", section
  "Gram assignment": the nearest centroid under the squared Euclidean distance.
* ``update``  -- same page, section "Full Lloyd step": the mean of the members.
* ``kmeanspp`` -- "004 — tile sizes, a Cython Lloyd step, and k-means++",
  section "k-means++": greedy D^2 seeding with 2 + log(n_clusters) trials.
* ``relocate_empty`` -- same page, section "Cython timing": the Lloyd step
  there relocates empty clusters.  The page gives no rule; this is the plain
  reading (each empty cluster takes one of the samples farthest from their
  centroid).  It is pure selection, written here in numpy.
* ``philox4x32_10`` / ``uniform`` -- the counter-based generator of Salmon et
  al. (SC'11), from its published definition.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kmeans_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_P = ctypes.c_void_p


def build(force: bool = False) -> str:
    """Compile ``kmeans_oracle.c`` into ``liboracle.so`` (gcc, OpenMP).

    ``-ffp-contract=off`` keeps every multiply and add separately rounded, so
    x86-64 and aarch64 builds give identical bits.
    """
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
           "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            lib.oracle_philox4x32_10.argtypes = [_P, _P, _P]
            lib.oracle_philox4x32_10.restype = None
            lib.oracle_uniform.argtypes = [_U64, _U64]
            lib.oracle_uniform.restype = ctypes.c_double
            lib.oracle_sqdist.argtypes = [_P, _P, _I64]
            lib.oracle_sqdist.restype = ctypes.c_double
            lib.oracle_max_threads.argtypes = []
            lib.oracle_max_threads.restype = ctypes.c_int
            lib.oracle_assign.argtypes = [_P, _P, _I64, _I64, _I64, _P, _P, _P, ctypes.c_int]
            lib.oracle_assign.restype = ctypes.c_double
            lib.oracle_update.argtypes = [_P, _P, _P, _I64, _I64, _I64, _P, _P, ctypes.c_int]
            lib.oracle_update.restype = ctypes.c_int
            lib.oracle_kmeanspp.argtypes = [_P, _I64, _I64, _I64, ctypes.c_int, _U64,
                                            _P, _P, _P, _P, ctypes.c_int]
            lib.oracle_kmeanspp.restype = ctypes.c_int
            _lib = lib
    return _lib


def _f32(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def max_threads() -> int:
    """Threads OpenMP will use (all cores in the process affinity mask)."""
    return int(_load().oracle_max_threads())


def philox4x32_10(counter, key) -> np.ndarray:
    """One Philox4x32-10 block: 4 x uint32 counter, 2 x uint32 key -> 4 x uint32."""
    c = np.ascontiguousarray(counter, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    _load().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, draw: int) -> float:
    """The k-means++ uniform for ``draw`` under ``seed`` (53-bit, in [0, 1))."""
    return float(_load().oracle_uniform(seed & (2**64 - 1), draw))


def sqdist(x, c) -> float:
    x = _f32(x)
    c = _f32(c)
    return float(_load().oracle_sqdist(_ptr(x), _ptr(c), x.shape[-1]))


def assign(X, C, nthreads: int = 0):
    """Brute-force nearest centroid.

    Returns ``(labels int64 (n,), best float64 (n,), second float64 (n,),
    inertia float)``: the winning index (lowest on ties), its squared distance,
    the runner-up distance (+inf when k == 1) and the sum of the winners.
    """
    X = _f32(X)
    C = _f32(C)
    n, d = X.shape
    k = C.shape[0]
    assert C.shape[1] == d
    labels = np.empty(n, dtype=np.int64)
    best = np.empty(n, dtype=np.float64)
    second = np.empty(n, dtype=np.float64)
    inertia = _load().oracle_assign(_ptr(X), _ptr(C), n, k, d, _ptr(labels), _ptr(best),
                                    _ptr(second), nthreads)
    return labels, best, second, float(inertia)


def update(X, labels, C_old, nthreads: int = 0):
    """Mean of members, empty cluster keeps its old row.

    Returns ``(C_new float32 (k, d), counts int64 (k,))``.
    """
    X = _f32(X)
    C_old = _f32(C_old)
    labels = np.ascontiguousarray(labels, dtype=np.int64)
    n, d = X.shape
    k = C_old.shape[0]
    C_new = np.empty((k, d), dtype=np.float32)
    counts = np.empty(k, dtype=np.int64)
    rc = _load().oracle_update(_ptr(X), _ptr(labels), _ptr(C_old), n, k, d, _ptr(C_new),
                               _ptr(counts), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_update failed ({rc}): label out of range or no memory")
    return C_new, counts


def lloyd_iter(X, C_old, nthreads: int = 0):
    """One Lloyd iteration: assign, then update with those labels."""
    labels, best, second, inertia = assign(X, C_old, nthreads)
    C_new, counts = update(X, labels, C_old, nthreads)
    return C_new, labels, best, second, inertia, counts


def relocate_empty(labels, best, k: int):
    """Give every empty cluster a member.

    "004 — tile sizes, a Cython Lloyd step, and k-means++", section "Cython
    timing", says only that the Lloyd step relocates empty clusters.  Reading:
    with m clusters that have no member, the m samples farthest from the
    centroid they were assigned to (largest ``best``; equal distances: lower
    sample index first) leave their clusters; taken in increasing sample
    index, they become the only members of the empty clusters taken in
    increasing cluster index.  A cluster that loses all its members this way
    is empty afterwards (and keeps its centroid in the update).

    ``labels`` (n,) int64 in [0, k) and ``best`` (n,) the assigned squared
    distances (no NaN).  Returns ``(new_labels int64 (n,), moved int64 (m,))``
    with ``moved`` the relocated samples in increasing index."""
    labels = np.array(labels, dtype=np.int64)
    best = np.asarray(best, dtype=np.float64)
    n = labels.shape[0]
    assert best.shape == (n,)
    counts = np.bincount(labels, minlength=k)
    assert counts.shape == (k,), "label outside [0, k)"
    empty = np.flatnonzero(counts == 0)
    m = empty.size
    if m == 0:
        return labels, np.empty(0, dtype=np.int64)
    # primary key: distance, largest first; then sample index, lowest first
    farthest = np.lexsort((np.arange(n), -best))[:m]
    moved = np.sort(farthest)
    labels[moved] = empty
    return labels, moved


def fit(X, C0, max_iter: int, tol: float, nthreads: int = 0, relocate: bool = False):
    """Lloyd iterations from C0 until the relative inertia improvement is at
    most ``tol`` or ``max_iter`` iterations have run (the pages fix no
    stopping rule; this is the plain one, the same as the library's).
    Iteration t assigns X to C_t (inertia_t) and updates to C_{t+1}; the fit
    stops after iteration t when inertia_t >= (1 - tol) * inertia_{t-1}.
    With ``relocate`` each assignment's labels pass through
    ``relocate_empty`` before the update (the inertia stays the
    assignment's).
    Returns ``(C_last, labels_last, best_last, inertia_history, n_iter)``."""
    C = _f32(C0)
    k = C.shape[0]
    hist = []
    labels = best = None
    for it in range(max_iter):
        labels, best, _, inertia = assign(X, C, nthreads)
        if relocate:
            labels, _ = relocate_empty(labels, best, k)
        C_new, _ = update(X, labels, C, nthreads)
        hist.append(inertia)
        C = C_new
        if it > 0 and inertia >= hist[-2] * (1.0 - tol):
            break
    return C, labels, best, np.array(hist), len(hist)


def n_trials_for(k: int) -> int:
    """2 + floor(ln k): the candidate count per new center."""
    import math
    return 2 + int(math.floor(math.log(k)))


def kmeanspp(X, k: int, seed: int, n_trials: int = 0, nthreads: int = 0):
    """Greedy D^2 seeding.

    Returns ``(indices int64 (k,), margins float64 (1 + (k-1) T,),
    potentials float64 (k,))``.  ``margins[draw]`` is how far that draw's
    target lay from the nearest running-sum boundary, over the total.
    """
    X = _f32(X)
    n, d = X.shape
    T = n_trials if n_trials > 0 else n_trials_for(k)
    indices = np.empty(k, dtype=np.int64)
    margins = np.zeros(1 + (k - 1) * T, dtype=np.float64)
    pots = np.zeros(k, dtype=np.float64)
    rc = _load().oracle_kmeanspp(_ptr(X), n, d, k, T, seed & (2**64 - 1), _ptr(indices), None,
                                 _ptr(margins), _ptr(pots), nthreads)
    if rc != 0:
        raise ValueError(f"oracle_kmeanspp failed ({rc})")
    return indices, margins, pots

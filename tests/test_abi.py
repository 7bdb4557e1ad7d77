"""Host-side checks of the C ABI: the library loads, exports what the header
declares, validates arguments before touching the GPU, and sizes workspaces
with no n*k term.  No kernel runs here (no GPU needed)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kmeans_gb300.h")
GOLDEN = os.path.join(ROOT, "tests", "golden", "probe_byte_counts.txt")


@pytest.fixture(scope="module")
def km():
    from distance_argmin_gb300 import build as b
    b.build()
    import distance_argmin_gb300 as km
    km.load()
    return km


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^[A-Za-z_][\w\s\*]*?\b(\w+)\s*\(", text, flags=re.M)))


def test_library_exports_every_declared_symbol(km):
    declared = _declared_functions()
    assert "kmeans_assign" in declared and "kmeanspp_init" in declared
    lib = ctypes.CDLL(km.LIB_PATH)
    for name in declared:
        assert hasattr(lib, name), f"{name} declared in the header but not exported"
    assert set(km.EXPORTS) == set(declared)


def test_binding_constants_match_the_header(km):
    # every integer #define of the header that the binding mirrors
    text = open(HEADER).read()
    defines = dict(re.findall(r"^#define KMEANS_(\w+) (\d+)\s*$", text, flags=re.M))
    assert {"HOST_MAX_SLICES", "HOST_OVERLAP_PREVIOUS", "HOST_READBACK_ON_COPY_STREAM"} <= set(defines)
    for name, value in defines.items():
        if hasattr(km, name):
            assert getattr(km, name) == int(value), name


def test_kmeanspp_rows_read_rejects_null_pointers(km):
    lib = _lib(km)
    out = ctypes.c_int64(0)
    assert lib.kmeanspp_rows_read(None, None, ctypes.byref(out)) == km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeanspp_rows_read(ctypes.c_void_p(0x10000), None, None) == km.KMEANS_ERR_INVALID_ARG


def test_status_strings(km):
    for st in range(8):
        s = km.kmeans_status_string(st)
        assert isinstance(s, str) and s and s != "unknown status"
    assert km.kmeans_status_string(99) == "unknown status"
    assert "sm_103a" in km.kmeans_build_info()


def _lib(km):
    return km.load()


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: validation fails first
FAKE_WS = ctypes.c_void_p(0x100000)  # 256-byte aligned


def test_invalid_arguments_are_rejected_on_the_host(km):
    lib = _lib(km)
    n, k, d = 100, 10, 16
    ws_need = km.kmeans_workspace_bytes(km.OP_ASSIGN, n, k, d)
    args = lambda X, C, n, k, d, ws=FAKE_WS, wsb=ws_need: (X, C, n, k, d, FAKE, FAKE, None, ws, wsb, 0, None)
    assert lib.kmeans_assign(*args(None, FAKE, n, k, d)) == km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_assign(*args(FAKE, FAKE, n, n + 1, d)) == km.KMEANS_ERR_INVALID_ARG  # k > n
    assert lib.kmeans_assign(*args(FAKE, FAKE, 0, 0, d)) == km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_assign(*args(FAKE, FAKE, n, k, 0)) == km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_assign(*args(FAKE, FAKE, n, k, 18)) == km.KMEANS_ERR_UNSUPPORTED    # d % 4
    assert lib.kmeans_assign(*args(FAKE, FAKE, n, k, d, wsb=ws_need - 1)) == km.KMEANS_ERR_WORKSPACE
    assert lib.kmeans_assign(*args(FAKE, FAKE, n, k, d, ws=ctypes.c_void_p(0x100010))) == \
        km.KMEANS_ERR_WORKSPACE  # misaligned
    assert lib.kmeans_assign(*args(FAKE, FAKE, 2**31, 10, d)) == km.KMEANS_ERR_INVALID_ARG
    # the FFMA comparator accepts any d, but still checks the workspace
    assert lib.kmeans_assign_ffma(*args(FAKE, FAKE, n, k, 18, wsb=1)) == km.KMEANS_ERR_WORKSPACE
    upd = lambda labels, ws, wsb: lib.kmeans_update(FAKE, labels, FAKE, FAKE, None, n, k, d, ws, wsb, 0, None)
    assert upd(None, FAKE_WS, 1 << 30) == km.KMEANS_ERR_INVALID_ARG
    assert upd(FAKE, FAKE_WS, 16) == km.KMEANS_ERR_WORKSPACE
    assert lib.kmeans_lloyd_iter(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, n, k, 6, FAKE_WS, 1 << 30, 0,
                                 None) == km.KMEANS_ERR_UNSUPPORTED
    assert lib.kmeanspp_init(FAKE, n, d, k, 33, 0, None, FAKE, FAKE_WS, 1 << 30, None) == \
        km.KMEANS_ERR_UNSUPPORTED  # more than 32 trials
    assert lib.kmeanspp_init(FAKE, n, d, k, 0, 0, None, None, FAKE_WS, 1 << 30, None) == \
        km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeans_device_status(None, None) == km.KMEANS_ERR_INVALID_ARG


@pytest.mark.parametrize("op", [0, 1, 2, 4])
@pytest.mark.parametrize("n", [1 << 12, 1 << 16])
def test_workspace_has_no_n_times_k_term(km, op, n):
    f = lambda n, k: km.kmeans_workspace_bytes(op, n, k, 512)
    k = n >> 4
    mixed = f(2 * n, 2 * k) - f(2 * n, k) - f(n, 2 * k) + f(n, k)
    assert abs(mixed) <= 16 * 1024  # only region alignment remains
    assert km.kmeans_workspace_bytes(op, 10, 11, 4) == 0  # k > n is invalid


def test_lloyd_workspace_is_the_larger_of_its_steps(km):
    for n, k, d in [(4096, 256, 512), (65536, 1024, 2048), (131072, 8192, 8192)]:
        a = km.kmeans_workspace_bytes(km.OP_ASSIGN, n, k, d)
        u = km.kmeans_workspace_bytes(km.OP_UPDATE, n, k, d)
        assert km.kmeans_workspace_bytes(km.OP_LLOYD, n, k, d) == max(a, u)


def test_fit_workspace_is_the_shared_scratch_plus_a_centroid_buffer(km):
    # the shared scratch, a second centroid buffer, the seeding's indices, the
    # inertia and the relocation's two k-long int32 arrays
    for n, k, d in [(4096, 256, 512), (65536, 1024, 2048), (131072, 8192, 8192)]:
        lloyd = km.kmeans_workspace_bytes(km.OP_LLOYD, n, k, d)
        fit = km.kmeans_workspace_bytes(km.OP_FIT, n, k, d)
        extra = fit - lloyd
        assert k * d * 4 + k * 16 <= extra <= k * d * 4 + k * 16 + 8 + 6 * 1024 + \
            max(0, km.kmeans_workspace_bytes(km.OP_KMEANSPP, n, k, d) - lloyd)
        assert fit < n * k * 4


def test_kmeanspp_slice_width_matches_the_library(km):
    # the workspace holds one float2 per (slice, 8 trials, sample): one more
    # feature than a whole slice adds exactly one slice of partial sums
    n, k, s = 65536, 1024, km.KPP_SLICE_FEATURES
    for d in (s, 2 * s):
        grow = km.kmeans_workspace_bytes(km.OP_KMEANSPP, n, k, d + 1) - km.kmeans_workspace_bytes(km.OP_KMEANSPP, n, k, d)
        assert grow == 8 * 8 * n
    assert km.kmeans_workspace_bytes(km.OP_KMEANSPP, n, k, s) == km.kmeans_workspace_bytes(km.OP_KMEANSPP, n, k, s - 1)


def test_relocate_workspace_and_argument_checks(km):
    lib = _lib(km)
    for n, k in [(10, 1), (4096, 256), (131072, 8192)]:
        b = km.kmeans_workspace_bytes(km.OP_RELOCATE, n, k, 1)
        assert 256 + 8 * k <= b <= 256 + 8 * k + 512      # header, counts, empty list
        assert b == km.kmeans_workspace_bytes(km.OP_RELOCATE, 2 * n, k, 7)  # independent of n and d
    need = km.kmeans_workspace_bytes(km.OP_RELOCATE, 100, 10, 1)
    rel = lambda labels, best, n, k, ws=FAKE_WS, wsb=need: lib.kmeans_relocate_empty(labels, best, n, k, ws, wsb,
                                                                                      None)
    assert rel(None, FAKE, 100, 10) == km.KMEANS_ERR_INVALID_ARG
    assert rel(FAKE, None, 100, 10) == km.KMEANS_ERR_INVALID_ARG
    assert rel(FAKE, FAKE, 100, 101) == km.KMEANS_ERR_INVALID_ARG       # k > n
    assert rel(FAKE, FAKE, 0, 0) == km.KMEANS_ERR_INVALID_ARG
    assert rel(FAKE, FAKE, 2**31, 10) == km.KMEANS_ERR_INVALID_ARG
    assert rel(ctypes.c_void_p(0x10004), FAKE, 100, 10) == km.KMEANS_ERR_INVALID_ARG   # labels not 8-aligned
    assert rel(FAKE, ctypes.c_void_p(0x10002), 100, 10) == km.KMEANS_ERR_INVALID_ARG   # best not 4-aligned
    assert rel(FAKE, FAKE, 100, 10, wsb=need - 1) == km.KMEANS_ERR_WORKSPACE
    assert rel(FAKE, FAKE, 100, 10, ws=ctypes.c_void_p(0x100010)) == km.KMEANS_ERR_WORKSPACE


def test_workspace_far_below_the_distance_matrix_at_every_workload(km):
    import synth
    for w in list(synth.WORKLOADS.values()) + [synth.KMEANSPP]:
        for op in (km.OP_ASSIGN, km.OP_LLOYD, km.OP_KMEANSPP):
            ws = km.kmeans_workspace_bytes(op, w.n, w.k, w.d)
            assert 0 < ws < w.n * w.k * 4, (w.name, op, ws)


def test_probe_byte_counts_from_the_page(km):
    # the fusion-probe page prints the sizes of the buffers a fused assignment
    # must avoid; check them against the shapes, and the workspace against them
    vals = {}
    for line in open(GOLDEN):
        if line.startswith("#") or not line.strip():
            continue
        name, v = line.split()
        vals[name] = float(v)
    n, k, d = 4096, 256, 512
    MiB = 1024 * 1024
    assert vals["distance_nk"] * MiB == n * k * 4
    assert vals["broadcast_nkd"] * MiB == n * k * d * 4
    assert vals["one_centroid_difference_nd"] * MiB == n * d * 4
    assert round(n * 8 / MiB, 3) == vals["labels_n_int64"]
    assert km.kmeans_workspace_bytes(km.OP_ASSIGN, n, k, d) < vals["distance_nk"] * MiB


def test_update_workspace_holds_every_chunks_partials(km):
    # The segmented mean cuts the member list into chunks sized for one wave
    # of 512-column slices (152 SMs x 12 blocks), at least 16 members, a
    # multiple of 16, at most 4096; every chunk keeps a head and a tail
    # partial row of d floats.  Small n with large d gives many short chunks.
    def chunk(n, d):
        slices = (d + 511) // 512
        chunks = (152 * 12 + slices - 1) // slices
        c = max(16, (n + chunks - 1) // chunks)
        return min(4096, (c + 15) // 16 * 16)

    for n, k, d in ((4096, 4, 8192), (65536, 1024, 2048), (1000, 10, 16384), (300, 3, 64)):
        n_chunks = (n + chunk(n, d) - 1) // chunk(n, d)
        assert km.kmeans_workspace_bytes(km.OP_UPDATE, n, k, d) >= 2 * n_chunks * d * 4 + 16 * n
    assert chunk(4096, 8192) == 48  # 86 chunks: one cluster of 4050 members crosses 85 of them


def test_shard_entry_points_validate_on_the_host(km):
    lib = _lib(km)
    F, W = FAKE, FAKE_WS
    # shard workspaces accept more centroids than samples; the others do not
    assert km.kmeans_workspace_bytes(km.OP_LLOYD_PARTIAL, 300, 700, 36) > 0
    assert km.kmeans_workspace_bytes(km.OP_UPDATE_PARTIAL, 300, 700, 36) > 0
    assert km.kmeans_workspace_bytes(km.OP_KMEANSPP_SHARD, 300, 700, 36) > 0
    assert km.kmeans_workspace_bytes(km.OP_LLOYD, 300, 700, 36) == 0
    n, k, d = 300, 700, 36
    need = km.kmeans_workspace_bytes(km.OP_UPDATE_PARTIAL, n, k, d)
    up = lambda sums, counts, labels=F, wsb=need: lib.kmeans_update_partial(F, labels, n, k, d, sums, counts, W, wsb,
                                                                            0, None)
    assert up(None, F) == km.KMEANS_ERR_INVALID_ARG
    assert up(F, None) == km.KMEANS_ERR_INVALID_ARG               # the counts are required
    assert up(F, F, labels=ctypes.c_void_p(0x10004)) == km.KMEANS_ERR_INVALID_ARG
    assert up(F, F, wsb=need - 1) == km.KMEANS_ERR_WORKSPACE       # k > n passed the size checks
    need = km.kmeans_workspace_bytes(km.OP_LLOYD_PARTIAL, n, k, d)
    lp = lambda dd, counts=F, wsb=need: lib.kmeans_lloyd_iter_partial(F, F, F, F, None, F, counts, n, k, dd, W, wsb,
                                                                      0, None)
    assert lp(34) == km.KMEANS_ERR_UNSUPPORTED                     # d % 4
    assert lp(d, counts=None) == km.KMEANS_ERR_INVALID_ARG
    assert lp(d, wsb=need - 1) == km.KMEANS_ERR_WORKSPACE
    rp = lambda pin, world, rows, parts=F, inertia=None: lib.kmeans_reduce_partials(parts, F, pin, world, rows, 8, F,
                                                                                    F, None, inertia, None)
    assert rp(None, 0, 4) == km.KMEANS_ERR_INVALID_ARG             # world 0
    assert rp(None, 2, -1) == km.KMEANS_ERR_INVALID_ARG
    assert rp(F, 2, 4) == km.KMEANS_ERR_INVALID_ARG                # part inertia without an output
    assert rp(None, 2, 4, inertia=F) == km.KMEANS_ERR_INVALID_ARG  # and the reverse
    assert rp(None, 2, 4, parts=None) == km.KMEANS_ERR_INVALID_ARG
    assert rp(None, 2, 0) == km.KMEANS_OK                          # nothing to reduce, nothing enqueued


def test_kmeanspp_shard_steps_validate_on_the_host(km):
    lib = _lib(km)
    F, W = FAKE, FAKE_WS
    assert km.kmeanspp_shard_exchange_bytes(8, 8192) == 64 + 8 * 8192 * 4
    assert km.kmeanspp_shard_exchange_bytes(3, 5) == 32 + 64       # indices and rows, each rounded to 16 bytes
    assert km.kmeanspp_shard_exchange_bytes(0, 8) == 0 and km.kmeanspp_shard_exchange_bytes(33, 8) == 0
    n, d, T = 1000, 64, 8
    need = km.kmeans_workspace_bytes(km.OP_KMEANSPP_SHARD, n, 10, d)
    first = lambda off, ng, send=F, T=T: lib.kmeanspp_shard_first(F, n, d, off, ng, T, 0, send, W, need, None)
    assert first(500, 1499) == km.KMEANS_ERR_INVALID_ARG           # the shard runs past n_global
    assert first(-1, 5000) == km.KMEANS_ERR_INVALID_ARG
    assert first(0, 5000, send=ctypes.c_void_p(0x10008)) == km.KMEANS_ERR_INVALID_ARG  # send not 16-aligned
    assert first(0, 5000, T=0) == km.KMEANS_ERR_INVALID_ARG
    assert first(0, 5000, T=33) == km.KMEANS_ERR_INVALID_ARG
    assert lib.kmeanspp_shard_first(F, n, d, 0, 5000, T, 0, F, W, need - 1, None) == km.KMEANS_ERR_WORKSPACE
    pick = lambda c, world, rank: lib.kmeanspp_shard_pick(F, n, d, 0, T, 0, c, F, world, rank, F, W, need, None)
    assert pick(0, 2, 0) == km.KMEANS_ERR_INVALID_ARG              # center 0 is the first step's
    assert pick(1, 2, 2) == km.KMEANS_ERR_INVALID_ARG              # rank outside the world
    assert pick(1, 0, 0) == km.KMEANS_ERR_INVALID_ARG
    dist = lambda first, pot: lib.kmeanspp_shard_dist(F, n, d, T, first, F, 2, pot, W, need, None)
    assert dist(0, None) == km.KMEANS_ERR_INVALID_ARG              # potentials needed after the first center
    assert dist(2, F) == km.KMEANS_ERR_INVALID_ARG
    commit = lambda first, pots, c: lib.kmeanspp_shard_commit(n, d, T, first, pots, 2, c, F, None, None, W, need, None)
    assert commit(1, None, 3) == km.KMEANS_ERR_INVALID_ARG         # the first center is center 0
    assert commit(0, None, 3) == km.KMEANS_ERR_INVALID_ARG
    assert commit(0, F, -1) == km.KMEANS_ERR_INVALID_ARG
    assert "exchange block" in km.kmeans_status_string(km.KMEANS_ERR_DEVICE_EXCHANGE)

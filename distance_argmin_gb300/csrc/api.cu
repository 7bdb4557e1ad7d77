// C ABI of the library (declared in include/kmeans_gb300.h): argument
// validation, workspace sizing and the order of kernel launches on the
// caller's stream.  Nothing here allocates memory or synchronises, except
// kmeans_device_status, whose job is to wait for the stream.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "../../include/kmeans_gb300.h"
#include "assign_common.cuh"
#include "common.cuh"
#include "kmeanspp.cuh"
#include "relocate.cuh"
#include "update.cuh"

using namespace km;

namespace {

constexpr int64_t kMaxIndex = 0x7fffffffLL;  // labels and member lists use 32-bit indices

bool sizes_ok(int64_t n, int64_t k, int64_t d) {
    return n >= 1 && k >= 1 && k <= n && d >= 1 && n <= kMaxIndex && k <= kMaxIndex && d <= kMaxIndex;
}

// A shard of the samples may hold fewer samples than there are centroids.
bool shard_sizes_ok(int64_t n, int64_t k, int64_t d) {
    return n >= 1 && k >= 1 && d >= 1 && n <= kMaxIndex && k <= kMaxIndex && d <= kMaxIndex;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int check_ws(const void *ws, size_t ws_bytes, size_t need) {
    if (ws == nullptr || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0) return KMEANS_ERR_WORKSPACE;
    if (ws_bytes < need) return KMEANS_ERR_WORKSPACE;
    return KMEANS_OK;
}

int cuda_status(cudaError_t e) { return e == cudaSuccess ? KMEANS_OK : KMEANS_ERR_CUDA; }

int tc_path_ok(const float *X, const float *C, int64_t d) {
    return (d % 4 == 0 && aligned16(X) && aligned16(C)) ? KMEANS_OK : KMEANS_ERR_UNSUPPORTED;
}

int default_trials(int64_t k) { return 2 + (int)floor(log((double)k)); }

// The three assignment paths: the bf16x3 tensor-core kernel, the 3xTF32
// tensor-core kernel and the float32 FFMA comparator.
enum class AssignPath { kBf16x3, kTf32x3, kFfma };

int run_assign(AssignPath path, const float *X, const float *C, int64_t n, int64_t k, int64_t d, int64_t *labels,
               float *best_dist, double *inertia, void *ws, size_t ws_bytes, cudaStream_t s) {
    if (!X || !C || !labels || !best_dist) return KMEANS_ERR_INVALID_ARG;
    if (!sizes_ok(n, k, d)) return KMEANS_ERR_INVALID_ARG;
    if (!aligned4(X) || !aligned4(C)) return KMEANS_ERR_INVALID_ARG;
    const bool tensor_cores = path != AssignPath::kFfma;
    if (tensor_cores) {
        const int st = tc_path_ok(X, C, d);
        if (st != KMEANS_OK) return st;
    } else if ((k + 127) / 128 > 65535) {
        return KMEANS_ERR_UNSUPPORTED;
    }
    const AssignLayout L = assign_layout(n, k, d, tensor_cores, path == AssignPath::kTf32x3 ? 4 : 2);
    const int wst = check_ws(ws, ws_bytes, (size_t)L.bytes);
    if (wst != KMEANS_OK) return wst;
    uint8_t *w = static_cast<uint8_t *>(ws);
    cudaError_t e;
    if (path == AssignPath::kBf16x3) {
        e = launch_prep_split(C, n, k, d, L, w, s);
        if (e == cudaSuccess) e = launch_assign_tc(X, n, k, d, L, w, s);
    } else if (path == AssignPath::kTf32x3) {
        e = launch_prep_split_tf32(C, n, k, d, L, w, s);
        if (e == cudaSuccess) e = launch_assign_tc(X, n, k, d, L, w, s, true, true);
    } else {
        e = launch_prep_norms(C, n, k, d, L, w, s);
        if (e == cudaSuccess) e = launch_assign_ffma(X, C, n, k, d, L, w, s);
    }
    if (e == cudaSuccess) e = launch_finalize(n, L, w, labels, best_dist, inertia, s);
    return cuda_status(e);
}

// kmeans_fit's workspace: the Lloyd / k-means++ scratch at the base (so the
// status word, and beside it the fit's inertia and empty count, sit in the
// header where kmeans_device_status looks), then the second centroid buffer
// of the ping-pong, the seeding's indices and the relocation's scratch.
struct FitLayout {
    int64_t shared;       // max(Lloyd, k-means++) scratch
    int64_t off_calt;     // k x d f32
    int64_t off_indices;  // k x i64
    RelocLayout reloc;    // counts and empty list, 2 x k x i32
    int64_t bytes;
};

FitLayout fit_layout(int64_t n, int64_t k, int64_t d) {
    FitLayout F{};
    const int64_t a = assign_layout(n, k, d, true).bytes;
    const int64_t u = update_layout(n, k, d).bytes;
    const int64_t p = kpp_layout(n, d, default_trials(k), k).bytes;
    F.shared = a > u ? a : u;
    if (p > F.shared) F.shared = p;
    int64_t o = align_up(F.shared, 1024);
    F.off_calt = o; o = align_up(o + k * d * 4, 1024);
    F.off_indices = o; o = align_up(o + k * 8, 1024);
    F.reloc = reloc_layout(k, o);
    F.bytes = align_up(F.reloc.end, 1024);
    return F;
}

// kmeans_lloyd_iter_fused's workspace: the assignment's scratch, then the
// zeroed accumulation area (sums, counts, per-32-row completion counters).
struct FusedLayout {
    AssignLayout A;
    int64_t off_sums;  // k x d f32
    int64_t off_cnt;   // k x i32
    int64_t off_done;  // ceil(n / 256) x 8 x u32
    int64_t bytes;
};

FusedLayout fused_layout(int64_t n, int64_t k, int64_t d) {
    FusedLayout F{};
    F.A = assign_layout(n, k, d, true, 2, false);  // the fused kernel never splits K
    int64_t o = align_up(F.A.bytes, 1024);
    F.off_sums = o; o = align_up(o + k * d * 4, 256);
    F.off_cnt = o; o = align_up(o + k * 4, 256);
    F.off_done = o; o += ((n + 255) / 256) * 8 * 4;
    F.bytes = align_up(o, 1024);
    return F;
}

// The Lloyd iteration after the tensor-core pass has written every sample's
// key: finalize (with the per-tile member count on the counting path), then
// the mean update.  The update reuses the assignment's workspace: its scratch
// is dead once the labels are written, and the count table and the fused
// finalize's block sums lie above the keys and norms that finalize still reads.
// With `sums_only` (a shard of the samples) C_new receives the clusters'
// sums instead of their means (see launch_update).
cudaError_t lloyd_finish(const float *X, const float *C_old, float *C_new, int64_t *labels, float *best_dist,
                         double *inertia, int32_t *counts, int64_t n, int64_t k, int64_t d, const AssignLayout &A,
                         uint8_t *w, cudaStream_t s, bool sums_only = false) {
    const UpdateLayout U = update_layout(n, k, d);
    const bool fused = U.counting && U.off_table >= A.off_xnorm + n * 4 && U.off_table >= A.off_keys + n * 8;
    cudaError_t e = fused ? launch_finalize_counting(n, k, A, U, w, labels, best_dist, inertia, s)
                          : launch_finalize(n, A, w, labels, best_dist, inertia, s);
    if (e == cudaSuccess) e = launch_update(X, labels, C_old, C_new, counts, n, k, d, U, w, false, s, fused, sums_only);
    return e;
}

int64_t lloyd_ws_bytes(int64_t n, int64_t k, int64_t d) {
    const int64_t a = assign_layout(n, k, d, true).bytes;
    const int64_t u = update_layout(n, k, d).bytes;
    return a > u ? a : u;
}

}  // namespace

extern "C" {

size_t kmeans_workspace_bytes(int op, int64_t n, int64_t k, int64_t d) {
    // the shard operations accept more centroids than samples
    if (op == KMEANS_OP_LLOYD_PARTIAL || op == KMEANS_OP_UPDATE_PARTIAL || op == KMEANS_OP_KMEANSPP_SHARD) {
        if (!shard_sizes_ok(n, k, d)) return 0;
        if (op == KMEANS_OP_LLOYD_PARTIAL) return (size_t)lloyd_ws_bytes(n, k, d);
        if (op == KMEANS_OP_UPDATE_PARTIAL) return (size_t)update_layout(n, k, d).bytes;
        return (size_t)kpp_shard_layout(n, d).bytes;
    }
    if (!sizes_ok(n, k, d)) return 0;
    switch (op) {
        case KMEANS_OP_ASSIGN:
            return (size_t)assign_layout(n, k, d, true).bytes;
        case KMEANS_OP_ASSIGN_FFMA:
            return (size_t)assign_layout(n, k, d, false).bytes;
        case KMEANS_OP_ASSIGN_3XTF32:
            return (size_t)assign_layout(n, k, d, true, 4).bytes;
        case KMEANS_OP_UPDATE:
            return (size_t)update_layout(n, k, d).bytes;
        case KMEANS_OP_LLOYD:
            return (size_t)lloyd_ws_bytes(n, k, d);
        case KMEANS_OP_KMEANSPP:
            return (size_t)kpp_layout(n, d, kKppMaxTrials, k).bytes;
        case KMEANS_OP_FIT:
            return (size_t)fit_layout(n, k, d).bytes;
        case KMEANS_OP_LLOYD_FUSED:
            return (size_t)fused_layout(n, k, d).bytes;
        case KMEANS_OP_RELOCATE:
            return (size_t)reloc_layout(k, sizeof(WsHeader)).end;
        default:
            return 0;
    }
}

int kmeans_assign(const float *X, const float *C, int64_t n, int64_t k, int64_t d, int64_t *labels,
                  float *best_dist, double *inertia, void *ws, size_t ws_bytes, uint64_t seed, void *stream) {
    (void)seed;
    return run_assign(AssignPath::kBf16x3, X, C, n, k, d, labels, best_dist, inertia, ws, ws_bytes,
                      static_cast<cudaStream_t>(stream));
}

int kmeans_assign_ffma(const float *X, const float *C, int64_t n, int64_t k, int64_t d, int64_t *labels,
                       float *best_dist, double *inertia, void *ws, size_t ws_bytes, uint64_t seed, void *stream) {
    (void)seed;
    return run_assign(AssignPath::kFfma, X, C, n, k, d, labels, best_dist, inertia, ws, ws_bytes,
                      static_cast<cudaStream_t>(stream));
}

int kmeans_assign_3xtf32(const float *X, const float *C, int64_t n, int64_t k, int64_t d, int64_t *labels,
                         float *best_dist, double *inertia, void *ws, size_t ws_bytes, uint64_t seed, void *stream) {
    (void)seed;
    return run_assign(AssignPath::kTf32x3, X, C, n, k, d, labels, best_dist, inertia, ws, ws_bytes,
                      static_cast<cudaStream_t>(stream));
}

int kmeans_update(const float *X, const int64_t *labels, const float *C_old, float *C_new, int32_t *counts,
                  int64_t n, int64_t k, int64_t d, void *ws, size_t ws_bytes, uint64_t seed, void *stream) {
    (void)seed;
    if (!X || !labels || !C_old || !C_new) return KMEANS_ERR_INVALID_ARG;
    if (!sizes_ok(n, k, d)) return KMEANS_ERR_INVALID_ARG;
    if (!aligned4(X) || !aligned4(C_old) || !aligned4(C_new) || (reinterpret_cast<uintptr_t>(labels) & 7u))
        return KMEANS_ERR_INVALID_ARG;
    const UpdateLayout L = update_layout(n, k, d);
    const int wst = check_ws(ws, ws_bytes, (size_t)L.bytes);
    if (wst != KMEANS_OK) return wst;
    return cuda_status(launch_update(X, labels, C_old, C_new, counts, n, k, d, L, static_cast<uint8_t *>(ws), true,
                                     static_cast<cudaStream_t>(stream)));
}

int kmeans_lloyd_iter(const float *X, const float *C_old, float *C_new, int64_t *labels, float *best_dist,
                      double *inertia, int32_t *counts, int64_t n, int64_t k, int64_t d, void *ws, size_t ws_bytes,
                      uint64_t seed, void *stream) {
    (void)seed;
    if (!X || !C_old || !C_new || !labels || !best_dist) return KMEANS_ERR_INVALID_ARG;
    if (!sizes_ok(n, k, d)) return KMEANS_ERR_INVALID_ARG;
    if (!aligned4(C_new) || (reinterpret_cast<uintptr_t>(labels) & 7u)) return KMEANS_ERR_INVALID_ARG;
    const int st = tc_path_ok(X, C_old, d);
    if (st != KMEANS_OK) return st;
    const size_t need = kmeans_workspace_bytes(KMEANS_OP_LLOYD, n, k, d);
    const int wst = check_ws(ws, ws_bytes, need);
    if (wst != KMEANS_OK) return wst;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    const AssignLayout A = assign_layout(n, k, d, true);
    cudaError_t e = launch_prep_split(C_old, n, k, d, A, w, s);
    if (e == cudaSuccess) e = launch_assign_tc(X, n, k, d, A, w, s);
    if (e == cudaSuccess) e = lloyd_finish(X, C_old, C_new, labels, best_dist, inertia, counts, n, k, d, A, w, s);
    return cuda_status(e);
}

int kmeans_lloyd_iter_fused(const float *X, const float *C_old, float *C_new, int64_t *labels, float *best_dist,
                            double *inertia, int32_t *counts, int64_t n, int64_t k, int64_t d, void *ws,
                            size_t ws_bytes, uint64_t seed, void *stream) {
    (void)seed;
    if (!X || !C_old || !C_new || !labels || !best_dist || C_new == C_old) return KMEANS_ERR_INVALID_ARG;
    if (!sizes_ok(n, k, d)) return KMEANS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(labels) & 7u)) return KMEANS_ERR_INVALID_ARG;
    const int st = tc_path_ok(X, C_old, d);
    if (st != KMEANS_OK) return st;
    if (!aligned16(C_new) || d > 4096) return KMEANS_ERR_UNSUPPORTED;
    const FusedLayout F = fused_layout(n, k, d);
    const int wst = check_ws(ws, ws_bytes, (size_t)F.bytes);
    if (wst != KMEANS_OK) return wst;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    FusedUpdate fu;
    fu.X = X;
    fu.sums = reinterpret_cast<float *>(w + F.off_sums);
    fu.counts = reinterpret_cast<int32_t *>(w + F.off_cnt);
    fu.row_done = reinterpret_cast<uint32_t *>(w + F.off_done);
    cudaError_t e = cudaMemsetAsync(w + F.off_sums, 0, (size_t)(F.bytes - F.off_sums), s);
    if (e == cudaSuccess) e = launch_prep_split(C_old, n, k, d, F.A, w, s);
    if (e == cudaSuccess) e = launch_assign_tc(X, n, k, d, F.A, w, s, true, false, &fu);
    if (e == cudaSuccess) e = launch_finalize(n, F.A, w, labels, best_dist, inertia, s);
    if (e == cudaSuccess) e = launch_fused_mean(fu.sums, fu.counts, C_old, C_new, counts, k, d, s);
    return cuda_status(e);
}

int kmeans_lloyd_iter_host(const float *X_host, const float *C_host, float *X, float *C_old, float *C_new,
                           int64_t *labels, float *best_dist, double *inertia, int32_t *counts, float *C_new_host,
                           int64_t *labels_host, double *inertia_host, int64_t n, int64_t k, int64_t d, int slices,
                           int flags, void *ws, size_t ws_bytes, void *stream, void *copy_stream) {
    if (!X_host || !C_host || !X || !C_old || !C_new || !labels || !best_dist) return KMEANS_ERR_INVALID_ARG;
    if (!sizes_ok(n, k, d)) return KMEANS_ERR_INVALID_ARG;
    if (slices < 1 || slices > KMEANS_HOST_MAX_SLICES) return KMEANS_ERR_INVALID_ARG;
    if (flags & ~(KMEANS_HOST_OVERLAP_PREVIOUS | KMEANS_HOST_READBACK_ON_COPY_STREAM)) return KMEANS_ERR_INVALID_ARG;
    if (stream == copy_stream || (inertia_host && !inertia)) return KMEANS_ERR_INVALID_ARG;
    if (!aligned4(C_new) || (reinterpret_cast<uintptr_t>(labels) & 7u)) return KMEANS_ERR_INVALID_ARG;
    const int st = tc_path_ok(X, C_old, d);
    if (st != KMEANS_OK) return st;
    const size_t need = kmeans_workspace_bytes(KMEANS_OP_LLOYD, n, k, d);
    const int wst = check_ws(ws, ws_bytes, need);
    if (wst != KMEANS_OK) return wst;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaStream_t cs = static_cast<cudaStream_t>(copy_stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    // slices of whole 256-sample pair blocks; where the tiles are wide units,
    // of whole rounds of the persistent schedule when that keeps at least
    // half the slices asked for (a part-filled last round in every slice
    // cost about 4% of the step on the sample-heavy shape)
    int64_t per = ((n + slices - 1) / slices + 255) / 256 * 256;
    const int64_t g = assign_round_rows(k, d);
    if (slices > 1 && g > 256) {
        const int64_t per_g = (per + g - 1) / g * g;
        if (2 * ((n + per_g - 1) / per_g) >= slices) per = per_g;
    }
    const int used = (int)((n + per - 1) / per);
    // ev[0 .. used-1]: slice i has landed; ev[used]: the entry point on
    // `stream`; ev[used + 1]: the centroids have landed; ev[used + 2]: the
    // update is done (read-back on the copy stream)
    cudaEvent_t ev[KMEANS_HOST_MAX_SLICES + 3];
    int made = 0;
    cudaError_t e = cudaSuccess;
    for (; made < used + 3 && e == cudaSuccess; ++made) e = cudaEventCreateWithFlags(&ev[made], cudaEventDisableTiming);
    if (e != cudaSuccess) --made;  // the failed one was not created
    // the copies wait for everything enqueued on `stream` before this call,
    // unless the caller vouches that X and C_old are free (then they may
    // overlap the previous call's update); the centroids go first on the
    // copy stream (a copy on `stream` could be scheduled behind all the
    // sample slices and hold back every slice)
    if (!(flags & KMEANS_HOST_OVERLAP_PREVIOUS)) {
        if (e == cudaSuccess) e = cudaEventRecord(ev[used], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[used], 0);
    }
    if (e == cudaSuccess) e = cudaMemcpyAsync(C_old, C_host, (size_t)(k * d) * sizeof(float), cudaMemcpyHostToDevice, cs);
    if (e == cudaSuccess) e = cudaEventRecord(ev[used + 1], cs);
    for (int i = 0; i < used && e == cudaSuccess; ++i) {
        const int64_t r0 = i * per, rows = (r0 + per <= n ? per : n - r0);
        e = cudaMemcpyAsync(X + r0 * d, X_host + r0 * d, (size_t)(rows * d) * sizeof(float), cudaMemcpyHostToDevice, cs);
        if (e == cudaSuccess) e = cudaEventRecord(ev[i], cs);
    }
    // the centroid split once, then each slice's tensor-core pass as soon as
    // its rows have landed, writing that slice's keys and norms
    const AssignLayout A = assign_layout(n, k, d, true);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(s, ev[used + 1], 0);
    if (e == cudaSuccess) e = launch_prep_split(C_old, n, k, d, A, w, s);
    for (int i = 0; i < used && e == cudaSuccess; ++i) {
        const int64_t r0 = i * per, rows = (r0 + per <= n ? per : n - r0);
        e = cudaStreamWaitEvent(s, ev[i], 0);
        AssignLayout Ai = A;
        Ai.off_keys += r0 * 8;
        Ai.off_xnorm += r0 * 4;
        if (e == cudaSuccess) e = launch_assign_tc(X + r0 * d, rows, k, d, Ai, w, s, false);
    }
    if (e == cudaSuccess) e = lloyd_finish(X, C_old, C_new, labels, best_dist, inertia, counts, n, k, d, A, w, s);
    // the read-backs: on `stream`, or on the copy stream once the update is done
    cudaStream_t rs = s;
    if (flags & KMEANS_HOST_READBACK_ON_COPY_STREAM) {
        rs = cs;
        if (e == cudaSuccess) e = cudaEventRecord(ev[used + 2], s);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cs, ev[used + 2], 0);
    }
    if (e == cudaSuccess && C_new_host)
        e = cudaMemcpyAsync(C_new_host, C_new, (size_t)(k * d) * sizeof(float), cudaMemcpyDeviceToHost, rs);
    if (e == cudaSuccess && labels_host)
        e = cudaMemcpyAsync(labels_host, labels, (size_t)n * sizeof(int64_t), cudaMemcpyDeviceToHost, rs);
    if (e == cudaSuccess && inertia_host)
        e = cudaMemcpyAsync(inertia_host, inertia, sizeof(double), cudaMemcpyDeviceToHost, rs);
    // released by the runtime once the work that uses them has completed
    for (int i = 0; i < made; ++i) cudaEventDestroy(ev[i]);
    return cuda_status(e);
}

int kmeans_fit(const float *X, float *C, int64_t *labels, float *best_dist, int32_t *counts, int64_t n, int64_t k,
               int64_t d, int init, uint64_t seed, int max_iter, double tol, int *n_iter, double *inertia_history,
               void *ws, size_t ws_bytes, void *stream) {
    if (!X || !C || !labels || !best_dist || !n_iter) return KMEANS_ERR_INVALID_ARG;
    if (!sizes_ok(n, k, d)) return KMEANS_ERR_INVALID_ARG;
    const bool relocate = (init & KMEANS_FIT_RELOCATE_EMPTY) != 0;
    init &= ~KMEANS_FIT_RELOCATE_EMPTY;
    if (init != KMEANS_INIT_GIVEN && init != KMEANS_INIT_KMEANSPP) return KMEANS_ERR_INVALID_ARG;
    if (relocate && !aligned4(best_dist)) return KMEANS_ERR_INVALID_ARG;
    if (max_iter < 1 || max_iter > 1000000 || !(tol >= 0.0) || tol > 1e300) return KMEANS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(labels) & 7u)) return KMEANS_ERR_INVALID_ARG;
    const int st = tc_path_ok(X, C, d);
    if (st != KMEANS_OK) return st;
    const FitLayout F = fit_layout(n, k, d);
    const int wst = check_ws(ws, ws_bytes, (size_t)F.bytes);
    if (wst != KMEANS_OK) return wst;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    float *calt = reinterpret_cast<float *>(w + F.off_calt);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(w);
    double *inertia_d = &hdr->fit_inertia;
    *n_iter = 0;
    cudaError_t e = cudaSuccess;
    if (init == KMEANS_INIT_KMEANSPP) {
        const int T = default_trials(k);
        if (T > kKppMaxTrials) return KMEANS_ERR_UNSUPPORTED;
        e = launch_kmeanspp(X, n, d, k, T, seed, C, reinterpret_cast<int64_t *>(w + F.off_indices),
                            kpp_layout(n, d, T, k), w, s);
    }
    const AssignLayout A = assign_layout(n, k, d, true);
    const UpdateLayout U = update_layout(n, k, d);
    // with relocation the update's counts show whether a cluster emptied;
    // without caller counts they go to the relocation's count scratch, which
    // the relocation itself rewrites only after they have been read
    int32_t *cnt = counts;
    if (relocate && !cnt) cnt = reinterpret_cast<int32_t *>(w + F.reloc.off_counts);
    uint32_t *nempty_d = &hdr->fit_nempty;
    float *cur = C, *nxt = calt;
    double prev = 0.0;
    int it = 0;
    while (e == cudaSuccess && it < max_iter) {
        e = launch_prep_split(cur, n, k, d, A, w, s);
        if (e == cudaSuccess) e = launch_assign_tc(X, n, k, d, A, w, s);
        if (e == cudaSuccess) e = lloyd_finish(X, cur, nxt, labels, best_dist, inertia_d, cnt, n, k, d, A, w, s);
        if (e == cudaSuccess && relocate) e = launch_count_empty(cnt, k, nempty_d, s);
        // status word, inertia and empty count in one read (each small
        // pageable copy costs a round trip while the GPU waits)
        WsHeader rec{};
        if (e == cudaSuccess) e = cudaMemcpyAsync(&rec, w, kFitRecordBytes, cudaMemcpyDeviceToHost, s);
        if (e == cudaSuccess) e = cudaStreamSynchronize(s);
        if (e != cudaSuccess) break;
        const double inertia = rec.fit_inertia;
        const uint32_t flags = rec.status;
        const uint32_t nempty = relocate ? rec.fit_nempty : 0u;
        ++it;
        *n_iter = it;
        if (flags & kFlagTimeout) return KMEANS_ERR_DEVICE_TIMEOUT;
        if (flags & kFlagBadLabel) return KMEANS_ERR_DEVICE_LABEL;
        if (nempty) {
            // a cluster is empty: move the farthest samples into the empty
            // clusters and redo the update with those labels (every row of
            // nxt is rewritten); an iteration without one pays only the check
            e = launch_relocate(labels, best_dist, n, k, F.reloc, w, s);
            if (e == cudaSuccess) e = launch_update(X, labels, cur, nxt, cnt, n, k, d, U, w, false, s);
            if (e != cudaSuccess) break;
        }
        if (inertia_history) inertia_history[it - 1] = inertia;
        float *t = cur;
        cur = nxt;
        nxt = t;
        // relative improvement over the previous iteration at most tol
        if (it > 1 && inertia >= prev * (1.0 - tol)) break;
        prev = inertia;
    }
    // the last update wrote `cur`; the caller's C must hold it
    if (e == cudaSuccess && cur != C) e = cudaMemcpyAsync(C, cur, (size_t)(k * d) * sizeof(float), cudaMemcpyDeviceToDevice, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    return cuda_status(e);
}

int kmeans_update_partial(const float *X, const int64_t *labels, int64_t n, int64_t k, int64_t d, float *sums,
                          int32_t *counts, void *ws, size_t ws_bytes, uint64_t seed, void *stream) {
    (void)seed;
    if (!X || !labels || !sums || !counts) return KMEANS_ERR_INVALID_ARG;
    if (!shard_sizes_ok(n, k, d)) return KMEANS_ERR_INVALID_ARG;
    if (!aligned4(X) || !aligned4(sums) || !aligned4(counts) || (reinterpret_cast<uintptr_t>(labels) & 7u))
        return KMEANS_ERR_INVALID_ARG;
    const UpdateLayout L = update_layout(n, k, d);
    const int wst = check_ws(ws, ws_bytes, (size_t)L.bytes);
    if (wst != KMEANS_OK) return wst;
    return cuda_status(launch_update(X, labels, nullptr, sums, counts, n, k, d, L, static_cast<uint8_t *>(ws), true,
                                     static_cast<cudaStream_t>(stream), false, true));
}

int kmeans_lloyd_iter_partial(const float *X, const float *C, int64_t *labels, float *best_dist, double *inertia,
                              float *sums, int32_t *counts, int64_t n, int64_t k, int64_t d, void *ws,
                              size_t ws_bytes, uint64_t seed, void *stream) {
    (void)seed;
    if (!X || !C || !labels || !best_dist || !sums || !counts) return KMEANS_ERR_INVALID_ARG;
    if (!shard_sizes_ok(n, k, d)) return KMEANS_ERR_INVALID_ARG;
    if (!aligned4(sums) || !aligned4(counts) || (reinterpret_cast<uintptr_t>(labels) & 7u))
        return KMEANS_ERR_INVALID_ARG;
    const int st = tc_path_ok(X, C, d);
    if (st != KMEANS_OK) return st;
    const int wst = check_ws(ws, ws_bytes, (size_t)lloyd_ws_bytes(n, k, d));
    if (wst != KMEANS_OK) return wst;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    const AssignLayout A = assign_layout(n, k, d, true);
    cudaError_t e = launch_prep_split(C, n, k, d, A, w, s);
    if (e == cudaSuccess) e = launch_assign_tc(X, n, k, d, A, w, s);
    if (e == cudaSuccess) e = lloyd_finish(X, nullptr, sums, labels, best_dist, inertia, counts, n, k, d, A, w, s, true);
    return cuda_status(e);
}

int kmeans_reduce_partials(const float *parts, const int32_t *part_counts, const double *part_inertia, int world,
                           int64_t rows, int64_t d, const float *C_old, float *C_new, int32_t *counts, double *inertia,
                           void *stream) {
    if (world < 1 || world > 65536 || rows < 0 || d < 1 || d > kMaxIndex) return KMEANS_ERR_INVALID_ARG;
    if ((part_inertia == nullptr) != (inertia == nullptr)) return KMEANS_ERR_INVALID_ARG;
    if (rows > 0 && (!parts || !part_counts || !C_old || !C_new)) return KMEANS_ERR_INVALID_ARG;
    if (rows == 0 && !inertia) return KMEANS_OK;
    if (!aligned4(parts) || !aligned4(part_counts) || !aligned4(C_old) || !aligned4(C_new) || !aligned4(counts) ||
        (reinterpret_cast<uintptr_t>(part_inertia) & 7u) || (reinterpret_cast<uintptr_t>(inertia) & 7u))
        return KMEANS_ERR_INVALID_ARG;
    return cuda_status(launch_reduce_partials(parts, part_counts, part_inertia, world, rows, d, C_old, C_new, counts,
                                              inertia, static_cast<cudaStream_t>(stream)));
}

size_t kmeanspp_shard_exchange_bytes(int n_trials, int64_t d) {
    if (n_trials < 1 || n_trials > kKppMaxTrials || d < 1 || d > kMaxIndex) return 0;
    return (size_t)kpp_exchange_bytes(n_trials, d);
}

namespace {
int kpp_shard_check(const float *X, int64_t n, int64_t d, int T, const void *ws, size_t ws_bytes, KppShardLayout &L) {
    if (n < 1 || d < 1 || n > kMaxIndex || d > kMaxIndex) return KMEANS_ERR_INVALID_ARG;
    if (T < 1 || T > kKppMaxTrials) return KMEANS_ERR_INVALID_ARG;
    if (X && !aligned4(X)) return KMEANS_ERR_INVALID_ARG;
    L = kpp_shard_layout(n, d);
    return check_ws(ws, ws_bytes, (size_t)L.bytes);
}
}  // namespace

int kmeanspp_shard_first(const float *X, int64_t n, int64_t d, int64_t row_offset, int64_t n_global, int n_trials,
                         uint64_t seed, void *send, void *ws, size_t ws_bytes, void *stream) {
    if (!X || !send || !aligned16(send)) return KMEANS_ERR_INVALID_ARG;
    if (row_offset < 0 || n_global < 1 || row_offset + n > n_global) return KMEANS_ERR_INVALID_ARG;
    KppShardLayout L;
    const int st = kpp_shard_check(X, n, d, n_trials, ws, ws_bytes, L);
    if (st != KMEANS_OK) return st;
    return cuda_status(launch_kpp_shard_first(X, n, d, row_offset, n_global, n_trials, seed,
                                              static_cast<uint8_t *>(send), static_cast<uint8_t *>(ws),
                                              static_cast<cudaStream_t>(stream)));
}

int kmeanspp_shard_pick(const float *X, int64_t n, int64_t d, int64_t row_offset, int n_trials, uint64_t seed,
                        int64_t c, const double *totals, int world, int rank, void *send, void *ws, size_t ws_bytes,
                        void *stream) {
    if (!X || !totals || !send || !aligned16(send) || (reinterpret_cast<uintptr_t>(totals) & 7u))
        return KMEANS_ERR_INVALID_ARG;
    if (world < 1 || world > 65536 || rank < 0 || rank >= world || c < 1 || row_offset < 0)
        return KMEANS_ERR_INVALID_ARG;
    KppShardLayout L;
    const int st = kpp_shard_check(X, n, d, n_trials, ws, ws_bytes, L);
    if (st != KMEANS_OK) return st;
    return cuda_status(launch_kpp_shard_pick(X, n, d, row_offset, n_trials, seed, c, totals, world, rank,
                                             static_cast<uint8_t *>(send), L, static_cast<uint8_t *>(ws),
                                             static_cast<cudaStream_t>(stream)));
}

int kmeanspp_shard_dist(const float *X, int64_t n, int64_t d, int n_trials, int first, const void *recv, int world,
                        double *pot, void *ws, size_t ws_bytes, void *stream) {
    if (!X || !recv || !aligned16(recv) || (!first && !pot) || (reinterpret_cast<uintptr_t>(pot) & 7u))
        return KMEANS_ERR_INVALID_ARG;
    if (world < 1 || world > 65536 || (first != 0 && first != 1)) return KMEANS_ERR_INVALID_ARG;
    KppShardLayout L;
    const int st = kpp_shard_check(X, n, d, n_trials, ws, ws_bytes, L);
    if (st != KMEANS_OK) return st;
    return cuda_status(launch_kpp_shard_dist(X, n, d, n_trials, first != 0, static_cast<const uint8_t *>(recv), world,
                                             pot, L, static_cast<uint8_t *>(ws), static_cast<cudaStream_t>(stream)));
}

int kmeanspp_shard_commit(int64_t n, int64_t d, int n_trials, int first, const double *pots, int world, int64_t c,
                          int64_t *indices, float *centers, double *total, void *ws, size_t ws_bytes, void *stream) {
    if (!indices || (!first && !pots) || (first != 0 && first != 1) || c < 0 || (first && c != 0))
        return KMEANS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(indices) & 7u) || (reinterpret_cast<uintptr_t>(pots) & 7u) ||
        (reinterpret_cast<uintptr_t>(total) & 7u) || (centers && !aligned4(centers)))
        return KMEANS_ERR_INVALID_ARG;
    if (world < 1 || world > 65536) return KMEANS_ERR_INVALID_ARG;
    KppShardLayout L;
    const int st = kpp_shard_check(nullptr, n, d, n_trials, ws, ws_bytes, L);
    if (st != KMEANS_OK) return st;
    return cuda_status(launch_kpp_shard_commit(n, d, n_trials, first != 0, pots, world, c, indices, centers, total, L,
                                               static_cast<uint8_t *>(ws), static_cast<cudaStream_t>(stream)));
}

int kmeans_relocate_empty(int64_t *labels, const float *best_dist, int64_t n, int64_t k, void *ws, size_t ws_bytes,
                          void *stream) {
    if (!labels || !best_dist) return KMEANS_ERR_INVALID_ARG;
    if (!sizes_ok(n, k, 1)) return KMEANS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(labels) & 7u) || !aligned4(best_dist)) return KMEANS_ERR_INVALID_ARG;
    const RelocLayout R = reloc_layout(k, sizeof(WsHeader));
    const int wst = check_ws(ws, ws_bytes, (size_t)R.end);
    if (wst != KMEANS_OK) return wst;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *w = static_cast<uint8_t *>(ws);
    cudaError_t e = cudaMemsetAsync(w, 0, sizeof(WsHeader), s);  // this call's status word
    if (e == cudaSuccess) e = launch_relocate(labels, best_dist, n, k, R, w, s);
    return cuda_status(e);
}

int kmeanspp_init(const float *X, int64_t n, int64_t d, int64_t k, int n_trials, uint64_t seed, float *centers,
                  int64_t *indices, void *ws, size_t ws_bytes, void *stream) {
    if (!X || !indices) return KMEANS_ERR_INVALID_ARG;
    if (!sizes_ok(n, k, d)) return KMEANS_ERR_INVALID_ARG;
    if (!aligned4(X) || (centers && !aligned4(centers)) || (reinterpret_cast<uintptr_t>(indices) & 7u))
        return KMEANS_ERR_INVALID_ARG;
    const int T = n_trials > 0 ? n_trials : default_trials(k);
    if (T > kKppMaxTrials) return KMEANS_ERR_UNSUPPORTED;
    const KppLayout L = kpp_layout(n, d, T, k);
    const int wst = check_ws(ws, ws_bytes, (size_t)L.bytes);
    if (wst != KMEANS_OK) return wst;
    return cuda_status(launch_kmeanspp(X, n, d, k, T, seed, centers, indices, L, static_cast<uint8_t *>(ws),
                                       static_cast<cudaStream_t>(stream)));
}

int kmeanspp_rows_read(const void *ws, void *stream, int64_t *rows) {
    if (ws == nullptr || rows == nullptr) return KMEANS_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KMEANS_ERR_CUDA;
    unsigned long long v = 0;
    if (cudaMemcpy(&v, static_cast<const uint8_t *>(ws) + offsetof(WsHeader, kpp_rows), sizeof(v),
                   cudaMemcpyDeviceToHost) != cudaSuccess)
        return KMEANS_ERR_CUDA;
    *rows = (int64_t)v;
    return KMEANS_OK;
}

int kmeans_device_status(const void *ws, void *stream) {
    if (ws == nullptr) return KMEANS_ERR_INVALID_ARG;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return KMEANS_ERR_CUDA;
    uint32_t st = 0;
    if (cudaMemcpy(&st, ws, sizeof(st), cudaMemcpyDeviceToHost) != cudaSuccess) return KMEANS_ERR_CUDA;
    if (st & kFlagTimeout) return KMEANS_ERR_DEVICE_TIMEOUT;
    if (st & kFlagBadLabel) return KMEANS_ERR_DEVICE_LABEL;
    if (st & kFlagExchange) return KMEANS_ERR_DEVICE_EXCHANGE;
    return KMEANS_OK;
}

const char *kmeans_status_string(int status) {
    switch (status) {
        case KMEANS_OK: return "ok";
        case KMEANS_ERR_INVALID_ARG: return "invalid argument";
        case KMEANS_ERR_UNSUPPORTED: return "unsupported by this build (see the header's requirements)";
        case KMEANS_ERR_WORKSPACE: return "workspace too small or not 256-byte aligned";
        case KMEANS_ERR_CUDA: return "CUDA runtime error";
        case KMEANS_ERR_DEVICE_TIMEOUT: return "a device pipeline wait ran out of time";
        case KMEANS_ERR_DEVICE_LABEL: return "a label outside [0, k) reached the update";
        case KMEANS_ERR_SCRATCH_LIMIT:
            return "problem too large for the built-in scratch of kmeans_assign_noalloc "
                   "(use kmeans_assign with a workspace)";
        case KMEANS_ERR_DEVICE_EXCHANGE: return "sharded k-means++: no rank's exchange block held a trial's candidate";
        default: return "unknown status";
    }
}

const char *kmeans_build_info(void) {
    return "kmeans_gb300 sm_103a: assign = tcgen05 cta_group::2 CTA pairs, bf16x3 split, BK 32, 8 split warps; "
           "d >= 2048 with k > 256: 256x512 wide units (one f32 accumulator per 256-column tile, X/C ring 3, "
           "split ring 5), K chunks of <= 8192 features above d = 8192, a soft barrier at each round start "
           "from 16 rounds; otherwise 256x256 tiles (one double-buffered accumulator up to d = 4096, separate "
           "hi.hi and correction accumulators above; X/C ring 4, split ring 6); comparator = FFMA 128x128; "
           "update = counting-scatter member list (k <= 32768; LSD radix above) + compensated segmented mean; "
           "sharded update = per-rank sums reduced in rank order; k-means++ = Philox4x32-10 greedy D^2 with "
           "triangle-inequality row pruning (single GPU; sharded steps without)";
}

}  // extern "C"

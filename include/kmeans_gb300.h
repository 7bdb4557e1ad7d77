/*
 * kmeans_gb300.h -- C ABI of the GB300 (sm_103a) k-means library.
 *
 * The library computes one Lloyd iteration of k-means and greedy k-means++
 * seeding on one GPU.  Every entry point takes caller-owned DEVICE pointers,
 * the sizes n (samples), k (centroids), d (features), a caller-owned device
 * workspace, a seed and a CUDA stream, enqueues its kernels on that stream and
 * returns without synchronising.  The library allocates no memory.
 *
 * Sources for what is computed (three pages of one benchmarking journal):
 *  [G] "Three shapes that fit an eager Gram assignment", section "Gram
 *      assignment": nearest centroid = argmin_c ||x - c||^2, evaluated through
 *      ||x||^2 + ||c||^2 - 2 x.c.
 *  [R] same page, section "Running argmin, one centroid": the assignment
 *      result is an int64 label and a float32 winning distance per sample
 *      (n * 12 bytes); no (n, k) distance matrix is ever stored.
 *  [U] same page, section "Full Lloyd step": each centroid becomes the mean of
 *      its members.
 *  [S] "004 — tile sizes, a Cython Lloyd step, and k-means++", section
 *      "Schedules added": ||x||^2 does not change the argmin and is left out of
 *      the comparison; ||c||^2 is computed once per centroid and reused.
 *  [K] same page, section "k-means++": greedy D^2 seeding with
 *      2 + log(n_clusters) candidate trials per new center.
 *  [L] same page, section "Cython timing": the Lloyd step measured there
 *      also relocates empty clusters (the page gives no rule).
 *
 * Conventions shared by every entry point
 *  - Layout: X is (n, d) float32 row-major, C is (k, d) float32 row-major,
 *    both contiguous.  labels are int64 (n), distances float32 (n).
 *  - Sizes: 1 <= k <= n, d >= 1, n < 2^31, k < 2^31.
 *  - Precision: inputs must be finite.  The assignment contraction runs on the
 *    tensor cores as three bf16 products of an error-compensated split of
 *    each float32 operand (hi = bf16(v), lo = bf16(v - hi)) with float32
 *    accumulation.  The three products share one accumulator per tile, over
 *    chunks of at most 8192 features whose sums are added in float32 (the
 *    error of the float32 tensor-core accumulation grows about linearly with
 *    the features an accumulator covers).  Where that does not apply (above
 *    4096 features with k <= 256, above 8192 in the built-in scratch of
 *    kmeans_assign_noalloc, and the 3xTF32 comparator above 2048) the two
 *    correction products keep an accumulator of their own, about three times
 *    more accurate than one shared over the same features.  The reported
 *    distance is within 1e-4 * (||x||^2 + ||c||^2) of the exact one (tested
 *    up to d = 24576 in chunks, whose error stays that of one 8192-feature
 *    chunk; up to about 16384 with separate accumulators).  Ties between
 *    centroids go to the lowest index.
 *  - Workspace: `ws` is a device buffer of at least
 *    kmeans_workspace_bytes(op, n, k, d) bytes, 256-byte aligned, owned by the
 *    caller.  Its size has no n*k term: no (n, k) buffer exists anywhere.
 *    One workspace must not be used by two calls that may run concurrently.
 *  - Errors: the return value reports argument validation
 *    (KMEANS_ERR_INVALID_ARG, KMEANS_ERR_UNSUPPORTED, KMEANS_ERR_WORKSPACE)
 *    and launch failures (KMEANS_ERR_CUDA).  Nothing is enqueued when a call
 *    returns an error.  Faults found on the device (a pipeline wait that ran
 *    out of time, a label outside [0, k)) are recorded in a status word in
 *    the workspace, which each call clears when it starts; read it with
 *    kmeans_device_status().
 *  - Streams: `stream` is a cudaStream_t passed as void* (NULL = legacy
 *    default stream).  A call may be captured into a CUDA graph and
 *    replayed (each replay redoes the whole call), except kmeans_fit, which
 *    synchronises, and the first kmeans_assign_noalloc call on a device.
 *    Make one ordinary call on the device before capturing, so that the
 *    one-time per-device set-up has run.
 */
#ifndef KMEANS_GB300_H
#define KMEANS_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    KMEANS_OK = 0,
    KMEANS_ERR_INVALID_ARG = 1,     /* null pointer, bad size, k > n, ...       */
    KMEANS_ERR_UNSUPPORTED = 2,     /* valid but outside this build's limits     */
    KMEANS_ERR_WORKSPACE = 3,       /* ws too small or misaligned                */
    KMEANS_ERR_CUDA = 4,            /* a CUDA runtime call failed                */
    KMEANS_ERR_DEVICE_TIMEOUT = 5,  /* a device pipeline wait ran out of time    */
    KMEANS_ERR_DEVICE_LABEL = 6,    /* kmeans_update saw a label outside [0, k)  */
    KMEANS_ERR_SCRATCH_LIMIT = 7,   /* kmeans_assign_noalloc: the problem needs more
                                       than KMEANS_NOALLOC_SCRATCH_BYTES of scratch */
    KMEANS_ERR_DEVICE_EXCHANGE = 8  /* kmeanspp_shard_dist: no rank's exchange block
                                       held a trial's candidate */
} kmeans_status;

/* Operation codes for kmeans_workspace_bytes. */
enum {
    KMEANS_OP_ASSIGN = 0,
    KMEANS_OP_ASSIGN_FFMA = 1,
    KMEANS_OP_UPDATE = 2,
    KMEANS_OP_LLOYD = 3,
    KMEANS_OP_KMEANSPP = 4,
    KMEANS_OP_FIT = 5,
    KMEANS_OP_ASSIGN_3XTF32 = 6,
    KMEANS_OP_LLOYD_FUSED = 7,
    KMEANS_OP_RELOCATE = 8,
    KMEANS_OP_KMEANSPP_SHARD = 9,  /* n = the shard's samples                   */
    KMEANS_OP_LLOYD_PARTIAL = 10,  /* kmeans_lloyd_iter_partial (k may exceed n) */
    KMEANS_OP_UPDATE_PARTIAL = 11  /* kmeans_update_partial (k may exceed n)     */
};

/* Initialisation of kmeans_fit. */
enum {
    KMEANS_INIT_GIVEN = 0,    /* start from the centroids in C            */
    KMEANS_INIT_KMEANSPP = 1  /* greedy k-means++ seeding (kmeanspp_init) */
};

/* Options of kmeans_fit, or-ed into its `init` argument. */
enum {
    KMEANS_FIT_RELOCATE_EMPTY = 0x100  /* kmeans_relocate_empty before each update */
};

/* Bytes of device workspace the operation needs for these sizes (0 when the
 * sizes are invalid).  Linear in n, in k*d and in n/4096; never in n*k.  The
 * tensor-core assignment adds a constant 10 MiB (40 parked 256 x 256 float32
 * tile halves) once the problem has more than 64 tiles of 256 x 256. */
size_t kmeans_workspace_bytes(int op, int64_t n, int64_t k, int64_t d);

/* Assignment [G][R][S].
 * For every sample i: labels[i] = the lowest j minimising ||x_i - c_j||^2,
 * best_dist[i] = max(0, ||x_i||^2 + ||c_j||^2 - 2 x_i.c_j) for that j, and
 * *inertia = sum_i best_dist[i] accumulated in float64 in a fixed order.
 * X, C: inputs (device).  labels, best_dist: outputs (device).
 * inertia: output (device, one double), may be NULL.
 * Extra requirement of this tensor-core path: d % 4 == 0 and X, C 16-byte
 * aligned (KMEANS_ERR_UNSUPPORTED otherwise; kmeans_assign_ffma has none).
 * Schedule: pairs of SMs work through 256 x 256 tiles of (samples,
 * centroids), or 256 x 512 units of two such tiles for d >= 2048 with
 * k > 256, in rounds; above 8192 features a unit runs its features in
 * chunks of at most 8192, adding each chunk's sums into a running sum kept
 * in the workspace.  When the last round of single tiles is at most half
 * full (d <= 4096), each of its tiles is computed as two halves of the
 * features on two pairs and the halves' sums are added at the end.  Those
 * tiles' distances carry a different (no larger) float32 accumulation error
 * than a single pass would, within the accuracy stated above; the results
 * are the same from run to run on a given GPU.
 * seed: unused (kept for a uniform signature). */
int kmeans_assign(const float *X, const float *C, int64_t n, int64_t k, int64_t d,
                  int64_t *labels, float *best_dist, double *inertia,
                  void *ws, size_t ws_bytes, uint64_t seed, void *stream);

/* The same assignment [G][R][S] computed with plain float32 FMA on the CUDA
 * cores (register-blocked tiles, the argmin fused into the same kernel).  It
 * exists to be measured against kmeans_assign; any d and any 4-byte alignment
 * are accepted. */
int kmeans_assign_ffma(const float *X, const float *C, int64_t n, int64_t k, int64_t d,
                       int64_t *labels, float *best_dist, double *inertia,
                       void *ws, size_t ws_bytes, uint64_t seed, void *stream);

/* The same assignment [G][R][S] on the tensor cores with the 3xTF32 split
 * instead of bf16x3 (a comparator of the operand split; the pages run
 * float32 with TF32 off): hi = v with its low 13 mantissa bits cleared, lo =
 * (v - hi) with its low 13 bits cleared, x.c = hi.hi + lo.hi + hi.lo from
 * kind::tf32 MMAs.  TF32 runs at half the bf16 rate, so about half the
 * throughput; and an MMA covers 8 features instead of 16, so the float32
 * accumulator takes twice the truncating adds: the operands are more exact
 * but the distances less (one accumulator up to d = 2048, separate ones
 * above; the 1e-4 bound holds for d up to about 8192).
 * Same requirements as kmeans_assign; workspace KMEANS_OP_ASSIGN_3XTF32. */
int kmeans_assign_3xtf32(const float *X, const float *C, int64_t n, int64_t k, int64_t d,
                         int64_t *labels, float *best_dist, double *inertia,
                         void *ws, size_t ws_bytes, uint64_t seed, void *stream);

/* Mean update [U].
 * C_new[j] = mean of the rows X[i] with labels[i] == j, summed in float32 with
 * compensation in a fixed order (bitwise reproducible run to run); a cluster
 * with no members keeps C_old[j] bit for bit.  counts (device int32, k) may
 * be NULL; it receives the member counts.  C_new may alias C_old.
 * labels must lie in [0, k); a label outside that range leaves C_new
 * unspecified and sets KMEANS_ERR_DEVICE_LABEL in the status word.
 * seed: unused. */
int kmeans_update(const float *X, const int64_t *labels, const float *C_old, float *C_new,
                  int32_t *counts, int64_t n, int64_t k, int64_t d,
                  void *ws, size_t ws_bytes, uint64_t seed, void *stream);

/* One Lloyd iteration [U]: kmeans_assign of X against C_old, then
 * kmeans_update into C_new with those labels.  labels, best_dist and
 * *inertia (device, may be NULL) receive the assignment; counts (device,
 * may be NULL) the member counts.  C_new must not alias C_old.
 * Same requirements as kmeans_assign. */
int kmeans_lloyd_iter(const float *X, const float *C_old, float *C_new, int64_t *labels,
                      float *best_dist, double *inertia, int32_t *counts,
                      int64_t n, int64_t k, int64_t d,
                      void *ws, size_t ws_bytes, uint64_t seed, void *stream);

/* One Lloyd iteration [U] with the update fused into the assignment (an
 * opt-in variant of kmeans_lloyd_iter; the pages have no counterpart).  As
 * soon as every centroid tile has merged its minimum into a group of 32
 * samples, the epilogue warp that merged last adds those samples' rows
 * (still in L2) into their clusters' sums with float atomics; a last pass
 * divides.  No sorted member list and no second pass over X in HBM.
 * Labels, best_dist and *inertia are kmeans_lloyd_iter's bit for bit, except
 * where kmeans_lloyd_iter computes a tile as two K halves (see kmeans_assign):
 * there best_dist and *inertia differ within the distance accuracy (labels
 * only at ties that close).  C_new differs: the sums are plain float32 in an order that varies from run
 * to run (not reproducible bit for bit), so a cluster of m members carries a
 * relative error up to about m * 2^-24 (within 1e-5 up to some 150 members
 * per cluster); empty clusters keep C_old bit for bit.  counts (may be NULL)
 * are exact.  Same requirements as kmeans_lloyd_iter plus d <= 4096 and
 * C_new 16-byte aligned (KMEANS_ERR_UNSUPPORTED otherwise); C_new must not
 * alias C_old; workspace KMEANS_OP_LLOYD_FUSED. */
int kmeans_lloyd_iter_fused(const float *X, const float *C_old, float *C_new, int64_t *labels,
                            float *best_dist, double *inertia, int32_t *counts,
                            int64_t n, int64_t k, int64_t d,
                            void *ws, size_t ws_bytes, uint64_t seed, void *stream);

/* Most slices kmeans_lloyd_iter_host splits the samples into. */
#define KMEANS_HOST_MAX_SLICES 64

/* kmeans_lloyd_iter_host flag: the copies into X and C_old do not wait for the
 * work enqueued on `stream` before the call, so they overlap the previous
 * iteration's update and read-back.  The caller guarantees that no earlier
 * unfinished work still uses X or C_old, for example by alternating two sets
 * of device buffers between successive calls. */
#define KMEANS_HOST_OVERLAP_PREVIOUS 1

/* kmeans_lloyd_iter_host flag: the copies to C_new_host, labels_host and
 * *inertia_host run on `copy_stream` once the update is done, instead of on
 * `stream`, so that `stream` can go on to the next iteration while they run.
 * The call's work is then complete when `copy_stream` (not `stream`) reaches
 * the point after it.  The caller leaves C_new, labels and inertia unchanged
 * until then, for example by alternating two sets of device buffers and two
 * copy streams between successive calls. */
#define KMEANS_HOST_READBACK_ON_COPY_STREAM 2

/* One Lloyd iteration [U] on inputs that live in host memory (the pages have
 * no counterpart: it serves callers whose data is not resident on the GPU).
 * X_host (n, d) and C_host (k, d) are host arrays, page-locked for the copies
 * to overlap; X and C_old are the device arrays they are copied into (and
 * then hold).  The samples travel in `slices` row slices (1 <= slices <=
 * KMEANS_HOST_MAX_SLICES, each a whole number of 256-sample blocks; where
 * the assignment runs wide units, of whole rounds of its schedule when that
 * keeps at least half as many slices) on `copy_stream`; on `stream` the centroids are copied and split once, and
 * each slice's tensor-core pass starts as soon as its rows have landed, so
 * the copies and the assignment overlap.  Finalize and the mean update then
 * run on `stream` exactly as in kmeans_lloyd_iter.  With slices = 1 the
 * outputs (C_new, labels, best_dist, *inertia, counts) are kmeans_lloyd_iter's
 * bit for bit; with more, each slice's pass may compute other tiles as two K
 * halves than the single call does (see kmeans_assign), so best_dist and
 * *inertia may differ within the distance accuracy (and labels, C_new and
 * counts only at ties that close).  Finally
 * C_new, the labels and *inertia are copied to C_new_host, labels_host and
 * *inertia_host (each may be NULL; inertia_host needs inertia).
 * The copies into X wait for the work enqueued on `stream` before the call
 * (without KMEANS_HOST_OVERLAP_PREVIOUS in flags) or not (with it, see
 * there); everything the call enqueues is complete when `stream` reaches the
 * point after it (the copy stream's part is joined back into `stream`),
 * unless flags has KMEANS_HOST_READBACK_ON_COPY_STREAM (see there).
 * copy_stream must differ from stream.  Same requirements as
 * kmeans_lloyd_iter; the workspace is the KMEANS_OP_LLOYD one. */
int kmeans_lloyd_iter_host(const float *X_host, const float *C_host, float *X, float *C_old, float *C_new,
                           int64_t *labels, float *best_dist, double *inertia, int32_t *counts,
                           float *C_new_host, int64_t *labels_host, double *inertia_host,
                           int64_t n, int64_t k, int64_t d, int slices, int flags,
                           void *ws, size_t ws_bytes, void *stream, void *copy_stream);

/* ---------------------------------------------------------------------------
 * Samples split by rows across GPUs (one process per GPU).  The update [U]
 * needs every member of a cluster, so the shards' unnormalised sums and
 * counts are combined before the divide; the collectives are the caller's
 * (e.g. NCCL through torch.distributed) and only move bytes, while every
 * addition across ranks happens in the library in rank order, so the result
 * does not depend on how the collective is scheduled.  One iteration:
 *   1. each rank: kmeans_lloyd_iter_partial on its rows (or, when the shard
 *      has at least k samples, kmeans_assign + kmeans_update_partial) ->
 *      sums (k, d), counts (k), its inertia;
 *   2. all-to-all: rank q receives every rank's rows [q*m, q*m + m) of the
 *      sums and counts (m = ceil(k / world), zero rows past k);
 *   3. each rank: kmeans_reduce_partials on its slice -> C_new rows, counts;
 *   4. all-gather of the C_new slices (and counts) -> C_new on every rank.
 * --------------------------------------------------------------------------- */

/* The mean update's sums [U] over one shard of the samples: sums[j] = the
 * sum of the rows X[i] with labels[i] == j (compensated float32 in a fixed
 * order, as kmeans_update sums before it divides), zeros for a cluster with
 * no member here; counts[j] (required) the member count.  X (n, d) and
 * labels (n) are this shard's; k is the global number of centroids (it may
 * exceed n).  Workspace KMEANS_OP_UPDATE_PARTIAL; requirements and label
 * checking as kmeans_update.  seed: unused. */
int kmeans_update_partial(const float *X, const int64_t *labels, int64_t n, int64_t k, int64_t d,
                          float *sums, int32_t *counts,
                          void *ws, size_t ws_bytes, uint64_t seed, void *stream);

/* One shard's part of a Lloyd iteration [U]: kmeans_assign of the shard's X
 * (n, d) against C (k, d, all centroids), then kmeans_update_partial of
 * those labels.  labels, best_dist, *inertia (the shard's, may be NULL) as
 * kmeans_assign; sums (k, d) and counts (k, required) as
 * kmeans_update_partial.  Requirements as kmeans_lloyd_iter, except that k
 * may exceed the shard's n; workspace KMEANS_OP_LLOYD_PARTIAL.  seed: unused. */
int kmeans_lloyd_iter_partial(const float *X, const float *C, int64_t *labels, float *best_dist,
                              double *inertia, float *sums, int32_t *counts,
                              int64_t n, int64_t k, int64_t d,
                              void *ws, size_t ws_bytes, uint64_t seed, void *stream);

/* The divide of the sharded update [U] for `rows` centroid rows.
 * parts (world, rows, d) float32 and part_counts (world, rows) int32 hold
 * every rank's sums and counts of those rows, rank-major.  For each row j:
 * count = sum over ranks of part_counts[r][j]; if count > 0, C_new[j] =
 * (sum over r of parts[r][j], added in rank order in float64, the first
 * rank's value as it is) / count, rounded once to float32; otherwise
 * C_new[j] = C_old[j].  With world = 1 this gives kmeans_update's bits.
 * counts (rows, may be NULL) receives the summed counts (the global count
 * of a cluster must be below 2^31).  part_inertia (world doubles) and
 * inertia (one double) are both NULL or both given: *inertia = the rank-order
 * sum of part_inertia.  C_new may alias C_old.  rows >= 0, 1 <= world <= 65536,
 * d >= 1.  One kernel, no workspace. */
int kmeans_reduce_partials(const float *parts, const int32_t *part_counts, const double *part_inertia,
                           int world, int64_t rows, int64_t d, const float *C_old, float *C_new,
                           int32_t *counts, double *inertia, void *stream);

/* Greedy k-means++ [K] over samples split by rows across ranks: the same
 * seeding as kmeanspp_init over the concatenated shards (rank order), as a
 * sequence of steps between which the caller all-gathers small buffers.
 * Rank r holds rows [row_offset, row_offset + n) of the n_global samples
 * (n >= 1; the offsets are the shards' sizes summed in rank order).
 * Exchange block: kmeanspp_shard_exchange_bytes(n_trials, d) bytes per rank
 * (16-byte aligned device memory): n_trials int64 global sample indices
 * (-1: not this rank's), then n_trials rows of d float32.
 * Workspace KMEANS_OP_KMEANSPP_SHARD with n = this shard's samples; it holds
 * the shard's D^2 between the steps, and its status word collects device
 * faults over the whole seeding (cleared by kmeanspp_shard_first).
 *   kmeanspp_shard_first   draw 0 picks the first center (uniform over
 *                          n_global); its owner fills slot 0 of `send`.
 *   (all-gather `send` of every rank -> recv, world blocks, rank order)
 *   kmeanspp_shard_dist    first = 1: distances to that center.
 *   kmeanspp_shard_commit  first = 1, c = 0: indices[0], centers[0], D^2,
 *                          and this shard's total of D^2 -> *total.
 *   (all-gather the totals -> world doubles, rank order)
 *   for c = 1 .. k-1:
 *     kmeanspp_shard_pick   draws 1 + (c-1)*n_trials + t: each trial's
 *                           target = u * (sum of the totals, rank order);
 *                           its owner is the first rank whose running total
 *                           exceeds it (the last rank's last sample when none
 *                           does), which finds the sample by its running sum
 *                           started at the earlier ranks' total and fills
 *                           the trial's slot of `send`.
 *     (all-gather `send`)
 *     kmeanspp_shard_dist   first = 0: distances to the n_trials candidates
 *                           and this shard's potentials -> pot (n_trials
 *                           doubles, device).
 *     (all-gather pot -> world x n_trials doubles)
 *     kmeanspp_shard_commit first = 0: the trial with the lowest potential
 *                           summed over ranks in rank order (lowest trial on
 *                           ties) becomes center c: indices[c] (device int64,
 *                           k), centers[c] (device float32 (k, d), may be
 *                           NULL), D^2 lowered; *total for the next draws
 *                           (total may be NULL after the last center).
 *     (all-gather the totals)
 * Every rank ends with the same indices and centers.  With world = 1 the
 * indices are kmeanspp_init's bit for bit.  Distances and sums as
 * kmeanspp_init.  kmeanspp_shard_dist sets KMEANS_ERR_DEVICE_EXCHANGE in the
 * status word if no block held a trial's candidate (inconsistent inputs).
 * n_trials: 1 .. 32 (use 2 + floor(ln k) for kmeanspp_init's default). */
size_t kmeanspp_shard_exchange_bytes(int n_trials, int64_t d);
int kmeanspp_shard_first(const float *X, int64_t n, int64_t d, int64_t row_offset, int64_t n_global,
                         int n_trials, uint64_t seed, void *send, void *ws, size_t ws_bytes, void *stream);
int kmeanspp_shard_pick(const float *X, int64_t n, int64_t d, int64_t row_offset, int n_trials, uint64_t seed,
                        int64_t c, const double *totals, int world, int rank, void *send,
                        void *ws, size_t ws_bytes, void *stream);
int kmeanspp_shard_dist(const float *X, int64_t n, int64_t d, int n_trials, int first, const void *recv,
                        int world, double *pot, void *ws, size_t ws_bytes, void *stream);
int kmeanspp_shard_commit(int64_t n, int64_t d, int n_trials, int first, const double *pots, int world,
                          int64_t c, int64_t *indices, float *centers, double *total,
                          void *ws, size_t ws_bytes, void *stream);

/* Empty-cluster relocation [L] (the rule is this library's reading; the
 * page names the step only).  With m clusters that no label names, the m
 * samples with the largest best_dist (equal distances: the lower sample
 * index first) are moved: taken in increasing sample index, their labels
 * become the empty clusters taken in increasing cluster index.  A cluster
 * whose every member moves is empty afterwards (kmeans_update then keeps
 * its centroid).  Nothing changes when no cluster is empty.
 * labels (device int64, n): in/out, values in [0, k).  best_dist (device
 * float32, n): each sample's squared distance to its assigned centroid, as
 * kmeans_assign writes it (no NaN; -0 counts as 0); read only.
 * A label outside [0, k) leaves every label as it was and sets
 * KMEANS_ERR_DEVICE_LABEL in the status word.  Cost: a counting pass over
 * the labels, then, only while a cluster is empty, six passes over best_dist
 * by one thread block.  Workspace KMEANS_OP_RELOCATE (d is ignored). */
int kmeans_relocate_empty(int64_t *labels, const float *best_dist, int64_t n, int64_t k,
                          void *ws, size_t ws_bytes, void *stream);

/* Greedy k-means++ seeding [K].
 * indices (device int64, k) receives the chosen sample indices, centers
 * (device float32 (k, d), may be NULL) the chosen rows of X.
 * n_trials <= 0 selects 2 + floor(ln k).  The draws come from Philox4x32-10
 * (Salmon et al., SC'11) keyed by `seed`: counter (draw, 0, 0, 0), uniform =
 * top 53 bits of the first two output words; draw 0 picks the first center
 * uniformly, draw 1 + (c-1)*n_trials + t is trial t of center c.  A trial
 * takes the first sample whose running sum of D^2 exceeds uniform * sum(D^2)
 * (the last sample if none does); the trial with the lowest potential
 * sum_i min(D^2_i, ||x_i - cand||^2) wins (lowest trial on ties).
 * Distances are float32 differences, squared and summed in float32 over
 * runs of at most 8 x 16 features per thread, the runs combined in
 * double-float; running sums and potentials are float64.
 * Rows that cannot change: each round skips the samples that every trial
 * provably leaves at their D^2 (by the triangle inequality through the
 * sample's nearest chosen center, with a 0.1% margin on the distance), so
 * the indices are those of the unpruned seeding while fewer rows of X are
 * read.  The workspace holds the bookkeeping for n <= 16,777,216; beyond
 * that every round reads every row. */
int kmeanspp_init(const float *X, int64_t n, int64_t d, int64_t k, int n_trials,
                  uint64_t seed, float *centers, int64_t *indices,
                  void *ws, size_t ws_bytes, void *stream);

/* Support for measurement (the pages have no counterpart): the rows of X
 * that the distance passes of the last kmeanspp_init (or kmeans_fit's
 * seeding) on `ws` read, summed over its passes: n for the first center,
 * then the rows each round could not skip, times the passes of a round
 * (ceil(n_trials / 8)).  0 when that seeding read every row (no pruning).
 * Synchronises `stream` first; *rows is host memory.  Returns
 * KMEANS_ERR_INVALID_ARG for a null ws or rows, KMEANS_ERR_CUDA when the
 * synchronisation or the copy fails. */
int kmeanspp_rows_read(const void *ws, void *stream, int64_t *rows);

/* A full fit: Lloyd iterations [U] until the inertia stops improving (the
 * pages fix no stopping rule; this is the plain one).  With
 * init == KMEANS_INIT_KMEANSPP, C is first seeded by kmeanspp_init with the
 * default trial count and `seed`; with KMEANS_INIT_GIVEN, C holds the
 * starting centroids.  With KMEANS_FIT_RELOCATE_EMPTY or-ed into init, the
 * labels of every iteration pass through kmeans_relocate_empty before the
 * update (best_dist and the inertia stay the assignment's); without it an
 * empty cluster keeps its centroid.  (The fit checks the update's counts for
 * an empty cluster, and only then relocates and updates again: an iteration
 * that empties no cluster pays one small kernel.)
 * Iteration t assigns X to C_t (inertia_t) and updates
 * to C_{t+1}; the fit stops after iteration t when
 * inertia_t >= (1 - tol) * inertia_{t-1} (relative improvement at most tol;
 * tol = 0 runs to a fixed point, where the inertia no longer drops), or after
 * max_iter iterations.  On return C holds the last updated centroids, labels,
 * best_dist and counts those of the last iteration (its assignment was to the
 * centroids before that update; at a fixed point they agree).
 * *n_iter (host) receives the iterations run and inertia_history (host,
 * max_iter doubles, may be NULL) each iteration's inertia.  Unlike the other
 * entry points this one synchronises `stream` once per iteration to read the
 * inertia; device faults end the fit with their status.  counts may be NULL.
 * Requirements as kmeans_lloyd_iter (C 16-byte aligned); 1 <= max_iter <=
 * 1000000, tol >= 0; workspace KMEANS_OP_FIT. */
int kmeans_fit(const float *X, float *C, int64_t *labels, float *best_dist, int32_t *counts,
               int64_t n, int64_t k, int64_t d, int init, uint64_t seed, int max_iter, double tol,
               int *n_iter, double *inertia_history, void *ws, size_t ws_bytes, void *stream);

/* Synchronises `stream` and returns the device status word of the last call
 * that used `ws` (KMEANS_OK, KMEANS_ERR_DEVICE_TIMEOUT or
 * KMEANS_ERR_DEVICE_LABEL), or KMEANS_ERR_CUDA if the stream reports an error. */
int kmeans_device_status(const void *ws, void *stream);

/* Human-readable text for a kmeans_status value (static storage). */
const char *kmeans_status_string(int status);

/* Size of the device array that kmeans_assign_noalloc uses as its scratch.
 * Every GPU that loads this library holds it until the process exits. */
#define KMEANS_NOALLOC_SCRATCH_BYTES (16u * 1024u * 1024u)

/* kmeans_assign without a workspace argument (the pages have no counterpart:
 * it exists for callers, not for the method).  Some callers cannot call
 * cudaMalloc when they need an assignment: code running under an allocator
 * that forbids new device allocations, plugins that are handed only their
 * input and output buffers, or real-time loops where an allocation and the
 * synchronisation it can imply are not allowed.  They pass only X, C and the
 * outputs; the scratch comes from one device array of
 * KMEANS_NOALLOC_SCRATCH_BYTES built into the library (16 MiB: enough for
 * 12 n + 4 k + 4 k ceil(d/64)*64 bytes plus 11 KiB, e.g. n = 65536, k = 1024,
 * d = 2048).  Larger problems are rejected with KMEANS_ERR_SCRATCH_LIMIT
 * before anything is enqueued; use kmeans_assign with a workspace for them.
 * Same inputs, outputs, requirements and results as kmeans_assign.  The
 * entry point allocates nothing and calls no allocating routine.
 * The first call on each device looks up the array's device address (one
 * cudaGetSymbolAddress): make that first call before any stream capture.
 * Every call, on every stream, shares the one array and leaves its contents
 * behind (each call resets what must start fresh); calls that can overlap on
 * the GPU race with each other and must be serialised by the caller.
 * Device-side timeouts are recorded in the array's status word, which
 * kmeans_device_status cannot reach; a call that returned KMEANS_OK and was
 * synchronised produced complete outputs unless labels hold -1. */
int kmeans_assign_noalloc(const float *X, const float *C, int64_t n, int64_t k, int64_t d,
                          int64_t *labels, float *best_dist, double *inertia, uint64_t seed,
                          void *stream);

/* Kernel timing for measurement tools (the pages have no counterpart: it
 * exists to hold each kernel against its roofline).
 * kmeans_trace_start(capacity) turns tracing on and clears earlier records.
 * From then on every call brackets its dominant kernel with a pair of CUDA
 * events recorded on the call's stream: the tensor-core assignment kernel
 * (kmeans_assign, kmeans_lloyd_iter, kmeans_assign_noalloc), the segmented
 * mean of the update (kmeans_update, kmeans_lloyd_iter) and the distance pass
 * of k-means++ seeding (kmeanspp_init).  Each kernel kind has `capacity`
 * event pairs (1 <= capacity <= KMEANS_TRACE_MAX_CAPACITY), created on the
 * current device; launches beyond the capacity are counted, not timed.
 * kmeans_trace_read waits for the recorded events of one kind and returns the
 * summed durations (milliseconds; each includes the kernel's launch latency
 * on the device), the number of timed launches and of all launches seen
 * (either count pointer may be NULL).  kmeans_trace_stop turns tracing off and
 * releases the events.  Tracing adds two stream operations per traced
 * launch; do not trace while a stream is being captured.  Start, read and
 * stop must not race with each other. */
#define KMEANS_TRACE_MAX_CAPACITY 65536
enum {
    KMEANS_KERNEL_ASSIGN_TC = 0,
    KMEANS_KERNEL_UPDATE_MEAN = 1,
    KMEANS_KERNEL_KMEANSPP_DIST = 2
};
int kmeans_trace_start(int capacity);
int kmeans_trace_read(int kernel, double *ms_total, int64_t *timed_launches, int64_t *launches);
int kmeans_trace_stop(void);

/* Build identification of the library: target architecture, tile shapes and
 * pipeline depth (static storage). */
const char *kmeans_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* KMEANS_GB300_H */

// Host launcher of the mean update.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace km {

// `sums_only`: write each cluster's unnormalised sum (zeros for an empty
// cluster) to C_new instead of its mean; C_old is then not read.
cudaError_t launch_update(const float *X, const int64_t *labels, const float *C_old, float *C_new,
                          int32_t *counts_out, int64_t n, int64_t k, int64_t d, const UpdateLayout &L,
                          uint8_t *ws, bool clear_header, cudaStream_t s, bool tile_counts_ready = false,
                          bool sums_only = false);

// Sample-sharded iteration: C_new[j] = (sum over ranks of parts[r][j], in
// rank order, in float64) / (sum over ranks of part_counts[r][j]), or C_old[j]
// when that count is 0; counts_out (nullable) the summed counts; inertia_out
// (nullable) the rank-order sum of part_inertia.  parts: world x rows x d
// float32, rank-major.
cudaError_t launch_reduce_partials(const float *parts, const int32_t *part_counts, const double *part_inertia,
                                   int world, int64_t rows, int64_t d, const float *C_old, float *C_new,
                                   int32_t *counts_out, double *inertia_out, cudaStream_t s);

// Assignment finalize fused with the update's per-tile cluster counts (one
// block per counting tile); used by the Lloyd iteration when the counting
// path applies.
cudaError_t launch_finalize_counting(int64_t n, int64_t k, const AssignLayout &A, const UpdateLayout &U,
                                     uint8_t *ws, int64_t *labels, float *best, double *inertia, cudaStream_t s);

// Mean step of kmeans_lloyd_iter_fused: C_new = sums / count (d % 4 == 0,
// 16-byte aligned rows), old rows for empty clusters, counts_out (may be null).
cudaError_t launch_fused_mean(const float *sums, const int32_t *cnt, const float *C_old, float *C_new,
                              int32_t *counts_out, int64_t k, int64_t d, cudaStream_t s);

}  // namespace km

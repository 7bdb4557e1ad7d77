// Host-side launchers shared by the assignment entry points.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace km {

int device_sm_count();
int assign_tc_smem_bytes();

// Clears the status word, splits C into bf16 hi / lo copies (row pitch
// L.d_pad), computes ||c_j||^2 and resets the per-sample keys.
cudaError_t launch_prep_split(const float *C, int64_t n, int64_t k, int64_t d, const AssignLayout &L,
                              uint8_t *ws, cudaStream_t s);

// Clears the status word, computes ||c_j||^2 and resets the keys (no split).
cudaError_t launch_prep_norms(const float *C, int64_t n, int64_t k, int64_t d, const AssignLayout &L,
                              uint8_t *ws, cudaStream_t s);

// Where the update fused into the assignment's epilogue accumulates
// (kmeans_lloyd_iter_fused): X, the (k, d) sums and (k) counts, zeroed
// beforehand, and one completion counter per 32 rows of every CTA.
struct FusedUpdate {
    const float *X;
    float *sums;
    int32_t *counts;
    uint32_t *row_done;
};

// `chained`: launched to overlap the tail of the kernel before it on `s`
// (the prologue's split); false after a wait on an event.  `tf32`: the
// 3xTF32 operand split (L from assign_layout(..., true, 4) and the centroid
// copies from launch_prep_split_tf32) instead of bf16x3.
cudaError_t launch_assign_tc(const float *X, int64_t n, int64_t k, int64_t d, const AssignLayout &L,
                             uint8_t *ws, cudaStream_t s, bool chained = true, bool tf32 = false,
                             const FusedUpdate *fused = nullptr);

// Sample rows whose wide units (bf16x3, d >= 2048, k > 256) fill whole
// rounds of the persistent schedule: a multiple of this many rows is
// assigned without a part-filled last round.  256 (one sample pair-block)
// where the tiles are not wide units.
int64_t assign_round_rows(int64_t k, int64_t d);

// launch_prep_split for the 3xTF32 path: C's hi (low 13 mantissa bits
// cleared) and lo (C - hi, low 13 bits cleared) as fp32, row pitch L.d_pad.
cudaError_t launch_prep_split_tf32(const float *C, int64_t n, int64_t k, int64_t d, const AssignLayout &L,
                                   uint8_t *ws, cudaStream_t s);

cudaError_t launch_assign_ffma(const float *X, const float *C, int64_t n, int64_t k, int64_t d,
                               const AssignLayout &L, uint8_t *ws, cudaStream_t s);

// Keys -> int64 labels, float32 distances (+ ||x||^2, clamped at 0) and the
// float64 inertia in a fixed reduction order.
cudaError_t launch_finalize(int64_t n, const AssignLayout &L, uint8_t *ws, int64_t *labels, float *best,
                            double *inertia, cudaStream_t s);

}  // namespace km

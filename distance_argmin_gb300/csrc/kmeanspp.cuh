// Host launcher of greedy k-means++ seeding.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace km {

cudaError_t launch_kmeanspp(const float *X, int64_t n, int64_t d, int64_t k, int T, uint64_t seed, float *centers,
                            int64_t *indices, const KppLayout &L, uint8_t *ws, cudaStream_t s);

}  // namespace km

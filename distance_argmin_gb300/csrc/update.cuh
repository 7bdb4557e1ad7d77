// Host launcher of the mean update.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace km {

cudaError_t launch_update(const float *X, const int64_t *labels, const float *C_old, float *C_new,
                          int32_t *counts_out, int64_t n, int64_t k, int64_t d, const UpdateLayout &L,
                          uint8_t *ws, bool clear_header, cudaStream_t s);

}  // namespace km

// Host launcher of greedy k-means++ seeding.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace km {

cudaError_t launch_kmeanspp(const float *X, int64_t n, int64_t d, int64_t k, int T, uint64_t seed, float *centers,
                            int64_t *indices, const KppLayout &L, uint8_t *ws, cudaStream_t s);

// The steps of greedy k-means++ on one shard of the samples (the
// kmeanspp_shard_* entry points of the C ABI).
cudaError_t launch_kpp_shard_first(const float *X, int64_t n_local, int64_t d, int64_t row_offset, int64_t n_global,
                                   int T, uint64_t seed, uint8_t *send, uint8_t *ws, cudaStream_t s);
cudaError_t launch_kpp_shard_dist(const float *X, int64_t n_local, int64_t d, int T, bool first, const uint8_t *recv,
                                  int world, double *pot_out, const KppShardLayout &L, uint8_t *ws, cudaStream_t s);
cudaError_t launch_kpp_shard_commit(int64_t n_local, int64_t d, int T, bool first, const double *recv_pot, int world,
                                    int64_t c, int64_t *indices, float *centers, double *total_out,
                                    const KppShardLayout &L, uint8_t *ws, cudaStream_t s);
cudaError_t launch_kpp_shard_pick(const float *X, int64_t n_local, int64_t d, int64_t row_offset, int T, uint64_t seed,
                                  int64_t c, const double *totals, int world, int rank, uint8_t *send,
                                  const KppShardLayout &L, uint8_t *ws, cudaStream_t s);

}  // namespace km

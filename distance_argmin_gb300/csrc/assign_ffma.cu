// The same fused assignment on the CUDA cores: a register-blocked float32 FMA
// tile (128 samples x 128 centroids per CTA, 8 x 8 per thread, pairs of
// columns in packed fp32x2 FMAs, double-buffered in shared memory) whose epilogue
// turns its scores ||c||^2 - 2 x.c into one (score, index) key per row and
// merges it with a 64-bit atomic minimum, so no (n, k) matrix is written.
// This is the measured comparator of the tensor-core path ("Three shapes that
// fit an eager Gram assignment", section "Gram assignment").
#include <cuda_runtime.h>
#include <stdint.h>

#include "assign_common.cuh"
#include "common.cuh"

namespace km {

namespace ff {
constexpr int BM = 128;
constexpr int BN = 128;
constexpr int BK = 16;
constexpr int THREADS = 256;
}  // namespace ff

template <bool VEC>
__device__ __forceinline__ float4 load4(const float *__restrict__ base, int row, int rows, int col, int cols) {
    if (row >= rows) return make_float4(0.f, 0.f, 0.f, 0.f);
    const float *p = base + (size_t)row * cols + col;
    if (VEC) {
        if (col + 3 < cols) return __ldg(reinterpret_cast<const float4 *>(p));
        return make_float4(0.f, 0.f, 0.f, 0.f);  // cols % 4 == 0 on this path
    }
    float4 v;
    v.x = col + 0 < cols ? __ldg(p + 0) : 0.f;
    v.y = col + 1 < cols ? __ldg(p + 1) : 0.f;
    v.z = col + 2 < cols ? __ldg(p + 2) : 0.f;
    v.w = col + 3 < cols ? __ldg(p + 3) : 0.f;
    return v;
}

// One block per SM: the paired accumulators want about 150 registers a thread
// (measured: 10.5% faster than scalar FMAs at two blocks, which spills).
template <bool VEC>
__global__ void __launch_bounds__(ff::THREADS, 1)
    assign_ffma_kernel(const float *__restrict__ X, const float *__restrict__ C,
                       const float *__restrict__ cnorm, int n, int k, int d, float *__restrict__ xnorm,
                       unsigned long long *__restrict__ keys) {
    __shared__ __align__(16) float As[2][ff::BK][ff::BM];
    __shared__ __align__(16) float Bs[2][ff::BK][ff::BN];
    const int tid = threadIdx.x;
    const int tx = tid & 15;
    const int ty = tid >> 4;
    const int m0 = blockIdx.x * ff::BM;
    const int n0 = blockIdx.y * ff::BN;
    const int lr = tid >> 2;         // load row 0..63 (and +64)
    const int lk = (tid & 3) * 4;    // load column 0,4,8,12
    const bool want_xnorm = blockIdx.y == 0;

    // acc[i][j] pairs columns 2j and 2j+1: one packed fp32x2 FMA per pair
    // (the same per-lane fma as two scalar ones, in half the issue slots)
    float2 acc[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = make_float2(0.f, 0.f);
    float xs[2] = {0.f, 0.f}, xc[2] = {0.f, 0.f};

    float4 ra[2], rb[2];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            ra[h] = load4<VEC>(X, m0 + lr + 64 * h, n, k0 + lk, d);
            rb[h] = load4<VEC>(C, n0 + lr + 64 * h, k, k0 + lk, d);
        }
    };
    auto stash = [&](int buf) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            As[buf][lk + 0][lr + 64 * h] = ra[h].x;
            As[buf][lk + 1][lr + 64 * h] = ra[h].y;
            As[buf][lk + 2][lr + 64 * h] = ra[h].z;
            As[buf][lk + 3][lr + 64 * h] = ra[h].w;
            Bs[buf][lk + 0][lr + 64 * h] = rb[h].x;
            Bs[buf][lk + 1][lr + 64 * h] = rb[h].y;
            Bs[buf][lk + 2][lr + 64 * h] = rb[h].z;
            Bs[buf][lk + 3][lr + 64 * h] = rb[h].w;
            if (want_xnorm) {
                float q = ra[h].x * ra[h].x;
                q = fmaf(ra[h].y, ra[h].y, q);
                q = fmaf(ra[h].z, ra[h].z, q);
                q = fmaf(ra[h].w, ra[h].w, q);
                const float y = q - xc[h];
                const float t = xs[h] + y;
                xc[h] = (t - xs[h]) - y;
                xs[h] = t;
            }
        }
    };

    const int ntiles = (d + ff::BK - 1) / ff::BK;
    fetch(0);
    stash(0);
    __syncthreads();
    for (int t = 0; t < ntiles; ++t) {
        const int buf = t & 1;
        if (t + 1 < ntiles) fetch((t + 1) * ff::BK);
#pragma unroll
        for (int kk = 0; kk < ff::BK; ++kk) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&As[buf][kk][ty * 4]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&As[buf][kk][ty * 4 + 64]);
            const float4 b0 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tx * 4]);
            const float4 b1 = *reinterpret_cast<const float4 *>(&Bs[buf][kk][tx * 4 + 64]);
            const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const float2 b[4] = {make_float2(b0.x, b0.y), make_float2(b0.z, b0.w), make_float2(b1.x, b1.y),
                                 make_float2(b1.z, b1.w)};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float2 ai = make_float2(a[i], a[i]);
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = __ffma2_rn(ai, b[j], acc[i][j]);
            }
        }
        if (t + 1 < ntiles) stash((t + 1) & 1);
        __syncthreads();
    }

    if (want_xnorm) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float v = xs[h] - xc[h];
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            const int row = m0 + lr + 64 * h;
            if ((tid & 3) == 0 && row < n) xnorm[row] = v;
        }
    }

    // fused epilogue: per-row min / argmin over this tile's 128 centroids
    float cn[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
        const int col = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
        cn[j] = col < k ? __ldg(cnorm + col) : 0.f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int row = m0 + (i < 4 ? ty * 4 + i : 64 + ty * 4 + i - 4);
        float best = __int_as_float(0x7f800000);
        int arg = -1;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int col = n0 + (j < 4 ? tx * 4 + j : 64 + tx * 4 + j - 4);
            const float s = fmaf(-2.f, (j & 1) ? acc[i][j >> 1].y : acc[i][j >> 1].x, cn[j]);
            if (col < k && s < best) {
                best = s;
                arg = col;
            }
        }
        unsigned long long key = arg >= 0 ? make_key(best, (uint32_t)arg) : kEmptyKey;
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) {
            const unsigned long long other = __shfl_xor_sync(0xffffffffu, key, o);
            key = other < key ? other : key;
        }
        if (tx == 0 && row < n && key != kEmptyKey) atomicMin(keys + row, key);
    }
}

cudaError_t launch_assign_ffma(const float *X, const float *C, int64_t n, int64_t k, int64_t d,
                               const AssignLayout &L, uint8_t *ws, cudaStream_t s) {
    const dim3 grid((unsigned)((n + ff::BM - 1) / ff::BM), (unsigned)((k + ff::BN - 1) / ff::BN));
    const bool vec = (d % 4 == 0) && ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(C)) & 15) == 0;
    const float *cnorm = reinterpret_cast<const float *>(ws + L.off_cnorm);
    float *xnorm = reinterpret_cast<float *>(ws + L.off_xnorm);
    unsigned long long *keys = reinterpret_cast<unsigned long long *>(ws + L.off_keys);
    if (vec)
        assign_ffma_kernel<true><<<grid, ff::THREADS, 0, s>>>(X, C, cnorm, (int)n, (int)k, (int)d, xnorm, keys);
    else
        assign_ffma_kernel<false><<<grid, ff::THREADS, 0, s>>>(X, C, cnorm, (int)n, (int)k, (int)d, xnorm, keys);
    return cudaGetLastError();
}

}  // namespace km

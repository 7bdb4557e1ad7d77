// Assignment prologue (centroid norms and bf16 split) and epilogue (labels,
// distances, inertia).
//
// ||c_j||^2 is computed once per call and reused by every sample tile
// ("004 — tile sizes, a Cython Lloyd step, and k-means++", section "Schedules
// added").  The reported distance adds ||x_i||^2 back to the winning score
// ||c||^2 - 2 x.c ("Three shapes that fit an eager Gram assignment", section
// "Gram assignment"), clamped at zero, and the result per sample is an int64
// label plus a float32 distance (same page, section "Running argmin, one
// centroid").
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "assign_common.cuh"
#include "common.cuh"

namespace km {

__device__ __forceinline__ void kahan_add(float &sum, float &comp, float v) {
    const float y = v - comp;
    const float t = sum + y;
    comp = (t - sum) - y;
    sum = t;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ uint32_t bf16x2_bits(__nv_bfloat162 h) {
    return *reinterpret_cast<uint32_t *>(&h);
}

// One 128-thread block per centroid row (grid-stride over rows); each thread
// converts up to 4 float4 groups per pass with its loads issued together.
// d % 4 == 0 and C 16-byte aligned (checked on the host for this path);
// columns d .. d_pad-1 of the copies are zeroed.
constexpr int kPrepThreads = 128;

// Per call, before the tensor-core pass: every key to "none yet"; with the
// K-split area, every ||x||^2 to 0 (the two halves of a split tile add their
// partial norms into it) and the split tickets and tags to 0.
__device__ __forceinline__ void reset_for_assign(unsigned long long *__restrict__ keys, int n,
                                                 float *__restrict__ xnorm_zero, uint32_t *__restrict__ ksync,
                                                 int ksync_words) {
    const int stride = gridDim.x * blockDim.x;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        keys[i] = kEmptyKey;
        if (xnorm_zero) xnorm_zero[i] = 0.f;
    }
    if (ksync)
        for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < ksync_words; i += stride) ksync[i] = 0u;
}

__global__ void __launch_bounds__(kPrepThreads)
    prep_split_kernel(const float *__restrict__ C, int k, int d, int d_pad, __nv_bfloat16 *__restrict__ chi,
                      __nv_bfloat16 *__restrict__ clo, float *__restrict__ cnorm,
                      unsigned long long *__restrict__ keys, int n, WsHeader *hdr, float *__restrict__ xnorm_zero,
                      uint32_t *__restrict__ ksync, int ksync_words) {
    __shared__ float red[kPrepThreads / 32];
    griddep_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        hdr->status = 0u;
        hdr->done_blocks = 0u;
        hdr->round_arrivals = 0u;
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int j = blockIdx.x; j < k; j += gridDim.x) {
        const float *row = C + (size_t)j * d;
        float sum = 0.f, comp = 0.f;
        for (int f0 = threadIdx.x * 4; f0 < d_pad; f0 += kPrepThreads * 16) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int f = f0 + u * kPrepThreads * 4;
                v[u] = f < d ? __ldg(reinterpret_cast<const float4 *>(row + f)) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int f = f0 + u * kPrepThreads * 4;
                if (f >= d_pad) break;
                const __nv_bfloat162 h01 = __floats2bfloat162_rn(v[u].x, v[u].y);
                const __nv_bfloat162 h23 = __floats2bfloat162_rn(v[u].z, v[u].w);
                const float2 f01 = __bfloat1622float2(h01);
                const float2 f23 = __bfloat1622float2(h23);
                const __nv_bfloat162 l01 = __floats2bfloat162_rn(v[u].x - f01.x, v[u].y - f01.y);
                const __nv_bfloat162 l23 = __floats2bfloat162_rn(v[u].z - f23.x, v[u].w - f23.y);
                const size_t o = (size_t)j * d_pad + f;
                *reinterpret_cast<uint2 *>(chi + o) = make_uint2(bf16x2_bits(h01), bf16x2_bits(h23));
                *reinterpret_cast<uint2 *>(clo + o) = make_uint2(bf16x2_bits(l01), bf16x2_bits(l23));
                float q = v[u].x * v[u].x;
                q = fmaf(v[u].y, v[u].y, q);
                q = fmaf(v[u].z, v[u].z, q);
                q = fmaf(v[u].w, v[u].w, q);
                kahan_add(sum, comp, q);
            }
        }
        const float part = warp_sum(sum - comp);
        if (lane == 0) red[wid] = part;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kPrepThreads / 32; ++w) tot += red[w];
            cnorm[j] = tot;
        }
        __syncthreads();
    }
    reset_for_assign(keys, n, xnorm_zero, ksync, ksync_words);
}

__device__ __forceinline__ float tf32_bits_trunc(float v) {
    return __uint_as_float(__float_as_uint(v) & 0xffffe000u);
}

// The 3xTF32 prologue: hi = c with its low 13 mantissa bits cleared, lo =
// (c - hi) with its low 13 bits cleared, both fp32 at row pitch d_pad (so the
// tensor cores read them exactly whether they round or truncate), ||c_j||^2
// from the exact c; otherwise as prep_split_kernel.
__global__ void __launch_bounds__(kPrepThreads)
    prep_split_tf32_kernel(const float *__restrict__ C, int k, int d, int d_pad, float *__restrict__ chi,
                           float *__restrict__ clo, float *__restrict__ cnorm,
                           unsigned long long *__restrict__ keys, int n, WsHeader *hdr, float *__restrict__ xnorm_zero,
                      uint32_t *__restrict__ ksync, int ksync_words) {
    __shared__ float red[kPrepThreads / 32];
    griddep_wait();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        hdr->status = 0u;
        hdr->done_blocks = 0u;
    }
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int j = blockIdx.x; j < k; j += gridDim.x) {
        const float *row = C + (size_t)j * d;
        float sum = 0.f, comp = 0.f;
        for (int f = threadIdx.x * 4; f < d_pad; f += kPrepThreads * 4) {
            const float4 v = f < d ? __ldg(reinterpret_cast<const float4 *>(row + f)) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 h = make_float4(tf32_bits_trunc(v.x), tf32_bits_trunc(v.y), tf32_bits_trunc(v.z),
                                         tf32_bits_trunc(v.w));
            const float4 l = make_float4(tf32_bits_trunc(v.x - h.x), tf32_bits_trunc(v.y - h.y),
                                         tf32_bits_trunc(v.z - h.z), tf32_bits_trunc(v.w - h.w));
            const size_t o = (size_t)j * d_pad + f;
            *reinterpret_cast<float4 *>(chi + o) = h;
            *reinterpret_cast<float4 *>(clo + o) = l;
            float q = v.x * v.x;
            q = fmaf(v.y, v.y, q);
            q = fmaf(v.z, v.z, q);
            q = fmaf(v.w, v.w, q);
            kahan_add(sum, comp, q);
        }
        const float part = warp_sum(sum - comp);
        if (lane == 0) red[wid] = part;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.f;
#pragma unroll
            for (int w = 0; w < kPrepThreads / 32; ++w) tot += red[w];
            cnorm[j] = tot;
        }
        __syncthreads();
    }
    reset_for_assign(keys, n, xnorm_zero, ksync, ksync_words);
}

// Norms only (any d, any 4-byte alignment).
__global__ void prep_norms_kernel(const float *__restrict__ C, int k, int d, float *__restrict__ cnorm,
                                  unsigned long long *__restrict__ keys, int n, WsHeader *hdr) {
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        hdr->status = 0u;
        hdr->done_blocks = 0u;
    }
    const int lane = threadIdx.x & 31;
    const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int nw = gridDim.x * (blockDim.x >> 5);
    for (int j = gw; j < k; j += nw) {
        const float *row = C + (size_t)j * d;
        float sum = 0.f, comp = 0.f;
        for (int f = lane; f < d; f += 32) {
            const float v = __ldg(row + f);
            kahan_add(sum, comp, v * v);
        }
        const float tot = warp_sum(sum - comp);
        if (lane == 0) cnorm[j] = tot;
    }
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        keys[i] = kEmptyKey;
}

constexpr int kFinThreads = 256;

// Rows are split into gridDim.x contiguous ranges (fixed by n), each summed in
// a fixed order; the last block to finish adds the block sums in index order.
__global__ void finalize_kernel(const unsigned long long *__restrict__ keys, const float *__restrict__ xnorm,
                                int n, int64_t *__restrict__ labels, float *__restrict__ best,
                                double *inertia, double *partial, WsHeader *hdr) {
    __shared__ double red[kFinThreads];
    __shared__ int is_last;
    griddep_wait();
    const int nb = gridDim.x;
    const int per = (n + nb - 1) / nb;
    const int r0 = blockIdx.x * per;
    const int r1 = min(n, r0 + per);
    double s = 0.0;
    for (int r = r0 + threadIdx.x; r < r1; r += kFinThreads) {
        const unsigned long long key = keys[r];
        if (key == kEmptyKey) {  // only for non-finite inputs
            labels[r] = -1;
            best[r] = __int_as_float(0x7fc00000);
            continue;
        }
        const float score = ord_to_float(static_cast<uint32_t>(key >> 32));
        const float b = fmaxf(0.f, xnorm[r] + score);
        labels[r] = static_cast<int64_t>(static_cast<uint32_t>(key & 0xffffffffu));
        best[r] = b;
        s += static_cast<double>(b);
    }
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = kFinThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (inertia == nullptr) return;
    if (threadIdx.x == 0) {
        partial[blockIdx.x] = red[0];
        __threadfence();
        const unsigned t = atomicAdd(&hdr->done_blocks, 1u);
        is_last = (t == (unsigned)nb - 1u);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    double v = 0.0;
    for (int b = threadIdx.x; b < nb; b += kFinThreads) v += __ldcg(partial + b);
    red[threadIdx.x] = v;
    __syncthreads();
    for (int w = kFinThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        *inertia = red[0];
        hdr->done_blocks = 0u;
    }
}

static int prep_grid(int64_t k, int64_t n) {
    const int64_t by_keys = (n + 1023) / 1024;
    int64_t g = k > by_keys ? k : by_keys;
    const int64_t cap = (int64_t)device_sm_count() * 16;
    if (g > cap) g = cap;
    return (int)(g < 1 ? 1 : g);
}

cudaError_t launch_prep_split(const float *C, int64_t n, int64_t k, int64_t d, const AssignLayout &L,
                              uint8_t *ws, cudaStream_t s) {
    const bool ks = L.off_ksync != 0;
    return launch_kernel(
        true, prep_split_kernel, dim3(prep_grid(k, n)), dim3(kPrepThreads), 0, s, C, (int)k, (int)d, (int)L.d_pad,
        reinterpret_cast<__nv_bfloat16 *>(ws + L.off_chi), reinterpret_cast<__nv_bfloat16 *>(ws + L.off_clo),
        reinterpret_cast<float *>(ws + L.off_cnorm), reinterpret_cast<unsigned long long *>(ws + L.off_keys), (int)n,
        reinterpret_cast<WsHeader *>(ws), ks ? reinterpret_cast<float *>(ws + L.off_xnorm) : nullptr,
        ks ? reinterpret_cast<uint32_t *>(ws + L.off_ksync) : nullptr, ks ? kKSplitSlots * kKSplitSyncWords : 0);
}

cudaError_t launch_prep_split_tf32(const float *C, int64_t n, int64_t k, int64_t d, const AssignLayout &L,
                                   uint8_t *ws, cudaStream_t s) {
    if (L.split_elem_bytes != 4) return cudaErrorInvalidValue;
    const bool ks = L.off_ksync != 0;
    return launch_kernel(
        true, prep_split_tf32_kernel, dim3(prep_grid(k, n)), dim3(kPrepThreads), 0, s, C, (int)k, (int)d,
        (int)L.d_pad, reinterpret_cast<float *>(ws + L.off_chi), reinterpret_cast<float *>(ws + L.off_clo),
        reinterpret_cast<float *>(ws + L.off_cnorm), reinterpret_cast<unsigned long long *>(ws + L.off_keys), (int)n,
        reinterpret_cast<WsHeader *>(ws), ks ? reinterpret_cast<float *>(ws + L.off_xnorm) : nullptr,
        ks ? reinterpret_cast<uint32_t *>(ws + L.off_ksync) : nullptr, ks ? kKSplitSlots * kKSplitSyncWords : 0);
}

cudaError_t launch_prep_norms(const float *C, int64_t n, int64_t k, int64_t d, const AssignLayout &L,
                              uint8_t *ws, cudaStream_t s) {
    prep_norms_kernel<<<prep_grid(k, n), 256, 0, s>>>(C, (int)k, (int)d,
                                                      reinterpret_cast<float *>(ws + L.off_cnorm),
                                                      reinterpret_cast<unsigned long long *>(ws + L.off_keys),
                                                      (int)n, reinterpret_cast<WsHeader *>(ws));
    return cudaGetLastError();
}

cudaError_t launch_finalize(int64_t n, const AssignLayout &L, uint8_t *ws, int64_t *labels, float *best,
                            double *inertia, cudaStream_t s) {
    int64_t nb = (n + kFinThreads - 1) / kFinThreads;
    if (nb > kMaxReduceBlocks) nb = kMaxReduceBlocks;
    return launch_kernel(true, finalize_kernel, dim3((unsigned)nb), dim3(kFinThreads), 0, s,
                         reinterpret_cast<const unsigned long long *>(ws + L.off_keys),
                         reinterpret_cast<const float *>(ws + L.off_xnorm), (int)n, labels, best, inertia,
                         reinterpret_cast<double *>(ws + L.off_partial), reinterpret_cast<WsHeader *>(ws));
}

}  // namespace km

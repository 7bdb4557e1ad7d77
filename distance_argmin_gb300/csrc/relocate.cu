// Empty-cluster relocation.
//
// "004 — tile sizes, a Cython Lloyd step, and k-means++", section "Cython
// timing": the Lloyd step there also relocates empty clusters, with no rule
// given.  The rule here is the plain reading: when m clusters have no member,
// the m samples farthest from the centroid they were assigned to (largest
// best distance; among equal distances the lower sample index first) leave
// their clusters and, taken in increasing sample index, become the only
// members of the empty clusters taken in increasing cluster index.  A cluster
// that loses every member this way is empty afterwards; the mean update then
// keeps its centroid.  Only labels change; the update that follows turns a
// relocated sample into its new cluster's centroid.
//
// Kernels:
//   reloc_count_kernel   member counts (int32 atomics, aggregated per warp
//                        over lanes holding the same label)
//   reloc_select_kernel  one CTA of 1024 threads.  (1) The empty clusters in
//                        increasing order, by a block scan over the counts;
//                        with none it returns here.  (2) The m-th largest
//                        distance key T, by a radix select over the 32-bit
//                        order-preserving image of the distances (4 passes of
//                        8 bits, most significant first), with `need` = how
//                        many samples whose key equals T are taken.  (3) Each
//                        thread owns a contiguous range of samples; a block
//                        scan of (count above T, count equal to T) per range
//                        gives every taken sample its rank in index order,
//                        and that rank picks its empty cluster.
//   reloc_count_empty_kernel  the number of empty clusters from counts an
//                        update already wrote (the fit's cheap check)
// Relocation is rare (it runs only while a cluster is empty), so one CTA is
// enough: its passes read the n distances six times from L2, with eight
// loads in flight per thread.  It is latency-bound on its one SM: about
// 140 us for n = 65536, paid only by an iteration that left a cluster empty.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "relocate.cuh"

namespace km {

namespace {

constexpr int kCountThreads = 256;
constexpr int kCountMaxBlocks = 152 * 8;
constexpr int kSelectThreads = 1024;
constexpr int kSelectWarps = kSelectThreads / 32;
constexpr int kBatch = 8;  // distance loads a select thread keeps in flight

// Order-preserving key of a non-negative distance, with -0 read as +0 so that
// the two zeros compare equal as they do as floats.
__device__ __forceinline__ uint32_t dist_key(float f) { return f == 0.0f ? 0x80000000u : float_to_ord(f); }

// Exclusive prefix sum of `v` over the block in thread order; `total`
// receives the block's sum.  Every thread of the block must call it.
__device__ __forceinline__ uint64_t block_exclusive_scan(uint64_t v, uint64_t *scratch, uint64_t &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const uint64_t o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint64_t x = lane < kSelectWarps ? scratch[lane] : 0ull;
        uint64_t xi = x;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const uint64_t o = __shfl_up_sync(0xffffffffu, xi, off);
            if (lane >= off) xi += o;
        }
        if (lane < kSelectWarps) scratch[lane] = xi - x;
        if (lane == 31) scratch[32] = xi;
    }
    __syncthreads();
    const uint64_t r = scratch[warp] + incl - v;
    total = scratch[32];
    __syncthreads();  // scratch is reused by the next call
    return r;
}

__global__ void __launch_bounds__(kCountThreads)
    reloc_count_kernel(const int64_t *__restrict__ labels, int64_t n, int k, int32_t *__restrict__ counts,
                       uint32_t *status) {
    const int64_t stride = (int64_t)gridDim.x * kCountThreads;
    // `base` is the same for the whole block, so whole warps reach the match
    for (int64_t base = (int64_t)blockIdx.x * kCountThreads; base < n; base += stride) {
        const int64_t i = base + threadIdx.x;
        int lab = -1;
        if (i < n) {
            const int64_t v = labels[i];
            if (v < 0 || v >= k)
                flag_error(status, kFlagBadLabel);
            else
                lab = (int)v;
        }
        const unsigned peers = __match_any_sync(0xffffffffu, lab);
        if (lab >= 0 && (int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&counts[lab], __popc(peers));
    }
}

__global__ void __launch_bounds__(kSelectThreads, 1)
    reloc_select_kernel(int64_t *__restrict__ labels, const float *__restrict__ best, int64_t n, int k,
                        const int32_t *__restrict__ counts, int32_t *__restrict__ empty, WsHeader *hdr) {
    __shared__ uint64_t scan[33];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_digit, s_need;
    const int t = threadIdx.x;
    // a bad label or an earlier fault: the labels stay as they are
    if (error_raised(&hdr->status)) return;

    // (1) the empty clusters, in increasing index
    const int64_t per_k = ((int64_t)k + kSelectThreads - 1) / kSelectThreads;
    const int64_t j0 = min((int64_t)k, t * per_k), j1 = min((int64_t)k, j0 + per_k);
    uint32_t zeros = 0;
    for (int64_t j = j0; j < j1; ++j) zeros += counts[j] == 0;
    uint64_t m64 = 0;
    uint64_t at = block_exclusive_scan(zeros, scan, m64);
    for (int64_t j = j0; j < j1; ++j)
        if (counts[j] == 0) empty[at++] = (int32_t)j;
    if (m64 == 0) return;  // uniform: every thread holds the same total
    // at least one cluster has a member, so m <= k - 1 <= n - 1

    // (2) radix select: T = the key of the m-th largest distance
    uint32_t prefix = 0u, mask = 0u, need = (uint32_t)m64;
    for (int shift = 24; shift >= 0; shift -= 8) {
        if (t < 256) hist[t] = 0u;
        __syncthreads();
        // kBatch loads in flight per thread before their histogram updates
        // (merging equal digits of a warp into one atomic measured slower)
        for (int64_t base = t; base < n; base += (int64_t)kSelectThreads * kBatch) {
            float v[kBatch];
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const int64_t i = base + (int64_t)q * kSelectThreads;
                v[q] = i < n ? best[i] : 0.0f;
            }
#pragma unroll
            for (int q = 0; q < kBatch; ++q) {
                const uint32_t u = dist_key(v[q]);
                if (base + (int64_t)q * kSelectThreads < n && (u & mask) == prefix)
                    atomicAdd(&hist[(u >> shift) & 255u], 1u);
            }
        }
        __syncthreads();
        if (t < 32) {
            // lane l holds digits 255 - 8l down to 248 - 8l: a scan over the
            // lanes runs through the digits from the largest down
            uint32_t c[8], sum = 0u;
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                c[q] = hist[255 - 8 * t - q];
                sum += c[q];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const uint32_t o = __shfl_up_sync(0xffffffffu, incl, off);
                if (t >= off) incl += o;
            }
            // the keys under the current prefix number at least `need`, so
            // some lane's running count reaches it
            const unsigned hit = __ballot_sync(0xffffffffu, incl >= need);
            if (t == __ffs(hit) - 1) {
                uint32_t run = incl - sum;
                int q = 0;
                while (q < 7 && run + c[q] < need) run += c[q++];
                s_digit = 255u - 8u * (uint32_t)t - (uint32_t)q;
                s_need = need - run;
            }
        }
        __syncthreads();
        prefix |= s_digit << shift;
        mask |= 255u << shift;
        need = s_need;
        __syncthreads();  // s_digit and hist are rewritten by the next pass
    }
    const uint32_t T = prefix;  // take every key above T and the first `need` equal to it

    // (3) ranks in sample order over contiguous per-thread ranges
    const int64_t per_n = (n + kSelectThreads - 1) / kSelectThreads;
    const int64_t i0 = min(n, t * per_n), i1 = min(n, i0 + per_n);
    uint32_t above = 0u, equal = 0u;
    for (int64_t i = i0; i < i1; i += kBatch) {
        float v[kBatch];
#pragma unroll
        for (int q = 0; q < kBatch; ++q) v[q] = i + q < i1 ? best[i + q] : 0.0f;
#pragma unroll
        for (int q = 0; q < kBatch; ++q) {
            const uint32_t u = dist_key(v[q]);
            const bool in = i + q < i1;
            above += in && u > T;
            equal += in && u == T;
        }
    }
    uint64_t both = 0;
    const uint64_t before = block_exclusive_scan(((uint64_t)above << 32) | equal, scan, both);
    uint32_t above_b = (uint32_t)(before >> 32), equal_b = (uint32_t)before;
    for (int64_t i = i0; i < i1; ++i) {
        const uint32_t u = dist_key(best[i]);  // L1-resident after the count above
        if (u > T) {
            labels[i] = empty[above_b + min(equal_b, need)];
            ++above_b;
        } else if (u == T) {
            if (equal_b < need) labels[i] = empty[above_b + equal_b];
            ++equal_b;
        }
    }
}

__global__ void __launch_bounds__(kSelectThreads)
    reloc_count_empty_kernel(const int32_t *__restrict__ counts, int k, uint32_t *__restrict__ n_empty) {
    __shared__ uint32_t sum;
    if (threadIdx.x == 0) sum = 0u;
    __syncthreads();
    uint32_t z = 0u;
    for (int j = threadIdx.x; j < k; j += kSelectThreads) z += counts[j] == 0;
    if (z) atomicAdd(&sum, z);
    __syncthreads();
    if (threadIdx.x == 0) *n_empty = sum;
}

}  // namespace

cudaError_t launch_count_empty(const int32_t *counts, int64_t k, uint32_t *n_empty, cudaStream_t s) {
    reloc_count_empty_kernel<<<1, kSelectThreads, 0, s>>>(counts, (int)k, n_empty);
    return cudaGetLastError();
}

cudaError_t launch_relocate(int64_t *labels, const float *best, int64_t n, int64_t k, const RelocLayout &R,
                            uint8_t *ws, cudaStream_t s) {
    int32_t *counts = reinterpret_cast<int32_t *>(ws + R.off_counts);
    int32_t *empty = reinterpret_cast<int32_t *>(ws + R.off_empty);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
    cudaError_t e = cudaMemsetAsync(counts, 0, (size_t)k * sizeof(int32_t), s);
    if (e != cudaSuccess) return e;
    const int64_t want = (n + kCountThreads - 1) / kCountThreads;
    const int blocks = (int)(want < kCountMaxBlocks ? want : kCountMaxBlocks);
    reloc_count_kernel<<<blocks, kCountThreads, 0, s>>>(labels, n, (int)k, counts, &hdr->status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    reloc_select_kernel<<<1, kSelectThreads, 0, s>>>(labels, best, n, (int)k, counts, empty, hdr);
    return cudaGetLastError();
}

}  // namespace km

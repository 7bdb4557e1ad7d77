// Mean update of the Lloyd iteration ("Three shapes that fit an eager Gram
// assignment", section "Full Lloyd step": every centroid becomes the mean of
// its members).  No (n, k) one-hot matrix: the labels are sorted into a member
// list and each centroid's members are summed as one contiguous segment.
//
// The member list, for k <= 32768 (the counting path):
//   1. per-cluster member counts of 256 fixed sample tiles (in a Lloyd
//      iteration the finalize of the assignment does this)
//   2. per-cluster prefixes over the tiles, and the totals
//   3. each tile's block scans the totals (-> segment offsets), then one warp
//      scatters the tile's samples in index order -> a stable member list
//      ordered by (label, sample index); the other warps write the counts
//      and the rows of empty clusters
// For larger k: a stable LSD radix sort of (label, sample index) with 8-bit
// digits (ceil(bits(k-1) / 8) passes: hist -> scan -> stable scatter), then
// the exclusive scan of the counts.
// Then, on both paths:
//   4. segmented sum over fixed chunks of the member list: a CTA owns one
//      chunk x one 512-column slice, sums each segment in member order with
//      compensated float32 additions and writes the mean when the segment is
//      inside its chunk, or a partial sum when it crosses the chunk boundary
//   5. fix-up: segments that crossed chunks add their partials in chunk order
// An empty cluster keeps its old row bit for bit (written by step 3 on the
// counting path, by step 5 on the radix path).
// Every step has a fixed order, so C_new is bitwise reproducible.
//
// The same kernels also serve a shard of the samples (the sample-sharded
// iteration): in sums mode the steps write each cluster's unnormalised
// sum, and zeros for an empty cluster, and reduce_partials_kernel later adds
// the shards' sums in rank order and divides.
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "common.cuh"
#include "trace.cuh"
#include "update.cuh"

namespace km {

__device__ __forceinline__ uint32_t clamp_label(int64_t lab, int k, uint32_t *status) {
    if (lab < 0 || lab >= k) {
        flag_error(status, kFlagBadLabel);
        return (uint32_t)(k - 1);
    }
    return (uint32_t)lab;
}

// counts[] = 0 (and header cleared when this call owns it)
__global__ void update_clear_kernel(int32_t *counts, int k, WsHeader *hdr, int clear_header) {
    griddep_wait();
    if (clear_header && blockIdx.x == 0 && threadIdx.x == 0) {
        hdr->status = 0u;
        hdr->done_blocks = 0u;
    }
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < k; j += gridDim.x * blockDim.x) counts[j] = 0;
}

// Per-tile digit histogram of pass `shift`; the first pass reads the int64
// labels directly (and counts members per cluster), later passes read the
// keys the previous pass wrote.
__global__ void __launch_bounds__(kSortThreads)
    radix_hist_kernel(const int64_t *__restrict__ labels, const uint32_t *__restrict__ keys_in, int n, int k,
                      int shift, int n_tiles, int32_t *__restrict__ hist, int32_t *__restrict__ counts,
                      uint32_t *status) {
    __shared__ int32_t h[kRadixBins];
    for (int b = threadIdx.x; b < kRadixBins; b += kSortThreads) h[b] = 0;
    __syncthreads();
    const int tile = blockIdx.x;
    const int base = tile * kSortTile;
    const int end = min(n, base + kSortTile);
    for (int i = base + threadIdx.x; i < end; i += kSortThreads) {
        uint32_t key;
        if (labels) {
            key = clamp_label(labels[i], k, status);
            // warp-aggregated member count
            const uint32_t active = __activemask();
            const uint32_t peers = __match_any_sync(active, key);
            const int leader = __ffs(peers) - 1;
            if ((int)(threadIdx.x & 31) == leader) atomicAdd(counts + key, __popc(peers));
        } else {
            key = keys_in[i];
        }
        atomicAdd(&h[(key >> shift) & 0xffu], 1);
    }
    __syncthreads();
    for (int b = threadIdx.x; b < kRadixBins; b += kSortThreads) hist[b * n_tiles + tile] = h[b];
}

// Exclusive scan of `len` int32 values, out[i] = sum of in[0..i-1] (one CTA,
// 1024 threads; `in` may equal `out`).  The total goes to *total_out if given.
__global__ void __launch_bounds__(1024) exclusive_scan_kernel(const int32_t *in, int32_t *out, int64_t len,
                                                              int32_t *total_out) {
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int64_t base = 0; base < len; base += 1024) {
        const int64_t i = base + threadIdx.x;
        const int32_t v = i < len ? in[i] : 0;
        int32_t incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += t;
        }
        if (lane == 31) warp_tot[wid] = incl;
        __syncthreads();
        if (wid == 0) {
            int32_t w = warp_tot[lane];
            int32_t wi = w;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int32_t t = __shfl_up_sync(0xffffffffu, wi, o);
                if (lane >= o) wi += t;
            }
            warp_tot[lane] = wi - w;  // exclusive prefix of warp totals
        }
        __syncthreads();
        const int32_t c = carry;
        if (i < len) out[i] = c + warp_tot[wid] + incl - v;
        __syncthreads();
        if (threadIdx.x == 1023) carry = c + warp_tot[wid] + incl;
        __syncthreads();
    }
    if (total_out && threadIdx.x == 0) *total_out = carry;
}

// Stable scatter of one radix pass.  The tile is walked in rounds of 256
// elements in index order; inside a round an element's rank among equal
// digits comes from its warp (match_any) and the warps before it.
__global__ void __launch_bounds__(kSortThreads)
    radix_scatter_kernel(const int64_t *__restrict__ labels, const uint32_t *__restrict__ keys_in,
                         const int32_t *__restrict__ vals_in, int n, int k, int shift, int n_tiles,
                         const int32_t *__restrict__ hist_scanned, uint32_t *__restrict__ keys_out,
                         int32_t *__restrict__ vals_out, uint32_t *status) {
    constexpr int W = kSortThreads / 32;
    __shared__ int32_t base_off[kRadixBins];
    __shared__ int32_t wcount[W][kRadixBins];
    const int tile = blockIdx.x;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int b = threadIdx.x; b < kRadixBins; b += kSortThreads) base_off[b] = hist_scanned[b * n_tiles + tile];
    const int tbase = tile * kSortTile;
    const int tend = min(n, tbase + kSortTile);
    for (int r0 = tbase; r0 < tend; r0 += kSortThreads) {
        for (int b = threadIdx.x; b < W * kRadixBins; b += kSortThreads) (&wcount[0][0])[b] = 0;
        __syncthreads();
        const int i = r0 + threadIdx.x;
        const bool valid = i < tend;
        uint32_t key = 0u;
        int32_t val = 0;
        if (valid) {
            if (labels) {
                key = clamp_label(labels[i], k, status);
                val = i;
            } else {
                key = keys_in[i];
                val = vals_in[i];
            }
        }
        const uint32_t digit = valid ? ((key >> shift) & 0xffu) : 0xffffffffu;
        const uint32_t peers = __match_any_sync(0xffffffffu, digit);
        const int rank_in_warp = __popc(peers & ((1u << lane) - 1u));
        if (valid && rank_in_warp == 0) wcount[wid][digit] = __popc(peers);
        __syncthreads();
        if (valid) {
            int32_t off = base_off[digit] + rank_in_warp;
            for (int w = 0; w < wid; ++w) off += wcount[w][digit];
            keys_out[off] = key;
            vals_out[off] = val;
        }
        __syncthreads();
        for (int b = threadIdx.x; b < kRadixBins; b += kSortThreads) {
            int32_t add = 0;
#pragma unroll
            for (int w = 0; w < W; ++w) add += wcount[w][b];
            base_off[b] += add;
        }
        __syncthreads();
    }
}

// ------------------------------------------- counting scatter (k <= 32768)
// The member list is the samples sorted by (label, index).  With per-tile
// cluster counts the position of sample i is
//   offsets[label_i] + (members of label_i in earlier tiles)
//                    + (members of label_i earlier in i's own tile),
// which three small kernels produce without a full sort.

// table[t][j] = members of cluster j among tile t's samples.
__global__ void __launch_bounds__(256)
    upd_tile_count_kernel(const int64_t *__restrict__ labels, int n, int k, int tile, int32_t *__restrict__ table,
                          uint32_t *status, WsHeader *hdr, int clear_header) {
    extern __shared__ int32_t cnt[];
    griddep_wait();
    if (clear_header && blockIdx.x == 0 && threadIdx.x == 0) {
        hdr->status = 0u;
        hdr->done_blocks = 0u;
    }
    for (int j = threadIdx.x; j < k; j += blockDim.x) cnt[j] = 0;
    __syncthreads();
    const int i0 = blockIdx.x * tile;
    const int i1 = min(n, i0 + tile);
    for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
        const uint32_t lab = clamp_label(labels[i], k, status);
        const uint32_t peers = __match_any_sync(__activemask(), lab);
        if ((int)(threadIdx.x & 31) == __ffs(peers) - 1) atomicAdd(&cnt[lab], __popc(peers));
    }
    __syncthreads();
    int32_t *row = table + (size_t)blockIdx.x * k;
    for (int j = threadIdx.x; j < k; j += blockDim.x) row[j] = cnt[j];
}

// The assignment's finalize step fused with the count above, for the Lloyd
// iteration: block t turns the packed keys of counting tile t into labels and
// distances (||x||^2 added back, clamped at 0), counts the tile's members per
// cluster, and adds its distances into a float64 block sum; the last block to
// finish adds the block sums in tile order.
constexpr int kFinCountThreads = 256;

__global__ void __launch_bounds__(kFinCountThreads)
    fin_tile_count_kernel(const unsigned long long *__restrict__ keys, const float *__restrict__ xnorm, int n, int k,
                          int tile, int64_t *__restrict__ labels, float *__restrict__ best, double *inertia,
                          double *partial, int32_t *__restrict__ table, WsHeader *hdr) {
    extern __shared__ int32_t cnt[];
    __shared__ double red[kFinCountThreads / 32];
    __shared__ int is_last;
    griddep_wait();
    for (int j = threadIdx.x; j < k; j += blockDim.x) cnt[j] = 0;
    __syncthreads();
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int i0 = blockIdx.x * tile;
    const int i1 = min(n, i0 + tile);
    double s = 0.0;
    for (int i = i0 + threadIdx.x; i < i1; i += blockDim.x) {
        const unsigned long long key = keys[i];
        uint32_t lab;
        if (key == kEmptyKey) {  // only for non-finite inputs
            labels[i] = -1;
            best[i] = __int_as_float(0x7fc00000);
            flag_error(&hdr->status, kFlagBadLabel);
            lab = (uint32_t)(k - 1);
        } else {
            lab = static_cast<uint32_t>(key & 0xffffffffu);
            const float b = fmaxf(0.f, xnorm[i] + ord_to_float(static_cast<uint32_t>(key >> 32)));
            labels[i] = static_cast<int64_t>(lab);
            best[i] = b;
            s += static_cast<double>(b);
        }
        const uint32_t peers = __match_any_sync(__activemask(), lab);
        if (lane == __ffs(peers) - 1) atomicAdd(&cnt[lab], __popc(peers));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_down_sync(0xffffffffu, s, o);
    if (lane == 0) red[wid] = s;
    __syncthreads();
    int32_t *row = table + (size_t)blockIdx.x * k;
    for (int j = threadIdx.x; j < k; j += blockDim.x) row[j] = cnt[j];
    if (inertia == nullptr) return;
    if (threadIdx.x == 0) {
        double b = 0.0;
        for (int w = 0; w < kFinCountThreads / 32; ++w) b += red[w];
        partial[blockIdx.x] = b;
        __threadfence();
        const unsigned t = atomicAdd(&hdr->done_blocks, 1u);
        is_last = (t == gridDim.x - 1u);
    }
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    // fixed order: strided per-thread sums, then the same warp and block tree
    double v = 0.0;
    for (int b = threadIdx.x; b < (int)gridDim.x; b += blockDim.x) v += __ldcg(partial + b);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    __syncthreads();
    if (lane == 0) red[wid] = v;
    __syncthreads();
    if (threadIdx.x == 0) {
        double t = 0.0;
        for (int w = 0; w < kFinCountThreads / 32; ++w) t += red[w];
        *inertia = t;
        hdr->done_blocks = 0u;
    }
}

// Per cluster: table[t][j] <- members of j in tiles before t; totals[j].
// One block covers kPrefixCols clusters; thread t holds tile t (the tile
// count equals the block size) and the tiles are scanned across the block.
// The exclusive offsets over the clusters are left to the scatter.
constexpr int kPrefixCols = 8;
__global__ void __launch_bounds__(kCountingTiles)
    upd_col_prefix_kernel(int32_t *__restrict__ table, int k, int32_t *__restrict__ totals) {
    __shared__ int32_t wsum[kCountingTiles / 32][kPrefixCols];
    griddep_wait();
    const int t = threadIdx.x;
    const int lane = t & 31, wid = t >> 5;
    const int j0 = blockIdx.x * kPrefixCols;
    int32_t v[kPrefixCols], incl[kPrefixCols];
#pragma unroll
    for (int u = 0; u < kPrefixCols; ++u) v[u] = (j0 + u < k) ? table[(size_t)t * k + j0 + u] : 0;
#pragma unroll
    for (int u = 0; u < kPrefixCols; ++u) {
        int32_t x = v[u];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        incl[u] = x;
        if (lane == 31) wsum[wid][u] = x;
    }
    __syncthreads();
#pragma unroll
    for (int u = 0; u < kPrefixCols; ++u) {
        int32_t before = 0, total = 0;
#pragma unroll
        for (int w = 0; w < kCountingTiles / 32; ++w) {
            const int32_t ws = wsum[w][u];
            if (w < wid) before += ws;
            total += ws;
        }
        if (j0 + u < k) {
            table[(size_t)t * k + j0 + u] = before + incl[u] - v[u];
            if (t == kCountingTiles - 1) totals[j0 + u] = total;
        }
    }
}

// Every block first scans the cluster totals (the exclusive offsets, which
// block 0 also writes out, k + 1 entries with the member total last) and adds
// its tile's column prefixes: the cursor of each cluster, in shared memory.
// One warp then walks the tile in index order, 32 samples at a time, the
// cursors giving the member-list positions; the whole block stages the tile's
// labels in shared memory first (the first round's labels are requested
// before the scan).  Meanwhile the other warps write the counts of the block's
// share of the clusters (j = block + i x blocks) and the rows of its empty
// clusters: the old row, or zeros with `mean` 0 (sums mode).
constexpr int kMaxCountingTile = 2048;  // samples per tile staged at once
constexpr int kScatterThreads = 256;
constexpr int kEmptyThreads = kScatterThreads - 32;
constexpr int kEmptyList = (int)((kCountingMaxK + kCountingTiles - 1) / kCountingTiles);  // clusters a block owns
constexpr int kEmptyUnroll = 8;

__global__ void __launch_bounds__(kScatterThreads)
    upd_tile_scatter_kernel(const int64_t *__restrict__ labels, int n, int k, int tile,
                            const int32_t *__restrict__ table, const int32_t *__restrict__ totals,
                            int32_t *__restrict__ offsets, int32_t *__restrict__ perm,
                            uint32_t *__restrict__ sorted_labels, uint32_t *status, const float *__restrict__ C_old,
                            float *__restrict__ C_new, int32_t *__restrict__ counts_out, int d, int mean) {
    constexpr int kPre = kMaxCountingTile / kScatterThreads;
    extern __shared__ int32_t cur[];
    __shared__ uint32_t lab_s[kMaxCountingTile];
    __shared__ int32_t wsum[kScatterThreads / 32];
    __shared__ int32_t empty_s[kEmptyList];
    __shared__ int n_empty;
    griddep_wait();
    const int32_t *row = table + (size_t)blockIdx.x * k;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    // warps 1.. take the block's share of the clusters for the counts and
    // empty rows, one each (a block owns at most kEmptyList <= kEmptyThreads
    // of them); their counts are requested now and used after the scan
    const int te = threadIdx.x - 32;
    const int64_t jl0 = blockIdx.x + (int64_t)(te < 0 ? 0 : te) * gridDim.x;
    const int32_t cnt0 = (te >= 0 && jl0 < k) ? totals[jl0] : -1;
    const int i0 = blockIdx.x * tile;
    const int i1 = min(n, i0 + tile);
    int64_t pre[kPre];
#pragma unroll
    for (int u = 0; u < kPre; ++u) {
        const int i = i0 + threadIdx.x + u * kScatterThreads;
        pre[u] = i < min(i1, i0 + kMaxCountingTile) ? labels[i] : 0;
    }
    // rounds of kScatterThreads x 8 clusters, thread t holding 8 consecutive
    // ones; `carry` is the member total of the rounds before
    int32_t carry = 0;
    for (int base = 0; base < k; base += kScatterThreads * 8) {
        const int j = base + threadIdx.x * 8;
        int32_t q[8], r[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            q[e] = j + e < k ? totals[j + e] : 0;
            r[e] = j + e < k ? row[j + e] : 0;
        }
        int32_t run = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) run += q[e];
        int32_t x = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) wsum[wid] = x;
        __syncthreads();
        int32_t before = carry + x - run, round_total = 0;
#pragma unroll
        for (int w = 0; w < kScatterThreads / 32; ++w) {
            const int32_t ws = wsum[w];
            if (w < wid) before += ws;
            round_total += ws;
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (j + e < k) {
                if (blockIdx.x == 0) offsets[j + e] = before;
                cur[j + e] = before + r[e];
            }
            before += q[e];
        }
        carry += round_total;
        __syncthreads();  // wsum is rewritten by the next round
    }
    if (blockIdx.x == 0 && threadIdx.x == 0) offsets[k] = carry;
    for (int c0 = i0; c0 < i1; c0 += kMaxCountingTile) {
        const int c1 = min(i1, c0 + kMaxCountingTile);
        __syncthreads();
        if (c0 == i0) {
#pragma unroll
            for (int u = 0; u < kPre; ++u) {
                const int i = c0 + threadIdx.x + u * kScatterThreads;
                if (i < c1) lab_s[i - c0] = clamp_label(pre[u], k, status);
            }
        } else {
            for (int i = c0 + threadIdx.x; i < c1; i += blockDim.x) lab_s[i - c0] = clamp_label(labels[i], k, status);
        }
        __syncthreads();
        if (threadIdx.x < 32) {
            for (int b = c0; b < c1; b += 32) {
                const int i = b + lane;
                const bool valid = i < c1;
                const uint32_t lab = valid ? lab_s[i - c0] : 0xffffffffu;
                const uint32_t peers = __match_any_sync(0xffffffffu, lab);
                const int rank = __popc(peers & ((1u << lane) - 1u));
                int32_t pos = 0;
                if (valid) pos = cur[lab] + rank;
                __syncwarp();
                if (valid && rank == 0) cur[lab] += __popc(peers);
                __syncwarp();
                if (valid) {
                    perm[pos] = i;
                    sorted_labels[pos] = lab;
                }
            }
        }
    }
    if (wid == 0) return;
    // warps 1.. (kEmptyThreads threads) meet on named barrier 1; warp 0 is
    // still walking
    if (te == 0) n_empty = 0;
    asm volatile("bar.sync 1, %0;" ::"n"(kEmptyThreads) : "memory");
    for (int64_t jl = jl0; jl < k; jl += (int64_t)kEmptyThreads * gridDim.x) {
        const int j = (int)jl;
        const int32_t cnt = jl == jl0 ? cnt0 : totals[j];
        if (counts_out) counts_out[j] = cnt;
        if (cnt == 0) {
            const int slot = atomicAdd(&n_empty, 1);
            if (slot < kEmptyList) {
                empty_s[slot] = j;
            } else {  // not reached with k <= kCountingMaxK over kCountingTiles blocks
                for (int f = 0; f < d; ++f) C_new[(size_t)j * d + f] = mean ? C_old[(size_t)j * d + f] : 0.f;
            }
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kEmptyThreads) : "memory");
    const int ne = min(n_empty, kEmptyList);
    if (ne == 0 || (mean && C_new == C_old)) return;
    // the listed rows as one flat range of ne x d floats (four at a time
    // where rows are whole aligned float4s), kEmptyUnroll loads in flight per
    // thread
    if ((d & 3) == 0 && ((reinterpret_cast<uintptr_t>(C_new) | reinterpret_cast<uintptr_t>(C_old)) & 15) == 0) {
        const int d4 = d >> 2;
        const int64_t total4 = (int64_t)ne * d4;
        for (int64_t g0 = te; g0 < total4; g0 += (int64_t)kEmptyThreads * kEmptyUnroll) {
            float4 v[kEmptyUnroll];
#pragma unroll
            for (int u = 0; u < kEmptyUnroll; ++u) {
                const int64_t g = g0 + (int64_t)u * kEmptyThreads;
                v[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                if (mean && g < total4)
                    v[u] = reinterpret_cast<const float4 *>(C_old + (size_t)empty_s[g / d4] * d)[g % d4];
            }
#pragma unroll
            for (int u = 0; u < kEmptyUnroll; ++u) {
                const int64_t g = g0 + (int64_t)u * kEmptyThreads;
                if (g < total4) reinterpret_cast<float4 *>(C_new + (size_t)empty_s[g / d4] * d)[g % d4] = v[u];
            }
        }
        return;
    }
    const int64_t total = (int64_t)ne * d;
    for (int64_t g0 = te; g0 < total; g0 += (int64_t)kEmptyThreads * kEmptyUnroll) {
        float v[kEmptyUnroll];
#pragma unroll
        for (int u = 0; u < kEmptyUnroll; ++u) {
            const int64_t g = g0 + (int64_t)u * kEmptyThreads;
            v[u] = 0.f;
            if (mean && g < total) v[u] = C_old[(size_t)empty_s[g / d] * d + g % d];
        }
#pragma unroll
        for (int u = 0; u < kEmptyUnroll; ++u) {
            const int64_t g = g0 + (int64_t)u * kEmptyThreads;
            if (g < total) C_new[(size_t)empty_s[g / d] * d + g % d] = v[u];
        }
    }
}

__device__ __forceinline__ void kahan4(float4 &s, float4 &c, const float4 v) {
    float y, t;
    y = v.x - c.x; t = s.x + y; c.x = (t - s.x) - y; s.x = t;
    y = v.y - c.y; t = s.y + y; c.y = (t - s.y) - y; s.y = t;
    y = v.z - c.z; t = s.z + y; c.z = (t - s.z) - y; s.z = t;
    y = v.w - c.w; t = s.w + y; c.w = (t - s.w) - y; s.w = t;
}

constexpr int kMeanThreads = 128;

// One CTA = one chunk of the member list x one slice of columns.
// VEC: 4 columns per thread with 16-byte loads (d % 4 == 0, X aligned).
// MEAN: a segment inside the chunk writes its mean; otherwise its sum.
template <bool VEC, bool MEAN>
__global__ void __launch_bounds__(kMeanThreads)
    segmented_mean_kernel(const float *__restrict__ X, const int32_t *__restrict__ perm,
                          const uint32_t *__restrict__ sorted_labels, const int32_t *__restrict__ offsets,
                          int n, int d, int chunk, float *__restrict__ C_new, float *__restrict__ head,
                          float *__restrict__ tail, int4 *__restrict__ tailc) {
    extern __shared__ int32_t s_members[];  // [chunk] sample indices, then [chunk] labels
    griddep_wait();
    int32_t *s_perm = s_members;
    uint32_t *s_lab = reinterpret_cast<uint32_t *>(s_members + chunk);
    const int c = blockIdx.x;
    if (tailc && blockIdx.y == 0 && threadIdx.x == 0) tailc[c] = make_int4(-1, 0, 0, 0);
    const int p0 = c * chunk;
    const int p1 = min(n, p0 + chunk);
    for (int p = p0 + threadIdx.x; p < p1; p += kMeanThreads) {
        s_perm[p - p0] = perm[p];
        s_lab[p - p0] = sorted_labels[p];
    }
    __syncthreads();
    constexpr int CPT = VEC ? 4 : 1;  // columns per thread
    const int col = (blockIdx.y * kMeanThreads + threadIdx.x) * CPT;
    if (col >= d) return;
    int p = p0;
    while (p < p1) {
        const uint32_t j = s_lab[p - p0];
        const int seg0 = offsets[j];
        const int seg1 = offsets[j + 1];
        int q = min(seg1, p1);
        if (q <= p) q = p + 1;  // only reachable with inconsistent (invalid) labels
        float4 s = make_float4(0.f, 0.f, 0.f, 0.f), cmp = make_float4(0.f, 0.f, 0.f, 0.f);
        int r = p;
        if (VEC) {
            // 32 member rows in flight, then 16, 8, 4, 1 (measured: 32 over 8
            // is 7-9% faster on every workload; the sums keep member order)
            for (; r + 32 <= q; r += 32) {
                float4 v[32];
#pragma unroll
                for (int u = 0; u < 32; ++u)
                    v[u] = __ldg(reinterpret_cast<const float4 *>(X + (size_t)s_perm[r + u - p0] * d + col));
#pragma unroll
                for (int u = 0; u < 32; ++u) kahan4(s, cmp, v[u]);
            }
            for (; r + 16 <= q; r += 16) {
                float4 v[16];
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    v[u] = __ldg(reinterpret_cast<const float4 *>(X + (size_t)s_perm[r + u - p0] * d + col));
#pragma unroll
                for (int u = 0; u < 16; ++u) kahan4(s, cmp, v[u]);
            }
            for (; r + 8 <= q; r += 8) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u)
                    v[u] = __ldg(reinterpret_cast<const float4 *>(X + (size_t)s_perm[r + u - p0] * d + col));
#pragma unroll
                for (int u = 0; u < 8; ++u) kahan4(s, cmp, v[u]);
            }
            for (; r + 4 <= q; r += 4) {
                const float4 v0 = __ldg(reinterpret_cast<const float4 *>(X + (size_t)s_perm[r - p0] * d + col));
                const float4 v1 = __ldg(reinterpret_cast<const float4 *>(X + (size_t)s_perm[r + 1 - p0] * d + col));
                const float4 v2 = __ldg(reinterpret_cast<const float4 *>(X + (size_t)s_perm[r + 2 - p0] * d + col));
                const float4 v3 = __ldg(reinterpret_cast<const float4 *>(X + (size_t)s_perm[r + 3 - p0] * d + col));
                kahan4(s, cmp, v0);
                kahan4(s, cmp, v1);
                kahan4(s, cmp, v2);
                kahan4(s, cmp, v3);
            }
            for (; r < q; ++r)
                kahan4(s, cmp, __ldg(reinterpret_cast<const float4 *>(X + (size_t)s_perm[r - p0] * d + col)));
        } else {
            for (; r < q; ++r) {
                const float v = __ldg(X + (size_t)s_perm[r - p0] * d + col);
                const float y = v - cmp.x;
                const float t = s.x + y;
                cmp.x = (t - s.x) - y;
                s.x = t;
            }
        }
        const float4 tot = make_float4(s.x - cmp.x, s.y - cmp.y, s.z - cmp.z, s.w - cmp.w);
        float *dst;
        bool mean = false;
        if (seg0 >= p0 && seg1 <= p1) {
            dst = C_new + (size_t)j * d + col;
            mean = true;
        } else if (seg0 < p0) {
            dst = head + (size_t)c * d + col;
        } else {
            dst = tail + (size_t)c * d + col;
            if (tailc && blockIdx.y == 0 && threadIdx.x == 0) tailc[c] = make_int4((int)j, seg0, seg1, 0);
        }
        if (MEAN && mean) {
            const float cnt = (float)(seg1 - seg0);
            if (VEC) *reinterpret_cast<float4 *>(dst) = make_float4(tot.x / cnt, tot.y / cnt, tot.z / cnt, tot.w / cnt);
            else *dst = tot.x / cnt;
        } else {
            if (VEC) *reinterpret_cast<float4 *>(dst) = tot;
            else *dst = tot.x;
        }
        p = q;
    }
}

// Segments that crossed chunk boundaries, empty clusters, and the counts.
// With `mean` 0 (sums mode) crossing segments write their sum and empty
// clusters zeros.
__global__ void __launch_bounds__(kMeanThreads)
    mean_fixup_kernel(const int32_t *__restrict__ offsets, const float *__restrict__ head,
                      const float *__restrict__ tail, const float *__restrict__ C_old, float *__restrict__ C_new,
                      int32_t *__restrict__ counts_out, int k, int d, int chunk, int mean) {
    for (int j = blockIdx.x; j < k; j += gridDim.x) {
        const int seg0 = offsets[j];
        const int seg1 = offsets[j + 1];
        const int cnt = seg1 - seg0;
        if (counts_out && threadIdx.x == 0) counts_out[j] = cnt;
        if (cnt == 0) {
            if (!mean)
                for (int f = threadIdx.x; f < d; f += kMeanThreads) C_new[(size_t)j * d + f] = 0.f;
            else if (C_new != C_old)
                for (int f = threadIdx.x; f < d; f += kMeanThreads) C_new[(size_t)j * d + f] = C_old[(size_t)j * d + f];
            continue;
        }
        const int cs = seg0 / chunk;
        const int ce = (seg1 - 1) / chunk;
        if (cs == ce) continue;
        for (int f = threadIdx.x; f < d; f += kMeanThreads) {
            float s = tail[(size_t)cs * d + f], cmp = 0.f;
            for (int c = cs + 1; c <= ce; ++c) {
                const float v = head[(size_t)c * d + f];
                const float y = v - cmp;
                const float t = s + y;
                cmp = (t - s) - y;
                s = t;
            }
            C_new[(size_t)j * d + f] = mean ? (s - cmp) / (float)cnt : s - cmp;
        }
    }
}

// Fix-up of the counting path: block c finishes the cluster that leaves
// chunk c (its tail partial plus the head partials of the chunks it covers, in
// chunk order).  A thread keeps kFixUnroll column groups (four columns each
// when VEC) in flight at once.  (The counts and the empty clusters' rows are
// written by the scatter.)
constexpr int kFixThreads = 256;
constexpr int kFixUnroll = 4;

template <bool VEC, bool MEAN>
__global__ void __launch_bounds__(kFixThreads)
    mean_fixup_chunks_kernel(const float *__restrict__ head, const float *__restrict__ tail,
                             const int4 *__restrict__ tailc, int n_chunks, float *__restrict__ C_new, int d,
                             int chunk) {
    using V = typename std::conditional<VEC, float4, float>::type;
    griddep_wait();
    constexpr int W = VEC ? 4 : 1;
    const int dv = d / W;  // VEC: d % 4 == 0
    for (int c = blockIdx.x; c < n_chunks; c += gridDim.x) {
        const int4 tc = tailc[c];  // {cluster, its first member, one past its last}
        const int j = tc.x;
        if (j < 0) continue;
        const int seg0 = tc.y;
        const int seg1 = tc.z;
        const int ce = (seg1 - 1) / chunk;
        const float cnt = (float)(seg1 - seg0);
        const V *tl = reinterpret_cast<const V *>(tail + (size_t)c * d);
        V *out = reinterpret_cast<V *>(C_new + (size_t)j * d);
        for (int g0 = threadIdx.x; g0 < dv; g0 += kFixThreads * kFixUnroll) {
            float s[kFixUnroll][W], cmp[kFixUnroll][W];
#pragma unroll
            for (int u = 0; u < kFixUnroll; ++u) {
                const int g = g0 + u * kFixThreads;
                V x;
                if (g < dv) x = tl[g]; else x = V{};
                const float *xf = reinterpret_cast<const float *>(&x);
#pragma unroll
                for (int e = 0; e < W; ++e) {
                    s[u][e] = xf[e];
                    cmp[u][e] = 0.f;
                }
            }
            for (int cc = c + 1; cc <= ce; ++cc) {
                const V *hd = reinterpret_cast<const V *>(head + (size_t)cc * d);
                V v[kFixUnroll];
#pragma unroll
                for (int u = 0; u < kFixUnroll; ++u) {
                    const int g = g0 + u * kFixThreads;
                    if (g < dv) v[u] = hd[g]; else v[u] = V{};
                }
#pragma unroll
                for (int u = 0; u < kFixUnroll; ++u) {
                    const float *vf = reinterpret_cast<const float *>(&v[u]);
#pragma unroll
                    for (int e = 0; e < W; ++e) {
                        const float y = vf[e] - cmp[u][e];
                        const float t = s[u][e] + y;
                        cmp[u][e] = (t - s[u][e]) - y;
                        s[u][e] = t;
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kFixUnroll; ++u) {
                const int g = g0 + u * kFixThreads;
                if (g >= dv) continue;
                V r;
                float *rf = reinterpret_cast<float *>(&r);
#pragma unroll
                for (int e = 0; e < W; ++e) rf[e] = MEAN ? (s[u][e] - cmp[u][e]) / cnt : s[u][e] - cmp[u][e];
                out[g] = r;
            }
        }
    }
}

// The mean step after the update fused into the assignment: C_new = sums /
// count per cluster (the same division as the sorted path), the old row for
// an empty cluster, and the counts.
__global__ void __launch_bounds__(256)
    fused_mean_kernel(const float4 *__restrict__ sums, const int32_t *__restrict__ cnt, const float *__restrict__ C_old,
                      float *__restrict__ C_new, int32_t *__restrict__ counts_out, int k, int d4) {
    griddep_wait();
    const int64_t total = (int64_t)k * d4;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < total; g += (int64_t)gridDim.x * blockDim.x) {
        const int j = (int)(g / d4);
        const int c = cnt[j];
        float4 v;
        if (c > 0) {
            const float4 sv = sums[g];
            const float f = (float)c;
            v = make_float4(sv.x / f, sv.y / f, sv.z / f, sv.w / f);
        } else {
            v = reinterpret_cast<const float4 *>(C_old)[g];
        }
        reinterpret_cast<float4 *>(C_new)[g] = v;
        if (counts_out && g - (int64_t)j * d4 == 0) counts_out[j] = c;
    }
}

cudaError_t launch_fused_mean(const float *sums, const int32_t *cnt, const float *C_old, float *C_new,
                              int32_t *counts_out, int64_t k, int64_t d, cudaStream_t s) {
    const int64_t total = k * (d / 4);
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    return launch_kernel(true, fused_mean_kernel, dim3((unsigned)(blocks < 1 ? 1 : blocks)), dim3(256), 0, s,
                         reinterpret_cast<const float4 *>(sums), cnt, C_old, C_new, counts_out, (int)k, (int)(d / 4));
}

// The sample-sharded iteration's reduction of one slice of centroid rows:
// every rank's partial sum of row j, added in rank order in float64 (the
// first rank's value taken as it is, so one rank gives the same bits as the
// single-GPU mean), divided once by the summed count and rounded to float32;
// the old row when no rank has a member.  The inertia is the rank-order sum
// of the ranks' inertias.
template <bool VEC>
__global__ void __launch_bounds__(256)
    reduce_partials_kernel(const float *__restrict__ parts, const int32_t *__restrict__ pcounts,
                           const double *__restrict__ pinertia, int world, int64_t rows, int d,
                           const float *__restrict__ C_old, float *__restrict__ C_new,
                           int32_t *__restrict__ counts_out, double *__restrict__ inertia_out) {
    using V = typename std::conditional<VEC, float4, float>::type;
    constexpr int W = VEC ? 4 : 1;
    const int64_t dv = d / W;
    const int64_t total = rows * dv;
    const int64_t plane = rows * (int64_t)d;  // floats per rank
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < total;
         g += (int64_t)gridDim.x * blockDim.x) {
        const int64_t j = g / dv;
        const int64_t off = j * d + (g - j * dv) * W;
        int64_t cnt = 0;
        for (int r = 0; r < world; ++r) cnt += pcounts[(int64_t)r * rows + j];
        if (cnt == 0) {
            *reinterpret_cast<V *>(C_new + off) = *reinterpret_cast<const V *>(C_old + off);
        } else if constexpr (VEC) {
            float4 v = *reinterpret_cast<const float4 *>(parts + off);
            double a0 = v.x, a1 = v.y, a2 = v.z, a3 = v.w;
            for (int r = 1; r < world; ++r) {
                v = *reinterpret_cast<const float4 *>(parts + (int64_t)r * plane + off);
                a0 += v.x;
                a1 += v.y;
                a2 += v.z;
                a3 += v.w;
            }
            const double c = (double)cnt;
            *reinterpret_cast<float4 *>(C_new + off) =
                make_float4((float)(a0 / c), (float)(a1 / c), (float)(a2 / c), (float)(a3 / c));
        } else {
            double a = parts[off];
            for (int r = 1; r < world; ++r) a += parts[(int64_t)r * plane + off];
            C_new[off] = (float)(a / (double)cnt);
        }
        if (counts_out && off == j * d) counts_out[j] = (int32_t)cnt;
    }
    if (inertia_out && blockIdx.x == 0 && threadIdx.x == 0) {
        double acc = pinertia[0];
        for (int r = 1; r < world; ++r) acc += pinertia[r];
        *inertia_out = acc;
    }
}

cudaError_t launch_reduce_partials(const float *parts, const int32_t *part_counts, const double *part_inertia,
                                   int world, int64_t rows, int64_t d, const float *C_old, float *C_new,
                                   int32_t *counts_out, double *inertia_out, cudaStream_t s) {
    const bool vec = (d % 4 == 0) && ((reinterpret_cast<uintptr_t>(parts) | reinterpret_cast<uintptr_t>(C_old) |
                                       reinterpret_cast<uintptr_t>(C_new)) & 15) == 0;
    const int64_t total = rows * (vec ? d / 4 : d);
    int64_t blocks = (total + 255) / 256;
    if (blocks > 152 * 16) blocks = 152 * 16;
    if (blocks < 1) blocks = 1;
    if (vec)
        reduce_partials_kernel<true><<<(unsigned)blocks, 256, 0, s>>>(parts, part_counts, part_inertia, world, rows,
                                                                      (int)d, C_old, C_new, counts_out, inertia_out);
    else
        reduce_partials_kernel<false><<<(unsigned)blocks, 256, 0, s>>>(parts, part_counts, part_inertia, world, rows,
                                                                       (int)d, C_old, C_new, counts_out, inertia_out);
    return cudaGetLastError();
}

// Per device, once: allow the per-cluster shared-memory counters of the
// counting path above the 48 KiB default.
static void set_counting_smem_limits(int64_t k) {
    if (k * 4 <= 48 * 1024) return;
    static std::once_flag attr_once[kMaxDevices];
    once_per_device(attr_once, [] {
        cudaFuncSetAttribute(upd_tile_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kCountingMaxK * 4));
        cudaFuncSetAttribute(fin_tile_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kCountingMaxK * 4));
        cudaFuncSetAttribute(upd_tile_scatter_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)(kCountingMaxK * 4));
    });
}

static int radix_passes(int64_t k) {
    int bits = 0;
    while (bits < 32 && ((int64_t)1 << bits) < k) ++bits;  // labels 0..k-1 need `bits` bits
    const int p = (bits + 7) / 8;
    return p < 1 ? 1 : p;
}

cudaError_t launch_update(const float *X, const int64_t *labels, const float *C_old, float *C_new,
                          int32_t *counts_out, int64_t n, int64_t k, int64_t d, const UpdateLayout &L,
                          uint8_t *ws, bool clear_header, cudaStream_t s, bool tile_counts_ready, bool sums_only) {
    WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + L.off_counts);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.off_offsets);
    int32_t *hist = reinterpret_cast<int32_t *>(ws + L.off_hist);
    uint32_t *ka = reinterpret_cast<uint32_t *>(ws + L.off_keys_a);
    int32_t *va = reinterpret_cast<int32_t *>(ws + L.off_vals_a);
    uint32_t *kb = reinterpret_cast<uint32_t *>(ws + L.off_keys_b);
    int32_t *vb = reinterpret_cast<int32_t *>(ws + L.off_vals_b);
    float *head = reinterpret_cast<float *>(ws + L.off_head);
    float *tail = reinterpret_cast<float *>(ws + L.off_tail);
    uint32_t *status = &hdr->status;
    const int tiles = (int)L.n_tiles;
    const bool vec = (d % 4 == 0) && ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(C_new)) & 15) == 0;
    const int cols_per_cta = kMeanThreads * (vec ? 4 : 1);
    const dim3 mgrid((unsigned)L.n_chunks, (unsigned)((d + cols_per_cta - 1) / cols_per_cta));
    const size_t msmem = (size_t)L.chunk * 8;
    // sums mode (a shard of the samples): sums instead of means, zeros for an
    // empty cluster
    const bool mean = !sums_only;
    auto *mean_k = vec ? (mean ? segmented_mean_kernel<true, true> : segmented_mean_kernel<true, false>)
                       : (mean ? segmented_mean_kernel<false, true> : segmented_mean_kernel<false, false>);
    auto *fix_k = vec ? (mean ? mean_fixup_chunks_kernel<true, true> : mean_fixup_chunks_kernel<true, false>)
                      : (mean ? mean_fixup_chunks_kernel<false, true> : mean_fixup_chunks_kernel<false, false>);

    if (L.counting) {
        int32_t *table = reinterpret_cast<int32_t *>(ws + L.off_table);
        int32_t *perm = va;
        uint32_t *slab = ka;
        int4 *tailc = reinterpret_cast<int4 *>(ws + L.off_tailc);
        const int ut = (int)L.n_utiles;
        const size_t csmem = (size_t)k * 4;
        set_counting_smem_limits(k);
        cudaError_t e = cudaSuccess;
        if (!tile_counts_ready)
            e = launch_kernel(true, upd_tile_count_kernel, dim3(ut), dim3(256), csmem, s, labels, (int)n,
                              (int)k, (int)L.utile, table, status, hdr, clear_header ? 1 : 0);
        if (e == cudaSuccess)
            e = launch_kernel(true, upd_col_prefix_kernel, dim3((unsigned)((k + kPrefixCols - 1) / kPrefixCols)),
                              dim3(kCountingTiles), 0, s, table, (int)k, counts);
        if (e == cudaSuccess)
            e = launch_kernel(true, upd_tile_scatter_kernel, dim3(ut), dim3(kScatterThreads), csmem, s, labels,
                              (int)n, (int)k, (int)L.utile, (const int32_t *)table, (const int32_t *)counts, offsets,
                              perm, slab, status, C_old, C_new, counts_out, (int)d, mean ? 1 : 0);
        trace_mark(kTraceUpdateMean, false, s);
        if (e == cudaSuccess)
            e = launch_kernel(true, mean_k, mgrid, dim3(kMeanThreads), msmem, s, X, (const int32_t *)perm,
                              (const uint32_t *)slab, (const int32_t *)offsets, (int)n, (int)d, (int)L.chunk, C_new,
                              head, tail, tailc);
        trace_mark(kTraceUpdateMean, true, s);
        if (e == cudaSuccess)
            e = launch_kernel(true, fix_k, dim3((unsigned)L.n_chunks), dim3(kFixThreads), 0, s,
                              (const float *)head, (const float *)tail,
                              (const int4 *)tailc, (int)L.n_chunks, C_new, (int)d, (int)L.chunk);
        return e;
    }

    const unsigned clear_grid = (unsigned)((k + 255) / 256 < 1024 ? (k + 255) / 256 : 1024);
    cudaError_t ce = launch_kernel(true, update_clear_kernel, dim3(clear_grid), dim3(256), 0, s, counts, (int)k, hdr,
                                   clear_header ? 1 : 0);
    if (ce != cudaSuccess) return ce;
    const int passes = radix_passes(k);
    uint32_t *kin = nullptr, *kout = ka;
    int32_t *vin = nullptr, *vout = va;
    for (int ps = 0; ps < passes; ++ps) {
        const int shift = 8 * ps;
        const int64_t *lab = ps == 0 ? labels : nullptr;
        radix_hist_kernel<<<tiles, kSortThreads, 0, s>>>(lab, kin, (int)n, (int)k, shift, tiles, hist, counts,
                                                          status);
        exclusive_scan_kernel<<<1, 1024, 0, s>>>(hist, hist, (int64_t)kRadixBins * tiles, nullptr);
        radix_scatter_kernel<<<tiles, kSortThreads, 0, s>>>(lab, kin, vin, (int)n, (int)k, shift, tiles, hist,
                                                             kout, vout, status);
        kin = kout;
        vin = vout;
        kout = (kout == ka) ? kb : ka;
        vout = (vout == va) ? vb : va;
    }
    // counts -> offsets (k + 1 entries: the scan writes the total at [k])
    exclusive_scan_kernel<<<1, 1024, 0, s>>>(counts, offsets, k, offsets + k);

    trace_mark(kTraceUpdateMean, false, s);
    mean_k<<<mgrid, kMeanThreads, msmem, s>>>(X, vin, kin, offsets, (int)n, (int)d, (int)L.chunk, C_new, head, tail,
                                              nullptr);
    trace_mark(kTraceUpdateMean, true, s);
    const int fix_grid = (int)(k < 4096 ? k : 4096);
    mean_fixup_kernel<<<fix_grid, kMeanThreads, 0, s>>>(offsets, head, tail, C_old, C_new, counts_out, (int)k,
                                                       (int)d, (int)L.chunk, mean ? 1 : 0);
    return cudaGetLastError();
}

cudaError_t launch_finalize_counting(int64_t n, int64_t k, const AssignLayout &A, const UpdateLayout &U,
                                     uint8_t *ws, int64_t *labels, float *best, double *inertia, cudaStream_t s) {
    set_counting_smem_limits(k);
    return launch_kernel(true, fin_tile_count_kernel, dim3((unsigned)U.n_utiles), dim3(kFinCountThreads),
                         (size_t)k * 4, s, reinterpret_cast<const unsigned long long *>(ws + A.off_keys),
                         reinterpret_cast<const float *>(ws + A.off_xnorm), (int)n, (int)k, (int)U.utile, labels,
                         best, inertia, reinterpret_cast<double *>(ws + U.off_fin_partial),
                         reinterpret_cast<int32_t *>(ws + U.off_table), reinterpret_cast<WsHeader *>(ws));
}

}  // namespace km

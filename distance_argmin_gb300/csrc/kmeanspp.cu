// Greedy k-means++ seeding ("004 — tile sizes, a Cython Lloyd step, and
// k-means++", section "k-means++": 2 + log(n_clusters) candidate trials per new
// center).  The centers are chosen one after the other; each round is:
//
//   K1 blocksum  D^2 <- min(D^2, distances to the previous winner); per-block
//                sums of D^2 (fixed order)
//   K2 pick      per trial: uniform from Philox4x32-10, target = u * sum D^2,
//                candidate = first sample whose running sum exceeds the target
//   K3 dist      one pass over X: squared distance of every sample to every
//                trial candidate; per-CTA partial potentials
//                sum_i min(D^2_i, dist_ti)
//   K4 select    potential per trial, lowest wins (lowest trial on ties)
//
// Distances: float32 differences, squared and summed in runs of 8 features,
// runs added with compensation, lanes combined in float64.  Running sums and
// potentials are float64.  Every reduction has a fixed order.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kmeanspp.cuh"

namespace km {

// ------------------------------------------- Philox4x32-10 (Salmon et al.)
__device__ __forceinline__ void philox_round(uint32_t &c0, uint32_t &c1, uint32_t &c2, uint32_t &c3, uint32_t k0,
                                             uint32_t k1) {
    const uint32_t lo0 = 0xD2511F53u * c0;
    const uint32_t hi0 = __umulhi(0xD2511F53u, c0);
    const uint32_t lo1 = 0xCD9E8D57u * c2;
    const uint32_t hi1 = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi1 ^ c1 ^ k0;
    const uint32_t n2 = hi0 ^ c3 ^ k1;
    c0 = n0;
    c1 = lo1;
    c2 = n2;
    c3 = lo0;
}

__device__ double philox_uniform(uint64_t seed, uint64_t draw) {
    uint32_t c0 = (uint32_t)draw, c1 = (uint32_t)(draw >> 32), c2 = 0u, c3 = 0u;
    uint32_t k0 = (uint32_t)seed, k1 = (uint32_t)(seed >> 32);
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r) {
            k0 += 0x9E3779B9u;
            k1 += 0xBB67AE85u;
        }
        philox_round(c0, c1, c2, c3, k0, k1);
    }
    const uint64_t bits = ((static_cast<uint64_t>(c0) << 32) | c1) >> 11;
    return static_cast<double>(bits) * 1.1102230246251565404236316680908203125e-16;  // 2^-53
}

// -------------------------------------------------------------- first center
__global__ void kpp_first_kernel(int64_t n, uint64_t seed, int64_t *cand, int64_t *indices, WsHeader *hdr) {
    hdr->status = 0u;
    hdr->done_blocks = 0u;
    const double u = philox_uniform(seed, 0);
    int64_t idx = static_cast<int64_t>(u * static_cast<double>(n));  // u >= 0: truncation is floor
    if (idx > n - 1) idx = n - 1;
    cand[0] = idx;
    indices[0] = idx;
}

// --------------------------------------------------------------- K1 blocksum
constexpr int kBsThreads = 256;

__global__ void __launch_bounds__(kBsThreads)
    kpp_blocksum_kernel(const double *__restrict__ dist, const int32_t *__restrict__ sel_t, int64_t n, int init,
                        double *__restrict__ D2, double *__restrict__ bsum) {
    __shared__ double red[kBsThreads];
    const double *db = dist + (init ? 0 : (int64_t)(*sel_t) * n);
    const int64_t base = (int64_t)blockIdx.x * kKppScanBlock;
    double s = 0.0;
#pragma unroll
    for (int q = 0; q < kKppScanBlock / kBsThreads; ++q) {
        const int64_t i = base + threadIdx.x + (int64_t)q * kBsThreads;
        if (i < n) {
            const double v = db[i];
            const double nd = init ? v : fmin(D2[i], v);
            D2[i] = nd;
            s += nd;
        }
    }
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = kBsThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) bsum[blockIdx.x] = red[0];
}

// ------------------------------------------------------------------ K2 pick
__device__ __forceinline__ double warp_incl_scan(double v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// The running sum at sample i is (sum of the block sums before its block) +
// (the in-block prefix up to i); the block-sum prefix is the same for every
// trial, so all trials see one consistent running sum.
__global__ void kpp_pick_kernel(const double *__restrict__ bsum, int64_t n_blocks, const double *__restrict__ D2,
                                int64_t n, uint64_t seed, uint64_t draw_base, int T, int64_t *__restrict__ cand) {
    const int lane = threadIdx.x & 31;
    const int t = threadIdx.x >> 5;
    if (t >= T) return;
    // total of D^2
    double total = 0.0;
    for (int64_t b0 = 0; b0 < n_blocks; b0 += 32) {
        const double v = (b0 + lane < n_blocks) ? bsum[b0 + lane] : 0.0;
        const double incl = warp_incl_scan(v, lane);
        total += __shfl_sync(0xffffffffu, incl, 31);
    }
    const double target = philox_uniform(seed, draw_base + (uint64_t)t) * total;
    // first block whose inclusive prefix exceeds the target
    double before = 0.0;  // sum of block sums before the current chunk
    int64_t blk = -1;
    double blk_before = 0.0;
    for (int64_t b0 = 0; b0 < n_blocks && blk < 0; b0 += 32) {
        const double v = (b0 + lane < n_blocks) ? bsum[b0 + lane] : 0.0;
        const double incl = before + warp_incl_scan(v, lane);
        const uint32_t hit = __ballot_sync(0xffffffffu, (b0 + lane < n_blocks) && incl > target);
        if (hit) {
            const int l = __ffs(hit) - 1;
            blk = b0 + l;
            blk_before = __shfl_sync(0xffffffffu, incl - v, l);
        }
        before += __shfl_sync(0xffffffffu, incl - before, 31);
    }
    int64_t pick = n - 1;
    // scan samples from that block on (later blocks only matter if rounding
    // put the target between the block's own running sum and its block sum)
    if (blk >= 0) {
        double run = blk_before;
        bool found = false;
        for (int64_t i0 = blk * kKppScanBlock; i0 < n && !found; i0 += 32) {
            const double v = (i0 + lane < n) ? D2[i0 + lane] : 0.0;
            const double incl = run + warp_incl_scan(v, lane);
            const uint32_t hit = __ballot_sync(0xffffffffu, (i0 + lane < n) && incl > target);
            if (hit) {
                pick = i0 + (__ffs(hit) - 1);
                found = true;
            }
            run = __shfl_sync(0xffffffffu, incl, 31);
        }
    }
    if (lane == 0) cand[t] = pick;
}

// ------------------------------------------------------------------ K3 dist
namespace kd {
constexpr int KT = 8;        // trial candidates per pass over X
constexpr int ROWS = 2;      // samples per warp at a time
constexpr int WARPS = 8;
constexpr int THREADS = WARPS * 32;
constexpr int SL = 1024;     // features of the candidates staged per slice
constexpr int GROUP = WARPS * ROWS;
}  // namespace kd

__device__ __forceinline__ void kahan(float &s, float &c, float v) {
    const float y = v - c;
    const float t = s + y;
    c = (t - s) - y;
    s = t;
}

template <bool VEC>
__device__ __forceinline__ void load8(const float *__restrict__ p, int avail, float (&v)[8]) {
    if (VEC && avail >= 8) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p + 4));
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) v[e] = e < avail ? __ldg(p + e) : 0.f;
    }
}

// dist[t][i] = ||x_i - x_cand[t]||^2 for t in [t0, min(T, t0 + KT)), and
// bpot[t][blockIdx.x] = sum over this CTA's samples of min(D2_i, dist[t][i])
// (skipped when D2 is null).
template <bool VEC>
__global__ void __launch_bounds__(kd::THREADS, 2)
    kpp_dist_kernel(const float *__restrict__ X, int64_t n, int d, const int64_t *__restrict__ cand, int T, int t0,
                    const double *__restrict__ D2, double *__restrict__ dist, double *__restrict__ bpot) {
    __shared__ __align__(16) float cs[kd::KT][kd::SL];
    __shared__ double wpot[kd::WARPS][kd::KT];
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nt = min(kd::KT, T - t0);
    double pot[kd::KT];
#pragma unroll
    for (int t = 0; t < kd::KT; ++t) pot[t] = 0.0;

    const int64_t n_groups = (n + kd::GROUP - 1) / kd::GROUP;
    for (int64_t g = blockIdx.x; g < n_groups; g += gridDim.x) {
        const int64_t r0 = g * kd::GROUP + warp * kd::ROWS;
        float s[kd::ROWS][kd::KT], c[kd::ROWS][kd::KT];
#pragma unroll
        for (int r = 0; r < kd::ROWS; ++r)
#pragma unroll
            for (int t = 0; t < kd::KT; ++t) s[r][t] = c[r][t] = 0.f;

        for (int f0 = 0; f0 < d; f0 += kd::SL) {
            const int width = min(kd::SL, d - f0);
            __syncthreads();
            for (int e = threadIdx.x; e < kd::KT * kd::SL; e += kd::THREADS) {
                const int t = e / kd::SL, f = e % kd::SL;
                float v = 0.f;
                if (t < nt && f < width) v = __ldg(X + cand[t0 + t] * (int64_t)d + f0 + f);
                cs[t][f] = v;
            }
            __syncthreads();
            for (int f = lane * 8; f < width; f += 256) {
                const int avail = width - f;
                float x[kd::ROWS][8];
#pragma unroll
                for (int r = 0; r < kd::ROWS; ++r) {
                    if (r0 + r < n) {
                        load8<VEC>(X + (r0 + r) * (int64_t)d + f0 + f, avail, x[r]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[r][e] = 0.f;
                    }
                }
#pragma unroll
                for (int t = 0; t < kd::KT; ++t) {
                    const float4 ca = *reinterpret_cast<const float4 *>(&cs[t][f]);
                    const float4 cb = *reinterpret_cast<const float4 *>(&cs[t][f + 4]);
                    const float cv[8] = {ca.x, ca.y, ca.z, ca.w, cb.x, cb.y, cb.z, cb.w};
#pragma unroll
                    for (int r = 0; r < kd::ROWS; ++r) {
                        float e0 = x[r][0] - cv[0];
                        float run = e0 * e0;
#pragma unroll
                        for (int e = 1; e < 8; ++e) {
                            const float de = x[r][e] - cv[e];
                            run = fmaf(de, de, run);
                        }
                        kahan(s[r][t], c[r][t], run);
                    }
                }
            }
        }
        // lanes -> one float64 distance per (row, trial), fixed tree order
#pragma unroll
        for (int r = 0; r < kd::ROWS; ++r) {
            const int64_t row = r0 + r;
#pragma unroll
            for (int t = 0; t < kd::KT; ++t) {
                double v = static_cast<double>(s[r][t]) - static_cast<double>(c[r][t]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (t < nt && row < n) {
                    if (lane == 0) dist[(int64_t)(t0 + t) * n + row] = v;
                    if (D2) pot[t] += fmin(D2[row], v);
                }
            }
        }
    }
    if (D2 == nullptr) return;
    if (lane == 0)
#pragma unroll
        for (int t = 0; t < kd::KT; ++t) wpot[warp][t] = pot[t];
    __syncthreads();
    if (threadIdx.x < nt) {
        double v = 0.0;
        for (int w = 0; w < kd::WARPS; ++w) v += wpot[w][threadIdx.x];
        bpot[(int64_t)(t0 + threadIdx.x) * gridDim.x + blockIdx.x] = v;
    }
}

// ----------------------------------------------------------------- K4 select
__global__ void kpp_select_kernel(const double *__restrict__ bpot, int n_cta, int T, const int64_t *__restrict__ cand,
                                  int64_t c, int64_t *__restrict__ indices, int32_t *__restrict__ sel_t) {
    __shared__ double pot[64];
    const int lane = threadIdx.x & 31;
    const int t = threadIdx.x >> 5;
    if (t < T) {
        double v = 0.0;
        for (int b0 = 0; b0 < n_cta; b0 += 32) {
            const double x = (b0 + lane < n_cta) ? bpot[(int64_t)t * n_cta + b0 + lane] : 0.0;
            v += __shfl_sync(0xffffffffu, warp_incl_scan(x, lane), 31);
        }
        if (lane == 0) pot[t] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int best = 0;
        for (int q = 1; q < T; ++q)
            if (pot[q] < pot[best]) best = q;
        *sel_t = best;
        indices[c] = cand[best];
    }
}

__global__ void gather_rows_kernel(const float *__restrict__ X, const int64_t *__restrict__ idx, int64_t k, int d,
                                   float *__restrict__ out) {
    for (int64_t j = blockIdx.x; j < k; j += gridDim.x) {
        const float *src = X + idx[j] * (int64_t)d;
        for (int f = threadIdx.x; f < d; f += blockDim.x) out[j * (int64_t)d + f] = src[f];
    }
}

static int dist_grid(int64_t n) {
    const int64_t groups = (n + kd::GROUP - 1) / kd::GROUP;
    int64_t g = groups < (int64_t)kKppMaxCtas ? groups : (int64_t)kKppMaxCtas;
    return (int)(g < 1 ? 1 : g);
}

template <bool VEC>
static void launch_dist(const float *X, int64_t n, int d, const int64_t *cand, int T, const double *D2, double *dist,
                        double *bpot, cudaStream_t s) {
    const int grid = dist_grid(n);
    for (int t0 = 0; t0 < T; t0 += kd::KT)
        kpp_dist_kernel<VEC><<<grid, kd::THREADS, 0, s>>>(X, n, d, cand, T, t0, D2, dist, bpot);
}

cudaError_t launch_kmeanspp(const float *X, int64_t n, int64_t d, int64_t k, int T, uint64_t seed, float *centers,
                            int64_t *indices, const KppLayout &L, uint8_t *ws, cudaStream_t s) {
    WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
    double *D2 = reinterpret_cast<double *>(ws + L.off_d2);
    double *dist = reinterpret_cast<double *>(ws + L.off_dist);
    double *bsum = reinterpret_cast<double *>(ws + L.off_bsum);
    double *bpot = reinterpret_cast<double *>(ws + L.off_bpot);
    int64_t *cand = reinterpret_cast<int64_t *>(ws + L.off_cand);
    int32_t *sel_t = reinterpret_cast<int32_t *>(ws + L.off_chosen);
    const bool vec = (d % 4 == 0) && (reinterpret_cast<uintptr_t>(X) & 15) == 0;
    auto dist_pass = [&](int Tn, const double *d2) {
        if (vec) launch_dist<true>(X, n, (int)d, cand, Tn, d2, dist, bpot, s);
        else launch_dist<false>(X, n, (int)d, cand, Tn, d2, dist, bpot, s);
    };
    const int n_cta = dist_grid(n);

    kpp_first_kernel<<<1, 1, 0, s>>>(n, seed, cand, indices, hdr);
    dist_pass(1, nullptr);  // distances to the first center
    for (int64_t c = 1; c < k; ++c) {
        kpp_blocksum_kernel<<<(int)L.n_blocks, kBsThreads, 0, s>>>(dist, sel_t, n, c == 1 ? 1 : 0, D2, bsum);
        kpp_pick_kernel<<<1, 32 * T, 0, s>>>(bsum, L.n_blocks, D2, n, seed, 1 + (uint64_t)(c - 1) * (uint64_t)T, T,
                                             cand);
        dist_pass(T, D2);
        kpp_select_kernel<<<1, 32 * T, 0, s>>>(bpot, n_cta, T, cand, c, indices, sel_t);
    }
    if (centers) {
        const int g = (int)(k < 4096 ? k : 4096);
        gather_rows_kernel<<<g, 256, 0, s>>>(X, indices, k, (int)d, centers);
    }
    return cudaGetLastError();
}

}  // namespace km

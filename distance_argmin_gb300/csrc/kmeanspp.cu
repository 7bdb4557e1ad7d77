// Greedy k-means++ seeding ("004 — tile sizes, a Cython Lloyd step, and
// k-means++", section "k-means++": 2 + log(n_clusters) candidate trials per new
// center).  The centers are chosen one after the other; each round is:
//
//   update   the winner of the previous round is the trial with the lowest
//            potential (lowest trial on ties); D^2 <- min(D^2, its distances);
//            per-block sums of D^2 (fixed order); each sample's nearest center
//   pick     per trial: uniform from Philox4x32-10, target = u * sum D^2,
//            candidate = first sample whose running sum exceeds the target
//   dcc      the trials' squared distances to the chosen centers
//   select   the rows some trial may bring below their D^2 (the others
//            provably keep it: see the row pruning below)
//   dist     one pass over the selected rows of X per 8 trials: each block
//            keeps one feature slice of the candidates in shared memory and
//            streams its samples once, writing per-slice partial squared
//            distances
//   combine  distances = slice partials added in slice order (+inf for rows
//            not read); per-block potentials sum_i min(D^2_i, dist_ti)
//
// Distances: float32 differences, squared and summed in runs of 8 features,
// a lane's runs added in float32, lanes and slices combined in double-float,
// then float64.  Running sums and potentials are float64.  Every reduction
// has a fixed order.
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kmeanspp.cuh"
#include "trace.cuh"

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
__global__ void kpp_first_kernel(int64_t n, uint64_t seed, int64_t *cand, int64_t *indices, WsHeader *hdr,
                                 int count_rows) {
    hdr->status = 0u;
    hdr->done_blocks = 0u;
    hdr->kpp_rows = count_rows ? (unsigned long long)n : 0ull;  // the first pass reads every row
    const double u = philox_uniform(seed, 0);
    int64_t idx = static_cast<int64_t>(u * static_cast<double>(n));  // u >= 0: truncation is floor
    if (idx > n - 1) idx = n - 1;
    cand[0] = idx;
    indices[0] = idx;
}

constexpr int kBsThreads = 256;

// ------------------------------------------------------------------ K2 pick
__device__ __forceinline__ double warp_incl_scan(double v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += t;
    }
    return v;
}

// Total of D^2 from its block sums, in chunks of 32 (one warp; every lane
// gets the same value).  The shard path computes its shard's total the same
// way, so one shard sees the single-GPU total bit for bit.
__device__ __forceinline__ double d2_total(const double *__restrict__ bsum, int64_t n_blocks, int lane) {
    double total = 0.0;
    for (int64_t b0 = 0; b0 < n_blocks; b0 += 32) {
        const double v = (b0 + lane < n_blocks) ? bsum[b0 + lane] : 0.0;
        const double incl = warp_incl_scan(v, lane);
        total += __shfl_sync(0xffffffffu, incl, 31);
    }
    return total;
}

// The D^2 draw (one warp): the first sample i whose running sum base + D2[0]
// + ... + D2[i] exceeds `target`, or n - 1 when none does.  The running sum
// at sample i is base + (sum of the block sums before its block) + (the
// in-block prefix up to i); the block-sum prefix is the same for every
// trial, so all trials see one consistent running sum.  `base` is 0 on one
// GPU and the sum of the earlier shards' totals on a shard.  Lane-uniform.
__device__ int64_t d2_search(const double *__restrict__ bsum, int64_t n_blocks, const double *__restrict__ D2,
                             int64_t n, double target, double base, int lane) {
    // first block whose inclusive prefix exceeds the target
    double before = base;  // running sum before the current chunk of blocks
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
    // put the target between the block's own running sum and its block sum):
    // lane l sums samples [32 l, 32 l + 32) of the 1024-sample block, one
    // warp scan of those totals finds the lane, which then walks its 32
    double run = blk_before;
    for (int64_t b = blk; b >= 0 && b < n_blocks; ++b) {
        const int64_t i0 = b * kKppScanBlock + lane * 32;
        double v[32];
        double tot = 0.0;
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = (i0 + e < n) ? D2[i0 + e] : 0.0;
#pragma unroll
        for (int e = 0; e < 32; ++e) tot += v[e];
        const double incl = run + warp_incl_scan(tot, lane);
        const uint32_t hit = __ballot_sync(0xffffffffu, incl > target);
        if (hit) {
            const int l = __ffs(hit) - 1;
            if (lane == l) {
                double acc = incl - tot;
                int64_t found = i0 + 31;
                for (int e = 0; e < 32; ++e) {
                    acc += v[e];
                    if (acc > target) {
                        found = i0 + e;
                        break;
                    }
                }
                pick = found < n ? found : n - 1;
            }
            pick = __shfl_sync(0xffffffffu, pick, l);
            break;
        }
        run = __shfl_sync(0xffffffffu, incl, 31);
    }
    return pick;
}

// One warp per trial, each in a block of its own: the scans are float64, and
// this part's float64 pipe is narrow enough (about two FMAs per clock per SM)
// that eight trials sharing one SM took 14 us.
__global__ void __launch_bounds__(32)
    kpp_pick_kernel(const double *__restrict__ bsum, int64_t n_blocks, const double *__restrict__ D2, int64_t n,
                    uint64_t seed, uint64_t draw_base, int T, int64_t *__restrict__ cand) {
    griddep_wait();
    const int lane = threadIdx.x;
    const int t = blockIdx.x;
    if (t >= T) return;
    const double total = d2_total(bsum, n_blocks, lane);
    const double target = philox_uniform(seed, draw_base + (uint64_t)t) * total;
    const int64_t pick = d2_search(bsum, n_blocks, D2, n, target, 0.0, lane);
    if (lane == 0) cand[t] = pick;
}

// ------------------------------------------------------------------ K3 dist
namespace kd {
constexpr int KT = kKppGroupTrials;  // trial candidates per pass over X
constexpr int ROWS = 2;              // samples per warp at a time
constexpr int MIN_BLOCKS = 1;        // one block per SM: 128 KiB of candidates, 24 warps of up to 85 registers
constexpr int WARPS = 24;
constexpr int THREADS = WARPS * 32;
constexpr int GROUP = WARPS * ROWS;
}  // namespace kd

// Error-free sum: s + e == a + b exactly (Knuth's TwoSum).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
    s = a + b;
    const float bb = s - a;
    e = (a - (s - bb)) + (b - bb);
}

// (hi, lo) += (ohi, olo) in double-float: TwoSum of the high parts, the low
// parts added to its error, renormalised.  Symmetric in its operands, so two
// lanes that add each other's values get the same bits.
__device__ __forceinline__ void df_add(float &hi, float &lo, float ohi, float olo) {
    float s, e;
    two_sum(hi, ohi, s, e);
    e += lo + olo;
    hi = s + e;
    lo = e - (hi - s);
}

// One reduce-scatter level over 2H double-float values: the lane whose `bit`
// is set keeps the upper half, its partner (lane ^ bit) the lower half; each
// sends the half it drops and adds the half it receives.  Values 0..H-1 hold
// the result.
template <int N, int H>
__device__ __forceinline__ void reduce_scatter_level(float (&hi)[N], float (&lo)[N], int lane, int bit) {
    const bool up = (lane & bit) != 0;
#pragma unroll
    for (int i = 0; i < H; ++i) {
        const float kh = up ? hi[H + i] : hi[i], kl = up ? lo[H + i] : lo[i];
        const float sh = up ? hi[i] : hi[H + i], sl = up ? lo[i] : lo[H + i];
        const float rh = __shfl_xor_sync(0xffffffffu, sh, bit);
        const float rl = __shfl_xor_sync(0xffffffffu, sl, bit);
        hi[i] = kh;
        lo[i] = kl;
        df_add(hi[i], lo[i], rh, rl);
    }
}

// Features p[0..3] and p[128..131] of a row (zeros past `avail`, the
// features left in the slice from p on).
template <bool VEC>
__device__ __forceinline__ void load4x2(const float *__restrict__ p, int avail, float2 (&v)[4]) {
    if (VEC && avail >= 132) {
        const float4 a = __ldg(reinterpret_cast<const float4 *>(p));
        const float4 b = __ldg(reinterpret_cast<const float4 *>(p + 128));
        v[0] = make_float2(a.x, a.y);
        v[1] = make_float2(a.z, a.w);
        v[2] = make_float2(b.x, b.y);
        v[3] = make_float2(b.z, b.w);
    } else {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            v[e] = make_float2(2 * e < avail ? __ldg(p + 2 * e) : 0.f, 2 * e + 1 < avail ? __ldg(p + 2 * e + 1) : 0.f);
            v[2 + e] = make_float2(128 + 2 * e < avail ? __ldg(p + 128 + 2 * e) : 0.f,
                                   128 + 2 * e + 1 < avail ? __ldg(p + 128 + 2 * e + 1) : 0.f);
        }
    }
}

// Partial distances over one feature slice (blockIdx.y) to trials
// [t0, t0 + nt): dpart[slice][t][i] = sum over the slice of (x_if - cand_tf)^2.
// The candidates are the rows cand[] of X, or the rows of `crows` when it is
// given (the shard path, whose candidates may live on other GPUs).
// The block stages its slice of the candidates (negated) in shared memory once
// and then streams its share of the samples, each sample read exactly once.
// Differences and squares use the packed two-float instructions; each run of
// a lane's 8 features of a step is added to a per-lane sum, the two rows'
// sums paired in one packed add.  A lane adds at most W / 256 runs (16 for a
// 4096-feature slice); lanes and slices are combined in double-float.
// With `rows` the pass reads only the listed rows: block b of samples lists
// rcount[b] of them, ascending, at rows[b * kKppScanBlock ...] (the others
// cannot change this round, see kpp_select_rows_kernel); the list is walked
// in sample order.  A row's sums do not depend on which rows share its warp.
template <bool VEC>
__global__ void __launch_bounds__(kd::THREADS, kd::MIN_BLOCKS)
    kpp_dist_part_kernel(const float *__restrict__ X, int64_t n, int d, const int64_t *__restrict__ cand,
                         const float *__restrict__ crows, int T, int t0, int W, int rev,
                         const int32_t *__restrict__ rows, const int32_t *__restrict__ rcount, int nb,
                         float2 *__restrict__ dpart) {
    extern __shared__ __align__(16) float cs[];  // [KT][W], negated; with rows, then nb + 1 ints
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int nt = min(kd::KT, T - t0);
    const int slice = blockIdx.y;
    const int fb = slice * W;
    const int width = min(W, d - fb);
    static_assert(kd::ROWS == 2, "the two rows' sums are paired in float2");
    // entries of the list of rows to read: every row, or the listed ones
    // (their count is known after the wait, from the block counts' prefix)
    int *pref = reinterpret_cast<int *>(cs + kd::KT * W);
    int64_t count = n;
    if (rows) {
        griddep_wait();
        if (warp == 0) {
            int run = 0;
            for (int b0 = 0; b0 < nb; b0 += 32) {
                const int v = b0 + lane < nb ? rcount[b0 + lane] : 0;
                int incl = v;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int t = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += t;
                }
                if (b0 + lane < nb) pref[b0 + lane] = run + incl - v;
                run += __shfl_sync(0xffffffffu, incl, 31);
            }
            if (lane == 0) pref[nb] = run;
        }
        __syncthreads();
        count = pref[nb];
    }
    const int64_t n_groups = (count + kd::GROUP - 1) / kd::GROUP;
    // the sample of list entry e, or n past the list
    auto row_of = [&](int64_t e) -> int64_t {
        if (e >= count) return n;
        if (!rows) return e;
        int lo = 0, hi = nb;  // pref[lo] <= e < pref[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pref[mid] <= e) lo = mid;
            else hi = mid;
        }
        return rows[(int64_t)lo * kKppScanBlock + (e - pref[lo])];
    };

    // A lane owns features f .. f+3 and f+128 .. f+131 of each 256-feature
    // step, so every 16-byte load of the warp (global and shared) covers 512
    // contiguous bytes.  The next step's rows are loaded while this step is
    // computed (xn), and the last step of a group loads the first step of the
    // block's next group, so a group starts without waiting for memory.  One
    // block of 24 warps per SM fits it in 85 registers a thread; more resident
    // warps hide more of the loads (16, 20, 24 and 28 warps measured 397, 375,
    // 363 and 386 us a pass).
    //
    // With `rev` set the block visits its groups from the top of X down: the
    // pass then starts on the rows the previous pass read last, which are
    // still in L2.  The i-th group a block visits is group(i) either way.
    float2 x[kd::ROWS][4], xn[kd::ROWS][4];
    int64_t rn[kd::ROWS];  // the rows whose first step is in xn
    auto group = [&](int64_t i) { return rev ? n_groups - 1 - i : i; };
    auto load_first_step = [&](int64_t i) {
        const int64_t e0 = (i < n_groups ? group(i) : n_groups) * kd::GROUP + warp * kd::ROWS;
#pragma unroll
        for (int r = 0; r < kd::ROWS; ++r) {
            rn[r] = row_of(e0 + r);
            if (rn[r] < n) {  // past the last group every row is past n
                load4x2<VEC>(X + rn[r] * (int64_t)d + fb + lane * 4, width - lane * 4, xn[r]);
            } else {
#pragma unroll
                for (int e = 0; e < 4; ++e) xn[r][e] = make_float2(0.f, 0.f);
            }
        }
    };
    // X is an input of the whole entry point, never written by a kernel of
    // the chain, so without a row list its first rows are requested before
    // the wait for the kernel that chose the candidates
    load_first_step(blockIdx.x);
    if (!rows) griddep_wait();
    // the candidates are rows of X, or (a shard) rows of the exchange buffer
    if (VEC) {
        // W and width are multiples of 4: a 16-byte group never straddles a
        // trial or the slice's end
        for (int e = threadIdx.x * 4; e < kd::KT * W; e += kd::THREADS * 4) {
            const int t = e / W, f = e - t * W;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            if (t < nt && f < width) {
                const float *src = crows ? crows + (int64_t)(t0 + t) * d : X + cand[t0 + t] * (int64_t)d;
                v = __ldg(reinterpret_cast<const float4 *>(src + fb + f));
                v = make_float4(-v.x, -v.y, -v.z, -v.w);
            }
            *reinterpret_cast<float4 *>(&cs[e]) = v;
        }
    } else {
        for (int e = threadIdx.x; e < kd::KT * W; e += kd::THREADS) {
            const int t = e / W, f = e - t * W;
            float v = 0.f;
            if (t < nt && f < width)
                v = -__ldg((crows ? crows + (int64_t)(t0 + t) * d : X + cand[t0 + t] * (int64_t)d) + fb + f);
            cs[e] = v;
        }
    }
    __syncthreads();

    for (int64_t g = blockIdx.x; g < n_groups; g += gridDim.x) {
        int64_t rw[kd::ROWS];
#pragma unroll
        for (int r = 0; r < kd::ROWS; ++r) rw[r] = rn[r];
        float2 s2[kd::KT];  // .x row 0, .y row 1
#pragma unroll
        for (int t = 0; t < kd::KT; ++t) s2[t] = make_float2(0.f, 0.f);
        for (int f0 = 0; f0 < width; f0 += 256) {
            const int f = f0 + lane * 4;
#pragma unroll
            for (int r = 0; r < kd::ROWS; ++r)
#pragma unroll
                for (int e = 0; e < 4; ++e) x[r][e] = xn[r][e];
            if (f0 + 256 < width) {
#pragma unroll
                for (int r = 0; r < kd::ROWS; ++r) {
                    if (rw[r] < n) load4x2<VEC>(X + rw[r] * (int64_t)d + fb + f + 256, width - f - 256, xn[r]);
                }
            } else {
                load_first_step(g + gridDim.x);
            }
#pragma unroll
            for (int t = 0; t < kd::KT; ++t) {
                const float4 ca = *reinterpret_cast<const float4 *>(&cs[t * W + f]);
                const float4 cb = *reinterpret_cast<const float4 *>(&cs[t * W + f + 128]);
                const float2 nc[4] = {make_float2(ca.x, ca.y), make_float2(ca.z, ca.w), make_float2(cb.x, cb.y),
                                      make_float2(cb.z, cb.w)};
                float rs[kd::ROWS];
#pragma unroll
                for (int r = 0; r < kd::ROWS; ++r) {
                    const float2 e0 = __fadd2_rn(x[r][0], nc[0]);
                    float2 run = __fmul2_rn(e0, e0);
#pragma unroll
                    for (int e = 1; e < 4; ++e) {
                        const float2 de = __fadd2_rn(x[r][e], nc[e]);
                        run = __ffma2_rn(de, de, run);
                    }
                    rs[r] = run.x + run.y;
                }
                s2[t] = __fadd2_rn(s2[t], make_float2(rs[0], rs[1]));
            }
        }
        // lanes -> one partial per (row, trial), as double-float values in
        // float32 (the float64 pipe of this part is far too slow for it).  A
        // reduce-scatter over the ROWS x KT sums: at each level (lane xor 16,
        // 8, 4, 2) a lane keeps half of its values, sends the other half to
        // its partner and adds what it receives; the last level (xor 1) is a
        // full exchange.  Every sum gets the same pairing tree as a full
        // butterfly, with far fewer shuffles and additions.
        constexpr int NS = kd::ROWS * kd::KT;
        static_assert(NS == 16 || NS == 32, "the reduce-scatter below handles 16 or 32 sums");
        float hi[NS], lo[NS];
#pragma unroll
        for (int r = 0; r < kd::ROWS; ++r)
#pragma unroll
            for (int t = 0; t < kd::KT; ++t) {
                hi[r * kd::KT + t] = r == 0 ? s2[t].x : s2[t].y;
                lo[r * kd::KT + t] = 0.f;
            }
        reduce_scatter_level<NS, NS / 2>(hi, lo, lane, 16);
        reduce_scatter_level<NS, NS / 4>(hi, lo, lane, 8);
        reduce_scatter_level<NS, NS / 8>(hi, lo, lane, 4);
        reduce_scatter_level<NS, NS / 16>(hi, lo, lane, 2);
        if constexpr (NS == 32) {
            reduce_scatter_level<NS, 1>(hi, lo, lane, 1);
        } else {
            const float ohi = __shfl_xor_sync(0xffffffffu, hi[0], 1);
            const float olo = __shfl_xor_sync(0xffffffffu, lo[0], 1);
            df_add(hi[0], lo[0], ohi, olo);
        }
        // lane l holds sum v = row * KT + trial: v = l (32 sums) or l / 2 (16
        // sums, held by both lanes of a pair)
        const int v = NS == 32 ? lane : lane >> 1;
        const int t = v % kd::KT;
        const int64_t row = v < kd::KT ? rw[0] : rw[1];
        if ((NS == 32 || (lane & 1) == 0) && t < nt && row < n)
            dpart[((int64_t)slice * kd::KT + t) * n + row] = make_float2(hi[0], lo[0]);
    }
}

// dist[t0 + t][i] = sum of the S slice partials (slice order, double-float); with D2, the
// block potentials bpot[t0 + t][block] = sum over the block's samples of
// min(D2_i, dist) in a fixed order.  Grid: (sample blocks, trials).
// With `flag`, a row the pass did not read (flag 0) is at distance +inf from
// every trial: no trial can lower its D^2 this round.
__global__ void __launch_bounds__(kBsThreads)
    kpp_combine_kernel(const float2 *__restrict__ dpart, int S, int64_t n, int t0, const double *__restrict__ D2,
                       const uint8_t *__restrict__ flag, double *__restrict__ dist, double *__restrict__ bpot,
                       int64_t n_blocks) {
    griddep_wait();
    __shared__ double red[kBsThreads];
    const int t = blockIdx.y;
    const int64_t base = (int64_t)blockIdx.x * kKppScanBlock;
    double pot = 0.0;
#pragma unroll
    for (int q = 0; q < kKppScanBlock / kBsThreads; ++q) {
        const int64_t i = base + threadIdx.x + (int64_t)q * kBsThreads;
        if (i < n) {
            // slice partials added as double-float values, one conversion at the end
            float hi = 0.f, lo = 0.f;
            if (flag && !flag[i]) {
                hi = __int_as_float(0x7f800000);  // +inf
            } else {
                for (int sl = 0; sl < S; ++sl) {
                    const float2 pv = dpart[((int64_t)sl * kd::KT + t) * n + i];
                    float s2, e;
                    two_sum(hi, pv.x, s2, e);
                    e += lo + pv.y;
                    hi = s2 + e;
                    lo = e - (hi - s2);
                }
            }
            const double v = static_cast<double>(hi) + static_cast<double>(lo);
            dist[(int64_t)(t0 + t) * n + i] = v;
            if (D2) pot += fmin(D2[i], v);
        }
    }
    if (D2 == nullptr) return;
    red[threadIdx.x] = pot;
    __syncthreads();
    for (int w = kBsThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) bpot[(int64_t)(t0 + t) * n_blocks + blockIdx.x] = red[0];
}

// The winning trial of the previous center: lowest total potential (lowest
// trial on ties), every block computing the same sums in the same order.
// Potential of trial t (one warp, every lane gets it): its block
// potentials summed lane-strided, then a butterfly.
__device__ __forceinline__ double trial_potential(const double *__restrict__ bpot, int t, int64_t n_blocks,
                                                  int lane) {
    double v = 0.0;
    for (int64_t b = lane; b < n_blocks; b += 32) v += bpot[(int64_t)t * n_blocks + b];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ int select_best_trial(const double *__restrict__ bpot, int T, int64_t n_blocks) {
    __shared__ int best_s;
    __shared__ double pot_s[kKppMaxTrials];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    for (int t = w; t < T; t += blockDim.x / 32) {
        const double v = trial_potential(bpot, t, n_blocks, lane);
        if (lane == 0) pot_s[t] = v;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int best = 0;
        for (int q = 1; q < T; ++q)
            if (pot_s[q] < pot_s[best]) best = q;
        best_s = best;
    }
    __syncthreads();
    return best_s;
}

// K1 of center c: choose the winner of center c-1 (from c = 2 on), lower D^2
// by its distances, and the per-block sums of D^2 for the draws of center c.
// With `near`, a sample whose D^2 the winner lowers records center c-1 as
// its nearest (every sample records center 0 at c = 1), and the rows of the
// center-candidate table for centers 0 .. c-1 are cleared for this round.
__global__ void __launch_bounds__(kBsThreads)
    kpp_update_kernel(const double *__restrict__ dist, const double *__restrict__ bpot, int T, int64_t n,
                      int64_t n_blocks, const int64_t *__restrict__ cand, int64_t *__restrict__ indices,
                      int64_t prev, int init, double *__restrict__ D2, double *__restrict__ bsum,
                      int32_t *__restrict__ near, float *__restrict__ dcc, int64_t kst) {
    griddep_wait();
    __shared__ double red[kBsThreads];
    if (dcc) {
        const int64_t cells = (int64_t)T * (prev + 1);
        for (int64_t e = (int64_t)blockIdx.x * kBsThreads + threadIdx.x; e < cells;
             e += (int64_t)gridDim.x * kBsThreads)
            dcc[(e / (prev + 1)) * kst + e % (prev + 1)] = 0.f;
    }
    int best = 0;
    if (!init) {
        best = select_best_trial(bpot, T, n_blocks);
        if (blockIdx.x == 0 && threadIdx.x == 0) indices[prev] = cand[best];
    }
    const double *db = dist + (int64_t)best * n;
    const int64_t base = (int64_t)blockIdx.x * kKppScanBlock;
    double s = 0.0;
#pragma unroll
    for (int q = 0; q < kKppScanBlock / kBsThreads; ++q) {
        const int64_t i = base + threadIdx.x + (int64_t)q * kBsThreads;
        if (i < n) {
            const double v = db[i];
            const double old = init ? 0.0 : D2[i];
            const double nd = init ? v : fmin(old, v);
            D2[i] = nd;
            if (near && (init || v < old)) near[i] = (int32_t)prev;
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

// ------------------------------------------------------- row pruning
// A sample x whose nearest committed center is c_j (D(x) = ||x - c_j||, so
// D^2(x) is its current D^2) is at least ||c_j - y|| - D(x) from a trial
// candidate y (triangle inequality).  When ||c_j - y|| >= 2.001 D(x), y is
// more than 1.0009 D(x) from x, and min(D^2(x), ||x - y||^2) is D^2(x)
// whatever rounding either distance carries (float32 sums are good to about
// 1e-6 relative, far inside the 0.2% margin on the squares).  A row that
// this clears for every trial of the round cannot change D^2, a potential or
// a draw: the distance pass skips it and the combine puts it at +inf.  The
// seeding's indices are therefore the same as without pruning.
constexpr double kKppPruneSq = 4.004;  // (2 + 0.001)^2, rounded up
constexpr int kDccChunk = 1024;        // features of one block of the center-candidate distances

// dcc[t][j] += sum over features [f0, f0 + 1024) of (X[indices[j]] - X[cand[t]])^2
// for the committed centers j < c, in float32, onto zeros the update kernel
// left (the feature chunks of a (t, j) pair add in any order: the table only
// decides which rows are read, never a value).  Grid (centers / 8, chunks):
// warp w takes center 8 * blockIdx.x + w; the block stages the chunk of every
// candidate.  Needs d % 4 == 0 and 16-byte aligned rows.
__global__ void __launch_bounds__(kBsThreads)
    kpp_dcc_kernel(const float *__restrict__ X, int d, const int64_t *__restrict__ indices, int64_t c,
                   const int64_t *__restrict__ cand, int T, int64_t kst, float *__restrict__ dcc) {
    constexpr int V = kDccChunk / 4;  // float4 per chunk of a row
    static_assert(V == kBsThreads, "one float4 of every candidate per thread");
    extern __shared__ float4 ys[];    // [T][V]
    griddep_wait();
    const int lane = threadIdx.x & 31;
    const int64_t j = (int64_t)blockIdx.x * (kBsThreads / 32) + (threadIdx.x >> 5);
    const int f0 = blockIdx.y * kDccChunk;
    const int w4 = min(kDccChunk, d - f0) / 4;
    // this warp's center chunk and every candidate's chunk, all in flight
    // together (the centers come from DRAM, the candidates mostly from L2)
    float4 xv[V / 32];
    const float4 *cj = j < c ? reinterpret_cast<const float4 *>(X + indices[j] * (int64_t)d + f0) : nullptr;
#pragma unroll
    for (int m = 0; m < V / 32; ++m) {
        const int q = lane + 32 * m;
        xv[m] = cj && q < w4 ? __ldg(cj + q) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int t = 0; t < kKppMaxTrials; ++t) {
        if (t < T) {
            const float4 *src = reinterpret_cast<const float4 *>(X + cand[t] * (int64_t)d + f0);
            ys[t * V + threadIdx.x] = threadIdx.x < w4 ? __ldg(src + threadIdx.x) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    __syncthreads();
    if (j >= c) return;
    // eight trials at a time, their butterflies interleaved
    constexpr int G = kKppGroupTrials;
#pragma unroll 1
    for (int t0 = 0; t0 < T; t0 += G) {
        float acc[G];
#pragma unroll
        for (int q = 0; q < G; ++q) acc[q] = 0.f;
#pragma unroll
        for (int m = 0; m < V / 32; ++m) {
#pragma unroll
            for (int q = 0; q < G; ++q) {
                if (t0 + q < T) {
                    const float4 y = ys[(t0 + q) * V + lane + 32 * m];
                    const float dx = xv[m].x - y.x, dy = xv[m].y - y.y, dz = xv[m].z - y.z, dw = xv[m].w - y.w;
                    acc[q] = fmaf(dx, dx, acc[q]);
                    acc[q] = fmaf(dy, dy, acc[q]);
                    acc[q] = fmaf(dz, dz, acc[q]);
                    acc[q] = fmaf(dw, dw, acc[q]);
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
#pragma unroll
            for (int q = 0; q < G; ++q) acc[q] += __shfl_xor_sync(0xffffffffu, acc[q], o);
        if (lane == 0) {
#pragma unroll
            for (int q = 0; q < G; ++q)
                if (t0 + q < T) atomicAdd(dcc + (int64_t)(t0 + q) * kst + j, acc[q]);
        }
    }
}

// Per block of kKppScanBlock samples, one a thread: flag[i] = 1 when some
// trial is closer than 2.001 D(x) to the sample's nearest center (the pass
// must read the row), and the flagged rows listed in ascending order at
// rows[block * 1024 ...], their number in rcount[block].  The table entries
// of eight trials are loaded before any is compared.
__global__ void __launch_bounds__(kKppScanBlock)
    kpp_select_rows_kernel(int64_t n, const int32_t *__restrict__ near, const double *__restrict__ D2,
                           const float *__restrict__ dcc, int T, int64_t kst, uint8_t *__restrict__ flag,
                           int32_t *__restrict__ rows, int32_t *__restrict__ rcount, int passes, WsHeader *hdr) {
    constexpr int WARPS = kKppScanBlock / 32;
    constexpr int G = kKppGroupTrials;
    __shared__ int wsum[WARPS];
    griddep_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    const int64_t i = (int64_t)blockIdx.x * kKppScanBlock + threadIdx.x;
    bool need = false;
    if (i < n) {
        const double lim = kKppPruneSq * D2[i];
        const float *dj = dcc + near[i];
        for (int t0 = 0; t0 < T; t0 += G) {
            float v[G];
#pragma unroll
            for (int q = 0; q < G; ++q) v[q] = t0 + q < T ? dj[(int64_t)(t0 + q) * kst] : __int_as_float(0x7f800000);
#pragma unroll
            for (int q = 0; q < G; ++q) need |= (double)v[q] < lim;
        }
        flag[i] = need ? 1 : 0;
    }
    // ascending positions: a ballot per warp, the warps' counts before it
    const unsigned m = __ballot_sync(0xffffffffu, need);
    if (lane == 0) wsum[w] = __popc(m);
    __syncthreads();
    int before = 0, total = 0;
#pragma unroll
    for (int q = 0; q < WARPS; ++q) {
        if (q < w) before += wsum[q];
        total += wsum[q];
    }
    if (need) rows[(int64_t)blockIdx.x * kKppScanBlock + before + __popc(m & ((1u << lane) - 1u))] = (int32_t)i;
    if (threadIdx.x == 0) {
        rcount[blockIdx.x] = total;
        atomicAdd(&hdr->kpp_rows, (unsigned long long)total * (unsigned long long)passes);
    }
}

// Winner of the last center.
__global__ void kpp_select_last_kernel(const double *__restrict__ bpot, int T, int64_t n_blocks,
                                       const int64_t *__restrict__ cand, int64_t *__restrict__ indices, int64_t c) {
    griddep_wait();
    const int best = select_best_trial(bpot, T, n_blocks);
    if (threadIdx.x == 0) indices[c] = cand[best];
}

__global__ void gather_rows_kernel(const float *__restrict__ X, const int64_t *__restrict__ idx, int64_t k, int d,
                                   float *__restrict__ out) {
    griddep_wait();
    for (int64_t j = blockIdx.x; j < k; j += gridDim.x) {
        const float *src = X + idx[j] * (int64_t)d;
        for (int f = threadIdx.x; f < d; f += blockDim.x) out[j * (int64_t)d + f] = src[f];
    }
}

// One pass over X for the candidates of trials [0, Tn): the per-slice
// partial distances, then their combination (with D2: and the block
// potentials).  Candidates: rows cand[] of X, or the rows of `crows`.
// `prune`: read only the rows kpp_select_rows_kernel listed (the layout has
// the pruning regions).
static cudaError_t kpp_dist_pass(const float *X, int64_t n, int64_t d, const KppLayout &L, uint8_t *ws, int Tn,
                                 const int64_t *cand, const float *crows, const double *d2, bool chained_first,
                                 bool rev, bool prune, cudaStream_t s) {
    double *dist = reinterpret_cast<double *>(ws + L.off_dist);
    float2 *dpart = reinterpret_cast<float2 *>(ws + L.off_dpart);
    double *bpot = reinterpret_cast<double *>(ws + L.off_bpot);
    const int32_t *rows = prune ? reinterpret_cast<const int32_t *>(ws + L.off_rows) : nullptr;
    const int32_t *rcount = prune ? reinterpret_cast<const int32_t *>(ws + L.off_rcount) : nullptr;
    const uint8_t *flag = prune ? ws + L.off_flag : nullptr;
    const bool vec = (d % 4 == 0) && ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(crows)) & 15) == 0;
    // the candidates' slice, then (row list) the prefix of the block counts
    const size_t smem = (size_t)kd::KT * L.W * sizeof(float) + (prune ? (size_t)(L.n_blocks + 1) * sizeof(int) : 0);
    {
        static std::once_flag attr_once[kMaxDevices];
        once_per_device(attr_once, [] {
            const int most = (int)(kd::KT * kKppSliceFloats * sizeof(float) + (kKppPruneMaxBlocks + 1) * sizeof(int));
            cudaFuncSetAttribute(kpp_dist_part_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
            cudaFuncSetAttribute(kpp_dist_part_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
        });
    }
    static std::atomic<int> sm_cache[kMaxDevices];
    const int sms = cached_per_device(sm_cache, [] {
        int v = 0, dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        return v > 0 ? v : 1;
    });
    const int64_t groups = (n + kd::GROUP - 1) / kd::GROUP;
    // one resident block per SM over all slices
    int64_t gx = (kd::MIN_BLOCKS * (int64_t)sms + L.S - 1) / L.S;
    if (gx > groups) gx = groups;
    const dim3 dgrid((unsigned)(gx < 1 ? 1 : gx), (unsigned)L.S);
    cudaError_t e = cudaSuccess;
    for (int t0 = 0; t0 < Tn && e == cudaSuccess; t0 += kd::KT) {
        const bool chained = chained_first || t0 > 0;
        trace_mark(kTraceKppDist, false, s);
        e = vec ? launch_kernel(chained, kpp_dist_part_kernel<true>, dgrid, dim3(kd::THREADS), smem, s, X, n, (int)d,
                                cand, crows, Tn, t0, L.W, (int)rev, rows, rcount, (int)L.n_blocks, dpart)
                : launch_kernel(chained, kpp_dist_part_kernel<false>, dgrid, dim3(kd::THREADS), smem, s, X, n, (int)d,
                                cand, crows, Tn, t0, L.W, (int)rev, rows, rcount, (int)L.n_blocks, dpart);
        trace_mark(kTraceKppDist, true, s);
        const int nt = Tn - t0 < kd::KT ? Tn - t0 : kd::KT;
        if (e == cudaSuccess)
            e = launch_kernel(true, kpp_combine_kernel, dim3((unsigned)L.n_blocks, (unsigned)nt), dim3(kBsThreads), 0,
                              s, (const float2 *)dpart, L.S, n, t0, d2, flag, dist, bpot, L.n_blocks);
    }
    return e;
}

cudaError_t launch_kmeanspp(const float *X, int64_t n, int64_t d, int64_t k, int T, uint64_t seed, float *centers,
                            int64_t *indices, const KppLayout &L, uint8_t *ws, cudaStream_t s) {
    WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
    double *D2 = reinterpret_cast<double *>(ws + L.off_d2);
    double *dist = reinterpret_cast<double *>(ws + L.off_dist);
    double *bsum = reinterpret_cast<double *>(ws + L.off_bsum);
    double *bpot = reinterpret_cast<double *>(ws + L.off_bpot);
    int64_t *cand = reinterpret_cast<int64_t *>(ws + L.off_cand);

    // every kernel after the first is chained to the one before it (see
    // launch_kernel); each waits for its predecessor before touching memory
    cudaError_t e = cudaSuccess;
    auto chain = [&](cudaError_t r) {
        if (e == cudaSuccess) e = r;
    };

    // row pruning (see kpp_select_rows_kernel) where the layout reserves it
    // and the rows are whole 16-byte groups
    const bool prune = L.off_near != 0 && L.k >= k && d % 4 == 0 && (reinterpret_cast<uintptr_t>(X) & 15) == 0;
    int32_t *near = prune ? reinterpret_cast<int32_t *>(ws + L.off_near) : nullptr;
    float *dcc = prune ? reinterpret_cast<float *>(ws + L.off_dcc) : nullptr;
    const size_t dcc_smem = (size_t)T * kDccChunk * sizeof(float);
    const unsigned dcc_chunks = (unsigned)((d + kDccChunk - 1) / kDccChunk);
    if (prune) {
        static std::once_flag attr_once[kMaxDevices];
        once_per_device(attr_once, [] {
            cudaFuncSetAttribute(kpp_dcc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)(kKppMaxTrials * kDccChunk * sizeof(float)));
        });
    }

    kpp_first_kernel<<<1, 1, 0, s>>>(n, seed, cand, indices, hdr, prune ? 1 : 0);
    chain(cudaGetLastError());
    // distances to the first center
    if (e == cudaSuccess) chain(kpp_dist_pass(X, n, d, L, ws, 1, cand, nullptr, nullptr, true, false, false, s));
    for (int64_t c = 1; c < k && e == cudaSuccess; ++c) {
        chain(launch_kernel(true, kpp_update_kernel, dim3((unsigned)L.n_blocks), dim3(kBsThreads), 0, s,
                            (const double *)dist, (const double *)bpot, T, n, L.n_blocks, (const int64_t *)cand, indices,
                            c - 1, c == 1 ? 1 : 0, D2, bsum, near, dcc, L.k));
        chain(launch_kernel(true, kpp_pick_kernel, dim3((unsigned)T), dim3(32), 0, s, (const double *)bsum, L.n_blocks,
                            (const double *)D2, n, seed, 1 + (uint64_t)(c - 1) * (uint64_t)T, T, cand));
        if (prune) {
            // the trials' distances to the c committed centers, then the rows to read
            const unsigned dblocks = (unsigned)((c + kBsThreads / 32 - 1) / (kBsThreads / 32));
            chain(launch_kernel(true, kpp_dcc_kernel, dim3(dblocks, dcc_chunks), dim3(kBsThreads), dcc_smem, s, X, (int)d,
                                (const int64_t *)indices, c, (const int64_t *)cand, T, L.k, dcc));
            chain(launch_kernel(true, kpp_select_rows_kernel, dim3((unsigned)L.n_blocks), dim3(kKppScanBlock), 0, s, n,
                                (const int32_t *)near, (const double *)D2, (const float *)dcc, T, L.k,
                                ws + L.off_flag, reinterpret_cast<int32_t *>(ws + L.off_rows),
                                reinterpret_cast<int32_t *>(ws + L.off_rcount), (T + kd::KT - 1) / kd::KT, hdr));
        }
        // successive passes run in opposite directions over X (see the kernel)
        if (e == cudaSuccess) chain(kpp_dist_pass(X, n, d, L, ws, T, cand, nullptr, D2, true, (c & 1) != 0, prune, s));
    }
    if (k > 1)
        chain(launch_kernel(true, kpp_select_last_kernel, dim3(1), dim3(256), 0, s, (const double *)bpot, T,
                            L.n_blocks, (const int64_t *)cand, indices, k - 1));
    if (centers) {
        const int g = (int)(k < 4096 ? k : 4096);
        chain(launch_kernel(true, gather_rows_kernel, dim3(g), dim3(256), 0, s, X, (const int64_t *)indices, k, (int)d,
                            centers));
    }
    return e;
}

// ------------------------------------------------------------- shard path
// Greedy k-means++ over samples split by rows across ranks.  Each rank holds
// its shard's D^2 and calls the steps below in turn; between them the caller
// all-gathers small buffers (candidate blocks, potentials, shard totals).
// Every rank makes the same decisions from the same gathered values, summed
// in rank order.  Exchange block of one rank: T int64 global sample indices
// (-1: the trial's candidate is not in this shard), then T rows of d
// float32 (the candidates this shard owns).

__global__ void kpp_shard_first_kernel(const float *__restrict__ X, int64_t n_local, int d, int64_t row_offset,
                                       int64_t n_global, uint64_t seed, int T, uint8_t *__restrict__ send,
                                       int64_t idx_bytes, WsHeader *hdr) {
    if (threadIdx.x == 0) {
        hdr->status = 0u;
        hdr->done_blocks = 0u;
    }
    const double u = philox_uniform(seed, 0);
    int64_t g = static_cast<int64_t>(u * static_cast<double>(n_global));  // u >= 0: truncation is floor
    if (g > n_global - 1) g = n_global - 1;
    const int64_t loc = g - row_offset;
    const bool mine = loc >= 0 && loc < n_local;
    int64_t *idx = reinterpret_cast<int64_t *>(send);
    float *rows = reinterpret_cast<float *>(send + idx_bytes);
    for (int t = threadIdx.x; t < T; t += blockDim.x) idx[t] = (t == 0 && mine) ? g : -1;
    if (mine)
        for (int f = threadIdx.x; f < d; f += blockDim.x) rows[f] = X[loc * (int64_t)d + f];
}

// Trial t's candidate comes from the first rank whose block owns it (exactly
// one does; none sets the exchange flag and leaves a zero row).
__global__ void kpp_shard_gather_kernel(const uint8_t *__restrict__ recv, int world, int64_t blk_bytes,
                                        int64_t idx_bytes, int d, float *__restrict__ crow,
                                        int64_t *__restrict__ cglob, uint32_t *status) {
    __shared__ int owner_s;
    const int t = blockIdx.x;
    if (threadIdx.x == 0) {
        int owner = -1;
        int64_t g = -1;
        for (int r = 0; r < world && owner < 0; ++r) {
            const int64_t v = reinterpret_cast<const int64_t *>(recv + (int64_t)r * blk_bytes)[t];
            if (v >= 0) {
                owner = r;
                g = v;
            }
        }
        if (owner < 0) flag_error(status, kFlagExchange);
        cglob[t] = g;
        owner_s = owner;
    }
    __syncthreads();
    const int owner = owner_s;
    const float *src = owner < 0 ? nullptr
                                 : reinterpret_cast<const float *>(recv + (int64_t)owner * blk_bytes + idx_bytes) +
                                       (int64_t)t * d;
    for (int f = threadIdx.x; f < d; f += blockDim.x) crow[(int64_t)t * d + f] = src ? src[f] : 0.f;
}

// This shard's potential of every trial (the same sums as one GPU's choice).
__global__ void kpp_shard_potentials_kernel(const double *__restrict__ bpot, int T, int64_t n_blocks,
                                            double *__restrict__ pot_out) {
    griddep_wait();
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    for (int t = w; t < T; t += blockDim.x / 32) {
        const double v = trial_potential(bpot, t, n_blocks, lane);
        if (lane == 0) pot_out[t] = v;
    }
}

// The winner of center c: the trial whose potential, summed over the ranks
// in rank order, is lowest (lowest trial on ties; trial 0 for the first
// center).  indices[c] and centers[c] take its global index and row; D^2 is
// lowered by its distances and the shard's block sums rewritten.
__global__ void __launch_bounds__(kBsThreads)
    kpp_shard_commit_kernel(const double *__restrict__ dist, const double *__restrict__ recv_pot, int world, int T,
                            int first, int64_t n, const int64_t *__restrict__ cglob, const float *__restrict__ crow,
                            int d, int64_t c, int64_t *__restrict__ indices, float *__restrict__ centers,
                            double *__restrict__ D2, double *__restrict__ bsum, int64_t n_blocks) {
    griddep_wait();
    __shared__ double red[kBsThreads];
    __shared__ int best_s;
    if (threadIdx.x == 0) {
        int best = 0;
        if (!first) {
            double bp = 0.0;
            for (int t = 0; t < T; ++t) {
                double p = recv_pot[t];
                for (int r = 1; r < world; ++r) p += recv_pot[(int64_t)r * T + t];
                if (t == 0 || p < bp) {
                    bp = p;
                    best = t;
                }
            }
        }
        best_s = best;
    }
    __syncthreads();
    const int best = best_s;
    if (blockIdx.x == 0) {
        if (threadIdx.x == 0) indices[c] = cglob[best];
        if (centers)
            for (int f = threadIdx.x; f < d; f += kBsThreads)
                centers[c * (int64_t)d + f] = crow[(int64_t)best * d + f];
    }
    if (blockIdx.x >= n_blocks) return;
    const double *db = dist + (int64_t)best * n;
    const int64_t base = (int64_t)blockIdx.x * kKppScanBlock;
    double sum = 0.0;
#pragma unroll
    for (int q = 0; q < kKppScanBlock / kBsThreads; ++q) {
        const int64_t i = base + threadIdx.x + (int64_t)q * kBsThreads;
        if (i < n) {
            const double v = db[i];
            const double nd = first ? v : fmin(D2[i], v);
            D2[i] = nd;
            sum += nd;
        }
    }
    red[threadIdx.x] = sum;
    __syncthreads();
    for (int w = kBsThreads / 2; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) bsum[blockIdx.x] = red[0];
}

__global__ void kpp_shard_total_kernel(const double *__restrict__ bsum, int64_t n_blocks, double *__restrict__ out) {
    griddep_wait();
    const double t = d2_total(bsum, n_blocks, threadIdx.x);
    if (threadIdx.x == 0) *out = t;
}

// The draws of center c on a shard (one warp per trial).  From the ranks'
// totals, in rank order: the global sum S, target = u * S, and the owner,
// the first rank whose running total exceeds the target (the last rank's
// last sample when none does, as on one GPU).  The owner searches its shard
// with the earlier ranks' total as the running sum's start and fills its
// exchange slot; the other ranks mark the slot -1.
__global__ void __launch_bounds__(32)
    kpp_shard_pick_kernel(const double *__restrict__ bsum, int64_t n_blocks, const double *__restrict__ D2,
                          int64_t n_local, const float *__restrict__ X, int d, int64_t row_offset, uint64_t seed,
                          uint64_t draw_base, int T, const double *__restrict__ totals, int world, int rank,
                          uint8_t *__restrict__ send, int64_t idx_bytes) {
    const int lane = threadIdx.x;
    const int t = blockIdx.x;
    if (t >= T) return;
    double S = totals[0];
    for (int r = 1; r < world; ++r) S += totals[r];
    const double target = philox_uniform(seed, draw_base + (uint64_t)t) * S;
    int owner = world - 1;
    bool clip = true;
    double base = 0.0, run = 0.0;
    for (int r = 0; r < world; ++r) {
        const double next = r == 0 ? totals[0] : run + totals[r];
        if (next > target) {
            owner = r;
            base = run;
            clip = false;
            break;
        }
        run = next;
    }
    int64_t *idx = reinterpret_cast<int64_t *>(send);
    if (owner != rank) {
        if (lane == 0) idx[t] = -1;
        return;
    }
    const int64_t pick = clip ? n_local - 1 : d2_search(bsum, n_blocks, D2, n_local, target, base, lane);
    if (lane == 0) idx[t] = row_offset + pick;
    float *row = reinterpret_cast<float *>(send + idx_bytes) + (int64_t)t * d;
    for (int f = lane; f < d; f += 32) row[f] = X[pick * (int64_t)d + f];
}

cudaError_t launch_kpp_shard_first(const float *X, int64_t n_local, int64_t d, int64_t row_offset, int64_t n_global,
                                   int T, uint64_t seed, uint8_t *send, uint8_t *ws, cudaStream_t s) {
    kpp_shard_first_kernel<<<1, 256, 0, s>>>(X, n_local, (int)d, row_offset, n_global, seed, T, send,
                                             kpp_exchange_idx_bytes(T), reinterpret_cast<WsHeader *>(ws));
    return cudaGetLastError();
}

cudaError_t launch_kpp_shard_dist(const float *X, int64_t n_local, int64_t d, int T, bool first, const uint8_t *recv,
                                  int world, double *pot_out, const KppShardLayout &L, uint8_t *ws, cudaStream_t s) {
    const int Tn = first ? 1 : T;
    float *crow = reinterpret_cast<float *>(ws + L.off_crow);
    int64_t *cglob = reinterpret_cast<int64_t *>(ws + L.off_cglob);
    WsHeader *hdr = reinterpret_cast<WsHeader *>(ws);
    kpp_shard_gather_kernel<<<Tn, 256, 0, s>>>(recv, world, kpp_exchange_bytes(T, d), kpp_exchange_idx_bytes(T),
                                               (int)d, crow, cglob, &hdr->status);
    cudaError_t e = cudaGetLastError();
    const double *D2 = first ? nullptr : reinterpret_cast<const double *>(ws + L.K.off_d2);
    if (e == cudaSuccess) e = kpp_dist_pass(X, n_local, d, L.K, ws, Tn, nullptr, crow, D2, true, false, false, s);
    if (e == cudaSuccess && !first)
        e = launch_kernel(true, kpp_shard_potentials_kernel, dim3(1), dim3(256), 0, s,
                          (const double *)(ws + L.K.off_bpot), T, L.K.n_blocks, pot_out);
    return e;
}

cudaError_t launch_kpp_shard_commit(int64_t n_local, int64_t d, int T, bool first, const double *recv_pot, int world,
                                    int64_t c, int64_t *indices, float *centers, double *total_out,
                                    const KppShardLayout &L, uint8_t *ws, cudaStream_t s) {
    double *bsum = reinterpret_cast<double *>(ws + L.K.off_bsum);
    cudaError_t e = launch_kernel(false, kpp_shard_commit_kernel, dim3((unsigned)L.K.n_blocks), dim3(kBsThreads), 0, s,
                                  (const double *)(ws + L.K.off_dist), recv_pot, world, T, first ? 1 : 0, n_local,
                                  (const int64_t *)(ws + L.off_cglob), (const float *)(ws + L.off_crow), (int)d, c,
                                  indices, centers, reinterpret_cast<double *>(ws + L.K.off_d2), bsum, L.K.n_blocks);
    if (e == cudaSuccess && total_out)
        e = launch_kernel(true, kpp_shard_total_kernel, dim3(1), dim3(32), 0, s, (const double *)bsum, L.K.n_blocks,
                          total_out);
    return e;
}

cudaError_t launch_kpp_shard_pick(const float *X, int64_t n_local, int64_t d, int64_t row_offset, int T, uint64_t seed,
                                  int64_t c, const double *totals, int world, int rank, uint8_t *send,
                                  const KppShardLayout &L, uint8_t *ws, cudaStream_t s) {
    kpp_shard_pick_kernel<<<T, 32, 0, s>>>(reinterpret_cast<const double *>(ws + L.K.off_bsum), L.K.n_blocks,
                                           reinterpret_cast<const double *>(ws + L.K.off_d2), n_local, X, (int)d,
                                           row_offset, seed, 1 + (uint64_t)(c - 1) * (uint64_t)T, T, totals, world,
                                           rank, send, kpp_exchange_idx_bytes(T));
    return cudaGetLastError();
}

}  // namespace km

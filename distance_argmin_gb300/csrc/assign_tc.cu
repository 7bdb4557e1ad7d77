// Fused nearest-centroid assignment on the sm_103a tensor cores.
//
// What it computes ("Three shapes that fit an eager Gram assignment", section
// "Gram assignment"; "004 — tile sizes, a Cython Lloyd step, and k-means++",
// section "Schedules added"): for every sample x_i the centroid index j that
// minimises ||c_j||^2 - 2 x_i.c_j (||x_i||^2 is common to a row and left out
// of the comparison), lowest j on ties.  The (n, k) score matrix is never
// stored: each 128 x 256 tile of scores lives only in tensor memory, is
// reduced to one (score, index) key per row by the epilogue warps, and is
// merged across centroid tiles with a 64-bit atomic minimum.
//
// Precision: the pages run float32 with TF32 disabled.  Here each float32
// operand v is split as hi = bf16(v), lo = bf16(v - hi) (v = hi + lo to about
// 2^-16 relative) and x.c = hi_x.hi_c + (lo_x.hi_c + hi_x.lo_c), dropping the
// lo_x.lo_c term.  The tensor cores add each 16-wide partial product into the
// float32 accumulator with a truncating add, so every MMA into an accumulator
// of magnitude |x.c| costs up to one unit in its last place, always in the
// same direction.  Accumulator modes (templates DB, WIDE, CHUNKED):
//   DB    d < 2048 (and up to 4096 where wide units do not apply: k <= 256,
//         the fused update, 3xTF32 up to 2048): the three products share one
//         accumulator per tile, and two such accumulators are double-buffered
//         in tensor memory, so the epilogue of one tile overlaps the MMAs of
//         the next;
//   WIDE  d >= 2048 with k > 256: a CTA pair computes two adjacent 256-column
//         tiles at once, each with one accumulator, single-buffered: every X
//         k-block is split once for 512 centroids instead of 256.  Above
//         8192 features (CHUNKED) K runs in chunks of at most 8192: after
//         each chunk but the last the epilogue adds the raw accumulator into
//         a running sum the CTA keeps in the workspace and hands the
//         accumulator back, and the last chunk's epilogue adds the running
//         sum before the argmin.  The truncation error is then that of one
//         chunk, as at d = 8192, at any d;
//   else  (d > 4096 with k <= 256, the built-in scratch above 8192, or 3xTF32
//         above 2048): hi.hi gets an accumulator of its own and the two small
//         correction products another (only d/16 truncating adds act at the
//         magnitude of x.c, not 3 d/16; the corrections stay about 2^8
//         smaller), added in float32 in the epilogue, single-buffered.
// Template TF32 swaps the split for 3xTF32 (see Fmt), a comparator; template
// FUSED adds the mean update's accumulation to the epilogue
// (kmeans_lloyd_iter_fused), another comparator.
//
// Structure: CTA pairs (clusters of 2, tcgen05 cta_group::2), persistent over
// a grouped tile order.  A pair owns a 256-sample x 256-centroid tile (two
// side by side when wide; below, one tile): each
// CTA holds 128 samples (its half of A, the rows of its tensor memory) and
// 128 centroids (its half of B); the even CTA issues the M = 256 MMAs for both.
//   warp 16      TMA producer (each CTA): its X rows (fp32) and its C rows
//                (bf16 hi / lo), 4-deep ring
//   warps 0-7    split X into bf16 hi / lo in the UMMA shared-memory layout
//                (6-deep ring), accumulate ||x_i||^2 on a sample block's first
//                centroid tile, then signal the even CTA that this k-block of
//                A (and B) is ready
//   warp 17      allocates the pair's tensor memory (both CTAs); in the even
//                CTA issues tcgen05.mma (descriptors built before it waits for
//                the split stage): per 16-wide K step hi.hi, lo.hi and hi.lo
//                into the tile's accumulator(s); completions are multicast to
//                both CTAs
//   warps 8-15   epilogue (each CTA, its 128 rows): tcgen05.ld the
//                accumulator(s) (two warps per lane quarter, 128 columns
//                each), score = ||c||^2 - 2 x.c, row min / argmin, atomicMin
//                into the per-sample key
// The tiles go to the pairs in rounds.  A last round at most half full would
// leave most pairs idle for a whole tile; its tiles run instead as two halves
// of the k-blocks on two pairs (work units, see unit_at).  In the epilogue the
// half that takes the first ticket parks its raw accumulator in the workspace
// and tags it; the other waits for the tag and adds the parked part to its
// own before the argmin.  Whole tiles, split tiles and chunked units each
// keep an MMA issue loop of their own around one inlined k-block step.
// Every wait is bounded; a timeout raises a flag in the status word and both
// CTAs wind down without hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <cstdlib>
#include <mutex>

#include "assign_common.cuh"
#include "common.cuh"
#include "trace.cuh"
#include "ptx.cuh"

namespace km {

namespace tc {
constexpr int BM = 128;                        // samples per CTA (the pair's MMA has M = 256)
constexpr int BN = 256;                        // centroids per pair tile (UMMA N)
constexpr int BN_CTA = BN / 2;                 // centroid rows each CTA loads
constexpr int BK = 32;                         // features per pipeline stage
constexpr int SPLIT_WARPS = 8;                 // warps converting X to bf16 hi / lo
constexpr int EPI_WARPS = 8;                   // 4 or 8: one or two warps per tensor-memory lane quarter
constexpr int EPI_COLS = BN * 4 / EPI_WARPS;   // accumulator columns each epilogue warp reads
constexpr int EPI_CHUNK = 32;                  // columns per tensor-memory load (16 or 32)
constexpr int WARP_EPI = SPLIT_WARPS;
constexpr int WARP_TMA = SPLIT_WARPS + EPI_WARPS;
constexpr int WARP_MMA = WARP_TMA + 1;
constexpr int THREADS = (WARP_MMA + 1) * 32;
constexpr int SPLIT_THREADS = SPLIT_WARPS * 32;
constexpr int SPLIT_GROUPS = BK / 8;                            // 8-feature groups per row of a k-block
constexpr int ROWS_PER_SPLIT_THREAD = BM * SPLIT_GROUPS / SPLIT_THREADS;
constexpr int SPLIT_ROW_STRIDE = SPLIT_THREADS / SPLIT_GROUPS;
constexpr int X_BYTES = BM * BK * 4;           // fp32 X tile, 128-byte swizzle
constexpr int BAR_BYTES = 256;
constexpr int ACC_MAIN = 0;                    // tensor-memory columns (separate accumulators)
constexpr int ACC_CORR = BN;
constexpr int TMEM_COLS = 2 * BN;              // either main + corrections, or two single accumulators
// Where wide units (below) do not apply, up to this many features the three
// products share one accumulator per tile and the accumulators are
// double-buffered, so the epilogue of one tile overlaps the MMAs of the next.
// The tensor cores' truncating float32 accumulation then costs about
// 6e-9 * d relative (measured 1.01e-4 at d = 16384); the wide units keep one
// accumulator up to d = 8192, and beyond that the correction products keep
// their own accumulator (single-buffered), which is about 3x more accurate.
constexpr int SINGLE_ACC_MAX_D = 4096;
// 3xTF32 issues an MMA per 8 features instead of 16, twice the truncating
// adds (measured 8.4e-5 relative with one accumulator at d = 4096, against
// 2.7e-5 for bf16x3), so its single-accumulator limit is half as large.
constexpr int SINGLE_ACC_MAX_D_TF32 = 2048;
// From WIDE_MIN_D features, with more than one tile of centroids, bf16x3
// runs wide units: a CTA pair computes 256 samples x 512 centroids (two
// 256-column tiles), each tile's three products in one accumulator, the two
// filling the 512 tensor-memory columns (single-buffered).  Every split of an
// X k-block then feeds twice the MMAs: at the power cap the X split costs
// energy the tensor cores could use (halving its work measured about 5% on
// the sample-heavy shape; the wide units as a whole ran that shape's
// assignment 12.5% faster).  One accumulator over this many features carries
// about twice the truncation error of d = 4096 (about 6e-9 * d; measured
// 5.6e-5 over every row of the sample- and centroid-heavy shapes), inside the
// 1e-4 bound; above it the wide units run K in chunks of at most this size.
constexpr int WIDE_MAX_D = 8192;
// Wide units pay off from this many features (and more than one tile of
// centroids): on lloyd10 (d = 2048) they ran 3.7% faster than the
// double-buffered single tiles, whose overlapped epilogue matters less than
// halving the split; with fewer features the epilogue's share grows, and the
// double-buffered tiles (with their K split of a short last round) stay.
constexpr int WIDE_MIN_D = 2048;
// Pairs that read the same X block or centroid columns in a round share its
// k-blocks in L2 only while they read them within about the time L2 holds
// them; over a long launch the pairs drift apart and re-read from DRAM (35
// to 68 GB a launch on the sample-heavy shape against 25 GB in step).  So
// from this many rounds on, each CTA's producer waits at the start of a round
// until the round's CTAs have all started it, for at most
// ROUND_SYNC_WAIT_NS: a scheduling hint, never an error, so a CTA that is
// not resident yet (another kernel on the GPU) costs at most that wait.
// Measured back to back under the power cap: the sample-heavy shape 1.0 and
// 1.3% faster on two boxes, centroid-heavy +0.3 and -1.0%, feature-heavy
// +0.3% (a barrier without the time limit: -2.4% and -1.8%); with it on
// every launch, lloyd10 (7 rounds) was 3.5% slower, hence the lower bound.
// Longer limits (100 and 300 us) measured no better.
constexpr int ROUND_SYNC_MIN_ROUNDS = 16;
constexpr uint64_t ROUND_SYNC_WAIT_NS = 20000;
constexpr int GROUP_M = 8;                     // pair sample blocks per raster band
constexpr uint16_t PAIR_MASK = 0x3;
static_assert(SPLIT_WARPS % 4 == 0 && WARP_EPI % 4 == 0, "epilogue warps start on a lane-quarter boundary");
static_assert(kKSplitSlotBytes == 2 * BM * BN * 4 && kKSplitSyncWords == 2 * EPI_WARPS * 2,
              "the K-split parking area matches the tile and the epilogue warps");

// What depends on the operand format.
//  bf16x3: hi = bf16(v), lo = bf16(v - hi), both written by the split warps
//          (X) or the prologue (C) in the 64-byte-swizzled K-major layout;
//          an MMA covers K = 16.
//  3xTF32: hi = v with its low 13 mantissa bits cleared, lo = (v - hi) with
//          its low 13 bits cleared, both exact as TF32 values; the split
//          warps clear X's bits in place in the fp32 TMA tile (the A operand
//          hi) and write lo beside it, the prologue writes C's hi and lo as
//          fp32; everything keeps the 128-byte-swizzled K-major layout of
//          the fp32 tiles, and an MMA covers K = 8.
template <bool TF32, bool WIDE = false>
struct Fmt {
    static constexpr int NT = WIDE ? 2 : 1;                        // centroid tiles per work unit
    static constexpr int B_BYTES = BN_CTA * BK * (TF32 ? 4 : 2);  // one C part per CTA
    static constexpr int A_STAGE = TF32 ? BM * BK * 4 : 2 * BM * BK * 2;  // lo (tf32) or hi + lo (bf16)
    static constexpr int A_LO = TF32 ? 0 : BM * BK * 2;                   // offset of lo in an A stage
    static constexpr int XB_STAGE = X_BYTES + 2 * NT * B_BYTES;  // X, then hi and lo of each centroid tile
    // X + C stages (TMA ring) and split-X stages; a wide stage carries twice
    // the MMA work, so fewer stages cover as much time
    static constexpr int SXB = TF32 ? 3 : (WIDE ? 3 : 4);
    static constexpr int SA = TF32 ? 4 : (WIDE ? 5 : 6);
    static constexpr int A_BASE = SXB * XB_STAGE;
    static constexpr int BAR_BASE = A_BASE + SA * A_STAGE;
    static constexpr int SMEM_BYTES = BAR_BASE + BAR_BYTES + 1024;  // + alignment slack
    static constexpr int TX_BYTES = XB_STAGE;
    static constexpr int K_STEP_BYTES = 32;                  // one MMA's K extent: 16 bf16 or 8 tf32
    static constexpr int K_STEPS = BK * (TF32 ? 4 : 2) / K_STEP_BYTES;
    static constexpr uint32_t ROW_BYTES = TF32 ? 128u : 64u;  // K-major row of one tile
    static constexpr uint32_t SBO = 8 * ROW_BYTES;           // 8 rows per swizzle atom
    static constexpr uint32_t LAYOUT = TF32 ? kLayoutSW128 : kLayoutSW64;
    // barrier slots
    static constexpr int XB_FULL = 0, XB_EMPTY = SXB, A_FULL = 2 * SXB, A_EMPTY = 2 * SXB + SA;
    static constexpr int T_FULL = 2 * SXB + 2 * SA, T_EMPTY = T_FULL + 2, DRAIN = T_FULL + 4;  // 2 accumulator slots
    static constexpr int NUM_BARS = T_FULL + 5;
    static_assert(XB_STAGE % 1024 == 0 && A_STAGE % 1024 == 0, "stages stay 1 KiB aligned");
    static_assert(SMEM_BYTES <= 232448, "fits the 227 KiB opt-in limit");
    static_assert(NUM_BARS * 8 + 16 <= BAR_BYTES, "barriers fit");
};
}  // namespace tc

struct TcParams {
    int n, k, d;
    int num_m, num_n, num_kb, num_tiles;  // num_m counts 256-sample pair blocks
    const float *cnorm;
    float *xnorm;
    unsigned long long *keys;
    uint32_t *status;
    int test_starve;  // test hook: the producer issues no loads, so the pipeline waits run out
    int test_hold_tag;  // test hook: K-split halves park but never tag, so the other halves' waits run out
    FusedUpdate fu;   // the update fused into the epilogue (kmeans_lloyd_iter_fused), else all null
    // K split of the last round: units [0, num_full) are whole tiles; unit
    // num_full + 2 s + h is half h of tile num_full + s (h = 0: k-blocks
    // [0, kb_half), h = 1: [kb_half, num_kb)).  Without a split num_units =
    // num_full = num_tiles.
    int num_units, num_full, kb_half;
    uint32_t epoch;   // this launch's ready tag: nonzero, unlike any tag left in ksync
    float *kacc;      // parked accumulators [slot][CTA][BM rows][BN columns]
    uint32_t *ksync;  // [slot][CTA][epilogue warp] {ticket, ready tag}
    // Chunked wide units: K runs in chunks of kb_chunk k-blocks, and each CTA
    // keeps the running sum of its finished chunks in park (kChunkParkCtaBytes
    // per CTA, indexed by blockIdx.x).
    int kb_chunk;
    float *park;
    // Soft round barrier of the wide units (null: off): every CTA's producer
    // counts itself in when it starts a round and waits, at most
    // ROUND_SYNC_WAIT_NS, for the round's other CTAs
    uint32_t *rsync;
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int &mb, int &nb) {
    const int band = tile / (tc::GROUP_M * num_n);
    const int first = band * tc::GROUP_M;
    const int gs = min(tc::GROUP_M, num_m - first);
    const int r = tile - band * tc::GROUP_M * num_n;
    mb = first + r % gs;
    nb = r / gs;
}

struct KUnit {
    int tile, kb0, kb1, half;  // half -1: a whole tile
};

__device__ __forceinline__ KUnit unit_at(const TcParams &p, int u) {
    if (u < p.num_full) return {u, 0, p.num_kb, -1};
    const int v = u - p.num_full;
    const int h = v & 1;
    return {p.num_full + (v >> 1), h ? p.kb_half : 0, h ? p.num_kb : p.kb_half, h};
}

__device__ __forceinline__ uint32_t bf162_bits(__nv_bfloat162 h) {
    return *reinterpret_cast<uint32_t *>(&h);
}

// hi = bf16(a), lo = bf16(a - hi) for a pair of floats, packed two per word
// (the first float in the low half).  a - hi is exact; one packed fma forms
// both differences.
__device__ __forceinline__ void split_pair(float a, float b, uint32_t &hi, uint32_t &lo) {
    hi = bf162_bits(__floats2bfloat162_rn(a, b));
    const float2 hf = make_float2(__uint_as_float(hi << 16), __uint_as_float(hi & 0xffff0000u));
    const float2 d = __ffma2_rn(hf, make_float2(-1.f, -1.f), make_float2(a, b));
    lo = bf162_bits(__floats2bfloat162_rn(d.x, d.y));
}

// One k-block of the X split: 128 rows x 32 fp32 (128-byte swizzled TMA
// tile) -> bf16 hi and lo tiles in the 64-byte-swizzled K-major layout the
// tensor cores read.  Thread t handles the 8-feature group (t & 3) of rows
// (t >> 2) + SPLIT_ROW_STRIDE * i: two 16-byte loads, two 16-byte stores.
// With NORM it also adds the squares of its values into a compensated
// running sum per row.
template <bool NORM>
__device__ __forceinline__ void split_kblock(const uint8_t *xs, uint8_t *ahi, int t,
                                             float (&acc)[tc::ROWS_PER_SPLIT_THREAD],
                                             float (&comp)[tc::ROWS_PER_SPLIT_THREAD]) {
    uint8_t *alo = ahi + tc::Fmt<false>::A_LO;
    const int g = t & (tc::SPLIT_GROUPS - 1);
#pragma unroll
    for (int i = 0; i < tc::ROWS_PER_SPLIT_THREAD; ++i) {
        const int r = tc::SPLIT_ROW_STRIDE * i + t / tc::SPLIT_GROUPS;
        const float4 v0 = *reinterpret_cast<const float4 *>(xs + r * 128 + (((2 * g) ^ (r & 7)) << 4));
        const float4 v1 = *reinterpret_cast<const float4 *>(xs + r * 128 + (((2 * g + 1) ^ (r & 7)) << 4));
        uint4 h, l;
        split_pair(v0.x, v0.y, h.x, l.x);
        split_pair(v0.z, v0.w, h.y, l.y);
        split_pair(v1.x, v1.y, h.z, l.z);
        split_pair(v1.z, v1.w, h.w, l.w);
        const uint32_t off = r * 64 + ((g ^ ((r >> 1) & 3)) << 4);
        *reinterpret_cast<uint4 *>(ahi + off) = h;
        *reinterpret_cast<uint4 *>(alo + off) = l;
        if (NORM) {
            float q = v0.x * v0.x;
            q = fmaf(v0.y, v0.y, q);
            q = fmaf(v0.z, v0.z, q);
            q = fmaf(v0.w, v0.w, q);
            q = fmaf(v1.x, v1.x, q);
            q = fmaf(v1.y, v1.y, q);
            q = fmaf(v1.z, v1.z, q);
            q = fmaf(v1.w, v1.w, q);
            const float y = q - comp[i];
            const float tsum = acc[i] + y;
            comp[i] = (tsum - acc[i]) - y;
            acc[i] = tsum;
        }
    }
}

__device__ __forceinline__ float tf32_trunc(float v) { return __uint_as_float(__float_as_uint(v) & 0xffffe000u); }

// One k-block of the 3xTF32 split: the fp32 X tile (128 rows x 32,
// 128-byte swizzled) keeps hi = v with its low 13 mantissa bits cleared,
// written back in place (it is the A operand hi), and lo = (v - hi) with its
// low 13 bits cleared goes to the same position of the lo tile (v - hi is
// exact; clearing its low bits drops at most 2 of them).  Thread t owns row
// t / 2 and four of that row's eight 16-byte chunks, at swizzled positions so
// that the eight threads of a quarter-warp hit distinct banks.  With NORM it
// also adds the squares of its 16 values (the exact v) into a compensated
// running sum.
template <bool NORM>
__device__ __forceinline__ void split_kblock_tf32(uint8_t *xs, uint8_t *alo, int t, float &acc, float &comp) {
    const int r = t >> 1;
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t off = r * 128 + ((((t & 1) * 4 + i) ^ (r & 7)) << 4);
        const float4 v = *reinterpret_cast<const float4 *>(xs + off);
        const float4 h = make_float4(tf32_trunc(v.x), tf32_trunc(v.y), tf32_trunc(v.z), tf32_trunc(v.w));
        const float4 l = make_float4(tf32_trunc(v.x - h.x), tf32_trunc(v.y - h.y), tf32_trunc(v.z - h.z),
                                     tf32_trunc(v.w - h.w));
        *reinterpret_cast<float4 *>(xs + off) = h;
        *reinterpret_cast<float4 *>(alo + off) = l;
        if (NORM) {
            q = fmaf(v.x, v.x, q);
            q = fmaf(v.y, v.y, q);
            q = fmaf(v.z, v.z, q);
            q = fmaf(v.w, v.w, q);
        }
    }
    if (NORM) {
        const float y = q - comp;
        const float tsum = acc + y;
        comp = (tsum - acc) - y;
        acc = tsum;
    }
}

// The update fused into the epilogue: the warp that merged the last column
// tile into 32 rows' keys adds those rows of X (still in L2: every column
// tile of the row block has just streamed them) into their clusters' sums
// with vector float atomics, and counts them.  The keys are final: every
// merging warp fenced its atomicMin before counting itself done.
__device__ __forceinline__ void fused_accumulate_rows(const TcParams &p, int row0, int lane) {
    const int i = row0 + lane;
    int j = -1;
    if (i < p.n) {
        const unsigned long long key = __ldcg(p.keys + i);
        if (key != kEmptyKey) j = (int)(key & 0xffffffffu);
    }
    if (j >= 0) atomicAdd(p.fu.counts + j, 1);
    const int d4 = p.d >> 2;
    const float4 *X4 = reinterpret_cast<const float4 *>(p.fu.X);
    float4 *S4 = reinterpret_cast<float4 *>(p.fu.sums);
    // two rows at a time, 8 chunks of each per lane: 16 loads in flight
    // before their atomics (one at a time, the loads' latency dominates)
    constexpr int U = 8;
    for (int r = 0; r < 32; r += 2) {
        const int ja = __shfl_sync(0xffffffffu, j, r);
        const int jb = __shfl_sync(0xffffffffu, j, r + 1);
        const float4 *xa = X4 + (size_t)(row0 + r) * d4;
        const float4 *xb = X4 + (size_t)(row0 + r + 1) * d4;
        for (int c0 = lane; c0 < d4; c0 += 32 * U) {
            float4 va[U], vb[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * u;
                va[u] = (ja >= 0 && c < d4) ? __ldg(xa + c) : make_float4(0.f, 0.f, 0.f, 0.f);
                vb[u] = (jb >= 0 && c < d4) ? __ldg(xb + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int c = c0 + 32 * u;
                if (ja >= 0 && c < d4) atomicAdd(S4 + (size_t)ja * d4 + c, va[u]);
                if (jb >= 0 && c < d4) atomicAdd(S4 + (size_t)jb * d4 + c, vb[u]);
            }
        }
    }
}

// DB: one accumulator per tile, double-buffered (d <= SINGLE_ACC_MAX_D); TF32:
// the 3xTF32 operand split instead of bf16x3 (see Fmt); WIDE: 256 x 512
// units, one accumulator per 256-column tile, single-buffered (bf16x3,
// d >= WIDE_MIN_D, k > 256); CHUNKED: wide units whose K runs in chunks of
// p.kb_chunk k-blocks with a running sum per CTA (d > WIDE_MAX_D)
template <bool DB, bool TF32, bool FUSED = false, bool WIDE = false, bool CHUNKED = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(tc::THREADS, 1)
    assign_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmChi,
                     const __grid_constant__ CUtensorMap tmClo, const TcParams p) {
    using F = tc::Fmt<TF32, WIDE>;
    static_assert(!WIDE || (!DB && !TF32 && !FUSED), "wide units: bf16x3, single-buffered, no fused update");
    static_assert(!CHUNKED || WIDE, "K chunks are a form of the wide units");
    constexpr int UNIT_N = F::NT * tc::BN;  // centroid columns of one work unit
    constexpr int EPI_CHUNKS = tc::EPI_COLS / tc::EPI_CHUNK;  // tensor-memory loads per tile and epilogue warp
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + F::BAR_BASE);
    auto bar = [&](int i) { return smem_addr(bars + i); };
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + F::NUM_BARS);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();  // 0 = the CTA that issues the MMAs
    const int pair = blockIdx.x >> 1;
    const int num_pairs = gridDim.x >> 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < F::SXB; ++s) {
            mbar_init(bar(F::XB_FULL + s), 1);
            mbar_init(bar(F::XB_EMPTY + s), tc::SPLIT_WARPS + 1);  // split warps + the MMA commit
        }
        for (int s = 0; s < F::SA; ++s) {
            mbar_init(bar(F::A_FULL + s), 2 * tc::SPLIT_WARPS);  // split warps of both CTAs (even CTA's copy)
            mbar_init(bar(F::A_EMPTY + s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(F::T_FULL + b), 1);
            mbar_init(bar(F::T_EMPTY + b), 2 * tc::EPI_WARPS);  // epilogue warps of both CTAs (even CTA's copy)
        }
        mbar_init(bar(F::DRAIN), 1);
        fence_barrier_init();
    }
    if (warp == tc::WARP_MMA) {
        tmem_alloc_pair(smem_addr(tmem_holder), tc::TMEM_COLS);
        tmem_relinquish_pair();
        tc_fence_before();
    }
    cluster_sync();  // both CTAs' barriers exist before anyone arrives remotely
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;
    griddep_wait();  // the centroid copies, norms and reset keys are written

    if (warp < tc::SPLIT_WARPS) {
        // ------------------------------------------------ split X into hi / lo
        const int t = threadIdx.x;  // 0 .. SPLIT_THREADS-1
        int it = 0;
        bool ok = true;
        for (int unit = pair; unit < p.num_units && ok; unit += num_pairs) {
            const KUnit un = unit_at(p, unit);
            int mb, nb;
            tile_coords(un.tile, p.num_m, p.num_n, mb, nb);
            const int m0 = mb * (2 * tc::BM) + (int)rank * tc::BM;
            float acc[tc::ROWS_PER_SPLIT_THREAD], comp[tc::ROWS_PER_SPLIT_THREAD];
#pragma unroll
            for (int i = 0; i < tc::ROWS_PER_SPLIT_THREAD; ++i) acc[i] = comp[i] = 0.f;
            for (int kb = un.kb0; kb < un.kb1; ++kb, ++it) {
                const int s = it % F::SXB;
                const int as = it % F::SA;
                if (!mbar_wait_warp(bar(F::XB_FULL + s), (it / F::SXB) & 1, p.status) ||
                    !mbar_wait_warp(bar(F::A_EMPTY + as), ((it / F::SA) & 1) ^ 1, p.status)) {
                    ok = false;
                    break;
                }
                uint8_t *xs = smem + s * F::XB_STAGE;
                uint8_t *ast = smem + F::A_BASE + as * F::A_STAGE;
                if constexpr (TF32) {
                    if (nb == 0)
                        split_kblock_tf32<true>(xs, ast, t, acc[0], comp[0]);  // this tile also reports ||x||^2
                    else
                        split_kblock_tf32<false>(xs, ast, t, acc[0], comp[0]);
                } else {
                    if (nb == 0)
                        split_kblock<true>(xs, ast, t, acc, comp);  // this tile also reports ||x||^2
                    else
                        split_kblock<false>(xs, ast, t, acc, comp);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive_cluster(map_to_cta(bar(F::A_FULL + as), 0));
                    mbar_arrive(bar(F::XB_EMPTY + s));  // this warp is done with the X tile
                }
            }
            if (!ok) break;
            if constexpr (TF32) {
                // two threads per row
                float v = acc[0] - comp[0];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                const int row = m0 + (t >> 1);
                if (nb == 0 && (t & 1) == 0 && row < p.n) {
                    // the two K halves of a split tile each add their part (onto 0)
                    if (un.half < 0) p.xnorm[row] = v;
                    else atomicAdd(p.xnorm + row, v);
                }
            } else {
#pragma unroll
                for (int i = 0; i < tc::ROWS_PER_SPLIT_THREAD; ++i) {
                    float v = acc[i] - comp[i];
                    v += __shfl_xor_sync(0xffffffffu, v, 1);
                    v += __shfl_xor_sync(0xffffffffu, v, 2);
                    const int row = m0 + tc::SPLIT_ROW_STRIDE * i + t / tc::SPLIT_GROUPS;
                    if (nb == 0 && (t & (tc::SPLIT_GROUPS - 1)) == 0 && row < p.n) {
                        if (un.half < 0) p.xnorm[row] = v;
                        else atomicAdd(p.xnorm + row, v);  // a K half of a split tile, onto 0
                    }
                }
            }
        }
    } else if (warp < tc::WARP_EPI + tc::EPI_WARPS) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;              // tensor-memory lane quarter this warp may read
        const int part = (warp - tc::WARP_EPI) >> 2;  // which EPI_COLS of the tile's 256 columns
        const uint32_t lanes = (uint32_t)(q * 32) << 16;
        int tile_iter = 0;
        int acc_use = 0;  // single-buffered accumulator: hand-overs so far (one per K chunk of a unit)
        // chunked wide units: this warp's rows and columns of the CTA's running
        // sum, interleaved like the K-split parking area below (float4 u4 of
        // load ch of tile t2 of lane l at ((t2 * EPI_CHUNKS + ch) * 8 + u4) * 32 + l)
        static_assert(kChunkParkCtaBytes == tc::EPI_WARPS * 32 * 2 * tc::EPI_COLS * 4, "one CTA's running sum");
        float *const csum = CHUNKED ? p.park + (size_t)blockIdx.x * (kChunkParkCtaBytes / 4) +
                                          (size_t)(warp - tc::WARP_EPI) * (32 * F::NT * tc::EPI_COLS) + lane * 4
                                    : nullptr;
        for (int unit = pair; unit < p.num_units; unit += num_pairs, ++tile_iter) {
            const KUnit un = unit_at(p, unit);
            int mb, nb;
            tile_coords(un.tile, p.num_m, p.num_n, mb, nb);
            const int buf = DB ? (tile_iter & 1) : 0;
            const uint32_t phase = DB ? ((tile_iter >> 1) & 1) : (acc_use & 1);
            if (!mbar_wait_warp(bar(F::T_FULL + buf), phase, p.status)) break;
            tc_fence_after();
            if constexpr (!DB) ++acc_use;
            const uint32_t acc_base = tmem_base + (DB ? (uint32_t)(buf * tc::BN) : (uint32_t)tc::ACC_MAIN);
            const int n0 = nb * UNIT_N + part * tc::EPI_COLS;
            const float *parked = nullptr;  // the rest of K (other half or earlier chunks), to add before the argmin
            if constexpr (CHUNKED) {
                // every K chunk but the last: add the accumulator into the
                // running sum (the first chunk stores it) and hand it back for
                // the next chunk
                bool ok = true;
                for (int kb = p.kb_chunk; kb < p.num_kb; kb += p.kb_chunk) {
#pragma unroll 1
                    for (int t2 = 0; t2 < F::NT; ++t2) {
#pragma unroll 1
                        for (int ch = 0; ch < EPI_CHUNKS; ++ch) {
                            if (n0 + t2 * tc::BN + ch * tc::EPI_CHUNK >= p.k) break;
                            float vm[tc::EPI_CHUNK];
                            tmem_ld_one<tc::EPI_CHUNK>(
                                acc_base + lanes + (uint32_t)(t2 * tc::BN + part * tc::EPI_COLS + ch * tc::EPI_CHUNK),
                                vm);
                            float4 *dst = reinterpret_cast<float4 *>(csum) + (t2 * EPI_CHUNKS + ch) * (tc::EPI_CHUNK / 4) * 32;
#pragma unroll
                            for (int u4 = 0; u4 < tc::EPI_CHUNK / 4; ++u4) {
                                float4 v = make_float4(vm[4 * u4], vm[4 * u4 + 1], vm[4 * u4 + 2], vm[4 * u4 + 3]);
                                if (kb > p.kb_chunk) {
                                    const float4 o = __ldcg(dst + u4 * 32);
                                    v = make_float4(v.x + o.x, v.y + o.y, v.z + o.z, v.w + o.w);
                                }
                                dst[u4 * 32] = v;
                            }
                        }
                    }
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(map_to_cta(bar(F::T_EMPTY), 0));
                    if (!mbar_wait_warp(bar(F::T_FULL), acc_use & 1, p.status)) {
                        ok = false;
                        break;
                    }
                    ++acc_use;
                    tc_fence_after();
                }
                if (!ok) break;
                if (p.num_kb > p.kb_chunk) parked = csum;
            }
            if constexpr (DB && !FUSED) {
                if (un.half >= 0) {
                    // The two K halves of a split tile meet here, warp by warp.
                    // The first to take a ticket parks its raw accumulator and
                    // tags it; the second waits for the tag (the first is
                    // running and only storing) and adds the parked part to its
                    // own.  float addition commutes, so the sum does not depend
                    // on which half came first.
                    const int slot = un.tile - p.num_full;
                    uint32_t *sync = p.ksync + (((size_t)slot * 2 + rank) * tc::EPI_WARPS + (warp - tc::WARP_EPI)) * 2;
                    // this warp's 32 rows x EPI_COLS columns, interleaved so that
                    // every 16-byte access of the warp covers 512 contiguous
                    // bytes: float4 u4 of chunk ch of lane l at (ch * 8 + u4) * 32 + l
                    float *park = p.kacc + ((((size_t)slot * 2 + rank) * tc::EPI_WARPS + (warp - tc::WARP_EPI)) *
                                                (32 * tc::EPI_COLS)) + (size_t)lane * 4;
                    uint32_t ticket = 0;
                    if (lane == 0) ticket = atomicAdd(sync, 1u);
                    ticket = __shfl_sync(0xffffffffu, ticket, 0);
                    if (ticket == 0) {
#pragma unroll 1
                        for (int ch = 0; ch < EPI_CHUNKS; ++ch) {
                            if (n0 + ch * tc::EPI_CHUNK >= p.k) break;
                            float vm[tc::EPI_CHUNK];
                            tmem_ld_one<tc::EPI_CHUNK>(
                                acc_base + lanes + (uint32_t)(part * tc::EPI_COLS + ch * tc::EPI_CHUNK), vm);
                            float4 *dst = reinterpret_cast<float4 *>(park) + ch * (tc::EPI_CHUNK / 4) * 32;
#pragma unroll
                            for (int u4 = 0; u4 < tc::EPI_CHUNK / 4; ++u4)
                                dst[u4 * 32] = make_float4(vm[4 * u4], vm[4 * u4 + 1], vm[4 * u4 + 2], vm[4 * u4 + 3]);
                        }
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(map_to_cta(bar(F::T_EMPTY + buf), 0));
                        __threadfence();
                        __syncwarp();
                        if (lane == 0 && !p.test_hold_tag) st_release_gpu(sync + 1, p.epoch);
                        continue;
                    }
                    if (!flag_wait_warp(sync + 1, p.epoch, p.status)) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(map_to_cta(bar(F::T_EMPTY + buf), 0));
                        break;
                    }
                    __threadfence();
                    if (lane == 0) sync[0] = 0u;  // the next launch starts from ticket 0
                    parked = park;
                }
            }
            float best = __int_as_float(0x7f800000);  // +inf
            int arg = -1;
            // the unit's tiles in column order (one, or two when wide), so that
            // the strict comparison keeps the lowest index on ties
#pragma unroll 1
            for (int t2 = 0; t2 < F::NT; ++t2) {
#pragma unroll 1
            for (int ch = 0; ch < EPI_CHUNKS; ++ch) {
                const int j0 = n0 + t2 * tc::BN + ch * tc::EPI_CHUNK;
                if (j0 >= p.k) break;
                const uint32_t col = (uint32_t)(t2 * tc::BN + part * tc::EPI_COLS + ch * tc::EPI_CHUNK);
                // x.c of this chunk's columns: one accumulator, or main + corrections
                float vm[tc::EPI_CHUNK], vc[tc::EPI_CHUNK];
                if constexpr (DB || WIDE) {
                    tmem_ld_one<tc::EPI_CHUNK>(acc_base + lanes + col, vm);
                    if constexpr (!FUSED) {
                        if (parked) {
                            const float4 *src =
                                reinterpret_cast<const float4 *>(parked) + (t2 * EPI_CHUNKS + ch) * (tc::EPI_CHUNK / 4) * 32;
#pragma unroll
                            for (int u4 = 0; u4 < tc::EPI_CHUNK / 4; ++u4) {
                                const float4 pv = __ldcg(src + u4 * 32);
                                vm[4 * u4] += pv.x;
                                vm[4 * u4 + 1] += pv.y;
                                vm[4 * u4 + 2] += pv.z;
                                vm[4 * u4 + 3] += pv.w;
                            }
                        }
                    }
                } else {
                    tmem_ld_pair<tc::EPI_CHUNK>(acc_base + lanes + col, tmem_base + lanes + tc::ACC_CORR + col, vm, vc);
#pragma unroll
                    for (int u = 0; u < tc::EPI_CHUNK; ++u) vm[u] += vc[u];
                }
                const float4 *cn4 = reinterpret_cast<const float4 *>(p.cnorm + j0);
                if (j0 + tc::EPI_CHUNK <= p.k) {
#pragma unroll
                    for (int u4 = 0; u4 < tc::EPI_CHUNK / 4; ++u4) {
                        const float4 cn = __ldg(cn4 + u4);
                        const float s0 = fmaf(-2.f, vm[4 * u4 + 0], cn.x);
                        const float s1 = fmaf(-2.f, vm[4 * u4 + 1], cn.y);
                        const float s2 = fmaf(-2.f, vm[4 * u4 + 2], cn.z);
                        const float s3 = fmaf(-2.f, vm[4 * u4 + 3], cn.w);
                        if (s0 < best) { best = s0; arg = j0 + 4 * u4 + 0; }
                        if (s1 < best) { best = s1; arg = j0 + 4 * u4 + 1; }
                        if (s2 < best) { best = s2; arg = j0 + 4 * u4 + 2; }
                        if (s3 < best) { best = s3; arg = j0 + 4 * u4 + 3; }
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < tc::EPI_CHUNK; ++u) {
                        if (j0 + u < p.k) {
                            const float s = fmaf(-2.f, vm[u], __ldg(p.cnorm + j0 + u));
                            if (s < best) { best = s; arg = j0 + u; }
                        }
                    }
                }
            }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(map_to_cta(bar(F::T_EMPTY + buf), 0));
            const int row = mb * (2 * tc::BM) + (int)rank * tc::BM + q * 32 + lane;
            if (row < p.n && arg >= 0) atomicMin(p.keys + row, make_key(best, (uint32_t)arg));
            if constexpr (FUSED) {
                // two warps per lane quarter merge into these 32 rows for each
                // of the num_n column tiles; the last of them adds the rows
                static_assert(tc::EPI_WARPS == 8, "two epilogue warps per lane quarter");
                __threadfence();
                __syncwarp();
                unsigned done = 0;
                if (lane == 0) done = atomicAdd(p.fu.row_done + ((mb * 2 + (int)rank) * 4 + q), 1u);
                done = __shfl_sync(0xffffffffu, done, 0);
                if (done == 2u * (unsigned)p.num_n - 1u) {
                    __threadfence();
                    fused_accumulate_rows(p, mb * (2 * tc::BM) + (int)rank * tc::BM + q * 32, lane);
                }
            }
        }
    } else if (warp == tc::WARP_TMA) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0 && !p.test_starve) {
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmChi);
            tma_prefetch_desc(&tmClo);
            int it = 0;
            bool ok = true;
            for (int unit = pair; unit < p.num_units && ok; unit += num_pairs) {
                const KUnit un = unit_at(p, unit);
                int mb, nb;
                tile_coords(un.tile, p.num_m, p.num_n, mb, nb);
                const int m0 = mb * (2 * tc::BM) + (int)rank * tc::BM;
                const int c0 = nb * UNIT_N + (int)rank * tc::BN_CTA;
                if (WIDE && p.rsync) {
                    // both CTAs of every pair with a unit in this round
                    const int r = (unit - pair) / num_pairs;
                    const uint32_t target =
                        2u * (uint32_t)(num_pairs * r + min(num_pairs, p.num_units - r * num_pairs));
                    atomicAdd(p.rsync, 1u);
                    const uint64_t t0 = globaltimer_ns();
                    while (ld_acquire_gpu(p.rsync) < target && globaltimer_ns() - t0 < tc::ROUND_SYNC_WAIT_NS)
                        __nanosleep(64);
                }
                for (int kb = un.kb0; kb < un.kb1; ++kb, ++it) {
                    const int s = it % F::SXB;
                    if (!mbar_wait(bar(F::XB_EMPTY + s), ((it / F::SXB) & 1) ^ 1, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + s * F::XB_STAGE;
                    mbar_arrive_expect_tx(bar(F::XB_FULL + s), F::TX_BYTES);
                    tma_load_2d(st, &tmX, bar(F::XB_FULL + s), kb * tc::BK, m0);
                    tma_load_2d(st + tc::X_BYTES, &tmChi, bar(F::XB_FULL + s), kb * tc::BK, c0);
                    tma_load_2d(st + tc::X_BYTES + F::B_BYTES, &tmClo, bar(F::XB_FULL + s), kb * tc::BK, c0);
                    if constexpr (WIDE) {  // the unit's second centroid tile (zero rows past k)
                        tma_load_2d(st + tc::X_BYTES + 2 * F::B_BYTES, &tmChi, bar(F::XB_FULL + s), kb * tc::BK,
                                    c0 + tc::BN);
                        tma_load_2d(st + tc::X_BYTES + 3 * F::B_BYTES, &tmClo, bar(F::XB_FULL + s), kb * tc::BK,
                                    c0 + tc::BN);
                    }
                }
            }
            if (!ok) {
                // let copies already in flight land before the CTA exits
                for (int j = max(0, it - F::SXB); j < it; ++j)
                    mbar_wait_drain(bar(F::XB_FULL + (j % F::SXB)), (j / F::SXB) & 1);
            }
        }
    } else {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0 && rank == 0) {
            constexpr uint32_t idesc =
                TF32 ? umma_idesc_tf32_f32(2 * tc::BM, tc::BN) : umma_idesc_bf16_f32(2 * tc::BM, tc::BN);
            const uint32_t d_main = tmem_base + tc::ACC_MAIN;
            const uint32_t d_corr = tmem_base + tc::ACC_CORR;
            const uint32_t dw = tmem_base + tc::BN;  // wide: the second tile's accumulator
            // One k-block (pipeline step `it`): the stage's MMAs into dm (hi.hi)
            // and dc (the corrections), the first of them onto a cleared
            // accumulator unless `acc_kb`, then the commits that free the
            // stages.  False when the wait for the split stage ran out.
            auto kblock = [&](int it, uint32_t dm, uint32_t dc, bool acc_kb) -> bool {
                const int s = it % F::SXB;
                const int as = it % F::SA;
                // operands of this stage: bf16 hi and lo of X in the A stage;
                // 3xTF32 hi of X in place in the fp32 tile, lo in the A stage
                const uint32_t xb = sbase + s * F::XB_STAGE;
                const uint32_t bhi = xb + tc::X_BYTES;
                const uint32_t blo = bhi + F::B_BYTES;
                const uint32_t ast = sbase + F::A_BASE + as * F::A_STAGE;
                const uint32_t ahi = TF32 ? xb : ast;
                const uint32_t alo = TF32 ? ast : ast + F::A_LO;
                // descriptors first: once the split stage lands, only the
                // MMAs remain between it and the tensor pipe (measured: the
                // issue latency here is on the critical path)
                uint64_t dah[F::K_STEPS], dal[F::K_STEPS], dbh[F::K_STEPS], dbl[F::K_STEPS];
                uint64_t dwh[F::K_STEPS], dwl[F::K_STEPS];  // wide: the second tile's hi and lo
#pragma unroll
                for (int kk = 0; kk < F::K_STEPS; ++kk) {
                    dah[kk] = umma_smem_desc(ahi + kk * F::K_STEP_BYTES, F::SBO, F::LAYOUT);
                    dal[kk] = umma_smem_desc(alo + kk * F::K_STEP_BYTES, F::SBO, F::LAYOUT);
                    dbh[kk] = umma_smem_desc(bhi + kk * F::K_STEP_BYTES, F::SBO, F::LAYOUT);
                    dbl[kk] = umma_smem_desc(blo + kk * F::K_STEP_BYTES, F::SBO, F::LAYOUT);
                    if constexpr (WIDE) {
                        dwh[kk] = umma_smem_desc(blo + F::B_BYTES + kk * F::K_STEP_BYTES, F::SBO, F::LAYOUT);
                        dwl[kk] = umma_smem_desc(blo + 2 * F::B_BYTES + kk * F::K_STEP_BYTES, F::SBO, F::LAYOUT);
                    }
                }
                // both CTAs' split warps have seen their X and C stage land
                if (!mbar_wait_cluster(bar(F::A_FULL + as), (it / F::SA) & 1, p.status)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < F::K_STEPS; ++kk) {
                    const uint32_t acc = (acc_kb || kk != 0) ? 1u : 0u;
                    if constexpr (TF32) {
                        mma_tf32_ss_pair(dm, dah[kk], dbh[kk], idesc, acc);
                        mma_tf32_ss_pair(dc, dal[kk], dbh[kk], idesc, DB ? 1u : acc);
                        mma_tf32_ss_pair(dc, dah[kk], dbl[kk], idesc, 1u);
                    } else {
                        mma_bf16_ss_pair(dm, dah[kk], dbh[kk], idesc, acc);
                        mma_bf16_ss_pair(dc, dal[kk], dbh[kk], idesc, (DB || WIDE) ? 1u : acc);
                        mma_bf16_ss_pair(dc, dah[kk], dbl[kk], idesc, 1u);
                        if constexpr (WIDE) {
                            mma_bf16_ss_pair(dw, dah[kk], dwh[kk], idesc, acc);
                            mma_bf16_ss_pair(dw, dal[kk], dwh[kk], idesc, 1u);
                            mma_bf16_ss_pair(dw, dah[kk], dwl[kk], idesc, 1u);
                        }
                    }
                }
                mma_commit_pair_multicast(bar(F::XB_EMPTY + s), tc::PAIR_MASK);
                mma_commit_pair_multicast(bar(F::A_EMPTY + as), tc::PAIR_MASK);
                return true;
            };
            int it = 0, tile_iter = 0;
            int acc_use = 0;  // single-buffered accumulator: hand-overs so far (one per K chunk of a unit)
            bool ok = true;
            for (int unit = pair; unit < p.num_units && ok; unit += num_pairs, ++tile_iter) {
                const int buf = DB ? (tile_iter & 1) : 0;
                const uint32_t phase = DB ? ((tile_iter >> 1) & 1) : (acc_use & 1);
                if (!mbar_wait_cluster(bar(F::T_EMPTY + buf), phase ^ 1, p.status)) break;
                tc_fence_after();
                if constexpr (!DB) ++acc_use;
                const uint32_t dm = DB ? tmem_base + (uint32_t)(buf * tc::BN) : d_main;
                const uint32_t dc = (DB || WIDE) ? dm : d_corr;  // one accumulator per tile, or main + corrections
                if constexpr (CHUNKED) {
                    for (int c0 = 0; c0 < p.num_kb && ok; c0 += p.kb_chunk) {
                        if (c0 > 0) {
                            // the epilogue adds this chunk to the running sum
                            // and hands the accumulator back
                            mma_commit_pair_multicast(bar(F::T_FULL), tc::PAIR_MASK);
                            if (!mbar_wait_cluster(bar(F::T_EMPTY), (acc_use & 1) ^ 1, p.status)) {
                                ok = false;
                                break;
                            }
                            ++acc_use;
                            tc_fence_after();
                        }
                        const int c1 = min(c0 + p.kb_chunk, p.num_kb);
                        for (int kb = c0; kb < c1; ++kb, ++it) {
                            if (!kblock(it, dm, dc, kb != c0)) {
                                ok = false;
                                break;
                            }
                        }
                    }
                } else if (unit < p.num_full) {
                    // whole tiles keep a loop of their own: any per-unit logic in
                    // it measured 1.3% on the whole kernel
                    for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
                        if (!kblock(it, dm, dc, kb != 0)) {
                            ok = false;
                            break;
                        }
                    }
                } else {
                    const KUnit un = unit_at(p, unit);
                    for (int kb = un.kb0; kb < un.kb1; ++kb, ++it) {
                        if (!kblock(it, dm, dc, kb != un.kb0)) {
                            ok = false;
                            break;
                        }
                    }
                }
                if (!ok) break;
                mma_commit_pair_multicast(bar(F::T_FULL + buf), tc::PAIR_MASK);
            }
            // no MMA may still be writing tensor memory when it is released
            mma_commit_pair(bar(F::DRAIN));
            mbar_wait_drain(bar(F::DRAIN), 0);
        }
    }

    __syncwarp();
    cluster_sync();  // no CTA leaves while its peer may still signal it
    if (warp == tc::WARP_MMA) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, tc::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

static bool encode_2d(CUtensorMap *map, CUtensorMapDataType dtype, int elem_bytes, const void *base,
                      uint64_t inner, uint64_t outer, uint64_t row_pitch_elems, uint32_t box_inner,
                      uint32_t box_outer, CUtensorMapSwizzle swz) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_pitch_elems * (uint64_t)elem_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int device_sm_count() {
    static std::atomic<int> cached[kMaxDevices];
    return cached_per_device(cached, [] {
        int dev = 0, v = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        return v > 0 ? v : 1;
    });
}

int assign_tc_smem_bytes() { return tc::Fmt<false>::SMEM_BYTES; }

// CTA pairs that can be resident at once (the persistent grid never exceeds
// it, so no pair waits for another to finish).
static int resident_pairs() {
    static std::atomic<int> cached[kMaxDevices];
    return cached_per_device(cached, [] {
        int clusters = 0;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(2 * (device_sm_count() / 2), 1, 1);
        cfg.blockDim = dim3(tc::THREADS, 1, 1);
        cfg.dynamicSmemBytes = tc::Fmt<false>::SMEM_BYTES;
        cudaLaunchAttribute attr;
        attr.id = cudaLaunchAttributeClusterDimension;
        attr.val.clusterDim.x = 2;
        attr.val.clusterDim.y = 1;
        attr.val.clusterDim.z = 1;
        cfg.attrs = &attr;
        cfg.numAttrs = 1;
        if (cudaOccupancyMaxActiveClusters(&clusters, assign_tc_kernel<true, false>, &cfg) != cudaSuccess ||
            clusters < 1) {
            cudaGetLastError();  // clear
            clusters = device_sm_count() / 2;
        }
        return clusters < 1 ? 1 : clusters;
    });
}

int64_t assign_round_rows(int64_t k, int64_t d) {
    if (d < tc::WIDE_MIN_D || k <= tc::BN) return 2 * tc::BM;
    int64_t a = resident_pairs(), b = (k + 2 * tc::BN - 1) / (2 * tc::BN);  // pairs, unit columns
    const int64_t pairs = a;
    while (b) {
        const int64_t t = a % b;
        a = b;
        b = t;
    }
    return 2 * tc::BM * (pairs / a);  // pair blocks * unit columns a multiple of the pairs
}

// Ready tags of K-split tiles: one per launch, never 0 (the value the prologue
// leaves), so a tag from an earlier launch on the same workspace never reads
// as ready.
static uint32_t next_ksplit_epoch() {
    static std::atomic<uint32_t> counter{0};
    uint32_t e;
    do {
        e = counter.fetch_add(1u, std::memory_order_relaxed) + 1u;
    } while (e == 0u);
    return e;
}

template <bool DB, bool TF32>
static cudaError_t set_smem_limit() {
    return cudaFuncSetAttribute(assign_tc_kernel<DB, TF32>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                tc::Fmt<TF32>::SMEM_BYTES);
}

cudaError_t launch_assign_tc(const float *X, int64_t n, int64_t k, int64_t d, const AssignLayout &L,
                             uint8_t *ws, cudaStream_t stream, bool chained, bool tf32, const FusedUpdate *fused) {
    // the shared-memory opt-in, once per device; a failure is kept and
    // returned by every later launch on that device
    static std::once_flag attr_once[kMaxDevices];
    static std::atomic<int> attr_err[kMaxDevices];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) dev = -1;
    auto set_all = [] {
        cudaError_t e = set_smem_limit<true, false>();
        if (e == cudaSuccess) e = set_smem_limit<false, false>();
        if (e == cudaSuccess) e = set_smem_limit<true, true>();
        if (e == cudaSuccess) e = set_smem_limit<false, true>();
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(assign_tc_kernel<true, false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     tc::Fmt<false>::SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(assign_tc_kernel<false, false, false, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, tc::Fmt<false, true>::SMEM_BYTES);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(assign_tc_kernel<false, false, false, true, true>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, tc::Fmt<false, true>::SMEM_BYTES);
        return e;
    };
    if (dev < 0) {
        const cudaError_t e = set_all();
        if (e != cudaSuccess) return e;
    } else {
        std::call_once(attr_once[dev], [&] { attr_err[dev].store((int)set_all(), std::memory_order_release); });
        const cudaError_t e = (cudaError_t)attr_err[dev].load(std::memory_order_acquire);
        if (e != cudaSuccess) return e;
    }

    // C hi / lo: bf16 (64-byte swizzle) or, for 3xTF32, fp32 (128-byte swizzle)
    CUtensorMap tmX, tmChi, tmClo;
    const void *chi = ws + L.off_chi;
    const void *clo = ws + L.off_clo;
    const CUtensorMapDataType cdt = tf32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    const int cbytes = tf32 ? 4 : 2;
    const CUtensorMapSwizzle cswz = tf32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
    if (L.split_elem_bytes != cbytes) return cudaErrorInvalidValue;
    if (!encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, X, (uint64_t)d, (uint64_t)n, (uint64_t)d,
                   tc::BK, tc::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmChi, cdt, cbytes, chi, (uint64_t)L.d_pad, (uint64_t)k, (uint64_t)L.d_pad, tc::BK, tc::BN_CTA,
                   cswz) ||
        !encode_2d(&tmClo, cdt, cbytes, clo, (uint64_t)L.d_pad, (uint64_t)k, (uint64_t)L.d_pad, tc::BK, tc::BN_CTA,
                   cswz))
        return cudaErrorInvalidValue;

    // accumulator mode: bf16x3 runs wide units (two tiles, one accumulator
    // each) from WIDE_MIN_D features when there is more than one tile of
    // centroids, above WIDE_MAX_D in K chunks of at most WIDE_MAX_D features
    // (where the workspace holds the running sums); otherwise one
    // double-buffered accumulator per tile up to SINGLE_ACC_MAX_D, and
    // separate accumulators beyond
    static_assert(tc::WIDE_MAX_D == kWideChunkD, "the workspace reserves the running sums above WIDE_MAX_D");
    const bool chunked = !tf32 && !fused && d > tc::WIDE_MAX_D && k > tc::BN && L.off_park != 0;
    const bool wide = chunked || (!tf32 && !fused && d >= tc::WIDE_MIN_D && d <= tc::WIDE_MAX_D && k > tc::BN);
    const bool db = !wide && d <= (tf32 ? tc::SINGLE_ACC_MAX_D_TF32 : tc::SINGLE_ACC_MAX_D);
    TcParams p{};
    p.n = (int)n;
    p.k = (int)k;
    p.d = (int)d;
    p.num_m = (int)((n + 2 * tc::BM - 1) / (2 * tc::BM));
    p.num_n = (int)((k + (wide ? 2 : 1) * tc::BN - 1) / ((wide ? 2 : 1) * tc::BN));  // work-unit columns
    p.num_kb = (int)((d + tc::BK - 1) / tc::BK);
    p.num_tiles = p.num_m * p.num_n;
    p.cnorm = reinterpret_cast<const float *>(ws + L.off_cnorm);
    p.xnorm = reinterpret_cast<float *>(ws + L.off_xnorm);
    p.keys = reinterpret_cast<unsigned long long *>(ws + L.off_keys);
    p.status = &reinterpret_cast<WsHeader *>(ws)->status;
    // Test-only fault injection (no trap, no fault): with this variable set the
    // producer issues nothing, every consumer's bounded wait runs out, the
    // status word reports KMEANS_ERR_DEVICE_TIMEOUT and the outputs hold -1.
    const char *starve = getenv("KMEANS_GB300_TEST_STARVE_PIPELINE");
    p.test_starve = (starve != nullptr && starve[0] == '1') ? 1 : 0;
    // Test-only, likewise: the first K half of a split tile parks its
    // accumulator but never tags it, so the second half's bounded wait runs
    // out and the call reports KMEANS_ERR_DEVICE_TIMEOUT.
    const char *hold = getenv("KMEANS_GB300_TEST_HOLD_KSPLIT_TAG");
    p.test_hold_tag = (hold != nullptr && hold[0] == '1') ? 1 : 0;
    int max_pairs = resident_pairs();
    if (chunked && max_pairs > kChunkParkCtas / 2) max_pairs = kChunkParkCtas / 2;  // one running sum per CTA
    const int pairs = p.num_tiles < max_pairs ? p.num_tiles : max_pairs;
    const int grid = 2 * (pairs > 0 ? pairs : 1);
    // K split of a last round that is at most half full (double-buffered
    // accumulators only, not the fused update): its tiles run as two K halves
    // on two pairs each, about half a round instead of a whole one
    p.num_units = p.num_full = p.num_tiles;
    p.kb_half = p.num_kb / 2;
    p.epoch = 0;
    p.kacc = nullptr;
    p.ksync = nullptr;
    // K chunks of at most WIDE_MAX_D features, balanced
    p.kb_chunk = p.num_kb;
    p.park = nullptr;
    // the soft round barrier of long wide launches (its counter is cleared
    // by the prep kernel before each call's first launch)
    p.rsync = nullptr;
    if (wide && (p.num_units + pairs - 1) / pairs >= tc::ROUND_SYNC_MIN_ROUNDS)
        p.rsync = &reinterpret_cast<WsHeader *>(ws)->round_arrivals;
    if (chunked) {
        const int max_kb = tc::WIDE_MAX_D / tc::BK;
        const int chunks = (p.num_kb + max_kb - 1) / max_kb;
        p.kb_chunk = (p.num_kb + chunks - 1) / chunks;
        p.park = reinterpret_cast<float *>(ws + L.off_park);
    }
    if (db && !fused && L.off_kacc != 0 && p.num_kb >= 2 && p.num_tiles > pairs) {
        const int rounds = (p.num_tiles + pairs - 1) / pairs;
        const int tail = p.num_tiles - (rounds - 1) * pairs;
        if (2 * tail <= pairs && tail <= kKSplitSlots) {
            p.num_full = p.num_tiles - tail;
            p.num_units = p.num_full + 2 * tail;
            p.kacc = reinterpret_cast<float *>(ws + L.off_kacc);
            p.ksync = reinterpret_cast<uint32_t *>(ws + L.off_ksync);
            p.epoch = next_ksplit_epoch();
        }
    }
    trace_mark(kTraceAssignTc, false, stream);
    const dim3 g(grid), b(tc::THREADS);
    cudaError_t e;
    if (fused) {
        // bf16x3 with double-buffered accumulators only
        if (tf32 || !db) return cudaErrorInvalidValue;
        p.fu = *fused;
        e = launch_kernel(chained, assign_tc_kernel<true, false, true>, g, b, tc::Fmt<false>::SMEM_BYTES, stream, tmX,
                          tmChi, tmClo, p);
    } else if (tf32)
        e = db ? launch_kernel(chained, assign_tc_kernel<true, true>, g, b, tc::Fmt<true>::SMEM_BYTES, stream, tmX, tmChi,
                               tmClo, p)
               : launch_kernel(chained, assign_tc_kernel<false, true>, g, b, tc::Fmt<true>::SMEM_BYTES, stream, tmX,
                               tmChi, tmClo, p);
    else if (db)
        e = launch_kernel(chained, assign_tc_kernel<true, false>, g, b, tc::Fmt<false>::SMEM_BYTES, stream, tmX, tmChi,
                          tmClo, p);
    else if (chunked)
        e = launch_kernel(chained, assign_tc_kernel<false, false, false, true, true>, g, b,
                          tc::Fmt<false, true>::SMEM_BYTES, stream, tmX, tmChi, tmClo, p);
    else if (wide)
        e = launch_kernel(chained, assign_tc_kernel<false, false, false, true>, g, b, tc::Fmt<false, true>::SMEM_BYTES,
                          stream, tmX, tmChi, tmClo, p);
    else
        e = launch_kernel(chained, assign_tc_kernel<false, false>, g, b, tc::Fmt<false>::SMEM_BYTES, stream, tmX, tmChi,
                          tmClo, p);
    trace_mark(kTraceAssignTc, true, stream);
    return e;
}

}  // namespace km

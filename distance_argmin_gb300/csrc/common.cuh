// Shared device helpers of the GB300 k-means library: status word, bounded
// waits, order-preserving keys for the fused argmin, workspace layout.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <cstddef>

#include <atomic>
#include <mutex>
#include <utility>

#include "../../include/kmeans_gb300.h"

namespace km {

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  The kernels of the assignment, the update
// and the Lloyd iteration form a chain on one stream, the first kernel of a
// call included: each is launched so that it may be scheduled while the
// kernel before it on the stream drains (ours or the caller's), and each calls
// griddep_wait() before its first global read or write.  That wait returns
// once the previous kernel has completed and its writes are visible; since
// every kernel waits before it exits, completion is transitive along the
// chain, and a caller's kernel that wrote the inputs has finished before they
// are read.  (Chaining a call's first kernel measured 2.6 us less per call of
// back-to-back updates of 65536 x 2048 into 1024 clusters, the same bits.)
// No kernel signals its dependents early: a dependent that is resident while
// its predecessor still runs only takes resources from it (measured: early
// signals made the update slower).  The wait is a no-op for a kernel launched
// the ordinary way.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Launch `kernel`; with `chained` set it may overlap the tail of the kernel
// launched before it on `s` (see above).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(bool chained, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                 cudaStream_t s, Args &&...args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = chained ? attr : nullptr;
    cfg.numAttrs = chained ? 1u : 0u;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// ---------------------------------------------------------------------------
// Host: one-time setup per device.  Function attributes (the shared-memory
// opt-in) are per device, and the cached launch limits differ per device, so
// both are kept per device index and set up safely from any host thread.
// ---------------------------------------------------------------------------
constexpr int kMaxDevices = 64;

// Runs fn() once for the current device (every time for a device index
// beyond kMaxDevices, which has no slot).
template <typename Fn>
inline void once_per_device(std::once_flag (&flags)[kMaxDevices], Fn &&fn) {
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices)
        std::call_once(flags[dev], std::forward<Fn>(fn));
    else
        fn();
}

// cache[device] = compute() the first time it is asked for on a device (a
// positive value; races compute the same value twice).
template <typename Fn>
inline int cached_per_device(std::atomic<int> (&cache)[kMaxDevices], Fn &&compute) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return compute();
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v <= 0) {
        v = compute();
        cache[dev].store(v, std::memory_order_relaxed);
    }
    return v;
}

// ---------------------------------------------------------------------------
// Device status word.  Lives in the first bytes of the caller's workspace and
// is cleared by every entry point before its first kernel.  Kernels OR flags
// into it; the host maps them to kmeans_status codes.
// ---------------------------------------------------------------------------
enum : uint32_t {
    kFlagTimeout = 1u,   // a pipeline wait ran out of time
    kFlagBadLabel = 2u,  // update saw a label outside [0, k)
    kFlagExchange = 4u,  // sharded k-means++: no rank's exchange block owned a trial
};

struct WsHeader {
    uint32_t status;          // device status flags
    uint32_t done_blocks;     // "last block" counter of the inertia reduction
    double fit_inertia;       // kmeans_fit: the last iteration's inertia
    uint32_t fit_nempty;      // kmeans_fit: clusters left empty by the last update
    unsigned long long kpp_rows;  // k-means++ with row pruning: sample rows its distance passes read
    uint32_t round_arrivals;      // tensor-core assignment: CTAs that have started each round (soft barrier)
    uint32_t pad[55];
};
// kmeans_fit reads the status word, the inertia and the empty count back in
// one copy of the header's first bytes.
constexpr size_t kFitRecordBytes = 20;
static_assert(offsetof(WsHeader, fit_inertia) == 8 && offsetof(WsHeader, fit_nempty) + 4 == kFitRecordBytes,
              "the fit's record is the header's first bytes");
static_assert(sizeof(WsHeader) == 256, "header is 256 bytes");
static_assert(offsetof(WsHeader, kpp_rows) == 24, "8-byte aligned");

// Wall-clock limit of one pipeline wait.  A wait that legitimately takes this
// long does not exist (the slowest stage waits for one k-block of a tile).
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void flag_error(uint32_t *status, uint32_t flag) {
    atomicOr(status, flag);
}

__device__ __forceinline__ bool error_raised(const uint32_t *status) {
    return *reinterpret_cast<const volatile uint32_t *>(status) != 0u;
}

// ---------------------------------------------------------------------------
// Order-preserving 32-bit image of a float: a < b (as finite floats) iff
// ord(a) < ord(b) (as unsigned).  The fused argmin packs ord(score) above the
// centroid index into one 64-bit key, so an unsigned 64-bit minimum picks the
// smallest score and, among equal scores, the lowest index.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t float_to_ord(float f) {
    uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float ord_to_float(uint32_t o) {
    uint32_t u = (o & 0x80000000u) ? (o & 0x7fffffffu) : ~o;
    return __uint_as_float(u);
}

__device__ __forceinline__ uint64_t make_key(float score, uint32_t j) {
    return (static_cast<uint64_t>(float_to_ord(score)) << 32) | j;
}

constexpr uint64_t kEmptyKey = ~0ull;

// ---------------------------------------------------------------------------
// Workspace layout.  Every region is 1 KiB aligned.  Sizes depend on n, on
// k*d (the split centroids) and on n/4096 (sort tiles); never on n*k.
// ---------------------------------------------------------------------------
__host__ __device__ inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

struct AssignLayout {
    int64_t d_pad;       // row pitch (elements) of the split centroid copies
    int64_t off_keys;    // n x u64 packed (score, index) keys
    int64_t off_xnorm;   // n x f32 ||x_i||^2
    int64_t off_cnorm;   // k x f32 ||c_j||^2
    int64_t off_chi;     // k x d_pad bf16 hi part of C
    int64_t off_clo;     // k x d_pad bf16 lo part of C
    int64_t off_partial; // kMaxReduceBlocks x f64 inertia partial sums
    int64_t split_elem_bytes;  // 2: bf16 hi / lo of C; 4: fp32 (3xTF32) hi / lo
    int64_t off_kacc;    // K-split tiles: kKSplitSlots x kKSplitSlotBytes parked accumulators (0: none)
    int64_t off_ksync;   // K-split tiles: kKSplitSlots x kKSplitSyncWords tickets and ready tags
    int64_t off_park;    // chunked wide units: kChunkParkCtas x kChunkParkCtaBytes running sums (0: none)
    int64_t bytes;
};

constexpr int kMaxReduceBlocks = 1024;

// The tensor-core assignment runs a persistent schedule of 256 x 256 tiles
// over its CTA pairs.  When the last round is at most half full, its tiles
// run as two halves of K each on two pairs; the half that finishes first
// parks its raw accumulator (one CTA: 128 rows x 256 columns of float32) for
// the other.  The parking area exists only for problems with more than
// kKSplitMinTiles tiles (below that there are no more tiles than pairs), and
// is sized for at most kKSplitSlots split tiles.
constexpr int kKSplitSlots = 40;
constexpr int64_t kKSplitMinTiles = 64;
constexpr int64_t kKSplitSlotBytes = 2 * 128 * 256 * 4;  // both CTAs of a pair
constexpr int kKSplitSyncWords = 2 * 8 * 2;              // CTA x epilogue warp x (ticket, tag)

// Above kWideChunkD features the bf16x3 wide units (256 samples x 512
// centroids, one accumulator per 256-column tile) run K in chunks of at most
// kWideChunkD features, so that each accumulator's truncation error stays
// that of d = kWideChunkD.  Between chunks every CTA adds its raw accumulator
// (128 rows x 512 columns of float32) into a running sum of its own in the
// workspace; the persistent grid has at most kChunkParkCtas CTAs.
constexpr int64_t kWideChunkD = 8192;
constexpr int kChunkParkCtas = 160;
constexpr int64_t kChunkParkCtaBytes = 128 * 512 * 4;

inline int64_t assign_tiles(int64_t n, int64_t k) { return ((n + 255) / 256) * ((k + 255) / 256); }

// `park`: reserve the parking areas of the K-split tiles and of the chunked
// wide units (tensor-core paths that may use them; not the built-in scratch
// or the fused update).
inline AssignLayout assign_layout(int64_t n, int64_t k, int64_t d, bool split, int split_elem_bytes = 2,
                                  bool park = true) {
    AssignLayout L{};
    L.d_pad = align_up(d, 64);
    L.split_elem_bytes = split ? split_elem_bytes : 0;
    int64_t o = sizeof(WsHeader);
    o = align_up(o, 1024); L.off_keys = o; o += n * 8;
    o = align_up(o, 1024); L.off_xnorm = o; o += n * 4;
    o = align_up(o, 1024); L.off_cnorm = o; o += k * 4;
    if (split) {
        o = align_up(o, 1024); L.off_chi = o; o += k * L.d_pad * split_elem_bytes;
        o = align_up(o, 1024); L.off_clo = o; o += k * L.d_pad * split_elem_bytes;
    } else {
        L.off_chi = L.off_clo = 0;
    }
    o = align_up(o, 1024); L.off_partial = o; o += kMaxReduceBlocks * 8;
    L.off_kacc = L.off_ksync = L.off_park = 0;
    if (split && park && assign_tiles(n, k) > kKSplitMinTiles) {
        o = align_up(o, 1024); L.off_kacc = o; o += kKSplitSlots * kKSplitSlotBytes;
        o = align_up(o, 1024); L.off_ksync = o; o += kKSplitSlots * kKSplitSyncWords * 4;
    }
    if (split && park && split_elem_bytes == 2 && d > kWideChunkD && k > 256) {
        o = align_up(o, 1024); L.off_park = o; o += kChunkParkCtas * kChunkParkCtaBytes;
    }
    L.bytes = align_up(o, 1024);
    return L;
}

// Update: LSD radix sort of the labels (8-bit digits) into a member list,
// then a segmented mean over fixed chunks of that list.
constexpr int kSortTile = 4096;      // labels per radix tile
constexpr int kSortThreads = 256;
constexpr int kRadixBins = 256;

struct UpdateLayout {
    int64_t n_tiles;     // radix tiles
    int64_t chunk;       // members per segmented-mean chunk
    int64_t n_chunks;
    int64_t off_counts;  // k x i32 member counts
    int64_t off_offsets; // (k + 1) x i32 exclusive scan of counts
    int64_t off_hist;    // 256 x n_tiles x i32 digit histograms (scanned in place)
    int64_t off_keys_a;  // n x u32 sort keys (ping)
    int64_t off_vals_a;  // n x i32 sort values (ping)
    int64_t off_keys_b;  // n x u32 (pong)
    int64_t off_vals_b;  // n x i32 (pong)
    int64_t off_head;    // n_chunks x d f32 partial sums, cluster entering a chunk
    int64_t off_tail;    // n_chunks x d f32 partial sums, cluster leaving a chunk
    int64_t off_tailc;   // n_chunks x int4 {cluster leaving the chunk (-1: none), its segment's bounds}
    int64_t n_utiles;    // tiles of the counting scatter (a constant cap, not n-proportional)
    int64_t utile;       // samples per counting tile
    int64_t off_table;   // n_utiles x k x i32 per-tile cluster counts, then column prefixes
    int64_t off_fin_partial;  // n_utiles x f64 inertia block sums of the Lloyd iteration's finalize
    bool counting;       // counting scatter (k <= kCountingMaxK) instead of the radix sort
    int64_t bytes;
};

constexpr int64_t kCountingMaxK = 32768;  // per-tile counters fit in shared memory
constexpr int64_t kCountingTiles = 256;

inline int64_t update_chunk(int64_t n, int64_t d) {
    // members per chunk: enough chunks for one full wave of 512-column slices
    // (the mean kernel's 128 threads of 40 registers fit 12 blocks per SM;
    // 12 measured 3% faster than 8, the loads it keeps in flight being what
    // bounds it), at least 16 members per chunk (small problems get more
    // blocks: 64 as the minimum left 4096 samples 64 blocks, 25% slower)
    int64_t slices = (d + 511) / 512;
    int64_t target_ctas = 152 * 12;
    int64_t chunks = (target_ctas + slices - 1) / slices;
    int64_t c = (n + chunks - 1) / chunks;
    if (c < 16) c = 16;
    c = align_up(c, 16);
    return c > 4096 ? 4096 : c;  // the chunk's member list is staged in shared memory
}

inline UpdateLayout update_layout(int64_t n, int64_t k, int64_t d) {
    UpdateLayout L{};
    L.n_tiles = (n + kSortTile - 1) / kSortTile;
    L.chunk = update_chunk(n, d);
    L.n_chunks = (n + L.chunk - 1) / L.chunk;
    int64_t o = sizeof(WsHeader);
    o = align_up(o, 1024); L.off_counts = o; o += k * 4;
    o = align_up(o, 1024); L.off_offsets = o; o += (k + 1) * 4;
    o = align_up(o, 1024); L.off_hist = o; o += kRadixBins * L.n_tiles * 4;
    o = align_up(o, 1024); L.off_keys_a = o; o += n * 4;
    o = align_up(o, 1024); L.off_vals_a = o; o += n * 4;
    o = align_up(o, 1024); L.off_keys_b = o; o += n * 4;
    o = align_up(o, 1024); L.off_vals_b = o; o += n * 4;
    o = align_up(o, 1024); L.off_head = o; o += L.n_chunks * d * 4;
    o = align_up(o, 1024); L.off_tail = o; o += L.n_chunks * d * 4;
    o = align_up(o, 1024); L.off_tailc = o; o += L.n_chunks * 16;
    L.counting = k <= kCountingMaxK;
    L.n_utiles = kCountingTiles;  // fixed, so the table is O(k) for every n
    L.utile = (n + L.n_utiles - 1) / L.n_utiles;
    L.off_table = 0;
    L.off_fin_partial = 0;
    if (L.counting) {
        o = align_up(o, 1024); L.off_table = o; o += L.n_utiles * k * 4;
        // last: the Lloyd iteration writes it while the assignment's keys and
        // norms (which lie below the member lists) are still being read
        o = align_up(o, 1024); L.off_fin_partial = o; o += L.n_utiles * 8;
    }
    L.bytes = align_up(o, 1024);
    return L;
}

// k-means++: D^2, running sums, per-trial distances and potentials.
constexpr int kKppScanBlock = 1024;   // samples per scan / potential block
constexpr int kKppMaxTrials = 32;
constexpr int kKppGroupTrials = 8;    // trial candidates per pass over X
constexpr int kKppSliceFloats = 4096; // features of the 8 candidates a CTA keeps in shared memory (128 KiB)

struct KppLayout {
    int T;
    int64_t n_blocks;     // 1024-sample blocks of the scan / potential reductions
    int S;                // feature slices (the distance pass splits d so a slice of the candidates stays resident)
    int W;                // features per slice (multiple of 256: whole 256-feature steps of the distance pass)
    int64_t off_d2;       // n x f64 current D^2
    int64_t off_dist;     // T x n x f64 distances to the trial candidates
    int64_t off_dpart;    // S x 8 x n x (f32 hi, f32 lo) per-slice partial distances of one pass
    int64_t off_bsum;     // n_blocks x f64 block sums of D^2
    int64_t off_bpot;     // T x n_blocks x f64 block potentials
    int64_t off_cand;     // T x i64 candidates of the current center
    int64_t off_chosen;   // spare
    // Rows that no trial can change (see kmeanspp.cu); 0 offsets: not reserved
    int64_t k;            // row pitch of the center-candidate table
    int64_t off_near;     // n x i32 each sample's nearest committed center (its position in the indices)
    int64_t off_dcc;      // T x k x f32 squared distances between the trial candidates and the committed centers
    int64_t off_rows;     // n_blocks x kKppScanBlock x i32 rows each block of samples has to read, ascending
    int64_t off_rcount;   // n_blocks x i32 rows listed per block
    int64_t off_flag;     // n x u8 1: the distance pass reads the row this round
    int64_t bytes;
};

// The distance pass keeps the prefix of the per-block row counts in shared
// memory beside the candidates; past this many sample blocks (16.7 M
// samples) the seeding reads every row.
constexpr int64_t kKppPruneMaxBlocks = 16384;

// k > 0: also the regions of the row pruning (the single-GPU seeding).
inline KppLayout kpp_layout(int64_t n, int64_t d, int T, int64_t k = 0) {
    KppLayout L{};
    L.T = T;
    L.n_blocks = (n + kKppScanBlock - 1) / kKppScanBlock;
    L.S = (int)((d + kKppSliceFloats - 1) / kKppSliceFloats);
    L.W = (int)align_up((d + L.S - 1) / L.S, 256);
    int64_t o = sizeof(WsHeader);
    o = align_up(o, 1024); L.off_d2 = o; o += n * 8;
    o = align_up(o, 1024); L.off_dist = o; o += (int64_t)T * n * 8;
    o = align_up(o, 1024); L.off_dpart = o; o += (int64_t)L.S * kKppGroupTrials * n * 8;
    o = align_up(o, 1024); L.off_bsum = o; o += L.n_blocks * 8;
    o = align_up(o, 1024); L.off_bpot = o; o += (int64_t)T * L.n_blocks * 8;
    o = align_up(o, 1024); L.off_cand = o; o += (int64_t)T * 8;
    o = align_up(o, 1024); L.off_chosen = o; o += 8;
    L.k = 0;
    L.off_near = L.off_dcc = L.off_rows = L.off_rcount = L.off_flag = 0;
    if (k > 0 && L.n_blocks <= kKppPruneMaxBlocks) {
        L.k = k;
        o = align_up(o, 1024); L.off_near = o; o += n * 4;
        o = align_up(o, 1024); L.off_dcc = o; o += (int64_t)T * k * 4;
        o = align_up(o, 1024); L.off_rows = o; o += L.n_blocks * kKppScanBlock * 4;
        o = align_up(o, 1024); L.off_rcount = o; o += L.n_blocks * 4;
        o = align_up(o, 1024); L.off_flag = o; o += n;
    }
    L.bytes = align_up(o, 1024);
    return L;
}

// k-means++ on one shard of the samples: the seeding's scratch for the
// shard's rows (room for the largest trial count), then the current
// candidates' rows and global indices, gathered from the ranks' exchange
// blocks.
struct KppShardLayout {
    KppLayout K;
    int64_t off_crow;   // kKppMaxTrials x d f32 candidate rows
    int64_t off_cglob;  // kKppMaxTrials x i64 candidate global sample indices
    int64_t bytes;
};

inline KppShardLayout kpp_shard_layout(int64_t n_local, int64_t d) {
    KppShardLayout L{};
    L.K = kpp_layout(n_local, d, kKppMaxTrials);
    int64_t o = align_up(L.K.bytes, 1024);
    L.off_crow = o; o += (int64_t)kKppMaxTrials * d * 4;
    o = align_up(o, 1024); L.off_cglob = o; o += (int64_t)kKppMaxTrials * 8;
    L.bytes = align_up(o, 1024);
    return L;
}

// One rank's exchange block: T int64 indices, then T rows of d float32.
inline int64_t kpp_exchange_idx_bytes(int T) { return align_up((int64_t)T * 8, 16); }
inline int64_t kpp_exchange_bytes(int T, int64_t d) { return align_up(kpp_exchange_idx_bytes(T) + (int64_t)T * d * 4, 16); }

}  // namespace km

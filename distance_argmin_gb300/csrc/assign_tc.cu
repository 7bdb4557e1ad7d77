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
// 2^-16 relative) and x.c is accumulated in float32 tensor memory as
// hi_x.hi_c + hi_x.lo_c + lo_x.hi_c.  The dropped lo_x.lo_c term and the
// split residuals are below 3 * 2^-16 |x_f c_f| per feature.
//
// Structure (one CTA per SM, persistent over a grouped tile order):
//   warp 8      TMA producer: X (fp32) tile, C hi / C lo (bf16) tiles
//   warps 0-3   split X into bf16 hi / lo in the UMMA shared-memory layout,
//               accumulate ||x_i||^2 on the way
//   warp 9      allocates tensor memory, issues tcgen05.mma (3 products per
//               16-wide K step) into one of two 128 x 256 f32 accumulators
//   warps 4-7   epilogue: tcgen05.ld the accumulator, score = ||c||^2 - 2 acc,
//               row min / argmin, atomicMin into the per-sample key
// Every wait is bounded; a timeout raises a flag in the status word and the
// whole CTA winds down without hanging.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "assign_common.cuh"
#include "common.cuh"
#include "ptx.cuh"

namespace km {

namespace tc {
constexpr int BM = 128;                       // samples per tile (UMMA M)
constexpr int BN = 256;                       // centroids per tile (UMMA N)
constexpr int BK = 32;                        // features per pipeline stage
constexpr int STAGES = 3;
constexpr int THREADS = 320;
constexpr int X_BYTES = BM * BK * 4;          // fp32 X tile, 128-byte swizzle
constexpr int A_BYTES = BM * BK * 2;          // one bf16 X part, 64-byte swizzle
constexpr int B_BYTES = BN * BK * 2;          // one bf16 C part, 64-byte swizzle
constexpr int STAGE_BYTES = X_BYTES + 2 * A_BYTES + 2 * B_BYTES;
constexpr int TX_BYTES = X_BYTES + 2 * B_BYTES;
constexpr int BAR_BYTES = 256;
constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + BAR_BYTES + 1024;  // + alignment slack
constexpr int ACC_COLS = BN;                  // f32 columns per accumulator
constexpr int TMEM_COLS = 2 * ACC_COLS;       // double-buffered
constexpr int GROUP_M = 16;                   // sample blocks per raster band
constexpr uint32_t SBO_64B = 8 * 64;          // 8 rows x 64 bytes per swizzle atom
static_assert(STAGE_BYTES % 1024 == 0, "stages stay 1 KiB aligned");
static_assert(SMEM_BYTES <= 232448, "fits the 227 KiB opt-in limit");
}  // namespace tc

struct TcParams {
    int n, k, d;
    int num_m, num_n, num_kb, num_tiles;
    const float *cnorm;
    float *xnorm;
    unsigned long long *keys;
    uint32_t *status;
};

__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int &mb, int &nb) {
    const int band = tile / (tc::GROUP_M * num_n);
    const int first = band * tc::GROUP_M;
    const int gs = min(tc::GROUP_M, num_m - first);
    const int r = tile - band * tc::GROUP_M * num_n;
    mb = first + r % gs;
    nb = r / gs;
}

__device__ __forceinline__ uint32_t bf162_bits(__nv_bfloat162 h) {
    return *reinterpret_cast<uint32_t *>(&h);
}

__global__ void __launch_bounds__(tc::THREADS, 1)
    assign_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmChi,
                     const __grid_constant__ CUtensorMap tmClo, const TcParams p) {
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_addr(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    const uint32_t sbase = smem_addr(smem);

    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + tc::STAGES * tc::STAGE_BYTES);
    // barrier slots: full[3] afull[3] empty[3] tfull[2] tempty[2] drain[1]
    auto bar = [&](int i) { return smem_addr(bars + i); };
    const int FULL = 0, AFULL = 3, EMPTY = 6, TFULL = 9, TEMPTY = 11, DRAIN = 13;
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(bars + 16);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < tc::STAGES; ++s) {
            mbar_init(bar(FULL + s), 1);
            mbar_init(bar(AFULL + s), 4);
            mbar_init(bar(EMPTY + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(bar(TFULL + a), 1);
            mbar_init(bar(TEMPTY + a), 4);
        }
        mbar_init(bar(DRAIN), 1);
        fence_barrier_init();
    }
    if (warp == 9) {
        tmem_alloc(smem_addr(tmem_holder), tc::TMEM_COLS);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_holder;

    if (warp < 4) {
        // ------------------------------------------------ split X into hi / lo
        const int t = threadIdx.x;  // 0..127
        const int c = t & 7;        // 16-byte chunk (4 floats) of a 128-byte fp32 row
        int it = 0;
        bool ok = true;
        for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
            int mb, nb;
            tile_coords(tile, p.num_m, p.num_n, mb, nb);
            float acc[8], comp[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[i] = comp[i] = 0.f;
            for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
                const int s = it % tc::STAGES;
                const uint32_t ph = (it / tc::STAGES) & 1;
                if (!mbar_wait_warp(bar(FULL + s), ph, p.status)) {
                    ok = false;
                    break;
                }
                const uint8_t *xs = smem + s * tc::STAGE_BYTES;
                uint8_t *ahi = smem + s * tc::STAGE_BYTES + tc::X_BYTES;
                uint8_t *alo = ahi + tc::A_BYTES;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int r = 16 * i + (t >> 3);
                    const float4 v =
                        *reinterpret_cast<const float4 *>(xs + r * 128 + ((c ^ (r & 7)) << 4));
                    const __nv_bfloat162 h01 = __floats2bfloat162_rn(v.x, v.y);
                    const __nv_bfloat162 h23 = __floats2bfloat162_rn(v.z, v.w);
                    const float2 f01 = __bfloat1622float2(h01);
                    const float2 f23 = __bfloat1622float2(h23);
                    const __nv_bfloat162 l01 = __floats2bfloat162_rn(v.x - f01.x, v.y - f01.y);
                    const __nv_bfloat162 l23 = __floats2bfloat162_rn(v.z - f23.x, v.w - f23.y);
                    const uint32_t off =
                        r * 64 + ((((c >> 1) ^ ((r >> 1) & 3)) << 4) | ((c & 1) << 3));
                    *reinterpret_cast<uint2 *>(ahi + off) = make_uint2(bf162_bits(h01), bf162_bits(h23));
                    *reinterpret_cast<uint2 *>(alo + off) = make_uint2(bf162_bits(l01), bf162_bits(l23));
                    float q = v.x * v.x;
                    q = fmaf(v.y, v.y, q);
                    q = fmaf(v.z, v.z, q);
                    q = fmaf(v.w, v.w, q);
                    const float y = q - comp[i];
                    const float tsum = acc[i] + y;
                    comp[i] = (tsum - acc[i]) - y;
                    acc[i] = tsum;
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(AFULL + s));
            }
            if (!ok) break;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                float v = acc[i] - comp[i];
                v += __shfl_xor_sync(0xffffffffu, v, 1);
                v += __shfl_xor_sync(0xffffffffu, v, 2);
                v += __shfl_xor_sync(0xffffffffu, v, 4);
                const int row = mb * tc::BM + 16 * i + (t >> 3);
                if (nb == 0 && c == 0 && row < p.n) p.xnorm[row] = v;
            }
        }
    } else if (warp < 8) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;  // tensor-memory lane quarter this warp may read
        int tile_iter = 0;
        for (int tile = blockIdx.x; tile < p.num_tiles; tile += gridDim.x, ++tile_iter) {
            int mb, nb;
            tile_coords(tile, p.num_m, p.num_n, mb, nb);
            const int a = tile_iter & 1;
            const uint32_t ph = (tile_iter >> 1) & 1;
            if (!mbar_wait_warp(bar(TFULL + a), ph, p.status)) break;
            tc_fence_after();
            const int n0 = nb * tc::BN;
            float best = __int_as_float(0x7f800000);  // +inf
            int arg = -1;
#pragma unroll 1
            for (int ch = 0; ch < tc::BN / 32; ++ch) {
                const int j0 = n0 + ch * 32;
                if (j0 >= p.k) break;
                float v[32];
                tmem_ld_32x32b_x32(tmem_base + (uint32_t)(a * tc::ACC_COLS + ch * 32) +
                                       ((uint32_t)(q * 32) << 16),
                                   v);
                const float4 *cn4 = reinterpret_cast<const float4 *>(p.cnorm + j0);
                if (j0 + 32 <= p.k) {
#pragma unroll
                    for (int u4 = 0; u4 < 8; ++u4) {
                        const float4 cn = __ldg(cn4 + u4);
                        const float s0 = fmaf(-2.f, v[4 * u4 + 0], cn.x);
                        const float s1 = fmaf(-2.f, v[4 * u4 + 1], cn.y);
                        const float s2 = fmaf(-2.f, v[4 * u4 + 2], cn.z);
                        const float s3 = fmaf(-2.f, v[4 * u4 + 3], cn.w);
                        if (s0 < best) { best = s0; arg = j0 + 4 * u4 + 0; }
                        if (s1 < best) { best = s1; arg = j0 + 4 * u4 + 1; }
                        if (s2 < best) { best = s2; arg = j0 + 4 * u4 + 2; }
                        if (s3 < best) { best = s3; arg = j0 + 4 * u4 + 3; }
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        if (j0 + u < p.k) {
                            const float s = fmaf(-2.f, v[u], __ldg(p.cnorm + j0 + u));
                            if (s < best) { best = s; arg = j0 + u; }
                        }
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(TEMPTY + a));
            const int row = mb * tc::BM + q * 32 + lane;
            if (row < p.n && arg >= 0) atomicMin(p.keys + row, make_key(best, (uint32_t)arg));
        }
    } else if (warp == 8) {
        // ------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tmX);
            tma_prefetch_desc(&tmChi);
            tma_prefetch_desc(&tmClo);
            int it = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x) {
                int mb, nb;
                tile_coords(tile, p.num_m, p.num_n, mb, nb);
                for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
                    const int s = it % tc::STAGES;
                    const uint32_t ph = (it / tc::STAGES) & 1;
                    if (!mbar_wait(bar(EMPTY + s), ph ^ 1, p.status)) {
                        ok = false;
                        break;
                    }
                    const uint32_t st = sbase + s * tc::STAGE_BYTES;
                    mbar_arrive_expect_tx(bar(FULL + s), tc::TX_BYTES);
                    tma_load_2d(st, &tmX, bar(FULL + s), kb * tc::BK, mb * tc::BM);
                    tma_load_2d(st + tc::X_BYTES + 2 * tc::A_BYTES, &tmChi, bar(FULL + s), kb * tc::BK,
                                nb * tc::BN);
                    tma_load_2d(st + tc::X_BYTES + 2 * tc::A_BYTES + tc::B_BYTES, &tmClo, bar(FULL + s),
                                kb * tc::BK, nb * tc::BN);
                }
            }
            if (!ok) {
                // let copies already in flight land before the CTA exits
                const int issued = it;
                for (int j = max(0, issued - tc::STAGES); j < issued; ++j)
                    mbar_wait_drain(bar(FULL + (j % tc::STAGES)), (j / tc::STAGES) & 1);
            }
        }
    } else {
        // ---------------------------------------------------------- MMA issue
        if (lane == 0) {
            constexpr uint32_t idesc = umma_idesc_bf16_f32(tc::BM, tc::BN);
            int it = 0, tile_iter = 0;
            bool ok = true;
            for (int tile = blockIdx.x; tile < p.num_tiles && ok; tile += gridDim.x, ++tile_iter) {
                const int a = tile_iter & 1;
                if (!mbar_wait(bar(TEMPTY + a), ((tile_iter >> 1) & 1) ^ 1, p.status)) break;
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(a * tc::ACC_COLS);
                for (int kb = 0; kb < p.num_kb; ++kb, ++it) {
                    const int s = it % tc::STAGES;
                    const uint32_t ph = (it / tc::STAGES) & 1;
                    if (!mbar_wait(bar(FULL + s), ph, p.status) || !mbar_wait(bar(AFULL + s), ph, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t ahi = sbase + s * tc::STAGE_BYTES + tc::X_BYTES;
                    const uint32_t alo = ahi + tc::A_BYTES;
                    const uint32_t bhi = alo + tc::A_BYTES;
                    const uint32_t blo = bhi + tc::B_BYTES;
#pragma unroll
                    for (int kk = 0; kk < tc::BK / 16; ++kk) {
                        const uint64_t dah = umma_smem_desc(ahi + kk * 32, tc::SBO_64B, kLayoutSW64);
                        const uint64_t dal = umma_smem_desc(alo + kk * 32, tc::SBO_64B, kLayoutSW64);
                        const uint64_t dbh = umma_smem_desc(bhi + kk * 32, tc::SBO_64B, kLayoutSW64);
                        const uint64_t dbl = umma_smem_desc(blo + kk * 32, tc::SBO_64B, kLayoutSW64);
                        mma_bf16_ss(d_tmem, dal, dbh, idesc, (kb | kk) != 0 ? 1u : 0u);
                        mma_bf16_ss(d_tmem, dah, dbl, idesc, 1u);
                        mma_bf16_ss(d_tmem, dah, dbh, idesc, 1u);
                    }
                    mma_commit(bar(EMPTY + s));
                }
                if (!ok) break;
                mma_commit(bar(TFULL + a));
            }
            // no MMA may still be writing tensor memory when it is released
            mma_commit(bar(DRAIN));
            mbar_wait_drain(bar(DRAIN), 0);
        }
    }

    __syncthreads();
    if (warp == 9) {
        tc_fence_after();
        tmem_dealloc(tmem_base, tc::TMEM_COLS);
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
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (cached[dev] == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = v > 0 ? v : 1;
    }
    return cached[dev];
}

int assign_tc_smem_bytes() { return tc::SMEM_BYTES; }

cudaError_t launch_assign_tc(const float *X, int64_t n, int64_t k, int64_t d, const AssignLayout &L,
                             uint8_t *ws, cudaStream_t stream) {
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(assign_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        tc::SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return attr_err;

    CUtensorMap tmX, tmChi, tmClo;
    const void *chi = ws + L.off_chi;
    const void *clo = ws + L.off_clo;
    if (!encode_2d(&tmX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, X, (uint64_t)d, (uint64_t)n, (uint64_t)d,
                   tc::BK, tc::BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tmChi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, chi, (uint64_t)L.d_pad, (uint64_t)k,
                   (uint64_t)L.d_pad, tc::BK, tc::BN, CU_TENSOR_MAP_SWIZZLE_64B) ||
        !encode_2d(&tmClo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, clo, (uint64_t)L.d_pad, (uint64_t)k,
                   (uint64_t)L.d_pad, tc::BK, tc::BN, CU_TENSOR_MAP_SWIZZLE_64B))
        return cudaErrorInvalidValue;

    TcParams p{};
    p.n = (int)n;
    p.k = (int)k;
    p.d = (int)d;
    p.num_m = (int)((n + tc::BM - 1) / tc::BM);
    p.num_n = (int)((k + tc::BN - 1) / tc::BN);
    p.num_kb = (int)((d + tc::BK - 1) / tc::BK);
    p.num_tiles = p.num_m * p.num_n;
    p.cnorm = reinterpret_cast<const float *>(ws + L.off_cnorm);
    p.xnorm = reinterpret_cast<float *>(ws + L.off_xnorm);
    p.keys = reinterpret_cast<unsigned long long *>(ws + L.off_keys);
    p.status = &reinterpret_cast<WsHeader *>(ws)->status;
    const int grid = p.num_tiles < device_sm_count() ? p.num_tiles : device_sm_count();
    assign_tc_kernel<<<grid, tc::THREADS, tc::SMEM_BYTES, stream>>>(tmX, tmChi, tmClo, p);
    return cudaGetLastError();
}

}  // namespace km

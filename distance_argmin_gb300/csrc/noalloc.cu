// kmeans_assign_noalloc: the tensor-core assignment for callers that cannot
// allocate device memory.
//
// Some callers of this library cannot call cudaMalloc at the point where they
// need an assignment: code running under an allocator that forbids new
// device allocations, plugins handed only the input and output buffers of a
// host framework, or real-time loops where an allocation (or the implicit
// synchronisation it may cause) is not allowed.  This entry point takes only
// the inputs and outputs; the scratch the assignment needs (per-sample keys,
// norms, the bf16 hi/lo copies of the centroids) lives in one file-scope
// device array of fixed size that the CUDA runtime creates when the library
// is loaded and keeps until the process exits.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "../../include/kmeans_gb300.h"
#include "assign_common.cuh"
#include "common.cuh"

namespace {

// Every GPU that loads this library holds this array until the process ends.
__device__ __align__(256) static unsigned char g_noalloc_scratch[KMEANS_NOALLOC_SCRATCH_BYTES];

using km::kMaxDevices;
std::mutex g_setup_mutex;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of the array on the current device, looked up once per
// device (host code only sees a host-side stand-in under the array's name).
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return KMEANS_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return KMEANS_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
    return KMEANS_OK;
}

}  // namespace

extern "C" int kmeans_assign_noalloc(const float *X, const float *C, int64_t n, int64_t k, int64_t d,
                                     int64_t *labels, float *best_dist, double *inertia, uint64_t seed,
                                     void *stream) {
    (void)seed;
    if (!X || !C || !labels || !best_dist) return KMEANS_ERR_INVALID_ARG;
    if (n < 1 || k < 1 || k > n || d < 1 || n > 0x7fffffffLL || k > 0x7fffffffLL || d > 0x7fffffffLL)
        return KMEANS_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(X) & 3u) || (reinterpret_cast<uintptr_t>(C) & 3u)) return KMEANS_ERR_INVALID_ARG;
    if (d % 4 != 0 || (reinterpret_cast<uintptr_t>(X) & 15u) || (reinterpret_cast<uintptr_t>(C) & 15u))
        return KMEANS_ERR_UNSUPPORTED;
    const km::AssignLayout L = km::assign_layout(n, k, d, true, 2, false);  // no K-split area in the scratch
    if ((uint64_t)L.bytes > (uint64_t)KMEANS_NOALLOC_SCRATCH_BYTES) return KMEANS_ERR_SCRATCH_LIMIT;
    void *scratch = nullptr;
    const int st = scratch_address(&scratch);
    if (st != KMEANS_OK) return st;
    uint8_t *ws = static_cast<uint8_t *>(scratch);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the prologue resets everything that must start fresh (status word,
    // reduction counter, per-sample keys); the rest is overwritten
    cudaError_t e = km::launch_prep_split(C, n, k, d, L, ws, s);
    if (e == cudaSuccess) e = km::launch_assign_tc(X, n, k, d, L, ws, s);
    if (e == cudaSuccess) e = km::launch_finalize(n, L, ws, labels, best_dist, inertia, s);
    return e == cudaSuccess ? KMEANS_OK : KMEANS_ERR_CUDA;
}

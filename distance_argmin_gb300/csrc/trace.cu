// Kernel timing for measurement tools (kmeans_trace_start / _read / _stop).
// Each traced kernel kind owns `capacity` pairs of CUDA events, created on the
// device that is current when tracing starts.  A launcher records the start
// event of the next free pair right before its kernel and the end event right
// after it, on the launch stream, so the pair times the kernel on the device
// (plus its launch latency there).  Launches beyond the capacity are counted
// but not timed.  Reading synchronises on the recorded end events only.
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "../../include/kmeans_gb300.h"
#include "trace.cuh"

namespace km {

std::atomic<int> g_trace_on{0};

namespace {

struct KindLog {
    std::vector<cudaEvent_t> start, end;
    int64_t timed = 0;     // pairs with both events recorded
    int64_t launched = 0;  // launches seen while tracing, timed or not
    bool open = false;     // a start event was recorded and its end is due
};

std::mutex g_mutex;
KindLog g_log[kTraceKinds];
int g_capacity = 0;

void destroy_all() {
    for (auto &lg : g_log) {
        for (cudaEvent_t e : lg.start) cudaEventDestroy(e);
        for (cudaEvent_t e : lg.end) cudaEventDestroy(e);
        lg = KindLog{};
    }
    g_capacity = 0;
}

}  // namespace

void trace_record(int kind, bool end, cudaStream_t s) {
    if (kind < 0 || kind >= kTraceKinds) return;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_trace_on.load(std::memory_order_relaxed)) return;
    KindLog &lg = g_log[kind];
    if (!end) {
        ++lg.launched;
        lg.open = false;
        if (lg.timed < g_capacity && cudaEventRecord(lg.start[lg.timed], s) == cudaSuccess) lg.open = true;
    } else if (lg.open) {
        if (cudaEventRecord(lg.end[lg.timed], s) == cudaSuccess) ++lg.timed;
        lg.open = false;
    }
}

}  // namespace km

using namespace km;

extern "C" int kmeans_trace_start(int capacity) {
    if (capacity < 1 || capacity > KMEANS_TRACE_MAX_CAPACITY) return KMEANS_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mutex);
    g_trace_on.store(0);
    destroy_all();
    for (auto &lg : g_log) {
        lg.start.resize(capacity);
        lg.end.resize(capacity);
        for (int i = 0; i < capacity; ++i) {
            if (cudaEventCreate(&lg.start[i]) != cudaSuccess || cudaEventCreate(&lg.end[i]) != cudaSuccess) {
                cudaGetLastError();
                lg.start.resize(i);
                lg.end.resize(i);
                destroy_all();
                return KMEANS_ERR_CUDA;
            }
        }
    }
    g_capacity = capacity;
    g_trace_on.store(1);
    return KMEANS_OK;
}

extern "C" int kmeans_trace_read(int kernel, double *ms_total, int64_t *timed_launches, int64_t *launches) {
    if (kernel < 0 || kernel >= kTraceKinds || !ms_total) return KMEANS_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_mutex);
    const KindLog &lg = g_log[kernel];
    double total = 0.0;
    for (int64_t i = 0; i < lg.timed; ++i) {
        float ms = 0.f;
        if (cudaEventSynchronize(lg.end[i]) != cudaSuccess ||
            cudaEventElapsedTime(&ms, lg.start[i], lg.end[i]) != cudaSuccess) {
            cudaGetLastError();
            return KMEANS_ERR_CUDA;
        }
        total += ms;
    }
    *ms_total = total;
    if (timed_launches) *timed_launches = lg.timed;
    if (launches) *launches = lg.launched;
    return KMEANS_OK;
}

extern "C" int kmeans_trace_stop(void) {
    std::lock_guard<std::mutex> lock(g_mutex);
    g_trace_on.store(0);
    for (auto &lg : g_log)
        for (int64_t i = 0; i < lg.timed; ++i) cudaEventSynchronize(lg.end[i]);
    destroy_all();
    return KMEANS_OK;
}

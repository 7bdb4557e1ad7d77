// Kernel timing for measurement tools: when tracing is on, the launchers
// bracket their dominant kernel with a pair of CUDA events on the launch
// stream (see kmeans_trace_start in the public header).
#pragma once

#include <cuda_runtime.h>

#include <atomic>

namespace km {

enum TraceKernel { kTraceAssignTc = 0, kTraceUpdateMean = 1, kTraceKppDist = 2, kTraceKinds = 3 };

extern std::atomic<int> g_trace_on;

void trace_record(int kind, bool end, cudaStream_t s);

// Cheap when tracing is off: one relaxed load.
inline void trace_mark(int kind, bool end, cudaStream_t s) {
    if (g_trace_on.load(std::memory_order_relaxed)) trace_record(kind, end, s);
}

}  // namespace km

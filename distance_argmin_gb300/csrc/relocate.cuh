// Empty-cluster relocation: device scratch layout and launcher.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"

namespace km {

// Scratch of one relocation: member counts and the list of empty clusters,
// placed at `base` inside a workspace.
struct RelocLayout {
    int64_t off_counts;  // k x i32
    int64_t off_empty;   // k x i32
    int64_t end;         // first byte after the scratch
};

inline RelocLayout reloc_layout(int64_t k, int64_t base) {
    RelocLayout R{};
    int64_t o = align_up(base, 256);
    R.off_counts = o; o = align_up(o + k * 4, 256);
    R.off_empty = o; o = align_up(o + k * 4, 256);
    R.end = o;
    return R;
}

// Rewrites the labels of the samples that move to empty clusters (the rule
// is stated in relocate.cu).  Leaves the labels as they are when a label
// outside [0, k) is found (flagged in the status word) or when the status
// word already holds a flag.
cudaError_t launch_relocate(int64_t *labels, const float *best, int64_t n, int64_t k, const RelocLayout &R,
                            uint8_t *ws, cudaStream_t s);

// *n_empty (device) = the number of zeros among counts[0 .. k).
cudaError_t launch_count_empty(const int32_t *counts, int64_t k, uint32_t *n_empty, cudaStream_t s);

}  // namespace km

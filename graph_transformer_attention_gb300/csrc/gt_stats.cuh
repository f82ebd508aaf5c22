// gt_stats.cuh -- per-kernel launch counts and, when turned on, CUDA-event
// timing of every kernel the library launches (gt_kernel_stats_* in the C ABI).
#pragma once

#include <cuda_runtime.h>

namespace gt {

// Counts one launch of `name` and, in timing mode, records a start event on
// `s`; returns a slot for stats_end (-1 when nothing is timed).
int stats_begin(const char* name, cudaStream_t s);
void stats_end(int slot, cudaStream_t s);

// Brackets the kernel launches of one scope: LaunchScope ls("fwd_tc", s); k<<<...>>>;
struct LaunchScope {
    int slot;
    cudaStream_t s;
    LaunchScope(const char* name, cudaStream_t st) : slot(stats_begin(name, st)), s(st) {}
    ~LaunchScope() { stats_end(slot, s); }
    LaunchScope(const LaunchScope&) = delete;
    LaunchScope& operator=(const LaunchScope&) = delete;
};

}  // namespace gt

// gt_selftest.cu -- a self-test of the bounded waits (gt_selftest_wait_timeout
// in the C ABI).
//
// Every mbarrier wait of the tensor-core kernels goes through mbar_wait, which
// gives up after a wall-clock limit, records the timeout in the device status
// word and lets the kernel return.  This kernel waits on a barrier that nothing
// ever arrives at, so the wait can only end by giving up: the next
// gt_check_device_status must report GT_ERR_TIMEOUT, and the context stays
// usable.  No fault, trap or unbounded loop is involved.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gt_common.cuh"
#include "gt_stats.cuh"
#include "gt_sm100.cuh"
#include "gt_tc_common.cuh"

namespace gt {
namespace {

__global__ void wait_selftest(int* status, uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        sm100::mbar_init(&bar, 1);
        sm100::fence_barrier_init();
        abort_flag = 0;
    }
    __syncthreads();
    if (threadIdx.x == 0 && !sm100::mbar_wait(&bar, 0, &abort_flag, limit_ns)) tc::fail(&abort_flag, status);
    __syncthreads();
}

}  // namespace
}  // namespace gt

extern "C" int gt_selftest_wait_timeout(int64_t limit_ns, void* stream) {
    if (limit_ns < 1000000 || limit_ns > 1000000000) return GT_ERR_INVALID_ARG;
    int* status = gt::device_status_ptr();
    if (!status) return GT_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
        gt::LaunchScope ls("selftest_wait", s);
        gt::wait_selftest<<<1, 32, 0, s>>>(status, (uint64_t)limit_ns);
    }
    return gt::check_launch();
}

// gt_noalloc.cu -- gt_bias_attn_bwd_noalloc: the backward pass for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or any allocator: code that runs inside a
// host framework owning all device memory, real-time or embedded callers that
// forbid allocation after start-up, and plain C hosts with no caching allocator
// at hand.  For them the backward pass can use a scratch array compiled into the
// library instead of a caller-provided workspace.
//
// The scratch is one file-scope __device__ array of GT_NOALLOC_SCRATCH_BYTES.
// Every GPU that loads the library holds it until the process exits.  In host
// code the array's name is only a stand-in, so its device address is looked up
// with cudaGetSymbolAddress once per device (with that device current) and then
// passed on as the workspace of the regular backward entry point.
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "gt_attn.h"
#include "gt_common.cuh"

static __device__ __align__(256) unsigned char g_noalloc_scratch[GT_NOALLOC_SCRATCH_BYTES];

namespace gt {
size_t bwd_ws_unsplit(int n, int h, int d);   // gt_abi.cu
}  // namespace gt

namespace {

// Device address of g_noalloc_scratch on the current device, looked up on the
// first call per device and cached.  Returns nullptr if the lookup fails.
void* noalloc_scratch_ptr() {
    static std::mutex mu;
    static void* ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        ptrs[dev] = p;
    }
    return ptrs[dev];
}

}  // namespace

extern "C" int gt_bias_attn_bwd_noalloc(int32_t dtype, int32_t n, int32_t h, int32_t d,
                                        const void* q, const void* k, const void* v,
                                        const void* o, const void* dO, const float* lse,
                                        const int8_t* spd, int64_t ld_spd, const float* T,
                                        int32_t nb, float scale, void* dq, void* dk, void* dv,
                                        float* dT, void* stream) {
    if (gt_bias_attn_workspace_size(dtype, n, h, d, 0) == 0) return GT_ERR_INVALID_ARG;
    // the backward run unsplit is what has to fit; with room to spare it splits
    if (gt::bwd_ws_unsplit(n, h, d) > (size_t)GT_NOALLOC_SCRATCH_BYTES) return GT_ERR_WORKSPACE;
    void* scratch = noalloc_scratch_ptr();
    if (!scratch) return GT_ERR_CUDA;
    return gt_bias_attn_bwd(dtype, n, h, d, q, k, v, o, dO, lse, spd, ld_spd, T, nb, scale, dq, dk,
                            dv, dT, scratch, (size_t)GT_NOALLOC_SCRATCH_BYTES, stream);
}

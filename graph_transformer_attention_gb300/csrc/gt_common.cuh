// gt_common.cuh -- shared host/device helpers of libgt (status codes, launch checks).
#pragma once

#include <utility>

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "gt_attn.h"

namespace gt {

// Device-side status word (one per process and device).  Kernels that give up
// a bounded wait OR a code into it and return; gt_check_device_status reads
// and clears it.
enum DeviceStatusBits : int {
    kStatusTimeout = 1,
};

// Device address of the status word of the current device (cached per device).
int* device_status_ptr();

inline int check_launch() {
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? GT_OK : GT_ERR_CUDA;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline int num_sms() {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    return sms > 0 ? sms : 1;
}

// Launches `kern` so that it may overlap the kernel before it in the stream
// (programmatic dependent launch): its CTAs can be scheduled once every CTA of
// that kernel has executed griddepcontrol.launch_dependents or exited, while
// that kernel still runs.  A kernel launched this way reads nothing the one
// before it writes, and ends with griddepcontrol.wait, so that it completes
// after it and the stream's later work sees both.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_overlapped(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                     cudaStream_t s, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Element access for the two storage types.
template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
    return __bfloat162float(x);
}
template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
    return __float2bfloat16_rn(x);
}

// Workspace carving: 256-byte aligned sub-buffers.
// Leading dimension (floats) of the backward's [16][ld] table of per-node
// lse log2 e and D values: rows padded to 16 bytes for the TMA.
inline int bwd_ld_ld(int n) { return (n + 3) & ~3; }

struct Carve {
    char* base;
    size_t off;
    size_t cap;
    __host__ explicit Carve(void* p, size_t c) : base(static_cast<char*>(p)), off(0), cap(c) {}
    template <typename T> __host__ T* take(size_t count) {
        off = (off + 255) & ~size_t(255);
        T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
        off += count * sizeof(T);
        return p;
    }
    __host__ bool fits() const { return off <= cap; }
};

}  // namespace gt

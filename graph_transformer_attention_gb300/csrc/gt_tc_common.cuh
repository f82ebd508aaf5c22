// gt_tc_common.cuh -- pieces shared by the tensor-core attention kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "gt_common.cuh"
#include "gt_sm100.cuh"

namespace gt {
namespace tc {

constexpr int kH = 8;                        // heads handled by the tensor-core kernels
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kWaitNs = 2000000000ull;  // bound of every mbarrier wait

// Record a timeout in the CTA's abort flag and the device status word.
__device__ __forceinline__ void fail(int* abort_flag, int* status) {
    *(volatile int*)abort_flag = 1;
    atomicOr(status, kStatusTimeout);
}

// Row r of NH per-head K-major [128][16] bf16 MMA operands (32-byte swizzle,
// 4096 bytes per head) for heads h_first .. h_first + NH - 1 of one node's
// [8][HD] row of x.  Head dim 8 is zero-padded to 16 per head so that products
// with the neighbouring head's channels vanish; head dim 16 is copied as is.
template <int HD, int NH = kH>
__device__ __forceinline__ void write_head_operands(uint8_t* base, int r, const __nv_bfloat16* src,
                                                    bool live, int h_first = 0) {
    const uint4* s = reinterpret_cast<const uint4*>(src);
    const uint32_t sw = (uint32_t)((r >> 2) & 1);
    const uint4 zero = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int h = 0; h < NH; ++h) {
        const int hg = h_first + h;
        uint4 lo, hi;
        if (HD == 8) {
            const uint4 v = live ? s[hg] : zero;
            lo = (hg & 1) ? zero : v;
            hi = (hg & 1) ? v : zero;
        } else {
            lo = live ? s[2 * hg] : zero;
            hi = live ? s[2 * hg + 1] : zero;
        }
        uint8_t* dst = base + h * 4096 + r * 32;
        *reinterpret_cast<uint4*>(dst + ((0u ^ sw) << 4)) = lo;
        *reinterpret_cast<uint4*>(dst + ((1u ^ sw) << 4)) = hi;
    }
}

// Bias table in shared memory: 256 rows (every byte code) of 8 fp32 head
// biases in base-2 units; codes >= nb get 0.
__device__ __forceinline__ void fill_bias_table(float* Ts, const float* T, int nb, int tid, int nthreads) {
    for (int x = tid; x < 256 * kH; x += nthreads) {
        const int code = x / kH, h = x % kH;
        Ts[x] = code < nb ? T[h * nb + code] * kLog2e : 0.f;
    }
}

// Bias table of NH heads h_first .. h_first + NH - 1: 256 rows (every byte
// code) of NH fp32 biases in base-2 units; codes >= nb get 0.
template <int NH>
__device__ __forceinline__ void fill_bias_table_heads(float* Ts, const float* T, int nb, int h_first,
                                                      int tid, int nthreads) {
    for (int x = tid; x < 256 * NH; x += nthreads) {
        const int code = x / NH, h = h_first + x % NH;
        Ts[x] = code < nb ? T[h * nb + code] * kLog2e : 0.f;
    }
}

__device__ __forceinline__ void red_shared_add_u32(uint32_t addr, uint32_t v) {
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

__device__ __forceinline__ void red_shared_add(uint32_t addr, float v) {
    asm volatile("red.shared.add.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

}  // namespace tc
}  // namespace gt

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

// Balanced split of a streamed loop over a fixed number of CTAs.  The work is
// `tasks` tasks of `nblk` steps each; CTA c takes the steps
// [c W / ctas, (c + 1) W / ctas) of their concatenation (W = tasks nblk).  With
// ctas >= tasks a share is at most nblk steps long, so it meets at most two
// tasks: the end of one and the start of the next.
struct Balance {
    int ctas;   // 0: no balancing (one CTA per task, from the grid)
    int tasks;
    int nblk;
    __host__ __device__ int64_t total() const { return (int64_t)tasks * nblk; }
    __host__ __device__ int64_t lo(int c) const { return (int64_t)c * total() / ctas; }
    // the share whose steps hold step p: the largest c with lo(c) <= p
    __host__ __device__ int cta_of(int64_t p) const {
        return (int)(((p + 1) * ctas + total() - 1) / total()) - 1;
    }
    // The share CTA b takes (ctas even): CTAs 2k and 2k + 1 take shares k and
    // k + ctas / 2, the same steps of the two halves.  The block scheduler hands
    // consecutive CTAs to different SMs, so the two CTAs that share an SM do not
    // run the same steps in lockstep.
    __host__ __device__ int share_of(int b) const { return (b & 1) * (ctas / 2) + (b >> 1); }
};

// The balanced grid for tasks = halves x tiles tasks of nblk steps each: a whole
// number of waves of per_sm CTAs per SM, at least one CTA per task (so a share
// meets at most two tasks) and at most one per min_steps steps, and an even
// count, so that the two halves split at a share boundary and shares c and
// c + ctas / 2 take the same steps of the two halves (with halves = 2).
// ctas = 0 when one CTA per task already fills its waves exactly.
inline Balance balance_grid(int tiles, int halves, int nblk, int per_sm, int min_steps) {
    const int tasks = halves * tiles;
    const int64_t slots = (int64_t)per_sm * num_sms();
    int64_t g = slots * ((tasks + slots - 1) / slots);
    const int64_t cap = (int64_t)tasks * nblk / min_steps;
    if (g > cap) g = cap;
    g &= ~int64_t(1);
    return Balance{g > tasks ? (int)g : 0, tasks, nblk};
}

// Steps [b0, b1) of task `task`: piece `which` (0 or 1) of share c;
// returns false when the share has no such piece.
struct Piece {
    int task, b0, b1;
};
__host__ __device__ inline bool piece_of(const Balance& bl, int c, int which, Piece& p) {
    const int64_t lo = bl.lo(c), hi = bl.lo(c + 1);
    const int t0 = (int)(lo / bl.nblk);
    const int64_t e0 = (int64_t)(t0 + 1) * bl.nblk;
    if (which == 0) {
        p.task = t0;
        p.b0 = (int)(lo - (int64_t)t0 * bl.nblk);
        p.b1 = (int)((hi < e0 ? hi : e0) - (int64_t)t0 * bl.nblk);
        return true;
    }
    if (hi <= e0) return false;
    p.task = t0 + 1;
    p.b0 = 0;
    p.b1 = (int)(hi - e0);
    return true;
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

// One TMEM row (lane) of the A operand of a per-head product with K = 16, for
// global head hg of a node's [8][HD] row src: the head's channels as bf16 pairs; head dim 8 sits in
// the half of the 16-column slot it shares with its neighbour head (the other
// half zero, so the neighbour's channels of the B operand drop out of the sum).
template <int HD>
__device__ __forceinline__ void head_a_row(const __nv_bfloat16* src, int hg, bool live, uint32_t (&a)[8]) {
    const uint4* s4 = reinterpret_cast<const uint4*>(src);
    if (HD == 16) {
        const uint4 lo = live ? s4[2 * hg] : make_uint4(0, 0, 0, 0);
        const uint4 hi = live ? s4[2 * hg + 1] : make_uint4(0, 0, 0, 0);
        a[0] = lo.x; a[1] = lo.y; a[2] = lo.z; a[3] = lo.w;
        a[4] = hi.x; a[5] = hi.y; a[6] = hi.z; a[7] = hi.w;
    } else {
        const uint4 v = live ? s4[hg] : make_uint4(0, 0, 0, 0);
        const bool odd = hg & 1;
        a[0] = odd ? 0u : v.x; a[1] = odd ? 0u : v.y; a[2] = odd ? 0u : v.z; a[3] = odd ? 0u : v.w;
        a[4] = odd ? v.x : 0u; a[5] = odd ? v.y : 0u; a[6] = odd ? v.z : 0u; a[7] = odd ? v.w : 0u;
    }
}

// Three bf16 parts (bits) of v whose fp32 sum is v to about 2^-24 relative:
// hi = bf16(v), mid = bf16(v - hi), lo = bf16(v - hi - mid); both differences
// are exact in fp32.
__device__ __forceinline__ void split3_bf16(float v, uint32_t& hi, uint32_t& mid, uint32_t& lo) {
    hi = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(v));
    const float r1 = v - __uint_as_float(hi << 16);
    mid = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(r1));
    lo = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(r1 - __uint_as_float(mid << 16)));
}

__device__ __forceinline__ void red_shared_add_u32(uint32_t addr, uint32_t v) {
    asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}

// dst[0..3] += (a, b, c, d), one 16-byte reduction (dst 16-byte aligned)
__device__ __forceinline__ void red_add_v4(float* dst, float a, float b, float c, float d) {
    asm volatile("red.global.v4.f32.add [%0], {%1, %2, %3, %4};" ::"l"(dst), "f"(a), "f"(b), "f"(c), "f"(d)
                 : "memory");
}

}  // namespace tc
}  // namespace gt

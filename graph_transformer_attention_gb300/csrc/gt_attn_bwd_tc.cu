// gt_attn_bwd_tc.cu -- tensor-core backward of topology-biased graph attention
// (bf16 storage, H = 8 heads, head dim 8 or 16) for sm_103a: the host side that
// launches the backward kernels.
//
// The backward pass recomputes P = exp(S - lse) blockwise, as the forward forms
// it (MegaGraph paper, Fig. 4: KV blocks stream past a Q tile, the bias column
// slice of each block comes from the int8 bucket matrix), and returns
//   dq = scale dS K,  dk = scale dS^T Q,  dv = P^T dO,  dT[h][c] = sum_{spd=c} dS,
// with dS = P (dO V^T - D) and D_i = <dO_i, o_i>.
//
// Kernels, in launch order:
//   bwd_prep    D_i per head, the table LD [16][ld] fp32 (row h holds lse_i log2 e
//               of head h, row 8 + h holds D_i; one column per node), the table LB
//               (bf16 [n][8][16]: per node and head -lse_i / scale and -D_i, each
//               as three bf16 parts whose sum is the fp32 value), and per head the
//               largest row norm of v (bounds the dT sums, see bwd_dq).
//   bwd_dq      (gt_attn_bwd_dq.cu) Q-stationary: dq and dT.
//   bwd_dkdv    (gt_attn_bwd_dkdv.cu) KV-stationary: dk and dv.
//   bwd_finish  the fp32 sums of split work to bf16 and the fp64 bucket sums
//               to the fp32 output, in one launch.
// Everything runs on the caller's stream, in this order.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "gt_common.cuh"
#include "gt_stats.cuh"
#include "gt_sm100.cuh"
#include "gt_tc_common.cuh"

namespace gt {
namespace {

using tc::kH;
using tc::kLog2e;
using tc::split3_bf16;
using sm100::pdl_trigger;
using sm100::pdl_wait;

constexpr int kMaxNb = 128;

// One thread per (node, head), node-major (x = 8 i + h), so a warp reads 32
// consecutive rows of HD bf16 of o, dO and v with 16-byte loads.
template <int HD>
__global__ void bwd_prep(int n, int ldl, float inv_scale, const __nv_bfloat16* __restrict__ o,
                         const __nv_bfloat16* __restrict__ dO, const __nv_bfloat16* __restrict__ v,
                         const float* __restrict__ lse, float* __restrict__ LD, uint16_t* __restrict__ LB,
                         float* __restrict__ Dv, float* __restrict__ vmax, float* __restrict__ acc, int dq_row0,
                         int kv_row0, double* __restrict__ dT64, int dT_count) {
    pdl_trigger();   // the dq kernel's prologue may run meanwhile; it waits for this grid before reading
    const int64_t total = (int64_t)n * kH;
    // clear what the backward sums into: the fp32 sums of split work (acc [3][n][8][HD]:
    // dq rows >= dq_row0, dk and dv rows >= kv_row0; negative = none) and the fp64
    // bucket sums; the dq kernel reads them only after this grid has completed
    {
        const int64_t stride = (int64_t)gridDim.x * blockDim.x;
        const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
        const int64_t row4 = kH * HD / 4, elems4 = (int64_t)n * row4;
        float4* a4 = reinterpret_cast<float4*>(acc);
        const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
        if (dq_row0 >= 0)
            for (int64_t x = dq_row0 * row4 + t0; x < elems4; x += stride) a4[x] = z;
        if (kv_row0 >= 0)
            for (int64_t x = kv_row0 * row4 + t0; x < elems4; x += stride) {
                a4[elems4 + x] = z;
                a4[2 * elems4 + x] = z;
            }
        for (int64_t x = t0; x < dT_count; x += stride) dT64[x] = 0.0;
    }
    // the loop bound is the same for the whole block, so every lane reaches the shuffles
    for (int64_t base = blockIdx.x * (int64_t)blockDim.x; base < total; base += (int64_t)gridDim.x * blockDim.x) {
        const int64_t x = base + threadIdx.x;
        const bool live = x < total;
        const int h = (int)(x & (kH - 1));
        const int64_t i = x / kH;
        float acc = 0.f, vn = 0.f;
        if (live) {
            const uint4* a = reinterpret_cast<const uint4*>(o + x * HD);
            const uint4* b = reinterpret_cast<const uint4*>(dO + x * HD);
            const uint4* c = reinterpret_cast<const uint4*>(v + x * HD);
#pragma unroll
            for (int q = 0; q < HD / 8; ++q) {
                const uint4 ua = a[q], ub = b[q], uc = c[q];
                const uint32_t wa[4] = {ua.x, ua.y, ua.z, ua.w}, wb[4] = {ub.x, ub.y, ub.z, ub.w},
                               wc[4] = {uc.x, uc.y, uc.z, uc.w};
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    acc = fmaf(__uint_as_float(wa[k] << 16), __uint_as_float(wb[k] << 16), acc);
                    acc = fmaf(__uint_as_float(wa[k] & 0xffff0000u), __uint_as_float(wb[k] & 0xffff0000u), acc);
                    vn = fmaf(__uint_as_float(wc[k] << 16), __uint_as_float(wc[k] << 16), vn);
                    vn = fmaf(__uint_as_float(wc[k] & 0xffff0000u), __uint_as_float(wc[k] & 0xffff0000u), vn);
                }
            }
        }
        // lanes l, l ^ 8, l ^ 16, l ^ 24 hold the same head (the warp's first x is a
        // multiple of 32); lanes 0..7 then add their head's maximum (non-negative
        // floats order like their bit patterns)
        float m = sqrtf(vn);
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
        if ((threadIdx.x & 31) < kH && m > 0.f) atomicMax(reinterpret_cast<int*>(vmax) + h, __float_as_int(m));
        if (live) {
            const float l = lse[(int64_t)h * n + i];
            LD[(int64_t)h * ldl + i] = l * kLog2e;
            LD[(int64_t)(kH + h) * ldl + i] = acc;
            Dv[(int64_t)h * n + i] = acc;
            uint32_t a0, a1, a2, b0, b1, b2;
            split3_bf16(-l * inv_scale, a0, a1, a2);
            split3_bf16(-acc, b0, b1, b2);
            uint4* dst = reinterpret_cast<uint4*>(LB + x * 16);
            dst[0] = make_uint4(a0 | (a1 << 16), a2 | (b0 << 16), b1 | (b2 << 16), 0u);
            dst[1] = make_uint4(0u, 0u, 0u, 0u);
        }
    }
}

__device__ __forceinline__ uint2 bf16x4(float4 v) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    return make_uint2(*reinterpret_cast<uint32_t*>(&lo), *reinterpret_cast<uint32_t*>(&hi));
}

// The backward's last step, one launch: the fp32 sums of split work to bf16 --
// dq rows dq_row0 .. n - 1 (dq_row0 < 0: none), dk and dv rows kv_row0 .. n - 1
// of the (KV tile, head half) groups >= kv_g1 (kv_row0 < 0: none); acc holds
// [3][n][8][HD] (dq, dk, dv) -- and the fp64 bucket sums dT64 to fp32.  Grid-
// stride over 4-value pieces.
template <int HD>
__global__ void bwd_finish(int n, const float* __restrict__ acc, int dq_row0, int kv_row0, int kv_g1,
                           __nv_bfloat16* __restrict__ dq, __nv_bfloat16* __restrict__ dk,
                           __nv_bfloat16* __restrict__ dv, int dT_count, const double* __restrict__ dT64,
                           float* __restrict__ dT) {
    pdl_wait();   // launched to overlap the dk/dv kernel's end: its sums are complete after this
    constexpr int kRow4 = kH * HD / 4;   // 4-value pieces per node
    const int64_t elems4 = (int64_t)n * kRow4;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    const int64_t t0 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const float4* a4 = reinterpret_cast<const float4*>(acc);
    if (dq_row0 >= 0)
        for (int64_t x = (int64_t)dq_row0 * kRow4 + t0; x < elems4; x += stride)
            reinterpret_cast<uint2*>(dq)[x] = bf16x4(a4[x]);
    if (kv_row0 >= 0)
        for (int64_t x = (int64_t)kv_row0 * kRow4 + t0; x < elems4; x += stride) {
            const int64_t row = x / kRow4;
            const int h = (int)((x % kRow4) / (HD / 4));
            if ((int)(row / 128) * 2 + h / 4 < kv_g1) continue;   // a whole group, written by its CTA
            reinterpret_cast<uint2*>(dk)[x] = bf16x4(a4[elems4 + x]);
            reinterpret_cast<uint2*>(dv)[x] = bf16x4(a4[2 * elems4 + x]);
        }
    for (int64_t x = t0; x < dT_count; x += stride) dT[x] = (float)dT64[x];
}

}  // namespace

bool bwd_tc_supported(int h, int d, int nb) { return h == kH && (d == 8 || d == 16) && nb <= kMaxNb; }

int launch_bwd_dq(int n, int d, const void* q, const void* k, const void* v, const void* dO,
                  const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                  const float* LD, int ldl, const float* vmax, int tail, void* dq, float* dq_acc,
                  double* dT64, cudaStream_t s);
int bwd_dq_tail_row0(int n, int tail, bool have_acc);
int bwd_dkdv_tail_row0(int n, int tail, bool have_acc);
int launch_bwd_dkdv(int n, int d, const void* q, const void* k, const void* v, const void* dO,
                    const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                    const uint16_t* LB, int tail, void* dk, void* dv, float* dk_acc, float* dv_acc,
                    cudaStream_t s);

// Backward on the tensor cores.  Workspace: LD [16][bwd_ld_ld(n)] fp32, LB bf16
// [n][8][16], Dv [8][n] fp32, dT64 [8][nb] fp64, aux [16] fp32 (aux[h]: largest |v_j|
// of head h), and the fp32 sums acc [3][n][8][d] when either split applies
// (tail > 1: the dk/dv groups past the last full wave split along their query
// tiles, or, on a graph whose groups do not fill one wave, dk/dv's equal shares of
// all its steps; dq_tail > 1: the dq tasks past the last full wave split along
// their KV blocks, all of them on a graph too small to fill a wave), else null.
int attn_bwd_tc(int n, int d, const void* q, const void* k, const void* v, const void* o,
                const void* dO, const float* lse, const int8_t* spd, int64_t ld, const float* T,
                int nb, float scale, void* dq, void* dk, void* dv, float* dT, float* LD, uint16_t* LB,
                float* Dv, double* dT64, float* aux, int tail, int dq_tail, float* acc,
                cudaStream_t s) {
    const int ldl = bwd_ld_ld(n);
    if (cudaMemsetAsync(aux, 0, sizeof(float) * 16, s) != cudaSuccess) return GT_ERR_CUDA;   // prep's maxima
    const int64_t total = (int64_t)n * kH;
    const int pblocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    // the dk/dv kernel takes -lse / scale; a zero scale (scores = bias alone) uses a
    // scale far below any product's resolution instead, with the same results
    const float fold_scale = (scale == 0.f || !isfinite(scale)) ? 1e-30f : scale;
    const size_t elems = (size_t)n * kH * d;
    // the fp32 sums (the split tasks' rows) and the bucket sums are cleared by the
    // prep kernel, so that nothing
    // stands between the launches (dq's prologue overlaps prep; the dk/dv kernel
    // may start on the SMs the dq kernel's last wave leaves free)
    const int dq_row0 = bwd_dq_tail_row0(n, dq_tail, acc != nullptr);
    const int kv_row0 = bwd_dkdv_tail_row0(n, tail, acc != nullptr);
    {
        LaunchScope ls("bwd_prep", s);
        auto prep = d == 8 ? bwd_prep<8> : bwd_prep<16>;
        prep<<<pblocks, 256, 0, s>>>(n, ldl, 1.f / fold_scale, static_cast<const __nv_bfloat16*>(o),
                                     static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(v),
                                     lse, LD, LB, Dv, aux, acc, acc ? dq_row0 : -1, acc ? kv_row0 : -1, dT64,
                                     (int)(kH * nb));
    }
    int rc = launch_bwd_dq(n, d, q, k, v, dO, spd, ld, T, nb, scale, LD, ldl, aux, acc ? dq_tail : 1, dq, acc,
                           dT64, s);
    if (rc != GT_OK) return rc;
    rc = launch_bwd_dkdv(n, d, q, k, v, dO, spd, ld, T, nb, scale, LB, acc ? tail : 1, dk, dv,
                         acc ? acc + elems : nullptr, acc ? acc + 2 * elems : nullptr, s);
    if (rc != GT_OK) return rc;
    {
        LaunchScope ls("bwd_finish", s);
        auto fin = d == 8 ? bwd_finish<8> : bwd_finish<16>;
        if (launch_overlapped(fin, dim3(2 * num_sms()), dim3(512), 0, s, n, (const float*)acc, acc ? dq_row0 : -1,
                              acc ? kv_row0 : -1, kv_row0 >= 0 ? kv_row0 / 128 * 2 : 0,
                              static_cast<__nv_bfloat16*>(dq), static_cast<__nv_bfloat16*>(dk),
                              static_cast<__nv_bfloat16*>(dv), (int)(kH * nb), (const double*)dT64, dT) != cudaSuccess)
            return GT_ERR_CUDA;
    }
    return check_launch();
}

}  // namespace gt

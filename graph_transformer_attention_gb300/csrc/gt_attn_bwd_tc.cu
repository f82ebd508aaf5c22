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
//               of head h, row 8 + h holds D_i; one column per node) and per head
//               the largest row norm of v (bounds the dT sums, see bwd_dq).
//   bwd_dq      (gt_attn_bwd_dq.cu) Q-stationary: dq and dT.
//   bwd_dkdv    (gt_attn_bwd_dkdv.cu) KV-stationary: dk and dv.
//   dT_to_f32   the fp64 bucket sums to the fp32 output.
// bwd_dq and bwd_dkdv read the same inputs and write different outputs; when
// the graph has few 128-row tiles, bwd_dkdv runs on a second stream beside
// bwd_dq (fork and join by events on the caller's stream), so that both kernels'
// CTAs fill the SMs at once.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "gt_common.cuh"
#include "gt_stats.cuh"
#include "gt_tc_common.cuh"

namespace gt {
namespace {

using tc::kH;
using tc::kLog2e;

constexpr int kMaxNb = 128;

// One thread per (node, head), node-major (x = 8 i + h), so a warp reads 32
// consecutive rows of HD bf16 of o, dO and v with 16-byte loads.
template <int HD>
__global__ void bwd_prep(int n, int ldl, const __nv_bfloat16* __restrict__ o,
                         const __nv_bfloat16* __restrict__ dO, const __nv_bfloat16* __restrict__ v,
                         const float* __restrict__ lse, float* __restrict__ LD, float* __restrict__ Dv,
                         float* __restrict__ vmax) {
    const int64_t total = (int64_t)n * kH;
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
            LD[(int64_t)h * ldl + i] = lse[(int64_t)h * n + i] * kLog2e;
            LD[(int64_t)(kH + h) * ldl + i] = acc;
            Dv[(int64_t)h * n + i] = acc;
        }
    }
}

// the split backward's fp32 sums [3][elems] (dq, dk, dv) to the bf16 outputs
__global__ void acc_to_bf16(size_t elems, const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                            __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv) {
    for (size_t x = blockIdx.x * (size_t)blockDim.x + threadIdx.x; x < elems; x += (size_t)gridDim.x * blockDim.x) {
        dq[x] = __float2bfloat16_rn(acc[x]);
        dk[x] = __float2bfloat16_rn(acc[elems + x]);
        dv[x] = __float2bfloat16_rn(acc[2 * elems + x]);
    }
}

__global__ void dT_to_f32(int count, const double* __restrict__ dT64, float* __restrict__ dT) {
    for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < count; x += gridDim.x * blockDim.x)
        dT[x] = (float)dT64[x];
}

// The second stream and the fork / join events of a device, created on first
// use (the only CUDA objects the backward keeps besides the launch statistics).
// side_mu is held while a call enqueues its fork and join, so that two host
// threads sharing the device never interleave their event records.
struct Side {
    cudaStream_t s2 = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr;
};

std::mutex side_mu;

bool side_for_device(Side* out) {
    static Side per[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    Side& sd = per[dev];
    if (!sd.join) {
        if (!sd.s2 && cudaStreamCreateWithFlags(&sd.s2, cudaStreamNonBlocking) != cudaSuccess) return false;
        if (!sd.fork && cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess) return false;
        if (cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess) return false;
    }
    *out = sd;
    return true;
}

}  // namespace

bool bwd_tc_supported(int h, int d, int nb) { return h == kH && (d == 8 || d == 16) && nb <= kMaxNb; }

int launch_bwd_dq(int n, int d, const void* q, const void* k, const void* v, const void* dO,
                  const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                  const float* LD, int ldl, const float* vmax, int nsplit, void* dq, float* dq_acc,
                  double* dT64, cudaStream_t s);
int launch_bwd_dkdv(int n, int d, const void* q, const void* k, const void* v, const void* dO,
                    const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                    const float* LD, int ldl, int nsplit, void* dk, void* dv, float* dk_acc, float* dv_acc,
                    cudaStream_t s);

// Backward on the tensor cores.  Workspace: LD [16][bwd_ld_ld(n)] fp32,
// Dv [8][n] fp32, dT64 [8][nb] fp64, aux [16] fp32 (aux[h]: largest |v_j| of head h).
int attn_bwd_tc(int n, int d, const void* q, const void* k, const void* v, const void* o,
                const void* dO, const float* lse, const int8_t* spd, int64_t ld, const float* T,
                int nb, float scale, void* dq, void* dk, void* dv, float* dT, float* LD, float* Dv,
                double* dT64, float* aux, int nsplit, float* acc, cudaStream_t s) {
    const int ldl = bwd_ld_ld(n);
    if (cudaMemsetAsync(dT64, 0, sizeof(double) * (size_t)kH * nb, s) != cudaSuccess) return GT_ERR_CUDA;
    if (cudaMemsetAsync(aux, 0, sizeof(float) * 16, s) != cudaSuccess) return GT_ERR_CUDA;
    const int64_t total = (int64_t)n * kH;
    const int pblocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    {
        LaunchScope ls("bwd_prep", s);
        auto prep = d == 8 ? bwd_prep<8> : bwd_prep<16>;
        prep<<<pblocks, 256, 0, s>>>(n, ldl, static_cast<const __nv_bfloat16*>(o),
                                     static_cast<const __nv_bfloat16*>(dO), static_cast<const __nv_bfloat16*>(v),
                                     lse, LD, Dv, aux);
    }
    // side by side only while the two kernels' CTAs (one per 128-row tile and
    // head half each) fit about one per SM: two co-resident CTAs of different
    // kernels slow each other more than two of the same kernel do (measured:
    // N = 16384 backward 2.41 ms in sequence, 2.68 ms side by side; N = 4096
    // 0.74 ms in sequence, 0.44 ms side by side)
    const int ctas = 2 * ((n + 127) / 128);
    const size_t elems = (size_t)n * kH * d;
    if (nsplit > 1 && acc) {
        // split streams: fp32 sums, then bf16
        if (cudaMemsetAsync(acc, 0, sizeof(float) * 3 * elems, s) != cudaSuccess) return GT_ERR_CUDA;
        int rc = launch_bwd_dq(n, d, q, k, v, dO, spd, ld, T, nb, scale, LD, ldl, aux, nsplit, dq, acc, dT64, s);
        if (rc != GT_OK) return rc;
        rc = launch_bwd_dkdv(n, d, q, k, v, dO, spd, ld, T, nb, scale, LD, ldl, nsplit, dk, dv, acc + elems,
                             acc + 2 * elems, s);
        if (rc != GT_OK) return rc;
        {
            LaunchScope ls("bwd_acc_to_bf16", s);
            acc_to_bf16<<<2 * num_sms(), 256, 0, s>>>(elems, acc, static_cast<__nv_bfloat16*>(dq),
                                                     static_cast<__nv_bfloat16*>(dk),
                                                     static_cast<__nv_bfloat16*>(dv));
        }
    } else if (2 * ctas > 3 * num_sms() / 2) {
        int rc = launch_bwd_dq(n, d, q, k, v, dO, spd, ld, T, nb, scale, LD, ldl, aux, 1, dq, nullptr, dT64, s);
        if (rc != GT_OK) return rc;
        rc = launch_bwd_dkdv(n, d, q, k, v, dO, spd, ld, T, nb, scale, LD, ldl, 1, dk, dv, nullptr, nullptr, s);
        if (rc != GT_OK) return rc;
    } else {
        std::lock_guard<std::mutex> lock(side_mu);
        Side sd;
        if (!side_for_device(&sd)) return GT_ERR_CUDA;
        if (cudaEventRecord(sd.fork, s) != cudaSuccess || cudaStreamWaitEvent(sd.s2, sd.fork, 0) != cudaSuccess)
            return GT_ERR_CUDA;
        const int rc = launch_bwd_dkdv(n, d, q, k, v, dO, spd, ld, T, nb, scale, LD, ldl, 1, dk, dv, nullptr,
                                       nullptr, sd.s2);
        const int rc2 = launch_bwd_dq(n, d, q, k, v, dO, spd, ld, T, nb, scale, LD, ldl, aux, 1, dq, nullptr, dT64,
                                      s);
        // join even when a launch failed, so the caller's stream never runs ahead
        if (cudaEventRecord(sd.join, sd.s2) != cudaSuccess || cudaStreamWaitEvent(s, sd.join, 0) != cudaSuccess)
            return GT_ERR_CUDA;
        if (rc != GT_OK) return rc;
        if (rc2 != GT_OK) return rc2;
    }
    {
        LaunchScope ls("bwd_dT_to_f32", s);
        dT_to_f32<<<1, 256, 0, s>>>(kH * nb, dT64, dT);
    }
    return check_launch();
}

}  // namespace gt

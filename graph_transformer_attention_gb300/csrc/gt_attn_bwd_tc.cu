// gt_attn_bwd_tc.cu -- tensor-core backward of topology-biased graph attention
// (bf16 storage, H = 8 heads, head dim 8 or 16) for sm_103a.
//
// The backward pass recomputes P = exp(S - lse) blockwise, as the forward forms
// it (MegaGraph paper, Fig. 4: KV blocks stream past a Q tile, the bias column
// slice of each block comes from the int8 bucket matrix), and returns
//   dq = scale dS K,  dk = scale dS^T Q,  dv = P^T dO,  dT[h][c] = sum_{spd=c} dS,
// with dS = P (dO V^T - D) and D_i = <dO_i, o_i>.
//
// Kernels:
//   bwd_prep    D_i per head, and the row table LD[i] = (lse_i log2 e, D_i) for
//               all 8 heads (64 bytes per node).
//   bwd_dq      (gt_attn_bwd_dq.cu) Q-stationary: dq and dT.
//   bwd_dkdv    KV-stationary: dk and dv (below).
//   dT_to_f32   the fp64 bucket sums to the fp32 output.
//
// All waits are bounded as in the forward kernel (timeout -> device status
// word, orderly exit, TMEM freed).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gt_common.cuh"
#include "gt_sm100.cuh"
#include "gt_tc_common.cuh"
#include "gt_tma.cuh"

namespace gt {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kCH = 16;
constexpr int kKVST = 2;
constexpr uint32_t kTmemCols = 512;
constexpr int kThreads = 192;
constexpr int kMaxNb = 128;

// ------------------------------------------------------------------ prep

template <typename TE>
__global__ void bwd_prep(int n, int hd, const TE* __restrict__ o, const TE* __restrict__ dO,
                         const float* __restrict__ lse, float* __restrict__ LD,
                         float* __restrict__ Dv) {
    const int64_t total = (int64_t)n * kH;
    for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(x / kH), h = (int)(x % kH);
        const TE* a = o + x * hd;
        const TE* b = dO + x * hd;
        float acc = 0.f;
        for (int c = 0; c < hd; ++c) acc = fmaf(to_f32(a[c]), to_f32(b[c]), acc);
        LD[(int64_t)i * 16 + h] = lse[(int64_t)h * n + i] * kLog2e;
        LD[(int64_t)i * 16 + 8 + h] = acc;
        Dv[(int64_t)h * n + i] = acc;
    }
}

__global__ void dT_to_f32(int count, const double* __restrict__ dT64, float* __restrict__ dT) {
    for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < count; x += gridDim.x * blockDim.x)
        dT[x] = (float)dT64[x];
}

// ------------------------------------------------------------- dk and dv
//
// KV-stationary: one CTA per 128 KV rows (thread r owns KV row r = TMEM lane r),
// all heads, streaming every Q tile.  Per chunk of 16 query rows i:
//   S^T_h = K_h Q_h^T and dP^T_h = V_h dO_h^T (M=128, N=16, K=16) into TMEM;
//   P^T = 2^(s log2e scale + b - lse_i log2e), dS^T = P^T (dP^T - D_i) in registers,
//   with lse_i, D_i of the 8 heads read from a 64-byte row of the LD table and the
//   bucket code of (i, j) from column j of the int8 tile;
//   P^T and dS^T (bf16) back to TMEM; dv_h += P^T_h dO_h, dk_h += dS^T_h Q_h.
// TMEM: dk at columns 0..127, dv at 128..255, and two 128-column regions whose
// roles alternate: S^T(t) in X, dP^T(t) in Y, then P^T/dS^T(t) over S^T(t) in X,
// S^T(t+1) into Y once dP^T(t) has been read, dP^T(t+1) into X after the dv/dk
// products of chunk t (the tensor pipe runs them in order).

template <int HD>
struct KvCfg {
    static constexpr int BQ = HD == 8 ? 128 : 64;       // query rows per TMA tile
    static constexpr int NCH = BQ / kCH;
    static constexpr int NSLOT = kH * HD / 16;
    static constexpr uint32_t OP_BYTES = kH * 128 * 32;
    static constexpr uint32_t SPD_BYTES = BQ * 128;      // [BQ i][128 j], no swizzle
    static constexpr uint32_t SLOT_BYTES = BQ * 32;
    static constexpr uint32_t LD_BYTES = BQ * 64;
    static constexpr uint32_t STAGE_BYTES = SPD_BYTES + 2 * NSLOT * SLOT_BYTES + LD_BYTES;
    static constexpr uint32_t OFF_K = 0;
    static constexpr uint32_t OFF_V = OP_BYTES;
    static constexpr uint32_t OFF_STAGE = 2 * OP_BYTES;
    static constexpr uint32_t OFF_T = OFF_STAGE + kKVST * STAGE_BYTES;
    static constexpr uint32_t OFF_BAR = OFF_T + 256 * kH * 4;
    static constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;
};

struct KvBars {
    uint64_t q_full[kKVST];
    uint64_t q_empty[kKVST];
    uint64_t s_full;
    uint64_t dp_full;
    uint64_t dp_free;
    uint64_t ds_ready;
    uint64_t done;
    uint64_t fin;
    uint32_t tmem_base;
    int abort;
};

constexpr uint32_t kColDk = 0;
constexpr uint32_t kColDv = 128;
__device__ __forceinline__ uint32_t kv_region(int t, bool x) {
    // X_t is region (t & 1), Y_t the other one
    const int r = x ? (t & 1) : ((t & 1) ^ 1);
    return 256u + 128u * r;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapG,
                const __grid_constant__ CUtensorMap mapS, const __grid_constant__ CUtensorMap mapL,
                const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                const float* __restrict__ T, int nb, int n, float scale, float scale_log2,
                __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int* status) {
    using C = KvCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    KvBars* bars = reinterpret_cast<KvBars*>(smem + C::OFF_BAR);
    float* Ts = reinterpret_cast<float*>(smem + C::OFF_T);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int j0 = blockIdx.x * 128;
    const int ntiles = (n + C::BQ - 1) / C::BQ;
    const int nchunks = ntiles * C::NCH;

    if (tid == kThreads - 32) {
        for (int s = 0; s < kKVST; ++s) {
            mbar_init(&bars->q_full[s], 1);
            mbar_init(&bars->q_empty[s], 128 + 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->dp_full, 1);
        mbar_init(&bars->dp_free, 128);
        mbar_init(&bars->ds_ready, 128);
        mbar_init(&bars->done, 1);
        mbar_init(&bars->fin, 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&mapQ);
        tma_prefetch_desc(&mapG);
        tma_prefetch_desc(&mapS);
        tma_prefetch_desc(&mapL);
    }
    if (warp == 4) tmem_alloc(&bars->tmem_base, kTmemCols);
    for (int x = tid; x < 256 * kH; x += kThreads) {
        const int code = x / kH, h = x % kH;
        Ts[x] = code < nb ? T[h * nb + code] * kLog2e : 0.f;
    }
    if (warp < 4) {
        const int row = j0 + tid;
        const bool live = row < n;
        const int64_t off = (int64_t)(live ? row : 0) * kH * HD;
        write_head_operands<HD>(smem + C::OFF_K, tid, k + off, live);
        write_head_operands<HD>(smem + C::OFF_V, tid, v + off, live);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bars->tmem_base;
    volatile int* abort_flag = &bars->abort;

    if (warp == 5) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int b = 0; b < ntiles; ++b) {
                const int ks = b & 1;
                if (b >= kKVST &&
                    !mbar_wait(&bars->q_empty[ks], ((b >> 1) - 1) & 1, abort_flag, kWaitNs)) {
                    fail(&bars->abort, status);
                    break;
                }
                uint8_t* st = smem + C::OFF_STAGE + ks * C::STAGE_BYTES;
                const int i0 = b * C::BQ;
                mbar_arrive_expect_tx(&bars->q_full[ks], C::STAGE_BYTES);
                tma_load_2d(st, &mapS, j0, i0, &bars->q_full[ks]);
#pragma unroll
                for (int s = 0; s < C::NSLOT; ++s) {
                    tma_load_2d(st + C::SPD_BYTES + s * C::SLOT_BYTES, &mapQ, 16 * s, i0,
                                &bars->q_full[ks]);
                    tma_load_2d(st + C::SPD_BYTES + (C::NSLOT + s) * C::SLOT_BYTES, &mapG, 16 * s,
                                i0, &bars->q_full[ks]);
                }
                tma_load_2d(st + C::SPD_BYTES + 2 * C::NSLOT * C::SLOT_BYTES, &mapL, 0, i0,
                            &bars->q_full[ks]);
                issued = b + 1;
            }
            if (*abort_flag) {
                int never = 0;
                for (int b = issued - kKVST; b < issued; ++b)
                    if (b >= 0) mbar_wait(&bars->q_full[b & 1], (b >> 1) & 1, &never, kWaitNs);
            }
        }
    } else if (warp == 4) {
        // ----------------------------------------------------------- MMA
        if (lane == 0) {
            const uint32_t idKK = idesc_bf16(128, 16, false, false);
            const uint32_t idKM = idesc_bf16(128, 16, false, true);
            const uint32_t k_base = smem_u32(smem + C::OFF_K);
            const uint32_t v_base = smem_u32(smem + C::OFF_V);
            const uint32_t stage_base = smem_u32(smem + C::OFF_STAGE);
            auto qslot = [&](int ks, int c, int h) -> uint32_t {
                return stage_base + ks * C::STAGE_BYTES + C::SPD_BYTES + (h * HD / 16) * C::SLOT_BYTES + c * 512;
            };
            auto gslot = [&](int ks, int c, int h) -> uint32_t {
                return qslot(ks, c, h) + C::NSLOT * C::SLOT_BYTES;
            };
            auto issue_s = [&](int tt) -> bool {
                const int b = tt / C::NCH, c = tt % C::NCH, ks = b & 1;
                if (c == 0 && !mbar_wait(&bars->q_full[ks], (b >> 1) & 1, abort_flag, kWaitNs))
                    return false;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < kH; ++h)
                    mma_ss(tbase + kv_region(tt, true) + 16 * h, smem_desc(k_base + h * 4096, 16, 256, 6),
                           smem_desc(qslot(ks, c, h), 16, 256, 6), idKK, 0);
                mma_commit(&bars->s_full);
                return true;
            };
            auto issue_dp = [&](int tt) {
                const int b = tt / C::NCH, c = tt % C::NCH, ks = b & 1;
#pragma unroll
                for (int h = 0; h < kH; ++h)
                    mma_ss(tbase + kv_region(tt, false) + 16 * h, smem_desc(v_base + h * 4096, 16, 256, 6),
                           smem_desc(gslot(ks, c, h), 16, 256, 6), idKK, 0);
                mma_commit(&bars->dp_full);
            };
            bool ok = issue_s(0);
            if (ok) issue_dp(0);
            for (int tt = 0; ok && tt < nchunks; ++tt) {
                const int b = tt / C::NCH, c = tt % C::NCH, ks = b & 1;
                if (!mbar_wait(&bars->dp_free, tt & 1, abort_flag, kWaitNs)) { ok = false; break; }
                if (tt + 1 < nchunks && !issue_s(tt + 1)) { ok = false; break; }
                if (!mbar_wait(&bars->ds_ready, tt & 1, abort_flag, kWaitNs)) { ok = false; break; }
                tc_fence_after();
                const uint32_t x = kv_region(tt, true);
#pragma unroll
                for (int h = 0; h < kH; ++h) {
                    const uint32_t acc = tt > 0 ? 1u : 0u;
                    mma_ts(tbase + kColDv + 16 * h, tbase + x + 16 * h,
                           smem_desc(gslot(ks, c, h), 256, 256, 6), idKM, acc);
                    mma_ts(tbase + kColDk + 16 * h, tbase + x + 16 * h + 8,
                           smem_desc(qslot(ks, c, h), 256, 256, 6), idKM, acc);
                }
                if (c == C::NCH - 1) mma_commit(&bars->q_empty[ks]);
                if (tt + 1 < nchunks) issue_dp(tt + 1);
            }
            if (ok) {
                mma_commit(&bars->done);
            } else {
                fail(&bars->abort, status);
                int never = 0;
                mma_commit(&bars->fin);
                mbar_wait(&bars->fin, 0, &never, kWaitNs);
            }
        }
    } else {
        // ------------------------------------------------------- softmax
        const int r = tid;
        const int row = j0 + r;
        const uint32_t lrow = tbase + ((uint32_t)(warp * 32) << 16);
        const float4* T4 = reinterpret_cast<const float4*>(Ts);
        int t = 0;
        bool ok = true;
        for (int b = 0; ok && b < ntiles; ++b) {
            const int ks = b & 1;
            if (!mbar_wait(&bars->q_full[ks], (b >> 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
            const uint8_t* st = smem + C::OFF_STAGE + ks * C::STAGE_BYTES;
            const float4* LD4 = reinterpret_cast<const float4*>(st + C::SPD_BYTES + 2 * C::NSLOT * C::SLOT_BYTES);
            for (int c = 0; c < C::NCH; ++c, ++t) {
                if (!mbar_wait(&bars->s_full, t & 1, abort_flag, kWaitNs)) { ok = false; break; }
                tc_fence_after();
                const uint32_t x = kv_region(t, true), y = kv_region(t, false);
                // bucket codes of the 16 (i, j) pairs of this chunk: column j = r of the tile
                uint32_t code[16];
#pragma unroll
                for (int kk = 0; kk < 16; ++kk) code[kk] = st[(c * kCH + kk) * 128 + r];
                // heads in two groups of four: S^T and dP^T of a group (16 columns each)
                // fit in registers, and one 16-byte bias / lse / D load serves the group
#pragma unroll
                for (int hg = 0; hg < 2; ++hg) {
                    uint32_t rs[4][16], rd[4][16];
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) tmem_ld_x16(lrow + x + 16 * (4 * hg + hh), rs[hh]);
                    tmem_wait_ld();
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk) {
                        const int il = c * kCH + kk;              // query row within the tile
                        const float4 b = T4[code[kk] * 2 + hg];
                        const float4 l = LD4[il * 4 + hg];
                        const float bias[4] = {b.x - l.x, b.y - l.y, b.z - l.z, b.w - l.w};
#pragma unroll
                        for (int hh = 0; hh < 4; ++hh)
                            rs[hh][kk] = __float_as_uint(
                                ex2(fmaf(__uint_as_float(rs[hh][kk]), scale_log2, bias[hh])));
                    }
                    if (hg == 0) {
                        if (!mbar_wait(&bars->dp_full, t & 1, abort_flag, kWaitNs)) ok = false;
                        tc_fence_after();
                    }
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) tmem_ld_x16(lrow + y + 16 * (4 * hg + hh), rd[hh]);
                    tmem_wait_ld();
                    if (hg == 1) {
                        tc_fence_before();
                        mbar_arrive(&bars->dp_free);
                    }
#pragma unroll
                    for (int kk = 0; kk < 16; ++kk) {
                        const int il = c * kCH + kk;
                        const float4 dd = LD4[il * 4 + 2 + hg];
                        const float Dd[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
                        for (int hh = 0; hh < 4; ++hh)
                            rd[hh][kk] = __float_as_uint(__uint_as_float(rs[hh][kk]) *
                                                         (__uint_as_float(rd[hh][kk]) - Dd[hh]));
                    }
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        uint32_t pp[8], pd[8];
#pragma unroll
                        for (int k2 = 0; k2 < 8; ++k2) {
                            pp[k2] = pack_bf16x2(__uint_as_float(rs[hh][2 * k2]),
                                                 __uint_as_float(rs[hh][2 * k2 + 1]));
                            pd[k2] = pack_bf16x2(__uint_as_float(rd[hh][2 * k2]),
                                                 __uint_as_float(rd[hh][2 * k2 + 1]));
                        }
                        tmem_st_x8(lrow + x + 16 * (4 * hg + hh), pp);
                        tmem_st_x8(lrow + x + 16 * (4 * hg + hh) + 8, pd);
                    }
                }
                tmem_wait_st();
                if (!ok) break;
                tc_fence_before();
                mbar_arrive(&bars->ds_ready);
            }
            if (!ok) break;
            mbar_arrive(&bars->q_empty[ks]);
        }
        if (!ok) {
            fail(&bars->abort, status);
        } else if (!mbar_wait(&bars->done, 0, abort_flag, kWaitNs)) {
            fail(&bars->abort, status);
        } else {
            tc_fence_after();
            const bool live = row < n;
#pragma unroll
            for (int h = 0; h < kH; ++h) {
                uint32_t ok16[16], ov16[16];
                tmem_ld_x16(lrow + kColDk + 16 * h, ok16);
                tmem_ld_x16(lrow + kColDv + 16 * h, ov16);
                tmem_wait_ld();
                const int c0h = (HD == 8) ? (h & 1) * 8 : 0;
                if (live) {
                    uint32_t wk[HD / 2], wv[HD / 2];
#pragma unroll
                    for (int q2 = 0; q2 < HD / 2; ++q2) {
                        wk[q2] = pack_bf16x2(__uint_as_float(ok16[c0h + 2 * q2]) * scale,
                                             __uint_as_float(ok16[c0h + 2 * q2 + 1]) * scale);
                        wv[q2] = pack_bf16x2(__uint_as_float(ov16[c0h + 2 * q2]),
                                             __uint_as_float(ov16[c0h + 2 * q2 + 1]));
                    }
                    uint4* dstk = reinterpret_cast<uint4*>(dk + ((int64_t)row * kH + h) * HD);
                    uint4* dstv = reinterpret_cast<uint4*>(dv + ((int64_t)row * kH + h) * HD);
#pragma unroll
                    for (int q2 = 0; q2 < HD / 8; ++q2) {
                        dstk[q2] = make_uint4(wk[4 * q2], wk[4 * q2 + 1], wk[4 * q2 + 2], wk[4 * q2 + 3]);
                        dstv[q2] = make_uint4(wv[4 * q2], wv[4 * q2 + 1], wv[4 * q2 + 2], wv[4 * q2 + 3]);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

template <int HD>
int launch_dkdv(int n, const void* q, const void* k, const void* v, const void* dO,
                const int8_t* spd, int64_t ld, const float* T, int nb, float scale, const float* LD,
                void* dk, void* dv, cudaStream_t s) {
    using C = KvCfg<HD>;
    CUtensorMap mq, mg, ms, ml;
    const uint64_t cols = (uint64_t)kH * HD;
    if (!make_map_2d(&mq, const_cast<void*>(q), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n, cols, cols * 2,
                     C::BQ, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_2d(&mg, const_cast<void*>(dO), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n, cols, cols * 2,
                     C::BQ, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_2d(&ms, const_cast<int8_t*>(spd), CU_TENSOR_MAP_DATA_TYPE_UINT8, n, n, ld, C::BQ,
                     128, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map_2d(&ml, const_cast<float*>(LD), CU_TENSOR_MAP_DATA_TYPE_FLOAT32, n, 16, 64, C::BQ,
                     16, CU_TENSOR_MAP_SWIZZLE_NONE))
        return GT_ERR_CUDA;
    if (cudaFuncSetAttribute(bwd_dkdv_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM) != cudaSuccess)
        return GT_ERR_CUDA;
    int* status = device_status_ptr();
    if (!status) return GT_ERR_CUDA;
    dim3 grid((n + 127) / 128);
    bwd_dkdv_kernel<HD><<<grid, kThreads, C::SMEM, s>>>(
        mq, mg, ms, ml, static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v),
        T, nb, n, scale, scale * kLog2e, static_cast<__nv_bfloat16*>(dk),
        static_cast<__nv_bfloat16*>(dv), status);
    return check_launch();
}

}  // namespace

bool bwd_tc_supported(int h, int d, int nb) { return h == kH && (d == 8 || d == 16) && nb <= kMaxNb; }

int launch_bwd_dq(int n, int d, const void* q, const void* k, const void* v, const void* dO,
                  const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                  const float* LD, void* dq, double* dT64, cudaStream_t s);

int attn_bwd_cols_simt(int dtype, int n, int h, int d, const void* q, const void* k, const void* v,
                       const void* dO, const float* lse, const float* Dv, const int8_t* spd,
                       int64_t ld, const float* T, int nb, float scale, void* dk, void* dv,
                       cudaStream_t s);

// Backward on the tensor cores.  ws: LD [n][16] fp32, Dv [8][n] fp32, dT64 [8][nb].
int attn_bwd_tc(int n, int d, const void* q, const void* k, const void* v, const void* o,
                const void* dO, const float* lse, const int8_t* spd, int64_t ld, const float* T,
                int nb, float scale, void* dq, void* dk, void* dv, float* dT, float* LD, float* Dv,
                double* dT64, cudaStream_t s) {
    if (cudaMemsetAsync(dT64, 0, sizeof(double) * (size_t)kH * nb, s) != cudaSuccess) return GT_ERR_CUDA;
    const int64_t total = (int64_t)n * kH;
    const int pblocks = (int)((total + 255) / 256 < 4096 ? (total + 255) / 256 : 4096);
    bwd_prep<__nv_bfloat16><<<pblocks, 256, 0, s>>>(n, d, static_cast<const __nv_bfloat16*>(o),
                                                    static_cast<const __nv_bfloat16*>(dO), lse, LD, Dv);
    int rc = launch_bwd_dq(n, d, q, k, v, dO, spd, ld, T, nb, scale, LD, dq, dT64, s);
    if (rc != GT_OK) return rc;
    rc = d == 8 ? launch_dkdv<8>(n, q, k, v, dO, spd, ld, T, nb, scale, LD, dk, dv, s)
                : launch_dkdv<16>(n, q, k, v, dO, spd, ld, T, nb, scale, LD, dk, dv, s);
    if (rc != GT_OK) return rc;
    dT_to_f32<<<1, 256, 0, s>>>(kH * nb, dT64, dT);
    return check_launch();
}

}  // namespace gt

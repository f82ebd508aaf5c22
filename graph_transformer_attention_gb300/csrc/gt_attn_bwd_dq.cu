// gt_attn_bwd_dq.cu -- tensor-core backward, Q-stationary part: dq and the
// bias-table gradient dT (bf16 storage, H = 8 heads, head dim 8 or 16).
//
// The backward recomputes P = exp(S - lse) blockwise, KV block by KV block with
// the matching bias slice of the int8 bucket matrix (MegaGraph, Fig. 4), and
//   dS = P (dO V^T - D),  dq = scale dS K,  dT[h][c] = sum over spd = c of dS.
//
// One CTA = one task: a tile of 128 query rows and one half of the heads (4 of
// 8); two CTAs share an SM, so one's softmax runs while the other waits on its
// tensor-core products.  Tasks past the last full wave of two CTAs per SM are
// split over several CTAs along the KV blocks (grid.z), which sum dq in fp32;
// so are all tasks of a graph too small to give every SM two.  192 threads:
//   warps 0-3  thread r owns query row r (TMEM lane r).  Per chunk of 16 KV
//              columns: S'_h and dP'_h from TMEM (lse and D already taken out by
//              the tensor core, below), one 16-byte shared load of the 4 head
//              biases per bucket byte, P = 2^(s' scale log2 e + b), dS = P dP',
//              dS (bf16) back to TMEM over S, and dS summed per
//              bucket: in registers while the row's 16 codes are equal, else with
//              shared-memory reductions into bins [code][head][NCP copies]; lane l
//              adds into copy l mod NCP, so with NCP = 32 the 32 rows of a warp never
//              meet on one address or bank, whatever their codes.  The bins hold
//              fixed-point integers (a 32-bit shared-memory add is a single native
//              operation, a float add is not): a row's dS values satisfy
//              sum_j |dS_ij| <= |dO_i| max_j |v_j| + |D_i| (the P_ij of a row sum to
//              1), so one power-of-two scale 2^e per CTA keeps every copy's sum below
//              2^30; the copies are summed exactly in 64 bits at the end.  The
//              scale is folded into the exponent (P 2^e = 2^(x - lse log2 e + e):
//              e is added to the bias table), so dS is formed in fixed-point units;
//              dq drops the 2^e at the end.
//   warp 4     MMA issuer: S_h = Q_h K_h^T and dP_h = dO_h V_h^T (M=128, N=16,
//              K=16), each followed by one product over all 4 heads (N = 64) that
//              adds -lse log2 e / (scale log2 e), resp. -D, per row and head: A
//              holds them as three bf16 parts per value (written by the prologue),
//              B selects each head's parts; then dq_h += dS_h K_h (A = dS from TMEM).
//   warp 5     TMA producer: bucket tile and K / V column slots per KV block.
// TMEM (256 columns): dq at 0..63 (16 per head), two S/dS stages at 64 and
// 128, dP at 192.  All waits are bounded (timeout -> device status word, orderly
// exit, TMEM freed).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "gt_common.cuh"
#include "gt_stats.cuh"
#include "gt_sm100.cuh"
#include "gt_tc_common.cuh"
#include "gt_tma.cuh"

namespace gt {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kBQ = 128;
constexpr int kCH = 16;
constexpr int kKVST = 2;
constexpr int kHC = 4;                     // heads per CTA
constexpr int kSoft = 128;
constexpr int kThreads = kSoft + 64;
constexpr int kMmaWarp = 4;
constexpr int kTmaWarp = 5;
constexpr uint32_t kTmemCols = 256;
constexpr uint32_t kColDq = 0;
constexpr uint32_t kColDp = 192;

__device__ __forceinline__ uint32_t s_col(int stage) { return 64u + 64u * stage; }

template <int HD>
struct DqCfg {
    static constexpr int BKV = 64;                     // KV rows per TMA block
    static constexpr int NCH = BKV / kCH;
    static constexpr int NSLOT = kHC * HD / 16;        // 16-column slots of this CTA's heads
    static constexpr uint32_t OP_BYTES = kHC * kBQ * 32;
    static constexpr uint32_t SPD_BYTES = kBQ * BKV;
    static constexpr uint32_t SLOT_BYTES = BKV * 32;
    static constexpr uint32_t STAGE_BYTES = SPD_BYTES + 2 * NSLOT * SLOT_BYTES;
    static constexpr uint32_t OFF_Q = 0;
    static constexpr uint32_t OFF_G = OP_BYTES;
    static constexpr uint32_t OFF_STAGE = 2 * OP_BYTES;
    static constexpr uint32_t OFF_T = OFF_STAGE + kKVST * STAGE_BYTES;   // bias table of the CTA's 4 heads
    // the fold operands: A_S and A_D [128 rows][16] (per head h, columns 4h .. 4h + 2
    // hold -(lse log2 e - e) / (scale log2 e), resp. -D, as three bf16 parts whose
    // sum is the fp32 value) and the B selector [64][16] that adds, to the 16 S (dP)
    // columns of head h, A's columns 4h .. 4h + 2
    static constexpr uint32_t OFF_FA = OFF_T + 256 * kHC * 4;
    static constexpr uint32_t OFF_FD = OFF_FA + kBQ * 32;
    static constexpr uint32_t OFF_FB = OFF_FD + kBQ * 32;
    static constexpr uint32_t OFF_BAR = OFF_FB + 64 * 32;
    static constexpr uint32_t OFF_BIN = OFF_BAR + 256;
    // bins: [nb][4 heads][ncp] int32 fixed point, sized at launch
    static constexpr uint32_t smem_bytes(int nb, int ncp) { return OFF_BIN + (uint32_t)nb * kHC * ncp * 4 + 1024; }
};
constexpr uint32_t kSmemLimit = 232448;      // one CTA per SM
constexpr uint32_t kSmemPair = 115712;       // two CTAs per SM

struct Bars {
    uint64_t kv_full[kKVST];
    uint64_t kv_empty[kKVST];
    uint64_t s_full[2];
    uint64_t ds_ready[2];
    uint64_t dq_done[2];
    uint64_t dp_full;
    uint64_t dp_free;
    uint64_t fin;
    uint32_t tmem_base;
    int abort;
};

// round(v) for a pair of floats with |v| < 2^29, on the FP32 and integer pipes
// instead of the conversion unit (which shares its throughput with ex2 and
// runs at half its rate).  v = a + b with a the nearest multiple of 512: the sum
// h = v + C1, C1 = 1.70703... * 2^32 (bits 0x4FDA7FFF), has a unit in the last
// place of 512, so h = C1 + a and its low mantissa bits hold a / 512; |b| <= 256.
// u = (C1 + C2) - h = C2 - a is exact (C2 = 2^23 + 512; C2 - a is a multiple of
// 512 below 2^30), and v + u rounds once, to C2 + round(b), whose low mantissa
// bits hold round(b).  So round(v) = a + round(b) = 512 (bits(h) - bits(C1)) +
// bits(v + u) - bits(C2), and C1, C2 are chosen so that 512 bits(C1) + bits(C2)
// = 0 mod 2^32: three packed adds and one shift-add per value.
__device__ __forceinline__ uint2 round_fixed2(float x, float y) {
    constexpr float kC1 = 7331642880.f;    // bits 0x4FDA7FFF
    constexpr float kC12 = 7340032000.f;   // kC1 + 2^23 + 512, exact
    const float2 v = make_float2(x, y);
    const float2 h = __fadd2_rn(v, make_float2(kC1, kC1));                          // C1 + a
    const float2 u = __fadd2_rn(make_float2(kC12, kC12), make_float2(-h.x, -h.y));  // C2 - a, exact
    const float2 b = __fadd2_rn(v, u);                                              // C2 + round(b)
    return make_uint2((__float_as_uint(h.x) << 9) + __float_as_uint(b.x),
                      (__float_as_uint(h.y) << 9) + __float_as_uint(b.y));
}

template <int HD, int NCP>
__global__ void __launch_bounds__(kThreads, 2)
bwd_dq_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
              const __grid_constant__ CUtensorMap mapS, const __nv_bfloat16* __restrict__ q,
              const __nv_bfloat16* __restrict__ dO, const float* __restrict__ LD, int ldl,
              const float* __restrict__ vmax,
              const float* __restrict__ T, int nb, int n, float scale, float scale_log2,
              int task_first, int split_blocks, __nv_bfloat16* __restrict__ dq, float* __restrict__ dq_acc,
              double* __restrict__ dT64, int after_prep, int* status) {
    using C = DqCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
    float* Ts = reinterpret_cast<float*>(smem + C::OFF_T);
    int* bins = reinterpret_cast<int*>(smem + C::OFF_BIN);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // after_prep: launched to overlap the prep kernel, whose tables (LD, vmax) it
    // may read only after griddepcontrol.wait (below, once the prologue has run on
    // the inputs alone); its dependents, which read those tables too, are let in
    // only then.  Otherwise the kernel before it wrote nothing it reads.
    if (!after_prep) pdl_trigger();   // the next kernel may take SMs as this one's free
    // task task_first + blockIdx.x: query tile task / 2, head half task % 2 (heads
    // 4 hb .. 4 hb + 3), so that the two halves of a tile, which read the same
    // bucket rows, run side by side
    const int task = task_first + (int)blockIdx.x;
    const int i0 = (task >> 1) * kBQ;
    const int hb = task & 1;
    // KV blocks kb0 .. kb0 + nblocks - 1 (all of them unless the columns are split
    // over grid.z, in which case dq is summed into dq_acc in fp32)
    const int total_blocks = (n + C::BKV - 1) / C::BKV;
    const int kb0 = split_blocks > 0 ? blockIdx.z * split_blocks : 0;
    const int nblocks = split_blocks > 0 ? min(split_blocks, total_blocks - kb0) : total_blocks;
    const int nchunks = nblocks * C::NCH;

    if (tid == kTmaWarp * 32) {
        for (int s = 0; s < kKVST; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], kSoft + 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bars->s_full[s], 1);
            mbar_init(&bars->ds_ready[s], kSoft);
            mbar_init(&bars->dq_done[s], 1);
        }
        mbar_init(&bars->dp_full, 1);
        mbar_init(&bars->dp_free, kSoft);
        mbar_init(&bars->fin, 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&mapK);
        tma_prefetch_desc(&mapV);
        tma_prefetch_desc(&mapS);
    }
    if (warp == kMmaWarp) tmem_alloc(&bars->tmem_base, kTmemCols);
    fill_bias_table_heads<kHC>(Ts, T, nb, kHC * hb, tid, kThreads);
    for (int x = tid; x < nb * kHC * NCP; x += kThreads) bins[x] = 0;
    // the fold's B selector: row m (column m of the 64 S or dP columns, head m / 16)
    // holds ones at columns 4 (m / 16) .. 4 (m / 16) + 2; 32-byte swizzle
    for (int m = tid; m < 64; m += kThreads) {
        uint32_t w[8];
#pragma unroll
        for (int k2 = 0; k2 < 8; ++k2)
            w[k2] = k2 == 2 * (m >> 4) ? 0x3F803F80u : k2 == 2 * (m >> 4) + 1 ? 0x00003F80u : 0u;   // bf16 1.0
        uint8_t* dst = smem + C::OFF_FB + m * 32;
        const uint32_t sw = (uint32_t)((m >> 2) & 1);
        *reinterpret_cast<uint4*>(dst + ((0u ^ sw) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(dst + ((1u ^ sw) << 4)) = make_uint4(w[4], w[5], w[6], w[7]);
    }
    if (tid < kBQ) {
        const int row = i0 + tid;
        const bool live = row < n;
        const int64_t off = (int64_t)(live ? row : 0) * kH * HD;
        write_head_operands<HD, kHC>(smem + C::OFF_Q, tid, q + off, live, kHC * hb);
        write_head_operands<HD, kHC>(smem + C::OFF_G, tid, dO + off, live, kHC * hb);
    }
    if (after_prep) pdl_wait();
    // this row's lse log2 e and D per head go into the fold operands, so that the
    // tensor core forms s - lse log2 e / (scale log2 e) and dP - D
    float L2[4] = {0.f, 0.f, 0.f, 0.f}, Dh[4] = {0.f, 0.f, 0.f, 0.f};
    if (tid < kBQ) {
        const int row = i0 + tid;
        const bool live = row < n;
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
            L2[hh] = live ? LD[(int64_t)(kHC * hb + hh) * ldl + row] : 0.f;
            Dh[hh] = live ? LD[(int64_t)(kH + kHC * hb + hh) * ldl + row] : 0.f;
        }
        // each value as three bf16 parts (the value, then what each part leaves:
        // 8 + 8 + 8 bits, so the parts sum to the fp32 value)
        const float inv_c = 1.f / scale_log2;
        uint32_t wa[8], wd[8];
        auto parts = [](float v, uint32_t& w01, uint32_t& w2) {
            const float p1 = __bfloat162float(__float2bfloat16_rn(v));
            const float r1 = v - p1;
            const float p2 = __bfloat162float(__float2bfloat16_rn(r1));
            w01 = pack_bf16x2(p1, p2);
            w2 = pack_bf16x2(r1 - p2, 0.f);
        };
#pragma unroll
        for (int hh = 0; hh < 4; ++hh) {
            parts(-L2[hh] * inv_c, wa[2 * hh], wa[2 * hh + 1]);
            parts(-Dh[hh], wd[2 * hh], wd[2 * hh + 1]);
        }
        const uint32_t sw = (uint32_t)((tid >> 2) & 1);
        uint8_t* da = smem + C::OFF_FA + tid * 32;
        uint8_t* dd = smem + C::OFF_FD + tid * 32;
        *reinterpret_cast<uint4*>(da + ((0u ^ sw) << 4)) = make_uint4(wa[0], wa[1], wa[2], wa[3]);
        *reinterpret_cast<uint4*>(da + ((1u ^ sw) << 4)) = make_uint4(wa[4], wa[5], wa[6], wa[7]);
        *reinterpret_cast<uint4*>(dd + ((0u ^ sw) << 4)) = make_uint4(wd[0], wd[1], wd[2], wd[3]);
        *reinterpret_cast<uint4*>(dd + ((1u ^ sw) << 4)) = make_uint4(wd[4], wd[5], wd[6], wd[7]);
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (after_prep) pdl_trigger();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bars->tmem_base;
    int* abort_flag = &bars->abort;

    if (warp == kTmaWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int b = 0; b < nblocks; ++b) {
                const int ks = b & 1;
                if (b >= kKVST &&
                    !mbar_wait(&bars->kv_empty[ks], ((b >> 1) - 1) & 1, abort_flag, kWaitNs)) {
                    fail(abort_flag, status);
                    break;
                }
                uint8_t* st = smem + C::OFF_STAGE + ks * C::STAGE_BYTES;
                const int j0 = (kb0 + b) * C::BKV;
                mbar_arrive_expect_tx(&bars->kv_full[ks], C::STAGE_BYTES);
                tma_load_2d(st, &mapS, j0, i0, &bars->kv_full[ks]);
#pragma unroll
                for (int s = 0; s < C::NSLOT; ++s) {
                    tma_load_2d(st + C::SPD_BYTES + s * C::SLOT_BYTES, &mapK, 16 * (hb * C::NSLOT + s),
                                j0, &bars->kv_full[ks]);
                    tma_load_2d(st + C::SPD_BYTES + (C::NSLOT + s) * C::SLOT_BYTES, &mapV,
                                16 * (hb * C::NSLOT + s), j0, &bars->kv_full[ks]);
                }
                issued = b + 1;
            }
            if (*(volatile int*)abort_flag) {
                int never = 0;
                for (int b = issued - kKVST; b < issued; ++b)
                    if (b >= 0) mbar_wait(&bars->kv_full[b & 1], (b >> 1) & 1, &never, kWaitNs);
            }
        }
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------- MMA
        // The whole warp runs the loop and waits; the elected lane issues (an MMA
        // from a converged warp through elect.sync costs a fraction of one from a
        // lane-0 branch), and descriptors are precomputed so that an MMA costs one add.
        {
            const uint32_t idKK = idesc_bf16(128, 16, false, false);
            const uint32_t idKM = idesc_bf16(128, 16, false, true);
            const uint32_t idFold = idesc_bf16(128, 64, false, false);   // the 4 heads' 64 columns at once
            const uint64_t dFA = desc_at(smem_desc_split(smem_u32(smem + C::OFF_FA), 16, 256, 6), 0);
            const uint64_t dFD = desc_at(smem_desc_split(smem_u32(smem + C::OFF_FD), 16, 256, 6), 0);
            const uint64_t dFB = desc_at(smem_desc_split(smem_u32(smem + C::OFF_FB), 16, 256, 6), 0);
            const uint32_t stage_base = smem_u32(smem + C::OFF_STAGE);
            const SmemDesc dQ = smem_desc_split(smem_u32(smem + C::OFF_Q), 16, 256, 6);
            const SmemDesc dG = smem_desc_split(smem_u32(smem + C::OFF_G), 16, 256, 6);
            const SmemDesc dKk = smem_desc_split(stage_base + C::SPD_BYTES, 16, 256, 6);    // K-major K, V
            const SmemDesc dKm = smem_desc_split(stage_base + C::SPD_BYTES, 256, 256, 6);   // MN-major K
            constexpr uint32_t kVoff = C::NSLOT * C::SLOT_BYTES;                             // V after K
            auto koff = [&](int tt, int h) -> uint32_t {
                const int b = tt / C::NCH, c = tt % C::NCH;
                return (uint32_t)((b & 1) * C::STAGE_BYTES + (h * HD / 16) * C::SLOT_BYTES + c * 512);
            };
            auto issue_s = [&](int tt) -> bool {
                const int b = tt / C::NCH, c = tt % C::NCH, ks = b & 1, ss = tt & 1;
                if (c == 0 && !mbar_wait_all(&bars->kv_full[ks], (b >> 1) & 1, abort_flag, kWaitNs))
                    return false;
                // stage ss last held dS(tt - 2): the dq products that read it were issued
                // before this point and the tensor pipe runs one thread's MMAs in order,
                // so no wait is needed before overwriting it
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int h = 0; h < kHC; ++h)
                        mma_ss(tbase + s_col(ss) + 16 * h, desc_at(dQ, h * 4096), desc_at(dKk, koff(tt, h)), idKK, 0);
                    mma_ss(tbase + s_col(ss), dFA, dFB, idFold, 1);       // - (lse log2 e - e) / (scale log2 e)
                    mma_commit(&bars->s_full[ss]);
                }
                __syncwarp();
                return true;
            };
            auto issue_dp = [&](int tt) {
                if (elect_one()) {
#pragma unroll
                    for (int h = 0; h < kHC; ++h)
                        mma_ss(tbase + kColDp + 16 * h, desc_at(dG, h * 4096), desc_at(dKk, koff(tt, h) + kVoff),
                               idKK, 0);
                    mma_ss(tbase + kColDp, dFD, dFB, idFold, 1);          // - D
                    mma_commit(&bars->dp_full);
                }
                __syncwarp();
            };
            bool ok = issue_s(0);
            if (ok) issue_dp(0);
            for (int tt = 0; ok && tt < nchunks; ++tt) {
                const int b = tt / C::NCH, c = tt % C::NCH, ks = b & 1, ss = tt & 1;
                if (tt + 1 < nchunks) {
                    if (!issue_s(tt + 1)) { ok = false; break; }
                    if (!mbar_wait_all(&bars->dp_free, tt & 1, abort_flag, kWaitNs)) { ok = false; break; }
                    tc_fence_after();
                    issue_dp(tt + 1);
                }
                if (!mbar_wait_all(&bars->ds_ready[ss], (tt >> 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int h = 0; h < kHC; ++h)
                        mma_ts(tbase + kColDq + 16 * h, tbase + s_col(ss) + 16 * h, desc_at(dKm, koff(tt, h)), idKM,
                               tt > 0 ? 1u : 0u);
                    mma_commit(&bars->dq_done[ss]);
                    if (c == C::NCH - 1) mma_commit(&bars->kv_empty[ks]);
                }
                __syncwarp();
            }
            if (!ok) {
                fail(abort_flag, status);
                int never = 0;
                if (elect_one()) mma_commit(&bars->fin);
                __syncwarp();
                mbar_wait_all(&bars->fin, 0, &never, kWaitNs);
            }
        }
    } else {
        // ------------------------------------------------------- softmax
        const int r = tid & (kBQ - 1);
        const int row = i0 + r;
        const bool live = row < n;
        const uint32_t lrow = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t tbl = smem_u32(Ts);     // 16-byte rows: the CTA's 4 head biases of a code
        // bin address: binb + code * kCodeStride + hh * kHeadStride
        constexpr uint32_t kHeadStride = 4u * NCP, kCodeStride = kHC * kHeadStride;
        const uint32_t binb = smem_u32(bins) + 4u * (uint32_t)(lane & (NCP - 1));
        // fixed-point scale of the dT bins: 2^e with (rows per copy) * max_i B_i * 2^e
        // <= 2^30, B_i = |dO_i| max_j |v_j| + |D_i| bounding sum_j |dS_ij| (per head).
        // The scale rides in the exponent (P 2^e = 2^(x - lse log2 e + e)): e is
        // added to every entry of the bias table, so dS comes out in fixed-point
        // units (and dq carries 2^e, taken out in the epilogue)
        float bscale;
        {
            float bmax = 0.f;
            if (live) {
                const uint4* src = reinterpret_cast<const uint4*>(dO + ((int64_t)row * kH + kHC * hb) * HD);
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    float nn = 0.f;
#pragma unroll
                    for (int q8 = 0; q8 < HD / 8; ++q8) {
                        const uint4 u = src[hh * (HD / 8) + q8];
                        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const float lo = __uint_as_float(wv[k] << 16), hi = __uint_as_float(wv[k] & 0xffff0000u);
                            nn = fmaf(lo, lo, fmaf(hi, hi, nn));
                        }
                    }
                    bmax = fmaxf(bmax, sqrtf(nn) * vmax[kHC * hb + hh] + fabsf(Dh[hh]));
                }
            }
            for (int o = 16; o > 0; o >>= 1) bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, o));
            float* red = reinterpret_cast<float*>(smem + C::OFF_BAR + sizeof(Bars));
            if (lane == 0) red[warp] = bmax;
            asm volatile("bar.sync 1, %0;" ::"n"(kSoft) : "memory");
            bmax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
            const float bound = bmax * (float)(kBQ / NCP);
            int e = 60;
            if (bound > 0.f) e = (int)floorf(log2f(1073741824.f / bound));
            if (!(bound < INFINITY) || e < 0) e = 0;
            if (e > 60) e = 60;
            bscale = exp2f((float)e);
            for (int x = tid; x < 256 * kHC; x += kSoft) Ts[x] += (float)e;
            asm volatile("bar.sync 1, %0;" ::"n"(kSoft) : "memory");
        }
        auto fx = [&](float v) -> uint32_t { return (uint32_t)__float2int_rn(v); };
        const float qscale = scale / bscale;
        // a uniform row's dS sums per head, kept as column pairs until the bin is flushed
        float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        int acc_code = -1;
        int t = 0;
        bool ok = true;
        for (int b = 0; ok && b < nblocks; ++b) {
            const int ks = b & 1;
            if (!mbar_wait(&bars->kv_full[ks], (b >> 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
            const uint32_t sp = smem_u32(smem + C::OFF_STAGE + ks * C::STAGE_BYTES) + r * C::BKV;
            const int j0 = (kb0 + b) * C::BKV;
            const bool tail_block = j0 + C::BKV > n;
            for (int c = 0; c < C::NCH; ++c, ++t) {
                const int ss = t & 1;
                if (!mbar_wait(&bars->s_full[ss], (t >> 1) & 1, abort_flag, kWaitNs) ||
                    !mbar_wait(&bars->dp_full, t & 1, abort_flag, kWaitNs)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t phys = C::BKV == 128 ? (uint32_t)(c ^ (r & 7)) : (uint32_t)(c ^ ((r >> 1) & 3));
                const uint4 cv = lds_u4(sp + (phys << 4));
                const uint32_t w[4] = {cv.x, cv.y, cv.z, cv.w};
                const uint32_t c0 = w[0] & 0xffu;
                const bool uniform = w[0] == c0 * 0x01010101u && w[1] == w[0] && w[2] == w[0] && w[3] == w[0];
                const bool wuni = __all_sync(0xffffffffu, uniform);
                if (uniform && (int)c0 != acc_code) {
                    if (acc_code >= 0 && acc_code < nb) {
#pragma unroll
                        for (int hh = 0; hh < 4; ++hh)
                            red_shared_add_u32(binb + acc_code * kCodeStride + hh * kHeadStride, fx(acc[hh].x + acc[hh].y));
                    }
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) acc[hh] = make_float2(0.f, 0.f);
                    acc_code = (int)c0;
                }
                const int jc = j0 + c * kCH;
                // One half chunk (8 columns).  The tensor core has already taken lse
                // log2 e (less the bins' e) out of S, in units of scale log2 e, and D out
                // of dP (the fold operand), so x - lse log2 e = s scale log2 e + b and dS =
                // P dP.  FAST: every row of the warp holds one code over the chunk (the
                // vote above), so a row takes its 4 head biases once, forms x with one
                // packed FMA per two columns and keeps its dS sums in registers; no row
                // needs the per-element bins.  Otherwise each
                // column takes its own code's biases, and rows with mixed codes add every
                // dS to the shared bins.  The two are separate code, so the uniform chunks
                // that dominate a graph of components run without the mixed path's branches.
                auto half = [&](int g, auto fast_tag) {
                    constexpr bool FAST = decltype(fast_tag)::value;
                    uint32_t rs[4][8], rd[4][8];
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        tmem_ld_x8(lrow + s_col(ss) + 16 * hh + 8 * g, rs[hh]);
                        tmem_ld_x8(lrow + kColDp + 16 * hh + 8 * g, rd[hh]);
                    }
                    tmem_wait_ld();
                    if (g == 1) {
                        tc_fence_before();
                        mbar_arrive(&bars->dp_free);
                    }
                    if constexpr (FAST) {
                        const float4 bv = lds_f4(tbl + c0 * 16u);
                        const float bb[4] = {bv.x, bv.y, bv.z, bv.w};
#pragma unroll
                        for (int hh = 0; hh < 4; ++hh) {
                            const float2 bl = make_float2(bb[hh], bb[hh]);
#pragma unroll
                            for (int k = 0; k < 8; k += 2) {
                                const float2 x = __ffma2_rn(
                                    make_float2(__uint_as_float(rs[hh][k]), __uint_as_float(rs[hh][k + 1])),
                                    make_float2(scale_log2, scale_log2), bl);
                                rs[hh][k] = __float_as_uint(x.x);
                                rs[hh][k + 1] = __float_as_uint(x.y);
                            }
                        }
                    } else {
                        // x = s scale log2 e + bias (scalar FMA), each column its own code
#pragma unroll
                        for (int k = 0; k < 8; ++k) {
                            const int kk = 8 * g + k;
                            const uint32_t code = __byte_perm(w[kk >> 2], 0u, 0x4440u + (kk & 3));
                            const float4 bv = lds_f4(tbl + code * 16u);
                            rs[0][k] = __float_as_uint(fmaf(__uint_as_float(rs[0][k]), scale_log2, bv.x));
                            rs[1][k] = __float_as_uint(fmaf(__uint_as_float(rs[1][k]), scale_log2, bv.y));
                            rs[2][k] = __float_as_uint(fmaf(__uint_as_float(rs[2][k]), scale_log2, bv.z));
                            rs[3][k] = __float_as_uint(fmaf(__uint_as_float(rs[3][k]), scale_log2, bv.w));
                        }
                    }
                    if (tail_block) {
#pragma unroll
                        for (int k = 0; k < 8; ++k)
                            if (jc + 8 * g + k >= n) {
#pragma unroll
                                for (int hh = 0; hh < 4; ++hh) rs[hh][k] = __float_as_uint(-INFINITY);
                            }
                    }
#pragma unroll
                    for (int hh = 0; hh < 4; ++hh) {
                        uint32_t pk[4];
#pragma unroll
                        for (int k = 0; k < 8; k += 2) {
                            const float2 p = make_float2(ex2(__uint_as_float(rs[hh][k])), ex2(__uint_as_float(rs[hh][k + 1])));
                            const float2 ds = __fmul2_rn(p, make_float2(__uint_as_float(rd[hh][k]),
                                                                        __uint_as_float(rd[hh][k + 1])));
                            rd[hh][k] = __float_as_uint(ds.x);
                            rd[hh][k + 1] = __float_as_uint(ds.y);
                            pk[k / 2] = pack_bf16x2(ds.x, ds.y);
                        }
                        if (FAST || uniform) {   // the row's sum for its register bin
#pragma unroll
                            for (int k = 0; k < 8; k += 2)
                                acc[hh] = __fadd2_rn(acc[hh], make_float2(__uint_as_float(rd[hh][k]),
                                                                         __uint_as_float(rd[hh][k + 1])));
                        }
                        tmem_st_x4(lrow + s_col(ss) + 16 * hh + 4 * g, pk);
                    }
                    if constexpr (!FAST) {
                        if (!uniform) {
                            // dS in fixed point (|dS| < 2^29 by the choice of the scale)
#pragma unroll
                            for (int hh = 0; hh < 4; ++hh)
#pragma unroll
                                for (int k = 0; k < 8; k += 2) {
                                    const uint2 fv =
                                        round_fixed2(__uint_as_float(rd[hh][k]), __uint_as_float(rd[hh][k + 1]));
                                    rd[hh][k] = fv.x;
                                    rd[hh][k + 1] = fv.y;
                                }
#pragma unroll
                            for (int k = 0; k < 8; ++k) {
                                const int kk = 8 * g + k;
                                const uint32_t code = __byte_perm(w[kk >> 2], 0u, 0x4440u + (kk & 3));
                                if (code < (uint32_t)nb) {
#pragma unroll
                                    for (int hh = 0; hh < 4; ++hh)
                                        red_shared_add_u32(binb + code * kCodeStride + hh * kHeadStride, rd[hh][k]);
                                }
                            }
                        }
                    }
                };
                if (wuni) {
                    half(0, std::true_type());
                    half(1, std::true_type());
                } else {
                    half(0, std::false_type());
                    half(1, std::false_type());
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&bars->ds_ready[ss]);
            }
            if (!ok) break;
            mbar_arrive(&bars->kv_empty[ks]);
        }
        if (acc_code >= 0 && acc_code < nb) {
#pragma unroll
            for (int hh = 0; hh < 4; ++hh)
                red_shared_add_u32(binb + acc_code * kCodeStride + hh * kHeadStride, fx(acc[hh].x + acc[hh].y));
        }
        if (!ok) {
            fail(abort_flag, status);
        } else {
            const int tp = nchunks - 1;
            if (!mbar_wait(&bars->dq_done[tp & 1], (tp >> 1) & 1, abort_flag, kWaitNs)) {
                fail(abort_flag, status);
            } else {
                tc_fence_after();
#pragma unroll
                for (int hh = 0; hh < 4; ++hh) {
                    const int h = kHC * hb + hh;
                    uint32_t ov[16];
                    tmem_ld_x16(lrow + kColDq + 16 * hh, ov);
                    tmem_wait_ld();
                    const int c0h = (HD == 8) ? (h & 1) * 8 : 0;
                    if (live && dq_acc) {
                        float* dst = dq_acc + ((int64_t)row * kH + h) * HD;
#pragma unroll
                        for (int k = 0; k < HD; k += 4)
                            asm volatile("red.global.v4.f32.add [%0], {%1, %2, %3, %4};" ::"l"(dst + k),
                                         "f"(__uint_as_float(ov[c0h + k]) * qscale),
                                         "f"(__uint_as_float(ov[c0h + k + 1]) * qscale),
                                         "f"(__uint_as_float(ov[c0h + k + 2]) * qscale),
                                         "f"(__uint_as_float(ov[c0h + k + 3]) * qscale)
                                         : "memory");
                    } else if (live) {
                        uint32_t wq[HD / 2];
#pragma unroll
                        for (int k = 0; k < HD / 2; ++k)
                            wq[k] = pack_bf16x2(__uint_as_float(ov[c0h + 2 * k]) * qscale,
                                                __uint_as_float(ov[c0h + 2 * k + 1]) * qscale);
                        uint4* dst = reinterpret_cast<uint4*>(dq + ((int64_t)row * kH + h) * HD);
#pragma unroll
                        for (int k = 0; k < HD / 8; ++k)
                            dst[k] = make_uint4(wq[4 * k], wq[4 * k + 1], wq[4 * k + 2], wq[4 * k + 3]);
                    }
                }
            }
        }
        // add the copies of each (code, head) bin to the global table
        asm volatile("bar.sync 1, %0;" ::"n"(kSoft) : "memory");
        for (int x = tid; x < nb * kHC; x += kSoft) {
            const int* cp = bins + (int64_t)x * NCP;
            long long s = 0;
#pragma unroll 8
            for (int l = 0; l < NCP; ++l) s += cp[(l + tid) & (NCP - 1)];
            const int code = x / kHC, h = kHC * hb + x % kHC;
            if (s != 0) atomicAdd(&dT64[h * nb + code], (double)s / (double)bscale);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
    if (tid == 0) pdl_wait();   // complete after the kernel before, if this one overlapped it
}

// First row of the tasks the tail split takes (tasks past the last full wave of
// two CTAs per SM, whose dq goes through dq_acc), or -1 when there is no such split.
int dq_tail_row0(int n, int tail, bool have_acc) {
    const int slots = 2 * num_sms();
    const int tasks = 2 * ((n + kBQ - 1) / kBQ);
    if (tail <= 1 || !have_acc || tasks % slots == 0) return -1;
    return (tasks / slots * slots / 2) * kBQ;
}

template <int HD>
int launch(int n, const void* q, const void* k, const void* v, const void* dO, const int8_t* spd,
           int64_t ld, const float* T, int nb, float scale, const float* LD, int ldl, const float* vmax,
           int tail, void* dq, float* dq_acc, double* dT64, cudaStream_t s) {
    using C = DqCfg<HD>;
    CUtensorMap mk, mv, ms;
    const uint64_t cols = (uint64_t)kH * HD;
    if (!make_map_2d(&mk, const_cast<void*>(k), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n, cols, cols * 2,
                     C::BKV, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_2d(&mv, const_cast<void*>(v), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n, cols, cols * 2,
                     C::BKV, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_2d(&ms, const_cast<int8_t*>(spd), CU_TENSOR_MAP_DATA_TYPE_UINT8, n, n, ld, kBQ,
                     C::BKV, C::BKV == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B))
        return GT_ERR_CUDA;
    int* status = device_status_ptr();
    if (!status) return GT_ERR_CUDA;
    // 32 bin copies (conflict-free) while two CTAs still fit on an SM, else 8
    const bool wide = C::smem_bytes(nb, 32) <= kSmemPair;
    auto kern = wide ? bwd_dq_kernel<HD, 32> : bwd_dq_kernel<HD, 8>;
    const uint32_t smem = C::smem_bytes(nb, wide ? 32 : 8);
    if (smem > kSmemLimit) return GT_ERR_UNSUPPORTED;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return GT_ERR_CUDA;
    const int total_blocks = (n + C::BKV - 1) / C::BKV;
    const int tasks = 2 * ((n + kBQ - 1) / kBQ);
    // tasks [first, first + count), each split over `split` CTAs (1: whole, into dq);
    // every launch may start while the one before it finishes: the first one
    // overlaps the prep kernel (and waits for it before reading its tables), the
    // split tail the whole tasks' last wave
    auto run = [&](int first, int count, int split, bool after_prep) -> int {
        const int per = split > 1 ? (total_blocks + split - 1) / split : 0;
        const int nz = per > 0 ? (total_blocks + per - 1) / per : 1;
        const dim3 grid(count, 1, nz);
        LaunchScope ls("bwd_dq", s);
        auto* qp = static_cast<const __nv_bfloat16*>(q);
        auto* gp = static_cast<const __nv_bfloat16*>(dO);
        auto* dqp = static_cast<__nv_bfloat16*>(dq);
        float* accp = per > 0 ? dq_acc : nullptr;
        if (launch_overlapped(kern, grid, dim3(kThreads), smem, s, mk, mv, ms, qp, gp, LD, ldl, vmax, T, nb, n,
                              scale, scale * kLog2e, first, per, dqp, accp, dT64, after_prep ? 1 : 0,
                              status) != cudaSuccess)
            return GT_ERR_CUDA;
        return check_launch();
    };
    const int row0 = dq_tail_row0(n, tail, dq_acc != nullptr);
    if (row0 >= 0) {
        // full waves of whole tasks (none on a graph too small to fill one), then
        // the rest split `tail` ways along the KV
        // blocks so that the last waves fill the SMs, overlapping the whole
        // tasks' last wave; the caller cleared their rows of dq_acc before and
        // converts them after
        const int g1 = (row0 / kBQ) * 2;
        if (g1 > 0) {
            const int rc = run(0, g1, 1, true);
            if (rc != GT_OK) return rc;
        }
        return run(g1, tasks - g1, tail, g1 == 0);
    }
    return run(0, tasks, 1, true);
}

}  // namespace

// KV split of the dq tasks (tile, head half) past the last full wave of two CTAs
// per SM (1 = none): the k in [2, 8] that makes the last, partial wave plus the
// split tail shortest, in units of one task's time; 1 when no k beats one more
// wave of whole tasks.
int bwd_dq_tail_split(int n) {
    const int slots = 2 * num_sms();
    const int tasks = 2 * ((n + kBQ - 1) / kBQ);
    if (tasks % slots == 0) return 1;
    const int rem = tasks % slots;
    int best = 1;
    double best_t = 1.0;
    for (int k = 2; k <= 8; ++k) {
        const double t = (double)((rem * k + slots - 1) / slots) / k;
        if (t < best_t - 1e-9) { best_t = t; best = k; }
    }
    return best;
}

int bwd_dq_tail_row0(int n, int tail, bool have_acc) { return dq_tail_row0(n, tail, have_acc); }

int launch_bwd_dq(int n, int d, const void* q, const void* k, const void* v, const void* dO,
                  const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                  const float* LD, int ldl, const float* vmax, int tail, void* dq, float* dq_acc,
                  double* dT64, cudaStream_t s) {
    return d == 8 ? launch<8>(n, q, k, v, dO, spd, ld, T, nb, scale, LD, ldl, vmax, tail, dq, dq_acc, dT64, s)
                  : launch<16>(n, q, k, v, dO, spd, ld, T, nb, scale, LD, ldl, vmax, tail, dq, dq_acc, dT64, s);
}

}  // namespace gt

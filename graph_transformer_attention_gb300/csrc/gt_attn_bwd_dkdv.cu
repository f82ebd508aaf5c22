// gt_attn_bwd_dkdv.cu -- tensor-core backward, KV-stationary part: dk and dv
// (bf16 storage, H = 8 heads, head dim 8 or 16).
//
// With P and dS recomputed as in the Q-stationary pass (MegaGraph, Fig. 4: the
// bias slice of each block comes from the int8 bucket matrix),
//   dv_j = sum_i P_ij dO_i,   dk_j = scale sum_i dS_ij Q_i.
//
// One CTA per SM = one group: a tile of 128 KV rows and one half of the heads
// (4 of 8), streaming every Q tile (or, for split groups, a range of them; or,
// in the balanced grid of a graph whose groups do not fill one wave, an equal
// share of all (group, Q tile) steps, the CTA switching groups as its share
// crosses them: dk and dv out, the next K and V in).  The CTA owns all 512 TMEM columns, so K and
// V sit in TMEM as the A operands of S^T = K Q^T and dP^T = V dO^T: every
// product reads only its small B operand from shared memory (an MMA with A in
// shared memory reads 4 KB of it, which both costs ~4x the tensor time and
// delays the softmax warps' own shared loads).  The work is cut into steps of
// one head pair and 32 query rows; the tensor core runs two steps ahead of the
// softmax warps.  576 threads:
//   warps 0-15 warp w owns KV rows 32 (w mod 4) .. + 31 (TMEM lanes), head
//              (w / 4) mod 2 of the pair and query rows 16 (w / 8) .. + 15 of each
//              step: it
//              reads S'^T and dP'^T from TMEM, the bucket codes from column r of the
//              int8 tile, forms P^T = 2^(s' scale log2 e + b) and dS^T = P^T dP'^T
//              and writes both (bf16) back over S'^T.  The tensor core has already
//              taken lse_i and D_i out: S'^T = K Q^T + 1 (-lse_i / scale) and
//              dP'^T = V dO^T + 1 (-D_i), the second product of each with a constant
//              A operand of ones in TMEM and B = the per-row values as three bf16
//              parts (exact to fp32 rounding), so the softmax warps load neither.
//   warp 16    MMA issuer (the whole warp waits, the elected lane issues): per
//              step, once its P^T and dS^T are in, dv_h += P^T_h dO_h and
//              dk_h += dS^T_h Q_h (A from TMEM), then S^T and dP^T of the step two
//              ahead into the same buffer (the tensor pipe runs one thread's MMAs
//              in order, so they land after the products that read the buffer).
//   warp 17    TMA producer: per Q tile the bucket tile and the Q, dO and LB
//              column slots (LB: -lse_i / scale and -D_i per head in three bf16
//              parts each); it also summarises each tile's codes.
// TMEM (512 columns): dk at 0, dv at 64, K at 128 and V at 160 (8 columns of
// bf16 pairs per head), the two ones operands at 192 and 200, and one
// 128-column buffer per head pair at 256 and 384: head e of the pair holds S'^T
// at +32e and dP'^T at +64 + 32e; the 16 columns of query rows 16u .. 16u + 15
// take P^T (columns +16u .. +7) and dS^T (+16u + 8 .. +15) over S'^T.  All waits are bounded (timeout -> device status word, orderly
// exit, TMEM freed).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
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

constexpr int kBKV = 128;
constexpr int kCH = 32;                    // query rows per step
constexpr int kQST = 2;
constexpr int kHC = 4;                     // heads per CTA
constexpr int kSoft = 512;                 // softmax threads: 128 KV rows x (2 heads x 2 row halves)
constexpr int kThreads = kSoft + 64;
constexpr int kMmaWarp = 16;
constexpr int kTmaWarp = 17;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColDk = 0;
constexpr uint32_t kColDv = 64;
constexpr uint32_t kColKA = 128;
constexpr uint32_t kColVA = 160;
constexpr uint32_t kColOnesL = 192;        // A = [1 1 1 0 ...]: picks -lse / scale from LB
constexpr uint32_t kColOnesD = 200;        // A = [0 0 0 1 1 1 0 ...]: picks -D
constexpr uint32_t kSmemOneCta = 120 * 1024;   // more than half an SM's shared memory: one CTA per SM

// TMEM buffer of head pair p
__device__ __forceinline__ uint32_t pair_buf(int p) { return 256u + 128u * (uint32_t)p; }

template <int HD>
struct KvCfg {
    static constexpr int BQ = 64;                         // query rows per TMA tile
    static constexpr int NCH = BQ / kCH;                  // steps of one head pair per tile
    static constexpr int NSLOT = kHC * HD / 16;           // 16-column slots of this CTA's heads
    static constexpr uint32_t SPD_BYTES = BQ * kBKV;      // [BQ i][128 j], no swizzle
    static constexpr uint32_t SLOT_BYTES = BQ * 32;
    static constexpr uint32_t LB_OFF = SPD_BYTES + 2 * NSLOT * SLOT_BYTES;   // one LB slot per head
    static constexpr uint32_t STAGE_BYTES = LB_OFF + kHC * SLOT_BYTES;
    static constexpr uint32_t OFF_STAGE = 0;
    static constexpr uint32_t OFF_T = OFF_STAGE + kQST * STAGE_BYTES;
    // per stage: one int per (32-row chunk, warp's 32 KV columns): the bucket code
    // when all 1024 codes of that block are equal, else -1
    static constexpr int NMETA = NCH * 4;
    static constexpr uint32_t OFF_META = OFF_T + 256 * kH * 4;
    static constexpr uint32_t OFF_BAR = OFF_META + kQST * NMETA * 4;
    static constexpr uint32_t SMEM_USED = OFF_BAR + 256 + 1024;
    static constexpr uint32_t SMEM = SMEM_USED > kSmemOneCta ? SMEM_USED : kSmemOneCta;
};

struct Bars {
    uint64_t q_full[kQST];
    uint64_t meta_ready[kQST];   // the stage's bucket summary is written (and its copies landed)
    uint64_t q_empty[kQST];
    uint64_t sd_full[2];         // S^T and dP^T of a step are in its head pair's buffer
    uint64_t ds_ready[2];        // P^T and dS^T of a step are in (dP^T read)
    uint64_t done;               // a group's last dk/dv products are complete (phase = its segment)
    uint64_t seg_ready;          // the next group's K and V are in TMEM, the last one's dk/dv read
    uint64_t fin;
    uint32_t tmem_base;
    int abort;
};

template <int HD, bool kBal>
__global__ void __launch_bounds__(kThreads, 1)
bwd_dkdv_kernel(const __grid_constant__ CUtensorMap mapQ, const __grid_constant__ CUtensorMap mapG,
                const __grid_constant__ CUtensorMap mapS, const __grid_constant__ CUtensorMap mapB,
                const __nv_bfloat16* __restrict__ k, const __nv_bfloat16* __restrict__ v,
                const float* __restrict__ T, int nb, int n, float scale, float scale_log2, int g0, int split_tiles,
                int bal_ctas, __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv,
                float* __restrict__ dk_acc, float* __restrict__ dv_acc, int* status) {
    using C = KvCfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    // 1024-byte aligned by pointer arithmetic on the shared array, so that the
    // compiler still knows plain accesses through it are shared-memory accesses
    uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
    float* Ts = reinterpret_cast<float*>(smem + C::OFF_T);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();   // the split tail may take SMs as this launch frees them
    // The CTA's work is a run of (group, Q tile) steps in group-major order: step
    // s = g T + qt, group g = KV tile g / 2 and head half g % 2 (heads 4 hb .. 4 hb
    // + 3), T Q tiles per group.  Balanced (kBal, bal_ctas CTAs): CTA x takes steps
    // [x S / bal_ctas, (x + 1) S / bal_ctas) of all S = groups T, so that every CTA
    // has the same work; the groups it shares with a neighbour (and, for
    // simplicity, all others) are summed into dk_acc / dv_acc in fp32.  Otherwise
    // one group g0 + blockIdx.x, its Q tiles split over grid.z when split_tiles > 0
    // (then summed in fp32 too).  The b-th tile of the CTA is step sb + b; a change
    // of group starts a new segment (K and V rewritten, dk and dv restarted).
    const int total_tiles = (n + C::BQ - 1) / C::BQ;
    int64_t sb, se;
    if (kBal) {
        const int64_t steps = (int64_t)(2 * ((n + kBKV - 1) / kBKV)) * total_tiles;
        sb = steps * blockIdx.x / bal_ctas;
        se = steps * (blockIdx.x + 1) / bal_ctas;
    } else {
        const int qt0 = split_tiles > 0 ? blockIdx.z * split_tiles : 0;
        sb = (int64_t)(g0 + (int)blockIdx.x) * total_tiles + qt0;
        se = sb + (split_tiles > 0 ? min(split_tiles, total_tiles - qt0) : total_tiles);
    }
    const int ntiles = (int)(se - sb);
    const int nchunks = ntiles * C::NCH;
    // the first tile's group and Q tile; the loops below walk the groups without
    // dividing: the k-th segment ends before tile T - q_first + k T
    const int g_first = (int)(sb / total_tiles);
    const int q_first = (int)(sb - (int64_t)g_first * total_tiles);

    if (tid == kTmaWarp * 32) {
        for (int s = 0; s < kQST; ++s) {
            mbar_init(&bars->q_full[s], 1);
            mbar_init(&bars->meta_ready[s], 32);
            mbar_init(&bars->q_empty[s], kSoft + 1);
        }
        for (int p = 0; p < 2; ++p) {
            mbar_init(&bars->sd_full[p], 1);
            mbar_init(&bars->ds_ready[p], kSoft);
        }
        mbar_init(&bars->done, 1);
        mbar_init(&bars->seg_ready, kSoft);
        mbar_init(&bars->fin, 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&mapQ);
        tma_prefetch_desc(&mapG);
        tma_prefetch_desc(&mapS);
        tma_prefetch_desc(&mapB);
    }
    if (warp == kMmaWarp) tmem_alloc(&bars->tmem_base, kTmemCols);
    fill_bias_table(Ts, T, nb, tid, kThreads);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bars->tmem_base;
    int* abort_flag = &bars->abort;
    // K and V rows of group g's heads into TMEM (A operands), one row per lane of
    // threads 0 .. 127 (again at each change of group)
    auto write_kv = [&](int g) {
        const int row = (g >> 1) * kBKV + tid;
        const bool live = row < n;
        const int64_t off = (int64_t)(live ? row : 0) * kH * HD;
        const uint32_t lr = tbase + ((uint32_t)((warp & 3) * 32) << 16);
#pragma unroll
        for (int hh = 0; hh < kHC; ++hh) {
            uint32_t a[8];
            head_a_row<HD>(k + off, kHC * (g & 1) + hh, live, a);
            tmem_st_x8(lr + kColKA + 8 * hh, a);
            head_a_row<HD>(v + off, kHC * (g & 1) + hh, live, a);
            tmem_st_x8(lr + kColVA + 8 * hh, a);
        }
    };
    if (tid < kBKV) {
        write_kv(g_first);
        // ones operands (bf16 1.0 = 0x3f80; element 2c in the low half of column c)
        const uint32_t lr = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        const uint32_t onesL[8] = {0x3f803f80u, 0x00003f80u, 0u, 0u, 0u, 0u, 0u, 0u};
        const uint32_t onesD[8] = {0u, 0x3f800000u, 0x3f803f80u, 0u, 0u, 0u, 0u, 0u};
        tmem_st_x8(lr + kColOnesL, onesL);
        tmem_st_x8(lr + kColOnesD, onesD);
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (warp == kTmaWarp) {
        // ------------------------------------------------------ TMA producer
        // Issues the copies of Q tile b + 2 once tile b is consumed, and summarises
        // each tile's bucket codes as soon as it lands (one tile ahead of the
        // softmax): per (32-row chunk, 32-column warp block) the common code or -1.
        int* meta = reinterpret_cast<int*>(smem + C::OFF_META);
        int issued = 0;
        bool ok = true;
        int ig = g_first, iq = q_first;   // group and Q tile of the next tile to issue (tiles in order)
        auto issue = [&](int b) -> bool {
            const int ks = b & 1;
            if (lane == 0) {
                if (b >= kQST && !mbar_wait(&bars->q_empty[ks], ((b >> 1) - 1) & 1, abort_flag, kWaitNs)) {
                    fail(abort_flag, status);
                } else {
                    uint8_t* st = smem + C::OFF_STAGE + ks * C::STAGE_BYTES;
                    const int i0 = iq * C::BQ, j0 = (ig >> 1) * kBKV, hb = ig & 1;
                    mbar_arrive_expect_tx(&bars->q_full[ks], C::STAGE_BYTES);
                    tma_load_2d(st, &mapS, j0, i0, &bars->q_full[ks]);
#pragma unroll
                    for (int s = 0; s < C::NSLOT; ++s) {
                        tma_load_2d(st + C::SPD_BYTES + s * C::SLOT_BYTES, &mapQ, 16 * (hb * C::NSLOT + s),
                                    i0, &bars->q_full[ks]);
                        tma_load_2d(st + C::SPD_BYTES + (C::NSLOT + s) * C::SLOT_BYTES, &mapG,
                                    16 * (hb * C::NSLOT + s), i0, &bars->q_full[ks]);
                    }
#pragma unroll
                    for (int hh = 0; hh < kHC; ++hh)
                        tma_load_2d(st + C::LB_OFF + hh * C::SLOT_BYTES, &mapB, 16 * (kHC * hb + hh), i0,
                                    &bars->q_full[ks]);
                }
            }
            __syncwarp();
            if (*(volatile int*)abort_flag) return false;
            issued = b + 1;
            if (++iq == total_tiles) {
                iq = 0;
                ++ig;
            }
            return true;
        };
        auto summarise = [&](int b) -> bool {
            const int ks = b & 1;
            if (!mbar_wait(&bars->q_full[ks], (b >> 1) & 1, abort_flag, kWaitNs)) {
                fail(abort_flag, status);
                return false;
            }
            const uint32_t st = smem_u32(smem + C::OFF_STAGE + ks * C::STAGE_BYTES);
            // per 32-row chunk: lane l checks 16-byte piece l & 7 of rows 4u + l / 8
            // (u = 0..7), so the eight lanes of a row cover all 32 banks; a warp
            // block w owns pieces 2w, 2w + 1 of every row
            const uint32_t piece = (uint32_t)(lane & 7), rsub = (uint32_t)(lane >> 3);
#pragma unroll 1
            for (int cc = 0; cc < C::NCH; ++cc) {
                const uint32_t row0 = st + (uint32_t)(kCH * cc) * kBKV;
                const uint32_t ref = lds_u8(row0 + 32u * (piece >> 1)) * 0x01010101u;
                bool same = true;
#pragma unroll
                for (int u = 0; u < kCH / 4; ++u) {
                    const uint4 vv = lds_u4(row0 + (4u * u + rsub) * kBKV + 16u * piece);
                    same = same && vv.x == ref && vv.y == ref && vv.z == ref && vv.w == ref;
                }
                const unsigned bal = __ballot_sync(0xffffffffu, same);
                const uint32_t wref = __shfl_sync(0xffffffffu, ref, 2 * (lane & 3));
                if (lane < 4) {
                    const unsigned mask = 0x03030303u << (2 * lane);
                    meta[ks * C::NMETA + 4 * cc + lane] = (bal & mask) == mask ? (int)(wref & 0xffu) : -1;
                }
            }
            __syncwarp();
            mbar_arrive(&bars->meta_ready[ks]);
            return true;
        };
        for (int b = 0; ok && b < kQST && b < ntiles; ++b) ok = issue(b);
        if (ok) ok = summarise(0);
        for (int b = 0; ok && b < ntiles; ++b) {
            if (b + 1 < ntiles && !summarise(b + 1)) { ok = false; break; }
            if (b + kQST < ntiles && !issue(b + kQST)) { ok = false; break; }
        }
        if (!ok && lane == 0) {
            int never = 0;
            for (int b = issued - kQST; b < issued; ++b)
                if (b >= 0) mbar_wait(&bars->q_full[b & 1], (b >> 1) & 1, &never, kWaitNs);
        }
    } else if (warp == kMmaWarp) {
        // ----------------------------------------------------------- MMA
        // Step s = 2 t + p: chunk t of 32 query rows, head pair p (heads 2p, 2p + 1
        // of this CTA), TMEM buffer p.  The whole warp runs the loop and waits; the
        // elected lane issues (an MMA from a converged warp through elect.sync costs
        // a fraction of one from a lane-0 branch), and descriptors are precomputed
        // so that an MMA costs one add.
        {
            const uint32_t idS = idesc_bf16(128, kCH, false, false);
            const uint32_t idKM = idesc_bf16(128, 16, false, true);
            const uint32_t stage_base = smem_u32(smem + C::OFF_STAGE);
            const SmemDesc dQk = smem_desc_split(stage_base + C::SPD_BYTES, 16, 256, 6);     // K-major Q
            const SmemDesc dQm = smem_desc_split(stage_base + C::SPD_BYTES, 256, 256, 6);    // MN-major Q
            constexpr uint32_t kG = C::NSLOT * C::SLOT_BYTES;                                 // dO after Q
            const int nsteps = 2 * nchunks;
            // offset of (stage, chunk, head) in the Q / dO column slots (32 rows = 1 KB)
            auto qoff = [&](int t, int h) -> uint32_t {
                const int b = t / C::NCH, c = t % C::NCH;
                return (uint32_t)((b & 1) * C::STAGE_BYTES + (h * HD / 16) * C::SLOT_BYTES + c * 1024);
            };
            // offset of (stage, chunk, head) in the LB slots
            auto boff = [&](int t, int h) -> uint32_t {
                const int b = t / C::NCH, c = t % C::NCH;
                return (uint32_t)((b & 1) * C::STAGE_BYTES + (C::LB_OFF - C::SPD_BYTES) + h * C::SLOT_BYTES + c * 1024);
            };
            auto issue_sd = [&](int st) -> bool {
                const int t = st >> 1, p = st & 1, b = t / C::NCH, c = t % C::NCH, ks = b & 1;
                if (c == 0 && p == 0 && !mbar_wait_all(&bars->q_full[ks], (b >> 1) & 1, abort_flag, kWaitNs))
                    return false;
                tc_fence_after();
                const uint32_t d = tbase + pair_buf(p);
                if (elect_one()) {
#pragma unroll
                    for (int e = 0; e < 2; ++e) {
                        const int h = 2 * p + e;
                        const uint32_t lb = boff(t, h);
                        mma_ts(d + 32 * e, tbase + kColKA + 8 * h, desc_at(dQk, qoff(t, h)), idS, 0);
                        mma_ts(d + 32 * e, tbase + kColOnesL, desc_at(dQk, lb), idS, 1);
                        mma_ts(d + 64 + 32 * e, tbase + kColVA + 8 * h, desc_at(dQk, qoff(t, h) + kG), idS, 0);
                        mma_ts(d + 64 + 32 * e, tbase + kColOnesD, desc_at(dQk, lb), idS, 1);
                    }
                    mma_commit(&bars->sd_full[p]);
                }
                __syncwarp();
                return true;
            };
            // a group's steps end with its dk / dv products and a commit of `done`;
            // the next group's S and dP wait for `seg_ready` (its K and V written,
            // the last group's dk and dv read), and its first products restart dk, dv
            // (the segment change sits outside the step loop, which stays as small
            // as with one group)
            int seg = 0;        // segments finished (the phase of done and seg_ready)
            int t_seg = 0;      // first chunk of the current segment
            int b_end = total_tiles - q_first;   // first tile past the current segment
            bool ok = true;
            int st = 0;
#pragma unroll 1
            for (int k0 = 0; ok && k0 < 2 && k0 < nsteps; ++k0) ok = issue_sd(k0);
            while (ok && st < nsteps) {
                const int st_end = kBal ? min(nsteps, 2 * C::NCH * b_end) : nsteps;   // the segment's steps
                for (; st < st_end; ++st) {
                    const int t = st >> 1, p = st & 1, b = t / C::NCH, c = t % C::NCH, ks = b & 1;
                    if (!mbar_wait_all(&bars->ds_ready[p], t & 1, abort_flag, kWaitNs)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t x = tbase + pair_buf(p);
                    if (elect_one()) {
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            const int h = 2 * p + e;
#pragma unroll
                            for (int k2 = 0; k2 < 2; ++k2) {
                                const uint32_t acc = (t > t_seg || k2 > 0) ? 1u : 0u;
                                mma_ts(tbase + kColDv + 16 * h, x + 32 * e + 16 * k2,
                                       desc_at(dQm, qoff(t, h) + kG + 512 * k2), idKM, acc);
                                mma_ts(tbase + kColDk + 16 * h, x + 32 * e + 16 * k2 + 8,
                                       desc_at(dQm, qoff(t, h) + 512 * k2), idKM, acc);
                            }
                        }
                        if (c == C::NCH - 1 && p == 1) mma_commit(&bars->q_empty[ks]);
                    }
                    __syncwarp();
                    if (st + 2 < st_end && !issue_sd(st + 2)) { ok = false; break; }
                }
                if (!kBal || !ok || st >= nsteps) break;
                // the segment's products are all issued: signal them, then wait for
                // the next group's K and V before its first S and dP
                if (elect_one()) mma_commit(&bars->done);
                __syncwarp();
                if (!mbar_wait_all(&bars->seg_ready, seg & 1, abort_flag, kWaitNs)) { ok = false; break; }
                tc_fence_after();
                ++seg;
                t_seg = st >> 1;
                b_end += total_tiles;
#pragma unroll 1
                for (int k0 = 0; ok && k0 < 2 && st + k0 < nsteps; ++k0) ok = issue_sd(st + k0);
            }
            if (ok) {
                if (elect_one()) mma_commit(&bars->done);
                __syncwarp();
            } else {
                fail(abort_flag, status);
                int never = 0;
                if (elect_one()) mma_commit(&bars->fin);
                __syncwarp();
                mbar_wait_all(&bars->fin, 0, &never, kWaitNs);
            }
        }
    } else {
        // ------------------------------------------------------- softmax
        // Warps w, w + 4, w + 8, w + 12 own the same 32 KV rows (TMEM lanes):
        // thread (r, e, half) takes head e of the pair and query rows 16 half ..
        // 16 half + 15 of every step.
        const int r = tid & (kBKV - 1);
        const int e = (tid >> 7) & 1;
        const int half = tid >> 8;
        const uint32_t lrow = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        // a group's dk and dv rows, after its last products (head 2 half + e of the
        // CTA's four, KV row r): into bf16, or added into the fp32 sums
        auto epilogue = [&](int g) {
            const int row = (g >> 1) * kBKV + r;
            const bool live = row < n;
            const int hh = 2 * half + e;
            const int h = kHC * (g & 1) + hh;
            uint32_t ok16[16], ov16[16];
            tmem_ld_x16(lrow + kColDk + 16 * hh, ok16);
            tmem_ld_x16(lrow + kColDv + 16 * hh, ov16);
            tmem_wait_ld();
            // head dim 8: the head's channels are columns 8 (h & 1) .. of the 16;
            // shift them down with constant register indices
            if (HD == 8 && (h & 1)) {
#pragma unroll
                for (int q2 = 0; q2 < 8; ++q2) {
                    ok16[q2] = ok16[q2 + 8];
                    ov16[q2] = ov16[q2 + 8];
                }
            }
            if (live && dk_acc) {
                float* gk = dk_acc + ((int64_t)row * kH + h) * HD;
                float* gv = dv_acc + ((int64_t)row * kH + h) * HD;
#pragma unroll
                for (int q4 = 0; q4 < HD / 4; ++q4) {
                    red_add_v4(gk + 4 * q4, __uint_as_float(ok16[4 * q4]) * scale, __uint_as_float(ok16[4 * q4 + 1]) * scale,
                               __uint_as_float(ok16[4 * q4 + 2]) * scale, __uint_as_float(ok16[4 * q4 + 3]) * scale);
                    red_add_v4(gv + 4 * q4, __uint_as_float(ov16[4 * q4]), __uint_as_float(ov16[4 * q4 + 1]),
                               __uint_as_float(ov16[4 * q4 + 2]), __uint_as_float(ov16[4 * q4 + 3]));
                }
            } else if (live) {
                uint32_t wk[HD / 2], wv[HD / 2];
#pragma unroll
                for (int q2 = 0; q2 < HD / 2; ++q2) {
                    wk[q2] = pack_bf16x2(__uint_as_float(ok16[2 * q2]) * scale,
                                         __uint_as_float(ok16[2 * q2 + 1]) * scale);
                    wv[q2] = pack_bf16x2(__uint_as_float(ov16[2 * q2]), __uint_as_float(ov16[2 * q2 + 1]));
                }
                uint4* dstk = reinterpret_cast<uint4*>(dk + ((int64_t)row * kH + h) * HD);
                uint4* dstv = reinterpret_cast<uint4*>(dv + ((int64_t)row * kH + h) * HD);
#pragma unroll
                for (int q2 = 0; q2 < HD / 8; ++q2) {
                    dstk[q2] = make_uint4(wk[4 * q2], wk[4 * q2 + 1], wk[4 * q2 + 2], wk[4 * q2 + 3]);
                    dstv[q2] = make_uint4(wv[4 * q2], wv[4 * q2 + 1], wv[4 * q2 + 2], wv[4 * q2 + 3]);
                }
            }
        };
        int t = 0;
        int seg = 0;    // segments finished
        int gb = g_first, qb = q_first;   // the tile's group and Q tile
        bool ok = true;
        int b = 0;
        while (ok) {
          // the segment's tiles; its end (dk and dv out, the next group's K and V in)
          // sits outside the tile loop, which stays as small as with one group
          const int b_stop = kBal ? min(ntiles, b + (total_tiles - qb)) : ntiles;
          for (; ok && b < b_stop; ++b, ++qb) {
            const int ks = b & 1;
            const uint32_t tbl = smem_u32(Ts) + 16u * (uint32_t)(gb & 1);
            // (the summary is written after the tile's copies have landed)
            if (!mbar_wait(&bars->meta_ready[ks], (b >> 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
            const uint8_t* stp = smem + C::OFF_STAGE + ks * C::STAGE_BYTES;
            const int* meta = reinterpret_cast<const int*>(smem + C::OFF_META) + ks * C::NMETA + (warp & 3);
            const int i0 = qb * C::BQ;
            const bool tail_tile = i0 + C::BQ > n;
            for (int c = 0; ok && c < C::NCH; ++c, ++t) {
                const int ir = c * kCH + 16 * half;       // this thread's first query row in the tile
                // bucket codes of the 16 (i, j) pairs: column r of the tile, unless the
                // warp's whole 32 x 32 block holds one code
                const int ucode = meta[4 * c];
                // One chunk, both head pairs.  FAST (the warp's 32 x 32 block holds one
                // code): one bias per head, x with one packed FMA per two rows; otherwise
                // each row's code and bias.  Separate instantiations, so the uniform
                // blocks run without the per-code path.  Returns false on a timeout.
                auto chunk = [&](auto fast_tag) -> bool {
                    constexpr bool FAST = decltype(fast_tag)::value;
                    uint32_t code[16];
                    float4 bu = make_float4(0.f, 0.f, 0.f, 0.f);
                    if constexpr (FAST) {
                        bu = lds_f4(tbl + (uint32_t)ucode * 32u);
                    } else {
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk) code[kk] = stp[(ir + kk) * kBKV + r];
                    }
#pragma unroll
                    for (int p = 0; p < 2; ++p) {
                        if (!mbar_wait(&bars->sd_full[p], t & 1, abort_flag, kWaitNs)) return false;
                        tc_fence_after();
                        const uint32_t x = lrow + pair_buf(p) + 32 * e + 16 * half;
                        uint32_t rs[16], rd[16];
                        tmem_ld_x16(x, rs);
                        tmem_ld_x16(x + 64, rd);
                        tmem_wait_ld();
                        // x = s' scale log2e + b(code); P = 2^x
                        float pf[16];
                        if constexpr (FAST) {
                            const float bh = p ? (e ? bu.w : bu.z) : (e ? bu.y : bu.x);
                            const float2 cc = make_float2(scale_log2, scale_log2);
#pragma unroll
                            for (int kk = 0; kk < 16; kk += 2) {
                                const float2 xa = __ffma2_rn(
                                    make_float2(__uint_as_float(rs[kk]), __uint_as_float(rs[kk + 1])), cc,
                                    make_float2(bh, bh));
                                pf[kk] = xa.x;
                                pf[kk + 1] = xa.y;
                            }
                        } else {
                            const uint32_t hofs = 4u * (uint32_t)(2 * p + e);
#pragma unroll
                            for (int kk = 0; kk < 16; ++kk) {
                                const float bv = __uint_as_float(lds_u32(tbl + code[kk] * 32u + hofs));
                                pf[kk] = fmaf(__uint_as_float(rs[kk]), scale_log2, bv);
                            }
                        }
#pragma unroll
                        for (int kk = 0; kk < 16; ++kk) pf[kk] = ex2(pf[kk]);
                        if (tail_tile) {
#pragma unroll
                            for (int kk = 0; kk < 16; ++kk)
                                if (i0 + ir + kk >= n) pf[kk] = 0.f;
                        }
                        uint32_t pp[8], pd[8];
#pragma unroll
                        for (int k2 = 0; k2 < 8; ++k2) {
                            pp[k2] = pack_bf16x2(pf[2 * k2], pf[2 * k2 + 1]);
                            const float2 ds = __fmul2_rn(
                                make_float2(pf[2 * k2], pf[2 * k2 + 1]),
                                make_float2(__uint_as_float(rd[2 * k2]), __uint_as_float(rd[2 * k2 + 1])));
                            pd[k2] = pack_bf16x2(ds.x, ds.y);
                        }
                        tmem_st_x8(x, pp);
                        tmem_st_x8(x + 8, pd);
                        tmem_wait_st();
                        tc_fence_before();
                        mbar_arrive(&bars->ds_ready[p]);
                    }
                    return true;
                };
                if (!(ucode >= 0 ? chunk(std::true_type()) : chunk(std::false_type()))) {
                    ok = false;
                    break;
                }
            }
            if (!ok) break;
            mbar_arrive(&bars->q_empty[ks]);
          }
          if (!ok) break;
          // the segment's last products are complete: its dk and dv
          if (!mbar_wait(&bars->done, seg & 1, abort_flag, kWaitNs)) { ok = false; break; }
          tc_fence_after();
          epilogue(gb);
          if (!kBal || b >= ntiles) break;
          // the next group's K and V, then let the MMA warp on
          qb = 0;
          ++gb;
          if (tid < kBKV) {
              write_kv(gb);
              tmem_wait_st();
          }
          tc_fence_before();
          mbar_arrive(&bars->seg_ready);
          ++seg;
        }
        if (!ok) fail(abort_flag, status);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
    if (tid == 0) pdl_wait();   // complete after the kernel before, which this one may overlap
}


// First KV row whose dk and dv are summed in fp32 (then turned into bf16 by the
// caller), or -1 when there are none.  Groups that do not fill one wave of one
// CTA per SM all go through the sums (the balanced grid); past one wave, the
// groups after the last full wave do (the split tail).
int dkdv_tail_row0(int n, int tail, bool have_acc) {
    const int sms = num_sms();
    const int groups = 2 * ((n + kBKV - 1) / kBKV);
    if (tail <= 1 || !have_acc || groups % sms == 0) return -1;
    return groups < sms ? 0 : (groups / sms * sms / 2) * kBKV;
}

template <int HD>
int launch(int n, const void* q, const void* k, const void* v, const void* dO, const int8_t* spd,
           int64_t ld, const float* T, int nb, float scale, float fold_scale, const uint16_t* LB,
           int tail, void* dk, void* dv, float* dk_acc, float* dv_acc, cudaStream_t s) {
    using C = KvCfg<HD>;
    CUtensorMap mq, mg, ms, ml;
    const uint64_t cols = (uint64_t)kH * HD;
    if (!make_map_2d(&mq, const_cast<void*>(q), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n, cols, cols * 2,
                     C::BQ, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_2d(&mg, const_cast<void*>(dO), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n, cols, cols * 2,
                     C::BQ, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_2d(&ms, const_cast<int8_t*>(spd), CU_TENSOR_MAP_DATA_TYPE_UINT8, n, n, ld, C::BQ,
                     kBKV, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map_2d(&ml, const_cast<uint16_t*>(LB), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n, (uint64_t)kH * 16,
                     (uint64_t)kH * 16 * 2, C::BQ, 16, CU_TENSOR_MAP_SWIZZLE_32B))
        return GT_ERR_CUDA;
    if (cudaFuncSetAttribute(bwd_dkdv_kernel<HD, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM) != cudaSuccess ||
        cudaFuncSetAttribute(bwd_dkdv_kernel<HD, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM) != cudaSuccess)
        return GT_ERR_CUDA;
    int* status = device_status_ptr();
    if (!status) return GT_ERR_CUDA;
    const int total_tiles = (n + C::BQ - 1) / C::BQ;
    const int groups = 2 * ((n + kBKV - 1) / kBKV);
    // the launch may overlap the kernel before it (the dq kernel): it reads only
    // the inputs and the prep tables
    auto run = [&](dim3 grid, int g_first, int per, int bal, bool sums) -> int {
        LaunchScope ls("bwd_dkdv", s);
        auto kern = bal > 0 ? bwd_dkdv_kernel<HD, true> : bwd_dkdv_kernel<HD, false>;
        if (launch_overlapped(kern, grid, dim3(kThreads), C::SMEM, s, mq, mg, ms, ml,
                              static_cast<const __nv_bfloat16*>(k), static_cast<const __nv_bfloat16*>(v), T, nb, n,
                              scale, fold_scale * kLog2e, g_first, per, bal, static_cast<__nv_bfloat16*>(dk),
                              static_cast<__nv_bfloat16*>(dv), sums ? dk_acc : nullptr, sums ? dv_acc : nullptr,
                              status) != cudaSuccess)
            return GT_ERR_CUDA;
        return check_launch();
    };
    const int row0 = dkdv_tail_row0(n, tail, dk_acc != nullptr);
    if (row0 == 0 && groups < num_sms()) {
        // fewer groups than SMs: the balanced grid, one CTA per SM, each an equal
        // share of the (group, Q tile) steps (the bucket matrix of such a graph
        // stays in L2 for the second head half's reads); the caller cleared the
        // sums before and turns them into bf16 after
        const int64_t steps = (int64_t)groups * total_tiles;
        const int ctas = (int)(steps < num_sms() ? steps : num_sms());
        return run(dim3(ctas), 0, 0, ctas, true);
    }
    if (row0 >= 0) {
        // full waves of whole groups, then the remaining groups split tail ways
        // over the SMs: the split CTAs are scheduled as SMs free up, which also
        // absorbs the uneven end of the dq kernel this launch overlaps (equal
        // static shares measured slower here)
        const int g1 = (row0 / kBKV) * 2;
        const int rc = run(dim3(g1), 0, 0, 0, false);
        if (rc != GT_OK) return rc;
        const int per = (total_tiles + tail - 1) / tail;
        return run(dim3(groups - g1, 1, (total_tiles + per - 1) / per), g1, per, 0, true);
    }
    return run(dim3(groups), 0, 0, 0, false);
}

}  // namespace

int bwd_dkdv_tail_row0(int n, int tail, bool have_acc) { return dkdv_tail_row0(n, tail, have_acc); }

int launch_bwd_dkdv(int n, int d, const void* q, const void* k, const void* v, const void* dO,
                    const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                    const uint16_t* LB, int tail, void* dk, void* dv, float* dk_acc, float* dv_acc,
                    cudaStream_t s) {
    // LB holds -lse / fold_scale with fold_scale = scale, or a tiny stand-in for a
    // zero scale; dk takes the true scale
    const float fold_scale = (scale == 0.f || !isfinite(scale)) ? 1e-30f : scale;
    return d == 8 ? launch<8>(n, q, k, v, dO, spd, ld, T, nb, scale, fold_scale, LB, tail, dk, dv, dk_acc,
                              dv_acc, s)
                  : launch<16>(n, q, k, v, dO, spd, ld, T, nb, scale, fold_scale, LB, tail, dk, dv, dk_acc,
                               dv_acc, s);
}

// How the dk/dv kernel fills the SMs: 1 when whole groups fill whole waves of
// one CTA per SM; 2 when the groups do not fill one wave (the balanced grid);
// otherwise the query-range split of the groups past the last full wave: the k
// in [2, 8] that makes the last waves the shortest, in units of one group's
// time, or 1 when no k beats one more wave of whole groups.
int bwd_dkdv_tail_split(int n) {
    const int sms = num_sms();
    const int groups = 2 * ((n + kBKV - 1) / kBKV);
    if (groups % sms == 0) return 1;
    if (groups < sms) return 2;
    const int rem = groups % sms;
    int best = 1;
    double best_t = 1.0;                        // the tail unsplit: one more wave of whole groups
    for (int k = 2; k <= 8; ++k) {
        const double t = (double)((rem * k + sms - 1) / sms) / k;
        if (t < best_t - 1e-9) { best_t = t; best = k; }
    }
    return best;
}

}  // namespace gt

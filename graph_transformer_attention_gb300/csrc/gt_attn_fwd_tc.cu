// gt_attn_fwd_tc.cu -- tensor-core forward of topology-biased graph attention
// (bf16 storage, H = 8 heads, head dim 8 or 16) for sm_103a.
//
// Blockwise form of the MegaGraph paper's Fig. 4: KV blocks of 64 nodes stream
// past a tile of 128 query rows; with each KV block comes the matching
// 128 x 64 slice of the int8 bucket matrix, and the bias b = T[h][code] is formed
// in registers from it.  Neither the scores nor the bias are ever stored.
//
// One CTA = one tile of 128 query rows and one half of the heads (4 of 8:
// grid.z); two CTAs share an SM, so one's softmax runs while the other waits on
// its tensor-core products.  192 threads:
//   warps 0-3  thread r owns query row r (TMEM lane r).  Per chunk of 32 KV
//              columns it reads S of the 4 heads from TMEM, gathers the 4 head
//              biases of each (i, j) with one 16-byte shared load per bucket byte,
//              exponentiates in base 2, writes P (bf16) to TMEM and keeps the row
//              sums.  When every row of the warp has 16 equal codes in a half chunk
//              (a warp vote), each head takes one bias and x - m is formed with one
//              packed fused multiply-add per two columns.
//   warp 4     MMA issuer: S_h = Q_h K_h^T (M=128, N=32, K=16) into TMEM, then
//              O_h += P_h V_h (A = P from TMEM, M=128, N=16, two K=16 steps).
//   warp 5     TMA producer: the bucket tile (128x64 int8, 64B swizzle) and the
//              K and V column slots (64 x 16 bf16, 32B swizzle) of each KV block,
//              double-buffered.
// TMEM (256 columns): O_h at 16h (64 columns), S for 4 heads x 32 columns at 64
// (128 columns), P (bf16) for 4 heads x 32 columns at 192 (64 columns).
// S is read into registers at the start of a chunk, so the next chunk's QK^T
// starts while this chunk is still being exponentiated.  Head dim 8 uses the
// 16-wide MMAs with the neighbouring head's channels riding along: Q is
// zero-padded per head so the extra K products vanish, and the extra output
// columns of O are ignored.
//
// Softmax statistics: the running maximum m is raised lazily.  P = 2^(x - m)
// is formed against the current m and a chunk is redone against a new maximum
// only when its row sum exceeds 2^8 (or is not finite); O is then rescaled in
// TMEM.  The first chunk sets m exactly.
//
// Every mbarrier wait is bounded; on timeout the CTA records GT_ERR_TIMEOUT in
// the device status word, all roles leave their loops, wait (bounded) for their
// own copies and MMAs in flight, free TMEM and return.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gt_common.cuh"
#include "gt_stats.cuh"
#include "gt_sm100.cuh"
#include "gt_tc_common.cuh"
#include "gt_tma.cuh"

namespace gt {
namespace {

using namespace sm100;
using namespace tc;

constexpr int kHC = 4;                  // heads per CTA
constexpr int kCtasPerSm = 2;
constexpr int kHalves = kH / kHC;       // head groups: tasks per query tile
constexpr int kBQ = 128;
constexpr int kBKV = 64;
constexpr int kCH = 32;                 // KV columns per MMA chunk
constexpr int kNCH = kBKV / kCH;
constexpr int kKVST = 2;
constexpr uint32_t kTmemCols = 64 * kHC;
constexpr int kNH = 2;                  // heads per softmax thread
constexpr int kSoftThreads = 128 * kHC / kNH;
constexpr int kThreads = kSoftThreads + 64;
constexpr int kMmaWarp = kSoftThreads / 32;
constexpr int kTmaWarp = kMmaWarp + 1;
constexpr float kRedoSum = 256.f;       // 2^8: redo a half chunk whose row sum exceeds this
constexpr uint32_t kColO = 0;                       // O: 16 columns per head
constexpr uint32_t kColS = 16 * kHC;                // S: 32 columns per head
constexpr uint32_t kColP = 16 * kHC + 32 * kHC;     // P (bf16 pairs): 16 columns per head

template <int HD>
struct Cfg {
    static constexpr int NSLOT = kHC * HD / 16;        // 16-column slots of this CTA's heads
    static constexpr uint32_t Q_BYTES = kHC * kBQ * 32;
    static constexpr uint32_t SPD_BYTES = kBQ * kBKV;
    static constexpr uint32_t SLOT_BYTES = kBKV * 32;
    static constexpr uint32_t STAGE_BYTES = SPD_BYTES + 2 * NSLOT * SLOT_BYTES;
    static constexpr uint32_t OFF_Q = 0;                  // Q of the first piece
    static constexpr uint32_t OFF_Q2 = Q_BYTES;           // Q of the second piece (balanced grid)
    static constexpr uint32_t OFF_STAGE = 2 * Q_BYTES;
    static constexpr uint32_t OFF_T = OFF_STAGE + kKVST * STAGE_BYTES;
    static constexpr uint32_t T_BYTES = 256 * kH * 4;
    static constexpr uint32_t OFF_BAR = OFF_T + T_BYTES;
    static constexpr uint32_t SMEM = OFF_BAR + 256 + 1024;   // + slack to align the base
};

struct Bars {
    uint64_t kv_full[kKVST];
    uint64_t kv_empty[kKVST];
    uint64_t s_full;
    uint64_t s_free;
    uint64_t p_ready;
    uint64_t pv_done;
    uint64_t fin;
    uint32_t tmem_base;
    int abort;
};

__device__ __forceinline__ void fail(Bars* bars, int* status) {
    *(volatile int*)&bars->abort = 1;
    atomicOr(status, kStatusTimeout);
}

__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

// One stretch of a CTA's work: query tile i0, head half hb, KV columns
// [j_begin, j_end) in nblocks blocks.  part < 0: the stretch is the task's whole
// KV range and its rows go to o and lse; else they go to partial slot `part`.
struct Seg {
    int i0, hb, j_begin, j_end, nblocks, part;
};

// Stretch si of this CTA.  Plain grid (bl.ctas == 0): one stretch, tile
// blockIdx.x, head half blockIdx.z, KV split blockIdx.y of kv_block columns.
// Balanced grid: task = head half * tiles + tile, nblk blocks of kBKV columns.
__device__ __forceinline__ bool seg_of(const Balance& bl, int si, int kv_begin, int kv_end, int kv_block,
                                       int parts, Seg& sg) {
    if (bl.ctas == 0) {
        if (si > 0) return false;
        sg.i0 = blockIdx.x * kBQ;
        sg.hb = blockIdx.z;
        sg.j_begin = kv_begin + (kv_block > 0 ? (int)blockIdx.y * kv_block : 0);
        sg.j_end = kv_block > 0 ? min(kv_end, sg.j_begin + kv_block) : kv_end;
        sg.nblocks = (sg.j_end - sg.j_begin + kBKV - 1) / kBKV;
        sg.part = parts ? (int)blockIdx.y : -1;
        return true;
    }
    Piece p;
    const int bl_share = bl.share_of(blockIdx.x);
    if (!piece_of(bl, bl_share, si, p)) return false;
    const int tiles = bl.tasks / kHalves;
    sg.i0 = (p.task % tiles) * kBQ;
    sg.hb = p.task / tiles;
    sg.j_begin = kv_begin + p.b0 * kBKV;
    sg.j_end = min(kv_end, kv_begin + p.b1 * kBKV);
    sg.nblocks = p.b1 - p.b0;
    sg.part = (p.b0 == 0 && p.b1 == bl.nblk) ? -1 : 2 * bl_share + si;
    return true;
}

// x = s * scale * log2(e) + T[h][code] * log2(e) for 4 heads and the 16 columns of
// half g of a chunk, in place over the raw S bits; one 16-byte load per code
// gives the four head biases (tbl: shared address of this head group's half of
// the first 32-byte table row).
template <int NH>
__device__ __forceinline__ void load_bias(uint32_t addr, float (&b)[NH]) {
    if constexpr (NH == 4) {
        const float4 v = lds_f4(addr);
        b[0] = v.x; b[1] = v.y; b[2] = v.z; b[3] = v.w;
    } else {
        const float2 v = lds_f2(addr);
        b[0] = v.x; b[1] = v.y;
    }
}

template <int NH>
__device__ __forceinline__ void score16(uint32_t (&sx)[NH][16], const uint4 cw, uint32_t tbl,
                                        float scale_log2) {
    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const uint32_t code = __byte_perm(w[k >> 2], 0u, 0x4440u + (k & 3));
        float bv[NH];
        load_bias<NH>(tbl + code * 32u, bv);
#pragma unroll
        for (int hh = 0; hh < NH; ++hh)
            sx[hh][k] = __float_as_uint(fmaf(__uint_as_float(sx[hh][k]), scale_log2, bv[hh]));
    }
}

// Columns at or beyond j_end (the tail of the last KV block) get x = -inf.
template <int NH>
__device__ __forceinline__ void mask16(uint32_t (&sx)[NH][16], int j, int j_end) {
#pragma unroll
    for (int k = 0; k < 16; ++k)
        if (j + k >= j_end) {
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) sx[hh][k] = __float_as_uint(-INFINITY);
        }
}

// p_k = 2^(x_k - m) for one head's 16 columns, packed to bf16 pairs; returns sum p.
// (two partial sums keep the dependent chain short)
__device__ __forceinline__ float exp_pack16(const uint32_t (&x)[16], float m, uint32_t (&pk)[8]) {
    float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
    const float2 mm = f2(-m, -m);
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
        const float2 d = __fadd2_rn(f2(__uint_as_float(x[k]), __uint_as_float(x[k + 1])), mm);
        const float2 p = f2(ex2(d.x), ex2(d.y));
        if (k & 2) acc1 = __fadd2_rn(acc1, p);
        else acc0 = __fadd2_rn(acc0, p);
        pk[k / 2] = pack_bf16x2(p.x, p.y);
    }
    const float2 acc = __fadd2_rn(acc0, acc1);
    return acc.x + acc.y;
}

// Rows whose 16 codes of a half chunk are all equal (in every row of the warp):
// x - m = s * scale * log2(e) + (b - m) in one packed fused multiply-add per two
// columns, the head's bias minus its running maximum taken once.
template <int NH>
__device__ __forceinline__ void score16_shifted(uint32_t (&sx)[NH][16], const float (&bb)[NH], const float (&m)[NH],
                                                float scale_log2) {
    const float2 cc = f2(scale_log2, scale_log2);
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        const float bm = bb[hh] - m[hh];
        const float2 bm2 = f2(bm, bm);
#pragma unroll
        for (int k = 0; k < 16; k += 2) {
            const float2 x = __ffma2_rn(f2(__uint_as_float(sx[hh][k]), __uint_as_float(sx[hh][k + 1])), cc, bm2);
            sx[hh][k] = __float_as_uint(x.x);
            sx[hh][k + 1] = __float_as_uint(x.y);
        }
    }
}

// p_k = 2^(x_k) for x already shifted by the running maximum; returns sum p.
__device__ __forceinline__ float exp_pack16_shifted(const uint32_t (&x)[16], uint32_t (&pk)[8]) {
    float2 acc0 = f2(0.f, 0.f), acc1 = f2(0.f, 0.f);
#pragma unroll
    for (int k = 0; k < 16; k += 2) {
        const float2 p = f2(ex2(__uint_as_float(x[k])), ex2(__uint_as_float(x[k + 1])));
        if (k & 2) acc1 = __fadd2_rn(acc1, p);
        else acc0 = __fadd2_rn(acc0, p);
        pk[k / 2] = pack_bf16x2(p.x, p.y);
    }
    const float2 acc = __fadd2_rn(acc0, acc1);
    return acc.x + acc.y;
}

template <int HD>
__global__ void __launch_bounds__(kThreads, kCtasPerSm)
fwd_tc_kernel(const __grid_constant__ CUtensorMap mapK, const __grid_constant__ CUtensorMap mapV,
              const __grid_constant__ CUtensorMap mapS, const __nv_bfloat16* __restrict__ q,
              const float* __restrict__ T, int nb, int n, float scale_log2, int kv_begin, int kv_end,
              int kv_block, int parts, __nv_bfloat16* __restrict__ o, float* __restrict__ lse,
              float* __restrict__ o_part,
              float* __restrict__ lse_part, const Balance bal, int* status) {
    using C = Cfg<HD>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    Bars* bars = reinterpret_cast<Bars*>(smem + C::OFF_BAR);
    float* Ts = reinterpret_cast<float*>(smem + C::OFF_T);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_trigger();   // the merge may launch meanwhile; it waits for this grid before reading
    // this CTA's one or two stretches (heads kHC hb .. kHC hb + kHC - 1 of each)
    // (recomputed from the parameters where needed: kept in registers they would
    // be live across the whole softmax loop)
    auto seg = [&](int si) {
        Seg sg{0, 0, 0, 0, 0, -1};
        seg_of(bal, si, kv_begin, kv_end, kv_block, parts, sg);
        return sg;
    };
    const int nblocks0 = seg(0).nblocks;
    const int nblocks1 = seg(1).nblocks;
    const int nseg = nblocks1 > 0 ? 2 : 1;
    const int nblocks = nblocks0 + nblocks1;
    const int nchunks0 = nblocks0 * kNCH;
    const int nchunks = nblocks * kNCH;

    if (tid == kTmaWarp * 32) {
        for (int s = 0; s < kKVST; ++s) {
            mbar_init(&bars->kv_full[s], 1);
            mbar_init(&bars->kv_empty[s], kSoftThreads + 1);
        }
        mbar_init(&bars->s_full, 1);
        mbar_init(&bars->s_free, kSoftThreads);
        mbar_init(&bars->p_ready, kSoftThreads);
        mbar_init(&bars->pv_done, 1);
        mbar_init(&bars->fin, 1);
        bars->abort = 0;
        fence_barrier_init();
        tma_prefetch_desc(&mapK);
        tma_prefetch_desc(&mapV);
        tma_prefetch_desc(&mapS);
    }
    if (warp == kMmaWarp) tmem_alloc(&bars->tmem_base, kTmemCols);
    // bias table in base-2 units, one 32-byte row of 8 heads per bucket code
    for (int x = tid; x < 256 * kH; x += kThreads) {
        const int code = x / kH, h = x % kH;
        Ts[x] = code < nb ? T[h * nb + code] * kLog2e : 0.f;
    }
    // per-head Q operands of this CTA's heads: [128 rows][16] bf16, 32-byte swizzle, K-major
    // (threads 0-127 the first stretch's tile, 128-255 the second's)
    if (tid < kBQ || (nseg > 1 && tid < 2 * kBQ)) {
        const Seg sg = seg(tid < kBQ ? 0 : 1);
        const int rr = tid & (kBQ - 1);
        const int row = sg.i0 + rr;
        const bool live = row < n;
        write_head_operands<HD, kHC>(smem + (tid < kBQ ? C::OFF_Q : C::OFF_Q2), rr,
                                     q + (int64_t)(live ? row : 0) * kH * HD, live, kHC * sg.hb);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = bars->tmem_base;
    volatile int* abort_flag = &bars->abort;

    if (warp == kTmaWarp) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;
            for (int b = 0; b < nblocks; ++b) {
                const int ks = b & 1;
                if (b >= kKVST &&
                    !mbar_wait(&bars->kv_empty[ks], ((b >> 1) - 1) & 1, abort_flag, kWaitNs)) {
                    fail(bars, status);
                    break;
                }
                const bool second = b >= nblocks0;
                const Seg sg = seg(second ? 1 : 0);
                const int i0 = sg.i0;
                const int hb = sg.hb;
                uint8_t* st = smem + C::OFF_STAGE + ks * C::STAGE_BYTES;
                const int j0 = sg.j_begin + (b - (second ? nblocks0 : 0)) * kBKV;
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
            if (*abort_flag) {
                // let the copies already issued land before the CTA goes away
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
            const uint32_t idQK = idesc_bf16(128, kCH, false, false);
            const uint32_t idPV = idesc_bf16(128, 16, false, true);
            const uint32_t stage_base = smem_u32(smem + C::OFF_STAGE);
            const SmemDesc dQ = smem_desc_split(smem_u32(smem + C::OFF_Q), 16, 256, 6);
            const SmemDesc dQ2 = smem_desc_split(smem_u32(smem + C::OFF_Q2), 16, 256, 6);
            const SmemDesc dKk = smem_desc_split(stage_base + C::SPD_BYTES, 16, 256, 6);     // K-major K
            const SmemDesc dVm = smem_desc_split(stage_base + C::SPD_BYTES, 256, 256, 6);    // MN-major V
            bool ok = true;
            // chunk tt covers KV rows 32c .. 32c+31 of block b: 1024 bytes into a slot
            auto koff = [&](int tt) -> uint32_t {
                const int b = tt / kNCH, c = tt % kNCH;
                return (uint32_t)((b & 1) * C::STAGE_BYTES + c * 1024);
            };
            auto issue_qk = [&](int tt) -> bool {
                const int b = tt / kNCH, c = tt % kNCH, ks = b & 1;
                if (c == 0 && !mbar_wait_all(&bars->kv_full[ks], (b >> 1) & 1, abort_flag, kWaitNs))
                    return false;
                if (tt > 0 && !mbar_wait_all(&bars->s_free, (tt - 1) & 1, abort_flag, kWaitNs))
                    return false;
                tc_fence_after();
                if (elect_one()) {
#pragma unroll
                    for (int h = 0; h < kHC; ++h) {
                        const int slot = h * HD / 16;
                        mma_ss(tbase + kColS + kCH * h, desc_at(tt < nchunks0 ? dQ : dQ2, h * 4096),
                               desc_at(dKk, koff(tt) + slot * C::SLOT_BYTES), idQK, 0);
                    }
                    mma_commit(&bars->s_full);
                }
                __syncwarp();
                return true;
            };
            ok = issue_qk(0);
            for (int tt = 0; ok && tt < nchunks; ++tt) {
                const int b = tt / kNCH, c = tt % kNCH, ks = b & 1;
                if (tt + 1 < nchunks && !issue_qk(tt + 1)) { ok = false; break; }
                if (!mbar_wait_all(&bars->p_ready, tt & 1, abort_flag, kWaitNs)) { ok = false; break; }
                tc_fence_after();
                const uint32_t voff = koff(tt) + C::NSLOT * C::SLOT_BYTES;
                if (elect_one()) {
#pragma unroll
                    for (int h = 0; h < kHC; ++h) {
                        const int slot = h * HD / 16;
#pragma unroll
                        for (int st = 0; st < 2; ++st)
                            mma_ts(tbase + kColO + 16 * h, tbase + kColP + 16 * h + 8 * st,
                                   desc_at(dVm, voff + slot * C::SLOT_BYTES + 512 * st), idPV,
                                   ((tt != 0 && tt != nchunks0) || st > 0) ? 1u : 0u);
                    }
                    mma_commit(&bars->pv_done);
                    if (c == kNCH - 1) mma_commit(&bars->kv_empty[ks]);
                }
                __syncwarp();
            }
            if (!ok) {
                fail(bars, status);
                int never = 0;
                if (elect_one()) mma_commit(&bars->fin);
                __syncwarp();
                mbar_wait_all(&bars->fin, 0, &never, kWaitNs);
            }
        }
    } else {
        // ------------------------------------------------------- softmax
        // warps w and w + 4 own the same 32 query rows (TMEM lanes) and split the
        // CTA's heads: thread (r, half) takes heads 2 half, 2 half + 1
        const int r = tid & (kBQ - 1);           // row within the tile = TMEM lane
        const int hl0 = kNH * (tid >> 7);        // this thread's first head among the CTA's
        const uint32_t lrow = tbase + ((uint32_t)((warp & 3) * 32) << 16);
        int t = 0;   // chunks so far (kNCH per KV block): the mbarrier phases
        bool ok = true;
        for (int si = 0; ok && si < nseg; ++si) {
            uint32_t tbl;    // 32-byte rows of 8 head biases
            int jb, je, nbs;  // the stretch's KV columns [jb, je) in nbs blocks
            {
                const Seg sg = seg(si);
                tbl = smem_u32(Ts) + 4u * (kHC * sg.hb + hl0);
                jb = sg.j_begin;
                je = sg.j_end;
                nbs = sg.nblocks;
            }
            float m[kNH], l[kNH];
#pragma unroll
            for (int h = 0; h < kNH; ++h) { m[h] = -INFINITY; l[h] = 0.f; }
            const int t0 = t;    // the stretch's first chunk
            int uni_skip = 0;    // half chunks left before the next uniformity vote (warp-uniform)
            for (int b = 0; ok && b < nbs; ++b) {
                const int bg = t / kNCH;   // KV blocks so far
                const int ks = bg & 1;
                if (!mbar_wait(&bars->kv_full[ks], (bg >> 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
                const uint32_t sp = smem_u32(smem + C::OFF_STAGE + ks * C::STAGE_BYTES) + r * kBKV;
                const int j0 = jb + b * kBKV;
                const bool tail_block = j0 + kBKV > je;
                for (int c = 0; c < kNCH; ++c, ++t) {
                    if (!mbar_wait(&bars->s_full, t & 1, abort_flag, kWaitNs)) { ok = false; break; }
                    tc_fence_after();
                    // codes of the 32 columns: two 16-byte chunks of the row (64-byte swizzle)
                    const uint32_t swz = (uint32_t)((r >> 1) & 3);
                    const uint4 c0 = lds_u4(sp + (((uint32_t)(2 * c) ^ swz) << 4));
                    const uint4 c1 = lds_u4(sp + (((uint32_t)(2 * c + 1) ^ swz) << 4));
                    const int jc = j0 + c * kCH;
                    if (t == t0) {
                        // the first chunk sets the running maximum exactly (both halves)
    #pragma unroll
                        for (int g = 0; g < 2; ++g) {
                            uint32_t sx[kNH][16];
    #pragma unroll
                            for (int hh = 0; hh < kNH; ++hh)
                                tmem_ld_x16(lrow + kColS + kCH * (hl0 + hh) + 16 * g, sx[hh]);
                            tmem_wait_ld();
                            score16<kNH>(sx, g ? c1 : c0, tbl, scale_log2);
                            if (tail_block) mask16<kNH>(sx, jc + 16 * g, je);
    #pragma unroll
                            for (int hh = 0; hh < kNH; ++hh)
    #pragma unroll
                                for (int k = 0; k < 16; ++k) m[hh] = fmaxf(m[hh], __uint_as_float(sx[hh][k]));
                        }
                    }
                    // P and O must not be touched before the previous chunk's PV is done with
                    // them; the wait is put off until the first write, so that the S loads and
                    // the first half's exponentials overlap that PV
                    bool pv_waited = t == t0;
                    auto wait_pv = [&]() {
                        if (pv_waited) return;
                        if (!mbar_wait(&bars->pv_done, (t - 1) & 1, abort_flag, kWaitNs)) ok = false;
                        tc_fence_after();
                        pv_waited = true;
                    };
    #pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        uint32_t sx[kNH][16];
    #pragma unroll
                        for (int hh = 0; hh < kNH; ++hh)
                            tmem_ld_x16(lrow + kColS + kCH * (hl0 + hh) + 16 * g, sx[hh]);
                        tmem_wait_ld();
                        if (g == 1) {
                            tc_fence_before();
                            mbar_arrive(&bars->s_free);      // S is consumed: the next QK^T may start
                        }
                        // exponentials of all heads first (independent chains), one vote on
                        // whether any head of any row needs a redo against a new maximum
                        uint32_t pk[kNH][8];
                        float ls[kNH];
                        bool need = false;
                        const uint4 cw = g ? c1 : c0;
                        const uint32_t code0 = cw.x & 0xffu;
                        bool wuni = false;
                        if (uni_skip > 0) {
                            --uni_skip;
                        } else if (t > t0) {
                            const bool uni = cw.x == code0 * 0x01010101u && cw.y == cw.x && cw.z == cw.x && cw.w == cw.x;
                            wuni = __all_sync(0xffffffffu, uni);
                            // after a failed vote the warp votes again 16 half chunks (256
                            // columns) later: where codes are mixed the vote seldom succeeds, and
                            // the mixed columns of a graph of small components come in runs
                            if (!wuni) uni_skip = 16;
                        }
                        if (wuni) {
                            float bb[kNH];
                            load_bias<kNH>(tbl + code0 * 32u, bb);
                            score16_shifted<kNH>(sx, bb, m, scale_log2);
                            if (tail_block) mask16<kNH>(sx, jc + 16 * g, je);
    #pragma unroll
                            for (int hh = 0; hh < kNH; ++hh) {
                                ls[hh] = exp_pack16_shifted(sx[hh], pk[hh]);
                                need |= !(ls[hh] <= kRedoSum);
                            }
                        } else {
                            score16<kNH>(sx, g ? c1 : c0, tbl, scale_log2);
                            if (tail_block) mask16<kNH>(sx, jc + 16 * g, je);
    #pragma unroll
                            for (int hh = 0; hh < kNH; ++hh) {
                                ls[hh] = exp_pack16(sx[hh], m[hh], pk[hh]);
                                need |= !(ls[hh] <= kRedoSum);
                            }
                        }
                        if (__any_sync(0xffffffffu, need)) {
                            wait_pv();
    #pragma unroll
                            for (int hh = 0; hh < kNH; ++hh) {
                                if (!__any_sync(0xffffffffu, !(ls[hh] <= kRedoSum))) continue;
                                // a new maximum for this head: redo, and rescale l, the P already
                                // written for this chunk, and O (TMEM columns hold this CTA's heads)
                                // (x of a uniform step is already shifted by m: its new maximum is
                                // m + the largest shifted x above 0)
                                float mx = wuni ? 0.f : m[hh];
    #pragma unroll
                                for (int k = 0; k < 16; ++k) mx = fmaxf(mx, __uint_as_float(sx[hh][k]));
                                const float alpha = wuni ? ex2(-mx) : ex2(m[hh] - mx);
                                m[hh] = wuni ? m[hh] + mx : mx;
                                l[hh] *= alpha;
                                ls[hh] = exp_pack16(sx[hh], mx, pk[hh]);
                                if (g == 1) {
                                    uint32_t pw[8];
                                    tmem_wait_st();   // the first half's P of this head is written
                                    tmem_ld_x8(lrow + kColP + 16 * (hl0 + hh), pw);
                                    tmem_wait_ld();
    #pragma unroll
                                    for (int k = 0; k < 8; ++k)
                                        pw[k] = pack_bf16x2(__uint_as_float(pw[k] << 16) * alpha,
                                                            __uint_as_float(pw[k] & 0xffff0000u) * alpha);
                                    tmem_st_x8(lrow + kColP + 16 * (hl0 + hh), pw);
                                }
                                if (t > t0) {
                                    uint32_t ov[16];
                                    tmem_ld_x16(lrow + kColO + 16 * (hl0 + hh), ov);
                                    tmem_wait_ld();
    #pragma unroll
                                    for (int k = 0; k < 16; ++k) ov[k] = __float_as_uint(__uint_as_float(ov[k]) * alpha);
                                    tmem_st_x16(lrow + kColO + 16 * (hl0 + hh), ov);
                                }
                            }
                        }
                        wait_pv();
    #pragma unroll
                        for (int hh = 0; hh < kNH; ++hh) {
                            l[hh] += ls[hh];
                            tmem_st_x8(lrow + kColP + 16 * (hl0 + hh) + 8 * g, pk[hh]);
                        }
                    }
                    tmem_wait_st();
                    tc_fence_before();
                    mbar_arrive(&bars->p_ready);
                    if (!ok) break;
                }
                if (!ok) break;
                mbar_arrive(&bars->kv_empty[ks]);
            }
            if (!ok) break;
            // ------------------------------------------ epilogue of the stretch
            // (the next stretch's first PV overwrites O only after every thread's
            // p_ready of that chunk, which follows these reads)
            if (!mbar_wait(&bars->pv_done, (t - 1) & 1, abort_flag, kWaitNs)) { ok = false; break; }
            tc_fence_after();
            const Seg sg = seg(si);
            const int row = sg.i0 + r;
            const bool live = row < n;
#pragma unroll
            for (int hh = 0; hh < kNH; ++hh) {
                const int h = kHC * sg.hb + hl0 + hh;
                uint32_t ov[16];
                tmem_ld_x16(lrow + kColO + 16 * (hl0 + hh), ov);
                tmem_wait_ld();
                const float inv = 1.f / l[hh];
                const int c0 = (HD == 8) ? (h & 1) * 8 : 0;
                const float lse_v = (m[hh] + log2f(l[hh])) * kLn2;
                if (!live) continue;
                if (sg.part < 0) {
                    uint32_t w[HD / 2];
#pragma unroll
                    for (int k = 0; k < HD / 2; ++k)
                        w[k] = pack_bf16x2(__uint_as_float(ov[c0 + 2 * k]) * inv,
                                           __uint_as_float(ov[c0 + 2 * k + 1]) * inv);
                    uint4* dst = reinterpret_cast<uint4*>(o + ((int64_t)row * kH + h) * HD);
#pragma unroll
                    for (int k = 0; k < HD / 8; ++k)
                        dst[k] = make_uint4(w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
                    lse[(int64_t)h * n + row] = lse_v;
                } else {
                    // KV-split partials: [split][n][8][HD] and [split][8][n]; balanced
                    // pieces: slot [128 rows][4 heads][HD] and [4 heads][128 rows]
                    const int64_t oo = bal.ctas == 0 ? (((int64_t)sg.part * n + row) * kH + h) * HD
                                                     : (((int64_t)sg.part * kBQ + r) * kHC + hl0 + hh) * HD;
                    const int64_t lo = bal.ctas == 0 ? ((int64_t)sg.part * kH + h) * n + row
                                                     : ((int64_t)sg.part * kHC + hl0 + hh) * kBQ + r;
                    float4* dst = reinterpret_cast<float4*>(o_part + oo);
#pragma unroll
                    for (int k = 0; k < HD / 4; ++k)
                        dst[k] = make_float4(__uint_as_float(ov[c0 + 4 * k]) * inv,
                                             __uint_as_float(ov[c0 + 4 * k + 1]) * inv,
                                             __uint_as_float(ov[c0 + 4 * k + 2]) * inv,
                                             __uint_as_float(ov[c0 + 4 * k + 3]) * inv);
                    lse_part[lo] = lse_v;
                }
            }
        }
        if (!ok) fail(bars, status);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tbase, kTmemCols);
    }
}

}  // namespace
}  // namespace gt

namespace gt {
namespace {

constexpr int kMinBlocks = 8;   // shortest balanced share: 8 KV blocks (512 columns)

Balance balance_for(int n) {
    return balance_grid((n + kBQ - 1) / kBQ, kHalves, (n + kBKV - 1) / kBKV, kCtasPerSm, kMinBlocks);
}

// Rows of the tasks that more than one CTA took: the pieces' normalised outputs
// and log-sum-exps combined exactly, o = sum_k e^(lse_k - M) o_k / sum_k e^(lse_k - M),
// lse = M + log sum_k e^(lse_k - M).  One thread per (row, head).
template <int HD>
__global__ void __launch_bounds__(256)
merge_pieces(const Balance bl, int n, const float* __restrict__ o_part, const float* __restrict__ lse_part,
             __nv_bfloat16* __restrict__ o, float* __restrict__ lse) {
    pdl_wait();   // launched to overlap the attention kernel's end: its partials are complete after this
    const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (int64_t)n * kH) return;
    const int row = (int)(idx / kH), h = (int)(idx % kH);
    const int tiles = bl.tasks / kHalves;
    const int r = row % kBQ, hl = h % kHC;
    const int64_t p0 = (int64_t)((h / kHC) * tiles + row / kBQ) * bl.nblk;
    const int c0 = bl.cta_of(p0), c1 = bl.cta_of(p0 + bl.nblk - 1);
    if (c0 == c1) return;   // one CTA took the whole task and wrote the row itself
    auto slot = [&](int c) { return 2 * c + ((c == c0 && bl.lo(c) < p0) ? 1 : 0); };
    float mx = -INFINITY;
    for (int c = c0; c <= c1; ++c) mx = fmaxf(mx, lse_part[((int64_t)slot(c) * kHC + hl) * kBQ + r]);
    float acc[HD];
#pragma unroll
    for (int k = 0; k < HD; ++k) acc[k] = 0.f;
    float wsum = 0.f;
    for (int c = c0; c <= c1; ++c) {
        const int sl = slot(c);
        const float w = __expf(lse_part[((int64_t)sl * kHC + hl) * kBQ + r] - mx);
        wsum += w;
        const float4* src = reinterpret_cast<const float4*>(o_part + (((int64_t)sl * kBQ + r) * kHC + hl) * HD);
#pragma unroll
        for (int k = 0; k < HD / 4; ++k) {
            const float4 v = src[k];
            acc[4 * k] += w * v.x;
            acc[4 * k + 1] += w * v.y;
            acc[4 * k + 2] += w * v.z;
            acc[4 * k + 3] += w * v.w;
        }
    }
    const float inv = 1.f / wsum;
    uint32_t pk[HD / 2];
#pragma unroll
    for (int k = 0; k < HD / 2; ++k) pk[k] = pack_bf16x2(acc[2 * k] * inv, acc[2 * k + 1] * inv);
    uint4* dst = reinterpret_cast<uint4*>(o + ((int64_t)row * kH + h) * HD);
#pragma unroll
    for (int k = 0; k < HD / 8; ++k) dst[k] = make_uint4(pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
    lse[(int64_t)h * n + row] = mx + __logf(wsum);
}

template <int HD>
int launch_fwd_tc(int n, const void* q, const void* k, const void* v, const int8_t* spd, int64_t ld,
                  const float* T, int nb, float scale, int kv_begin, int kv_end, int kv_block, int parts,
                  const Balance& bal, void* o, float* lse, float* o_part, float* lse_part, cudaStream_t s) {
    using C = Cfg<HD>;
    CUtensorMap mk, mv, ms;
    const uint64_t cols = (uint64_t)kH * HD;
    if (!make_map_2d(&mk, const_cast<void*>(k), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n, cols, cols * 2,
                     kBKV, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_2d(&mv, const_cast<void*>(v), CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, n, cols, cols * 2,
                     kBKV, 16, CU_TENSOR_MAP_SWIZZLE_32B) ||
        !make_map_2d(&ms, const_cast<int8_t*>(spd), CU_TENSOR_MAP_DATA_TYPE_UINT8, n, n, ld, kBQ,
                     kBKV, CU_TENSOR_MAP_SWIZZLE_64B))
        return GT_ERR_CUDA;
    if (cudaFuncSetAttribute(fwd_tc_kernel<HD>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)C::SMEM) != cudaSuccess)
        return GT_ERR_CUDA;
    int* status = device_status_ptr();
    if (!status) return GT_ERR_CUDA;
    const int nsplit = kv_block > 0 ? (kv_end - kv_begin + kv_block - 1) / kv_block : 1;
    const dim3 grid = bal.ctas > 0 ? dim3(bal.ctas) : dim3((n + kBQ - 1) / kBQ, nsplit, kHalves);
    {
        LaunchScope ls("fwd_tc", s);
        fwd_tc_kernel<HD><<<grid, kThreads, C::SMEM, s>>>(
            mk, mv, ms, static_cast<const __nv_bfloat16*>(q), T, nb, n, scale * kLog2e, kv_begin, kv_end,
            nsplit > 1 ? kv_block : 0, parts, static_cast<__nv_bfloat16*>(o), lse, o_part, lse_part, bal,
            status);
    }
    int rc = check_launch();
    if (rc != GT_OK || bal.ctas == 0) return rc;
    {
        LaunchScope ls("fwd_merge", s);
        const int64_t threads = (int64_t)n * kH;
        if (launch_overlapped(merge_pieces<HD>, dim3((unsigned)((threads + 255) / 256)), dim3(256), 0, s, bal, n,
                              (const float*)o_part, (const float*)lse_part, static_cast<__nv_bfloat16*>(o),
                              lse) != cudaSuccess)
            return GT_ERR_CUDA;
    }
    return check_launch();
}

}  // namespace

bool fwd_tc_supported(int h, int d) { return h == kH && (d == 8 || d == 16); }

int fwd_tc_balanced_ctas(int n) { return balance_for(n).ctas; }

// Floats of the balanced forward's partial slots (0: the plain grid needs none):
// two slots per CTA of [128 rows][4 heads][d] outputs and [4][128] log-sum-exps.
size_t fwd_tc_piece_floats(int n, int d) {
    const Balance bl = balance_for(n);
    return bl.ctas == 0 ? 0 : (size_t)2 * bl.ctas * kBQ * kHC * (d + 1);
}

int merge_partials(int dtype, int n, int h, int d, int nsplit, const float* o_part,
                   const float* lse_part, void* o, float* lse, cudaStream_t s);

// kv_block > 0: grid.y splits of kv_block columns merged by merge_partials;
// 0: the balanced grid, whose partial slots start at o_part (lse_part after
// the outputs: fwd_tc_piece_floats in all).
int attn_fwd_tc(int n, int d, const void* q, const void* k, const void* v, const int8_t* spd,
                int64_t ld, const float* T, int nb, float scale, int kv_block, void* o, float* lse,
                float* o_part, float* lse_part, cudaStream_t s) {
    const int nsplit = kv_block > 0 ? (n + kv_block - 1) / kv_block : 1;
    const int parts = nsplit > 1;
    Balance bal = parts ? Balance{0, 0, 0} : balance_for(n);
    if (bal.ctas > 0) {
        if (!o_part) return GT_ERR_WORKSPACE;
        lse_part = o_part + (size_t)2 * bal.ctas * kBQ * kHC * d;
    }
    int rc = d == 8 ? launch_fwd_tc<8>(n, q, k, v, spd, ld, T, nb, scale, 0, n, kv_block, parts, bal, o, lse,
                                       o_part, lse_part, s)
                    : launch_fwd_tc<16>(n, q, k, v, spd, ld, T, nb, scale, 0, n, kv_block, parts, bal, o, lse,
                                        o_part, lse_part, s);
    if (rc != GT_OK || nsplit == 1) return rc;
    return merge_partials(GT_BF16, n, kH, d, nsplit, o_part, lse_part, o, lse, s);
}

// Attention of every query row over the KV columns [kv_begin, kv_end) only:
// o_part [n][8][d] fp32 (normalised over those columns) and lse_part [8][n].
int attn_fwd_tc_range(int n, int d, const void* q, const void* k, const void* v, const int8_t* spd,
                      int64_t ld, const float* T, int nb, float scale, int kv_begin, int kv_end,
                      float* o_part, float* lse_part, cudaStream_t s) {
    const Balance none{0, 0, 0};
    return d == 8 ? launch_fwd_tc<8>(n, q, k, v, spd, ld, T, nb, scale, kv_begin, kv_end, 0, 1, none, nullptr,
                                     nullptr, o_part, lse_part, s)
                  : launch_fwd_tc<16>(n, q, k, v, spd, ld, T, nb, scale, kv_begin, kv_end, 0, 1, none, nullptr,
                                      nullptr, o_part, lse_part, s);
}

}  // namespace gt

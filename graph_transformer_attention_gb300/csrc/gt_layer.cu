// gt_layer.cu -- the GT encoder layer around the biased attention (width 64 =
// 8 heads x 8 channels, FFN width 64: the model of the MegaGraph paper's Fig. 8),
// forward and backward:
//
//   u = LN1(x); [q|k|v] = u W_qkv + b_qkv; o = A(q, k, v); hh = x + o W_o + b_o;
//   z = LN2(hh); a = z W_1 + b_1; y = hh + GELU(a) W_2 + b_2
//
// (LayerNorm before each sublayer, GELU(a) = a Phi(a): the Graphormer encoder
// layer; the pages give the widths, not the order of the steps.)
//
// Four tile kernels, one CTA of 256 threads per 128 node rows; row r of the tile
// is TMEM lane r, and threads r and r + 128 (warps w and w + 4, which reach the
// same lanes) each take half of its 64 features.  Every product with a layer
// matrix is a tcgen05.mma (M = 128 node rows): the activation rows go into TMEM
// as the A operand (tf32, fp32 storage), the matrix sits in shared memory as the
// B operand, the fp32 accumulator comes back with tcgen05.ld, and the threads do
// the LayerNorms (row sums passed between the two halves), GELU, residuals and
// the LayerNorm backward in registers.  Tiles of node rows and the weight
// matrices move between global and shared memory as whole-tile bulk copies on
// the TMA engine:
//   layer_ln_qkv    x -> LN1 -> u W_qkv + b -> q, k, v (bf16, the attention's inputs)
//   layer_out_ffn   o, x -> hh -> LN2 -> FFN -> y
//   layer_ffn_bwd   dy, and hh, z, a, GELU(a) recomputed from x and o -> dO for
//                   the attention backward (bf16) and d(hh); dW_2, dW_1, dW_o and
//                   their biases, dLN2
//   layer_qkv_bwd   dq, dk, dv, d(hh), and u recomputed from x -> dx; dW_qkv,
//                   db_qkv, dLN1
// Weight gradients are products over the node rows: each backward kernel writes
// the row vectors it needs transposed (features x node rows, bf16) into shared
// memory, and one bf16 MMA per 16 rows forms features x features sums in TMEM,
// two matrices per product (the M = 128 rows of A are two stacked 64-feature
// vectors).  A row of ones stacked under a vector gives its column sums (the
// bias and LayerNorm-shift gradients) in the same product.  The LayerNorm
// gains fold out: with z = zh g + s, sum_r z_i d_j = g_i sum_r zh_i d_j + s_i
// sum_r d_j, so the products take the normalised zh (whose diagonal with dz
// is the gain gradient).  Each CTA stores its sums in its own row of a partials
// buffer, which reduce_partials adds up in a fixed order (deterministic, no
// atomics).  The attention itself is the library's tensor-core forward and
// backward.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gt_common.cuh"
#include "gt_sm100.cuh"
#include "gt_stats.cuh"
#include "gt_tc_common.cuh"

namespace gt {
namespace {

using namespace sm100;

constexpr int kC = 64;          // width (8 heads x 8 channels)
constexpr int kF = 64;          // FFN width
constexpr int kTile = 128;      // node rows of a CTA
constexpr int kThreads = 2 * kTile;   // two threads per node row
constexpr float kLnEps = 1e-5f;

// GELU(a) = a Phi(a) and its derivative Phi(a) + a phi(a)
__device__ __forceinline__ float gelu(float a) { return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f)); }
__device__ __forceinline__ float gelu_grad(float a) {
    return 0.5f * (1.0f + erff(a * 0.70710678118654752f)) + a * 0.39894228040143268f * expf(-0.5f * a * a);
}

// ------------------------------------------------------------ MMA operands

// A K-major operand with R rows is stored as sub-tiles of [R][32 bytes] (8 fp32
// or 16 bf16 along K per row), 32-byte swizzle: the two 16-byte halves of row r
// trade places when bit 2 of r is set.  One MMA k-step reads one sub-tile.
// Byte offset of (row, kbyte):
__host__ __device__ constexpr uint32_t sw32(int R, int row, int kbyte) {
    return (uint32_t)((kbyte >> 5) * R * 32 + row * 32 + ((((kbyte >> 4) & 1) ^ ((row >> 2) & 1)) << 4) +
                      (kbyte & 15));
}

// Instruction descriptor of kind::tf32 (A and B tf32 read from fp32 storage), fp32 accumulate, K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[tmem] * B[smem], tf32, K = 8 per instruction (8 TMEM columns of A).
__device__ __forceinline__ void mma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}

__device__ __forceinline__ void st_shared_f32(uint32_t addr, float v) {
    asm volatile("st.shared.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Column k = r (this thread's node row) of rows rho .. rho + NV - 1 of a bf16
// operand with R rows per sub-tile (rho a multiple of 8): row rho + f gets v[f] * m.
template <int R, int NV>
__device__ __forceinline__ void put_col(uint32_t base, int rho, int r, const float (&v)[NV], float m) {
    const uint32_t a = base + (uint32_t)((r >> 4) * R * 32 + rho * 32 + (r & 7) * 2);
    const uint32_t c = (uint32_t)((r >> 3) & 1);
    const uint32_t a0 = a + (c << 4), a1 = a + ((c ^ 1u) << 4);
#pragma unroll
    for (int f = 0; f < NV; ++f)
        st_shared_u16((((f >> 2) & 1) ? a1 : a0) + 32u * f, __bfloat16_as_ushort(__float2bfloat16_rn(v[f] * m)));
}

// Rows rho .. rho + 63 of every sub-tile of a bf16 operand with R rows per
// sub-tile: row rho all ones, the rest zero (column sums in a product).
template <int R>
__device__ __forceinline__ void put_ones_block(uint8_t* base, int rho) {
    for (int i = threadIdx.x; i < 8 * 64 * 2; i += blockDim.x) {
        const int kk = i >> 7, row = (i >> 1) & 63, half = i & 1;
        const uint32_t v = row == 0 ? 0x3f803f80u : 0u;
        *reinterpret_cast<uint4*>(base + kk * R * 32 + (rho + row) * 32 + half * 16) = make_uint4(v, v, v, v);
    }
}

// ------------------------------------------------------------ rows and TMEM
//
// Two threads share a node row: warps w and w + 4 reach the same 32 TMEM lanes,
// so thread (row r, half h) takes features 32 h .. 32 h + 31 of row r, and the
// row sums of the LayerNorms pass between the two through shared memory.  Rows
// that must outlive a product wait in TMEM.  Only the GELU loops,
// whose per-element code is long, run in rolled 8-column chunks (the next chunk's
// read in flight while the current one is computed): a tile kernel runs its code
// once per CTA, so long unrolled loops spend their time fetching instructions.

constexpr int kHalf = kC / 2;   // features per thread

template <int NV>
__device__ __forceinline__ void tst(uint32_t t, const float (&v)[NV]) {
#pragma unroll
    for (int h = 0; h < NV / 16; ++h) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(v[16 * h + i]);
        tmem_st_x16(t + 16 * h, r);
    }
}

// a bf16 half row (16 words) into 32 fp32 TMEM columns
__device__ __forceinline__ void tst_bf16(uint32_t t, const uint32_t (&w)[kHalf / 2]) {
#pragma unroll
    for (int h = 0; h < kHalf / 16; ++h) {
        uint32_t r[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            r[2 * i] = w[8 * h + i] << 16;
            r[2 * i + 1] = w[8 * h + i] & 0xffff0000u;
        }
        tmem_st_x16(t + 16 * h, r);
    }
}

__device__ __forceinline__ void tld32(uint32_t t, float (&v)[32]) {
    uint32_t r[32];
    tmem_ld_x32(t, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// two 32-column reads behind one wait
__device__ __forceinline__ void tld32x2(uint32_t t0, float (&v0)[32], uint32_t t1, float (&v1)[32]) {
    uint32_t r0[32], r1[32];
    tmem_ld_x32(t0, r0);
    tmem_ld_x32(t1, r1);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) { v0[i] = __uint_as_float(r0[i]); v1[i] = __uint_as_float(r1[i]); }
}

__device__ __forceinline__ void tst8(uint32_t t, const float (&v)[8]) {
    uint32_t r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(v[i]);
    tmem_st_x8(t, r);
}

// Column k = r of rows rho .. rho + 2 NW - 1 of a bf16 operand from bf16 values
// held as NW words (no rounding: the values are bf16 already).
template <int R, int NW>
__device__ __forceinline__ void put_col_bf16(uint32_t base, int rho, int r, const uint32_t (&w)[NW]) {
    const uint32_t a = base + (uint32_t)((r >> 4) * R * 32 + rho * 32 + (r & 7) * 2);
    const uint32_t c = (uint32_t)((r >> 3) & 1);
    const uint32_t a0 = a + (c << 4), a1 = a + ((c ^ 1u) << 4);
#pragma unroll
    for (int f = 0; f < 2 * NW; ++f)
        st_shared_u16((((f >> 2) & 1) ? a1 : a0) + 32u * f,
                      (uint16_t)((f & 1) ? (w[f >> 1] >> 16) : (w[f >> 1] & 0xffffu)));
}

// Row sums over the two halves of a row: a thread adds its partner's partial
// (same row, other half) through shared memory.  The two buffers alternate, so
// one barrier per exchange suffices: a buffer is written again only after every
// thread has passed the next exchange's barrier, by which time it has read it.
// Callers keep exchanges in code that every thread of the CTA runs.
struct RowXch {
    float2* buf;   // [2][2][kTile]
    int k;
    __device__ __forceinline__ float2 sum(int hf, int r, float2 v) {
        float2* b = buf + (k & 1) * 2 * kTile;
        ++k;
        b[hf * kTile + r] = v;
        __syncthreads();
        const float2 o = b[(hf ^ 1) * kTile + r];
        return make_float2(v.x + o.x, v.y + o.y);
    }
};

// Mean and 1 / std of a row from its two halves (LayerNorm statistics, two passes).
__device__ __forceinline__ float2 ln_stats(RowXch& xc, int hf, int r, const float (&v)[kHalf]) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < kHalf; ++i) s += v[i];
    const float mu = xc.sum(hf, r, make_float2(s, 0.f)).x * (1.0f / kC);
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < kHalf; ++i) q = fmaf(v[i] - mu, v[i] - mu, q);
    return make_float2(mu, rsqrtf(xc.sum(hf, r, make_float2(q, 0.f)).x * (1.0f / kC) + kLnEps));
}

// v[j] by selects (no local memory)
template <int NV>
__device__ __forceinline__ float pick(const float (&v)[NV], int j) {
    float r = v[0];
#pragma unroll
    for (int i = 1; i < NV; ++i) r = j == i ? v[i] : r;
    return r;
}

// ------------------------------------------------------------ bulk tile copies
//
// A tile's node rows are contiguous in global memory, and so is each weight
// matrix: each moves between global and shared memory as one 1D bulk copy on the
// TMA engine (cp.async.bulk), issued by thread 0 (a thread-per-row global access
// would touch 32 rows per warp instruction; a copy per row would queue hundreds
// of small copies on the engine).  Loads complete on an mbarrier; stores are
// drained by thread 0 before the CTA exits.  Staged rows keep the global layout,
// so the 8 threads of a quarter warp, taking 16-byte chunk j of 8 consecutive
// rows, would all hit one bank group: a thread reads and writes the chunks of its
// row in an order rotated by its row number, and a select network puts them back
// in place in registers.

constexpr int kRow32 = kC * 4;   // an fp32 node row, bytes
constexpr int kRow16 = kC * 2;   // a bf16 node row

__device__ __forceinline__ void bulk_load(uint32_t sdst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(sdst),
                 "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void bulk_store(void* gdst, uint32_t ssrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc), "r"(bytes)
                 : "memory");
}

// this thread's bulk stores: committed, then waited for (their shared-memory
// sources may be reused or released afterwards)
__device__ __forceinline__ void bulk_store_drain() {
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Staged rows written with ordinary stores become visible to the bulk stores
// issued after this (every thread calls it).
__device__ __forceinline__ void staged_ready() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    __syncthreads();
}

// a 4-byte shared load ordered like ordinary memory accesses (staged data lands
// by bulk copy: its reads must stay behind the barrier wait)
__device__ __forceinline__ uint32_t lds_b32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

__device__ __forceinline__ void sts_u4(uint32_t addr, uint4 v) {
    asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
                 : "memory");
}

// out chunk j = in chunk (j + s) mod NC (NC chunks of 4 words, 0 <= s < NC), in
// log2 NC stages of selects
template <int NC>
__device__ __forceinline__ void rotate_chunks(uint32_t (&v)[4 * NC], int s) {
#pragma unroll
    for (int b = 1; b < NC; b <<= 1) {
        const bool on = (s & b) != 0;
        uint32_t t[4 * NC];
#pragma unroll
        for (int i = 0; i < 4 * NC; ++i) t[i] = v[(i + 4 * b) % (4 * NC)];
#pragma unroll
        for (int i = 0; i < 4 * NC; ++i) v[i] = on ? t[i] : v[i];
    }
}

// NC 16-byte chunks starting at `addr` (row r's part of a staged tile), in order
template <int NC>
__device__ __forceinline__ void lds_chunks(uint32_t addr, int r, uint32_t (&v)[4 * NC]) {
#pragma unroll
    for (int j = 0; j < NC; ++j) {
        const uint4 q = lds_u4(addr + 16 * ((j + r) & (NC - 1)));   // slot j = chunk (j + r)
        v[4 * j] = q.x; v[4 * j + 1] = q.y; v[4 * j + 2] = q.z; v[4 * j + 3] = q.w;
    }
    rotate_chunks<NC>(v, (NC - (r & (NC - 1))) & (NC - 1));
}

template <int NC>
__device__ __forceinline__ void sts_chunks(uint32_t addr, int r, uint32_t (&v)[4 * NC]) {
    rotate_chunks<NC>(v, r & (NC - 1));                   // slot j = chunk (j + r)
#pragma unroll
    for (int j = 0; j < NC; ++j)
        sts_u4(addr + 16 * ((j + r) & (NC - 1)), make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
}

// the half row (32 fp32) of row r from a staged fp32 tile (zeros for a dead row)
__device__ __forceinline__ void lds_half_f32(uint32_t stg, int r, int hf, bool live, float (&v)[kHalf]) {
    uint32_t w[kHalf];
    lds_chunks<8>(stg + r * kRow32 + hf * (kHalf * 4), r, w);
#pragma unroll
    for (int i = 0; i < kHalf; ++i) v[i] = live ? __uint_as_float(w[i]) : 0.f;
}

// the half row of row r from a staged bf16 tile, as 16 words (zeros for a dead row)
__device__ __forceinline__ void lds_half_bf16(uint32_t stg, int r, int hf, bool live, uint32_t (&w)[kHalf / 2]) {
    lds_chunks<4>(stg + r * kRow16 + hf * (kHalf * 2), r, w);
#pragma unroll
    for (int i = 0; i < kHalf / 2; ++i) w[i] = live ? w[i] : 0u;
}

// 32 fp32 values at byte offset `off` of row r of a staged tile with row pitch P
__device__ __forceinline__ void sts_f32x32(uint32_t stg, int P, int r, int off, const float (&v)[32]) {
    uint32_t w[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(v[i]);
    sts_chunks<8>(stg + r * P + off, r, w);
}

// 32 values as bf16 at byte offset `off` of row r of a staged bf16 tile
__device__ __forceinline__ void sts_bf16x32(uint32_t stg, int r, int off, const float (&v)[32]) {
    uint32_t w[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) w[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
    sts_chunks<4>(stg + r * kRow16 + off, r, w);
}

// B operand (n, k) = W[n][k] from a row-major [N][K] matrix staged as is: 16-byte
// moves, a warp filling 16 whole rows of one sub-tile.
template <int N, int K>
__device__ __forceinline__ void relayout_rows(uint8_t* dst, uint32_t nat) {
    static_assert(N % 16 == 0 && K % 8 == 0, "16 x 8 blocks");
    const uint32_t d = smem_u32(dst);
    const int lane = threadIdx.x & 31;
#pragma unroll 4
    for (int b = threadIdx.x >> 5; b < (N / 16) * (K / 8); b += kThreads / 32) {
        const int n = 16 * (b / (K / 8)) + (lane >> 1), k = 8 * (b % (K / 8)) + 4 * (lane & 1);
        sts_u4(d + sw32(N, n, 4 * k), lds_u4(nat + (n * K + k) * 4));
    }
}

// B operand (n, k) = W[k][n] from a row-major [K][N] matrix staged as is.  A warp
// step moves 32 consecutive n of 4 rows k: lane l takes n = n0 + l and k = k0 +
// ((l >> 3) + t) % 4 at turn t, so its loads (one row each, 32 consecutive words)
// and its stores (bank 8 (l % 4) + 4 (l / 4 % 2) + k % 4) both cover 32 banks.
template <int K, int N>
__device__ __forceinline__ void relayout_cols(uint8_t* dst, uint32_t nat) {
    static_assert(N % 32 == 0 && K % 8 == 0, "32 x 4 blocks");
    const int lane = threadIdx.x & 31;
#pragma unroll 2
    for (int b = threadIdx.x >> 5; b < (N / 32) * (K / 4); b += kThreads / 32) {
        const int n = 32 * (b % (N / 32)) + lane, k0 = 4 * (b / (N / 32));
#pragma unroll
        for (int t = 0; t < 4; ++t) {
            const int k = k0 + (((lane >> 3) + t) & 3);
            *reinterpret_cast<float*>(dst + sw32(N, n, 4 * k)) = __uint_as_float(lds_b32(nat + (k * N + n) * 4));
        }
    }
}

// ------------------------------------------------------------ CTA control

struct Ctl {
    uint64_t bar;      // one arrival per committed group of MMAs
    uint64_t ldbar;    // the bulk loads (thread 0 arrives with their bytes)
    uint32_t tbase;    // TMEM base address
    int abort;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

// Barriers and TMEM; ends with the CTA barrier that makes both visible.
__device__ __forceinline__ void ctl_init(Ctl& c, uint32_t cols) {
    if (threadIdx.x == 0) {
        mbar_init(&c.bar, 1);
        mbar_init(&c.ldbar, 1);
        c.abort = 0;
        fence_barrier_init();
    }
    if (threadIdx.x < 32) tmem_alloc(&c.tbase, cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Waits for the bulk loads, in every thread; one decision for the CTA.
__device__ __forceinline__ bool loads_wait(Ctl& c, int* status) {
    const bool ok = mbar_wait_all(&c.ldbar, 0, &c.abort, tc::kWaitNs);
    if (!ok && (threadIdx.x & 31) == 0) tc::fail(&c.abort, status);
    return __syncthreads_and(ok) != 0;
}

// This thread's TMEM stores and shared-memory operand stores are complete and
// visible to the tensor core, in every thread of the CTA; returns whether every
// thread's `ok` held (one uniform decision per phase).
__device__ __forceinline__ bool operands_ready(bool ok) {
    tmem_wait_st();
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    tc_fence_before();
    const bool all = __syncthreads_and(ok) != 0;
    tc_fence_after();
    return all;
}

// Waits for the last committed group (every lane of the warp); flips the phase.
__device__ __forceinline__ bool mma_wait(Ctl& c, uint32_t& phase, int* status) {
    const bool ok = mbar_wait_all(&c.bar, phase, &c.abort, tc::kWaitNs);
    if (!ok && (threadIdx.x & 31) == 0) tc::fail(&c.abort, status);
    phase ^= 1u;
    tc_fence_after();
    return ok;
}

// mma_wait in every warp, then one decision for the whole CTA (the row
// exchanges that follow need every thread at their barriers).
__device__ __forceinline__ bool mma_wait_cta(Ctl& c, uint32_t& phase, int* status) {
    const bool ok = mma_wait(c, phase, status);
    return __syncthreads_and(ok) != 0;
}

// End of a tile kernel: if a wait gave up, give the bulk loads and the last MMA
// group a second bounded wait so that nothing is still writing shared memory or
// TMEM, then free the columns.  (A bulk store is drained by its own thread.)
__device__ __forceinline__ void ctl_finish(Ctl& c, bool ok, uint32_t phase, uint32_t cols) {
    tc_fence_before();
    const bool all = __syncthreads_and(ok) != 0;
    if (threadIdx.x < 32) {
        if (!all) {
            int never = 0;
            mbar_wait(&c.ldbar, 0, &never, tc::kWaitNs);
            mbar_wait(&c.bar, phase ^ 1u, &never, tc::kWaitNs);
        }
        tc_fence_after();
        tmem_dealloc(c.tbase, cols);
    }
}

// ------------------------------------------------------------------ forward

struct SmemLnQkv {
    uint8_t w[3 * kC * kC * 4];                    // B (n, k) = W_qkv[k][n], n < 192
    uint8_t stg[3 * kC * kC * 4 + kTile * kRow32];   // W_qkv and the x tile as copied; then the q, k, v tiles
    float g1[kC], b1[kC], bq[3 * kC];
    float2 xch[4 * kTile];
};
static_assert(3 * kTile * kRow16 <= 3 * kC * kC * 4 + kTile * kRow32, "q, k, v staging");
constexpr uint32_t kLnQkvCols = 256;   // u (A, 64 columns), then the q | k | v accumulator (192)

__global__ void __launch_bounds__(kThreads)
layer_ln_qkv(int n, const float* __restrict__ x, const float* __restrict__ ln_g, const float* __restrict__ ln_b,
             const float* __restrict__ w_qkv, const float* __restrict__ b_qkv, __nv_bfloat16* __restrict__ q,
             __nv_bfloat16* __restrict__ k, __nv_bfloat16* __restrict__ v, int* status) {
    extern __shared__ uint8_t smem_raw[];
    SmemLnQkv& S = *reinterpret_cast<SmemLnQkv*>(align1024(smem_raw));
    __shared__ Ctl ctl;
    const int tid = threadIdx.x, warp = tid >> 5, hf = warp >> 2;
    const int r = ((warp & 3) << 5) | (tid & 31), c0 = kHalf * hf;
    const int row = blockIdx.x * kTile + r;
    const bool live = row < n;
    ctl_init(ctl, kLnQkvCols);
    const int row0 = blockIdx.x * kTile, rows = n - row0 < kTile ? n - row0 : kTile;
    const uint32_t stg = smem_u32(S.stg), xs = stg + 3 * kC * kC * 4;
    if (tid == 0) {
        mbar_arrive_expect_tx(&ctl.ldbar, 3 * kC * kC * 4 + rows * kRow32);
        bulk_load(stg, w_qkv, 3 * kC * kC * 4, &ctl.ldbar);
        bulk_load(xs, x + (size_t)row0 * kC, rows * kRow32, &ctl.ldbar);
    }
    for (int i = tid; i < kC; i += kThreads) { S.g1[i] = ln_g[i]; S.b1[i] = ln_b[i]; }
    for (int i = tid; i < 3 * kC; i += kThreads) S.bq[i] = b_qkv[i];
    bool ok = loads_wait(ctl, status);
    uint32_t phase = 0;
    const uint32_t tb = ctl.tbase, tl = tb + ((uint32_t)(32 * (warp & 3)) << 16);
    if (ok) {
        relayout_cols<kC, 3 * kC>(S.w, stg);
        float u[kHalf];
        lds_half_f32(xs, r, hf, live, u);
        RowXch xc{S.xch, 0};
        const float2 st = ln_stats(xc, hf, r, u);
#pragma unroll
        for (int i = 0; i < kHalf; ++i) u[i] = fmaf((u[i] - st.x) * st.y, S.g1[c0 + i], S.b1[c0 + i]);
        tst(tl + c0, u);
    }
    ok = operands_ready(ok);
    if (ok) {
        if (warp == 0) {
            if (elect_one()) {
                const SmemDesc dw = smem_desc_split(smem_u32(S.w), 16, 256, 6);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_tf32_ts(tb + 64, tb + 8 * kk, desc_at(dw, kk * 3 * kC * 32), idesc_tf32(128, 3 * kC),
                                kk > 0);
                mma_commit(&ctl.bar);
            }
            __syncwarp();
        }
        ok = mma_wait(ctl, phase, status);
    }
    if (ok) {
#pragma unroll 1
        for (int c = 3 * kHalf * hf; c < 3 * kHalf * (hf + 1); c += 32) {
            float t[32];
            tld32(tl + 64 + c, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] += S.bq[c + i];
            sts_bf16x32(stg + (c >> 6) * kTile * kRow16, r, (c & (kC - 1)) * 2, t);
        }
    }
    ok = __syncthreads_and(ok) != 0;
    staged_ready();
    if (tid == 0) {
        if (ok) {
            __nv_bfloat16* dst[3] = {q, k, v};
#pragma unroll
            for (int s = 0; s < 3; ++s) bulk_store(dst[s] + (size_t)row0 * kC, stg + s * kTile * kRow16, rows * kRow16);
        }
        bulk_store_drain();
    }
    ctl_finish(ctl, ok, phase, kLnQkvCols);
}

struct SmemOutFfn {
    uint8_t wo[kC * kC * 4], w1[kC * kF * 4], w2[kF * kC * 4];   // B (n, k) = W[k][n]
    uint8_t wn[3 * kC * kC * 4];                                 // W_o, W_1, W_2 as copied
    uint8_t os[kTile * kRow16];                                  // the o tile
    uint8_t xs[kTile * kRow32];                                  // the x tile, then the y tile
    float bo[kC], b1[kF], b2[kC], g2[kC], s2[kC];
    float2 xch[4 * kTile];
};
// TMEM: slot 0 (o, then a, then GELU(a)), slot 1 at 64 (t, then z, then f), hh at 128
constexpr uint32_t kOutFfnCols = 256;

__global__ void __launch_bounds__(kThreads)
layer_out_ffn(int n, const float* __restrict__ x, const __nv_bfloat16* __restrict__ o,
              const float* __restrict__ w_o, const float* __restrict__ b_o, const float* __restrict__ ln_g,
              const float* __restrict__ ln_b, const float* __restrict__ w_1, const float* __restrict__ b_1,
              const float* __restrict__ w_2, const float* __restrict__ b_2, float* __restrict__ y, int* status) {
    extern __shared__ uint8_t smem_raw[];
    SmemOutFfn& S = *reinterpret_cast<SmemOutFfn*>(align1024(smem_raw));
    __shared__ Ctl ctl;
    const int tid = threadIdx.x, warp = tid >> 5, hf = warp >> 2;
    const int r = ((warp & 3) << 5) | (tid & 31), c0 = kHalf * hf;
    const int row = blockIdx.x * kTile + r;
    const bool live = row < n;
    ctl_init(ctl, kOutFfnCols);
    const int row0 = blockIdx.x * kTile, rows = n - row0 < kTile ? n - row0 : kTile;
    const uint32_t wn = smem_u32(S.wn), os = smem_u32(S.os), xs = smem_u32(S.xs);
    if (tid == 0) {
        mbar_arrive_expect_tx(&ctl.ldbar, 3 * kC * kC * 4 + rows * (kRow16 + kRow32));
        const float* src[3] = {w_o, w_1, w_2};
#pragma unroll
        for (int m = 0; m < 3; ++m) bulk_load(wn + m * kC * kC * 4, src[m], kC * kC * 4, &ctl.ldbar);
        bulk_load(os, o + (size_t)row0 * kC, rows * kRow16, &ctl.ldbar);
        bulk_load(xs, x + (size_t)row0 * kC, rows * kRow32, &ctl.ldbar);
    }
    for (int i = tid; i < kC; i += kThreads) {
        S.bo[i] = b_o[i]; S.b1[i] = b_1[i]; S.b2[i] = b_2[i]; S.g2[i] = ln_g[i]; S.s2[i] = ln_b[i];
    }
    bool ok = loads_wait(ctl, status);
    uint32_t phase = 0;
    const uint32_t tb = ctl.tbase, tl = tb + ((uint32_t)(32 * (warp & 3)) << 16);
    RowXch xc{S.xch, 0};
    float hh[kHalf];
    if (ok) {
        relayout_cols<kC, kC>(S.wo, wn);
        uint32_t ow[kHalf / 2];
        lds_half_bf16(os, r, hf, live, ow);
        lds_half_f32(xs, r, hf, live, hh);
        tst_bf16(tl + c0, ow);                            // slot 0: o
    }
    ok = operands_ready(ok);
    const SmemDesc dwo = smem_desc_split(smem_u32(S.wo), 16, 256, 6);
    const SmemDesc dw1 = smem_desc_split(smem_u32(S.w1), 16, 256, 6);
    const SmemDesc dw2 = smem_desc_split(smem_u32(S.w2), 16, 256, 6);
    // three products in turn: slot 1 = slot 0 W_o, slot 0 = slot 1 W_1, slot 1 = slot 0 W_2
    auto issue = [&](uint32_t d, uint32_t a, const SmemDesc& w) {
        if (warp == 0) {
            if (elect_one()) {
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_tf32_ts(tb + d, tb + a + 8 * kk, desc_at(w, kk * 64 * 32), idesc_tf32(128, 64), kk > 0);
                mma_commit(&ctl.bar);
            }
            __syncwarp();
        }
    };
    if (ok) {
        issue(64, 0, dwo);
        relayout_cols<kC, kF>(S.w1, wn + kC * kC * 4);    // while the product runs
        relayout_cols<kF, kC>(S.w2, wn + 2 * kC * kC * 4);
        ok = mma_wait_cta(ctl, phase, status);
    }
    if (ok) {
        float t[kHalf];
        tld32(tl + 64 + c0, t);
#pragma unroll
        for (int i = 0; i < kHalf; ++i) hh[i] += t[i] + S.bo[c0 + i];
        tst(tl + 128 + c0, hh);                           // hh, for the last residual
        const float2 st = ln_stats(xc, hf, r, hh);
#pragma unroll
        for (int i = 0; i < kHalf; ++i) t[i] = fmaf((hh[i] - st.x) * st.y, S.g2[c0 + i], S.s2[c0 + i]);
        tst(tl + 64 + c0, t);                             // slot 1: z
    }
    ok = operands_ready(ok);
    if (ok) {
        issue(0, 64, dw1);
        ok = mma_wait(ctl, phase, status);
    }
    if (ok) {
        uint32_t cur[8], nxt[8] = {};
        tmem_ld_x8(tl + c0, cur);
        tmem_wait_ld();
#pragma unroll 1
        for (int c = c0; c < c0 + kHalf; c += 8) {
            if (c + 8 < c0 + kHalf) tmem_ld_x8(tl + c + 8, nxt);
            float a[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = gelu(__uint_as_float(cur[i]) + S.b1[c + i]);
            tst8(tl + c, a);                              // slot 0: GELU(a)
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
        }
    }
    ok = operands_ready(ok);
    if (ok) {
        issue(64, 0, dw2);
        ok = mma_wait(ctl, phase, status);
    }
    if (ok) {
        float f[kHalf];
        tld32x2(tl + 64 + c0, f, tl + 128 + c0, hh);
#pragma unroll
        for (int i = 0; i < kHalf; ++i) f[i] += hh[i] + S.b2[c0 + i];
        sts_f32x32(xs, kRow32, r, hf * kHalf * 4, f);    // the y tile (x is consumed)
    }
    ok = __syncthreads_and(ok) != 0;
    staged_ready();
    if (tid == 0) {
        if (ok) bulk_store(y + (size_t)row0 * kC, xs, rows * kRow32);
        bulk_store_drain();
    }
    ctl_finish(ctl, ok, phase, kOutFfnCols);
}

// ----------------------------------------------------------------- backward

// Per-CTA partial weight gradients: each CTA stores its sums in its own row of
// `part` ([nparts][kPartStride]); reduce_partials adds the rows in a fixed
// order (no atomics: no contention on the few thousand gradient entries, and
// the same result on every run) into the gradient arrays.
constexpr int kPartStride = kC * 3 * kC + 5 * kC;   // the larger of the two kernels' layouts (12608)

struct PartSegs {
    float* dst[12];
    int off[12];
    int nseg;
};

// Both backward kernels' partials in one launch: entries [0, kPartStride) sum
// the rows at `part` (layer_ffn_bwd's), entries [kPartStride, 2 kPartStride) the
// rows at part + nparts kPartStride (layer_qkv_bwd's).  One CTA per 32
// consecutive entries (kPartStride is a multiple of 32, so a CTA stays in one
// set): warp w adds partial rows w, w + 8, ... (coalesced along the entries),
// then warp 0 adds the 8 warp sums.
static_assert(kPartStride % 32 == 0, "a CTA of reduce_partials must not straddle the two partial sets");
__global__ void __launch_bounds__(256) reduce_partials(const float* __restrict__ part, int nparts, PartSegs sg,
                                                       int total) {
    __shared__ float red[8][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int i = blockIdx.x * 32 + tx;
    const int set = i >= kPartStride ? 1 : 0;
    const float* base = part + (size_t)set * nparts * kPartStride;
    const int e = i - set * kPartStride;
    float acc = 0.f;
    if (i < total) {
#pragma unroll 4
        for (int p = ty; p < nparts; p += 8) acc += base[(size_t)p * kPartStride + e];
    }
    red[ty][tx] = acc;
    __syncthreads();
    if (ty == 0 && i < total) {
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r) sum += red[r][tx];
        int seg = 0;
        while (seg + 1 < sg.nseg && i >= sg.off[seg + 1]) ++seg;
        sg.dst[seg][i - sg.off[seg]] = sum;
    }
}

// Transposed bf16 operands of the weight-gradient products: [256 rows][K = 128
// node rows], 8 sub-tiles of 256 x 32 bytes.
constexpr int kTR = 256;
constexpr int kTBytes = 8 * kTR * 32;

// At the start ta | tb stage the inputs as copied: W_o, W_2, W_1 and the o, dy, x
// tiles; at the end the image area stages dO and dh and ta the partial sums.
static_assert(3 * kC * kC * 4 + kTile * (kRow16 + 2 * kRow32) <= 2 * kTBytes, "input staging");

struct SmemFfnBwd {
    uint8_t wo_c[kC * kC * 4];   // (n = i, k = m) = W_o[m][i]:  t  = o W_o
    uint8_t w1_c[kC * kF * 4];   // (n = j, k = i) = W_1[i][j]:  a  = z W_1
    uint8_t w2_r[kF * kC * 4];   // (n = j, k = c) = W_2[j][c]:  dg = dy W_2^T
    uint8_t w1_r[kC * kF * 4];   // (n = i, k = j) = W_1[i][j]:  dz = da W_1^T
    uint8_t wo_r[kC * kC * 4];   // (n = m, k = i) = W_o[m][i]:  dO = dh W_o^T
    uint8_t ta[kTBytes];         // rows: GELU(a) | o | zh | ones (A of the gradient products)
    uint8_t tb[kTBytes];         // rows: da | dy | dh | dz       (B of the gradient products)
    float bo[kC], b1[kF], g2[kC], s2[kC];
    float vec[4 * kC];           // column sums: db_1 | db_2 | db_o | dLN2 shift
    float2 xch[4 * kTile];
};
static_assert(kTile * (kRow16 + kRow32) <= 5 * kC * kC * 4, "dO and dh staging");
static_assert(kPartStride * 4 <= kTBytes, "partial staging");
// TMEM columns: o then zh 0, dy 64 (A operands), t then z 128, dg 192, a then da
// 256, dz 320, dh 384, dO 448; once those are consumed the gradient products take
// 0..255 (zh | ones against da | dy | dh | dz) and 256..383 (GELU(a) | o against
// dy | dh).
constexpr uint32_t kFfnBwdCols = 512;

__global__ void __launch_bounds__(kThreads)
layer_ffn_bwd(int n, const float* __restrict__ x, const __nv_bfloat16* __restrict__ o,
              const float* __restrict__ dy, const float* __restrict__ w_o, const float* __restrict__ b_o,
              const float* __restrict__ ln_g, const float* __restrict__ ln_b, const float* __restrict__ w_1,
              const float* __restrict__ b_1, const float* __restrict__ w_2, __nv_bfloat16* __restrict__ dO,
              float* __restrict__ dh, float* __restrict__ part, int* status) {
    extern __shared__ uint8_t smem_raw[];
    SmemFfnBwd& S = *reinterpret_cast<SmemFfnBwd*>(align1024(smem_raw));
    __shared__ Ctl ctl;
    const int tid = threadIdx.x, warp = tid >> 5, hf = warp >> 2;
    const int r = ((warp & 3) << 5) | (tid & 31), c0 = kHalf * hf;
    const int row = blockIdx.x * kTile + r;
    const bool live = row < n;
    ctl_init(ctl, kFfnBwdCols);
    const uint32_t ta = smem_u32(S.ta), tbb = smem_u32(S.tb);
    const int row0 = blockIdx.x * kTile, rows = n - row0 < kTile ? n - row0 : kTile;
    const uint32_t wn = ta, os = wn + 3 * kC * kC * 4, dys = os + kTile * kRow16, xs = dys + kTile * kRow32;
    if (tid == 0) {
        mbar_arrive_expect_tx(&ctl.ldbar, 3 * kC * kC * 4 + rows * (kRow16 + 2 * kRow32));
        const float* src[3] = {w_o, w_2, w_1};
#pragma unroll
        for (int m = 0; m < 3; ++m) bulk_load(wn + m * kC * kC * 4, src[m], kC * kC * 4, &ctl.ldbar);
        bulk_load(os, o + (size_t)row0 * kC, rows * kRow16, &ctl.ldbar);
        bulk_load(dys, dy + (size_t)row0 * kC, rows * kRow32, &ctl.ldbar);
        bulk_load(xs, x + (size_t)row0 * kC, rows * kRow32, &ctl.ldbar);
    }
    for (int i = tid; i < kC; i += kThreads) {
        S.bo[i] = b_o[i]; S.b1[i] = b_1[i]; S.g2[i] = ln_g[i]; S.s2[i] = ln_b[i];
    }
    bool ok = loads_wait(ctl, status);
    uint32_t phase = 0;
    const uint32_t tb = ctl.tbase, tl = tb + ((uint32_t)(32 * (warp & 3)) << 16);
    RowXch xc{S.xch, 0};
    uint32_t ow[kHalf / 2];
    float v[kHalf], w[kHalf];
    if (ok) {
        relayout_cols<kC, kC>(S.wo_c, wn);
        relayout_rows<kC, kC>(S.wo_r, wn);
        relayout_rows<kF, kC>(S.w2_r, wn + kC * kC * 4);
        relayout_rows<kC, kF>(S.w1_r, wn + 2 * kC * kC * 4);
        relayout_cols<kC, kF>(S.w1_c, wn + 2 * kC * kC * 4);
        lds_half_bf16(os, r, hf, live, ow);
        lds_half_f32(dys, r, hf, live, v);
        lds_half_f32(xs, r, hf, live, w);
    }
    __syncthreads();                                      // the staged inputs are read: ta and tb are free
    if (ok) {
        put_ones_block<kTR>(S.ta, 192);
        // rows past the end are zeros, so their columns of the gradient operands are too
        tst_bf16(tl + 0 + c0, ow);
        tst(tl + 64 + c0, v);
        put_col_bf16<kTR>(ta, 64 + c0, r, ow);            // o^T
        put_col<kTR>(tbb, 64 + c0, r, v, 1.f);            // dy^T
    }
    ok = operands_ready(ok);
    const bool issuer = warp == 0;
    auto mma64 = [&](uint32_t d, uint32_t a, const uint8_t* wm) {   // D (64 columns) = A (TMEM, K = 64) W
        const SmemDesc dw = smem_desc_split(smem_u32(wm), 16, 256, 6);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_tf32_ts(tb + d, tb + a + 8 * kk, desc_at(dw, kk * 64 * 32), idesc_tf32(128, 64), kk > 0);
    };
    if (ok) {
        if (issuer) {
            if (elect_one()) {
                mma64(128, 0, S.wo_c);                    // t
                mma64(192, 64, S.w2_r);                   // dg = dy W_2^T
                mma_commit(&ctl.bar);
            }
            __syncwarp();
        }
        ok = mma_wait_cta(ctl, phase, status);
    }
    float r2 = 0.f;
    if (ok) {
        tld32(tl + 128 + c0, v);
#pragma unroll
        for (int i = 0; i < kHalf; ++i) w[i] += v[i] + S.bo[c0 + i];   // hh
        const float2 st = ln_stats(xc, hf, r, w);
        r2 = st.y;
#pragma unroll
        for (int i = 0; i < kHalf; ++i) {
            w[i] = (w[i] - st.x) * st.y;                  // zh
            v[i] = fmaf(w[i], S.g2[c0 + i], S.s2[c0 + i]);   // z
        }
        tst(tl + 0 + c0, w);                              // zh (o is consumed)
        tst(tl + 128 + c0, v);
        put_col<kTR>(ta, 128 + c0, r, w, 1.f);            // zh^T
    }
    ok = operands_ready(ok);
    if (ok) {
        if (issuer) {
            if (elect_one()) {
                mma64(256, 128, S.w1_c);                  // a = z W_1
                mma_commit(&ctl.bar);
            }
            __syncwarp();
        }
        ok = mma_wait(ctl, phase, status);
    }
    if (ok) {
        const float lm = live ? 1.f : 0.f;
        uint32_t ca[8], cg[8], na[8] = {}, ng[8] = {};
        tmem_ld_x8(tl + 256 + c0, ca);
        tmem_ld_x8(tl + 192 + c0, cg);
        tmem_wait_ld();
#pragma unroll 1
        for (int c = c0; c < c0 + kHalf; c += 8) {
            if (c + 8 < c0 + kHalf) {
                tmem_ld_x8(tl + 256 + c + 8, na);
                tmem_ld_x8(tl + 192 + c + 8, ng);
            }
            float a[8], g[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float av = __uint_as_float(ca[i]) + S.b1[c + i];
                a[i] = __uint_as_float(cg[i]) * gelu_grad(av);   // da
                g[i] = gelu(av);                                  // GELU(a)
            }
            tst8(tl + 256 + c, a);
            put_col<kTR>(ta, c, r, g, lm);                // GELU(a)^T (a dead row's GELU(b_1) is not zero)
            put_col<kTR>(tbb, c, r, a, 1.f);              // da^T
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) { ca[i] = na[i]; cg[i] = ng[i]; }
        }
    }
    ok = operands_ready(ok);
    if (ok) {
        if (issuer) {
            if (elect_one()) {
                mma64(320, 256, S.w1_r);                  // dz = da W_1^T
                mma_commit(&ctl.bar);
            }
            __syncwarp();
        }
        ok = mma_wait_cta(ctl, phase, status);
    }
    if (ok) {
        tld32x2(tl + 320 + c0, v, tl + 0 + c0, w);        // dz, zh
        put_col<kTR>(tbb, 192 + c0, r, v, 1.f);           // dz^T
        float m1 = 0.f, m2 = 0.f;
#pragma unroll
        for (int i = 0; i < kHalf; ++i) {
            v[i] *= S.g2[c0 + i];
            m1 += v[i];
            m2 = fmaf(v[i], w[i], m2);
        }
        const float2 m = xc.sum(hf, r, make_float2(m1, m2));
        m1 = m.x * (1.0f / kC);
        m2 = m.y * (1.0f / kC);
        float d[kHalf];
        tld32(tl + 64 + c0, d);                           // dy
#pragma unroll
        for (int i = 0; i < kHalf; ++i) d[i] += r2 * (v[i] - m1 - w[i] * m2);   // dh
        tst(tl + 384 + c0, d);
        put_col<kTR>(tbb, 128 + c0, r, d, 1.f);           // dh^T
    }
    ok = operands_ready(ok);
    if (ok) {
        if (issuer) {
            if (elect_one()) {
                mma64(448, 384, S.wo_r);                  // dO = dh W_o^T
                const SmemDesc da_ = smem_desc_split(ta, 16, 256, 6), db_ = smem_desc_split(tbb, 16, 256, 6);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)            // [GELU(a) | o]^T [dy | dh]
                    mma_ss(tb + 256, desc_at(da_, kk * kTR * 32), desc_at(db_, kk * kTR * 32 + 64 * 32),
                           idesc_bf16(128, 128, false, false), kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)            // [zh | ones]^T [da | dy | dh | dz]
                    mma_ss(tb + 0, desc_at(da_, kk * kTR * 32 + 128 * 32), desc_at(db_, kk * kTR * 32),
                           idesc_bf16(128, 256, false, false), kk > 0);
                mma_commit(&ctl.bar);
            }
            __syncwarp();
        }
        ok = mma_wait(ctl, phase, status);
    }
    // staging: dO and dh in the image area, the CTA's partial-sum row in ta (all
    // consumed now), laid out as in global memory: dW_2, dW_1, dW_o rows, then
    // db_2 | db_1 | db_o | dLN2 gain | shift
    const uint32_t dos = smem_u32(S.wo_c), dhs = dos + kTile * kRow16, ps = ta, pvec = ps + 3 * kC * kRow32;
    if (ok) {
        tld32x2(tl + 448 + c0, v, tl + 384 + c0, w);      // dO, dh
        sts_bf16x32(dos, r, hf * kHalf * 2, v);
        sts_f32x32(dhs, kRow32, r, hf * kHalf * 4, w);
        if ((warp & 3) == 2) {                            // lane 64: the column sums, 128 columns per half
#pragma unroll 1
            for (int c = 128 * hf; c < 128 * (hf + 1); c += 32) {
                tld32(tl + c, v);
                if (r == 64) sts_f32x32(smem_u32(S.vec), 0, r, 4 * c, v);
            }
        }
    }
    ok = __syncthreads_and(ok) != 0;
    if (ok) {
        if (r < 64) {
            tld32x2(tl + 256 + c0, v, tl + 0 + c0, w);
            sts_f32x32(ps, kRow32, r, 4 * c0, v);         // dW_2 row j
            const float gi = S.g2[r], si = S.s2[r];
#pragma unroll
            for (int j = 0; j < kHalf; ++j) w[j] = fmaf(gi, w[j], si * S.vec[c0 + j]);
            sts_f32x32(ps, kRow32, kC + r, 4 * c0, w);    // dW_1 row i
            tld32(tl + 192 + c0, v);
            if ((r >> 5) == hf) st_shared_f32(pvec + 4 * (3 * kC + r), pick(v, r - c0));   // gain: diag of zh^T dz
        } else {
            const int f = r - 64;
            tld32(tl + 256 + 64 + c0, v);
            sts_f32x32(ps, kRow32, 2 * kC + f, 4 * c0, v);   // dW_o row m
            if (hf == 0) {
                st_shared_f32(pvec + 4 * f, S.vec[64 + f]);            // db_2
                st_shared_f32(pvec + 4 * (kC + f), S.vec[f]);          // db_1
            } else {
                st_shared_f32(pvec + 4 * (2 * kC + f), S.vec[128 + f]);   // db_o
                st_shared_f32(pvec + 4 * (4 * kC + f), S.vec[192 + f]);   // dLN2 shift
            }
        }
    }
    ok = __syncthreads_and(ok) != 0;
    staged_ready();
    if (tid == 0) {
        if (ok) {
            bulk_store(dO + (size_t)row0 * kC, dos, rows * kRow16);
            bulk_store(dh + (size_t)row0 * kC, dhs, rows * kRow32);
            bulk_store(part + (size_t)blockIdx.x * kPartStride, ps, kPartStride * 4);
        }
        bulk_store_drain();
    }
    ctl_finish(ctl, ok, phase, kFfnBwdCols);
}

// At the start ta | tb | extra stage the inputs as copied: W_qkv and the dq, dk,
// dv, x, dh tiles; later the image area stages dx and ta the partial sums.
constexpr int kQkvIn = 3 * kC * kC * 4 + 3 * kTile * kRow16 + 2 * kTile * kRow32;
constexpr int kQkvExtra = kQkvIn - 8 * 128 * 32 - kTBytes;

struct SmemQkvBwd {
    uint8_t w[kC * 3 * kC * 4];  // (n = m, k = c) = W_qkv[m][c]: du = dqkv W_qkv^T (24 k-steps)
    uint8_t ta[8 * 128 * 32];    // rows: uh | ones (A of the gradient product)
    uint8_t tb[kTBytes];         // rows: dq | dk | dv | du
    uint8_t extra[kQkvExtra];
    float g1[kC], b1[kC];
    float vec[4 * kC];           // column sums: db_qkv | dLN1 shift
    float2 xch[4 * kTile];
};
static_assert(kTile * kRow32 <= kC * 3 * kC * 4, "dx staging");
static_assert(kPartStride * 4 <= 8 * 128 * 32 + kTBytes, "partial staging");
// TMEM columns: dq | dk | dv 0..191 (A operand), du 192; then the gradient product 0..255.
constexpr uint32_t kQkvBwdCols = 256;

__global__ void __launch_bounds__(kThreads)
layer_qkv_bwd(int n, const float* __restrict__ x, const float* __restrict__ ln_g, const float* __restrict__ ln_b,
              const float* __restrict__ w_qkv, const __nv_bfloat16* __restrict__ dq,
              const __nv_bfloat16* __restrict__ dk, const __nv_bfloat16* __restrict__ dv,
              const float* __restrict__ dh, float* __restrict__ dx, float* __restrict__ part, int* status) {
    extern __shared__ uint8_t smem_raw[];
    SmemQkvBwd& S = *reinterpret_cast<SmemQkvBwd*>(align1024(smem_raw));
    __shared__ Ctl ctl;
    const int tid = threadIdx.x, warp = tid >> 5, hf = warp >> 2;
    const int r = ((warp & 3) << 5) | (tid & 31), c0 = kHalf * hf;
    const int row = blockIdx.x * kTile + r;
    const bool live = row < n;
    ctl_init(ctl, kQkvBwdCols);
    const uint32_t ta = smem_u32(S.ta), tbb = smem_u32(S.tb);
    const int row0 = blockIdx.x * kTile, rows = n - row0 < kTile ? n - row0 : kTile;
    const uint32_t wn = ta, gs = wn + 3 * kC * kC * 4, xs = gs + 3 * kTile * kRow16, hs = xs + kTile * kRow32;
    if (tid == 0) {
        mbar_arrive_expect_tx(&ctl.ldbar, 3 * kC * kC * 4 + rows * (3 * kRow16 + 2 * kRow32));
        bulk_load(wn, w_qkv, 3 * kC * kC * 4, &ctl.ldbar);
        const __nv_bfloat16* src[3] = {dq, dk, dv};
#pragma unroll
        for (int s = 0; s < 3; ++s) bulk_load(gs + s * kTile * kRow16, src[s] + (size_t)row0 * kC, rows * kRow16, &ctl.ldbar);
        bulk_load(xs, x + (size_t)row0 * kC, rows * kRow32, &ctl.ldbar);
        bulk_load(hs, dh + (size_t)row0 * kC, rows * kRow32, &ctl.ldbar);
    }
    for (int i = tid; i < kC; i += kThreads) { S.g1[i] = ln_g[i]; S.b1[i] = ln_b[i]; }
    bool ok = loads_wait(ctl, status);
    uint32_t phase = 0;
    const uint32_t tb = ctl.tbase, tl = tb + ((uint32_t)(32 * (warp & 3)) << 16);
    RowXch xc{S.xch, 0};
    uint32_t gq[kHalf / 2], gk[kHalf / 2], gv[kHalf / 2];
    float u[kHalf], d[kHalf];
    if (ok) {
        relayout_rows<kC, 3 * kC>(S.w, wn);
        lds_half_bf16(gs, r, hf, live, gq);
        lds_half_bf16(gs + kTile * kRow16, r, hf, live, gk);
        lds_half_bf16(gs + 2 * kTile * kRow16, r, hf, live, gv);
        lds_half_f32(xs, r, hf, live, u);
        lds_half_f32(hs, r, hf, live, d);
    }
    __syncthreads();                                      // the staged inputs are read: ta and tb are free
    float2 st = make_float2(0.f, 0.f);
    if (ok) {
        put_ones_block<128>(S.ta, 64);
        // rows past the end are zeros, so their columns of the gradient operands are too
        tst_bf16(tl + 0 + c0, gq);
        tst_bf16(tl + 64 + c0, gk);
        tst_bf16(tl + 128 + c0, gv);
        put_col_bf16<kTR>(tbb, 0 + c0, r, gq);            // dq^T
        put_col_bf16<kTR>(tbb, 64 + c0, r, gk);           // dk^T
        put_col_bf16<kTR>(tbb, 128 + c0, r, gv);          // dv^T
        st = ln_stats(xc, hf, r, u);
#pragma unroll
        for (int i = 0; i < kHalf; ++i) u[i] = (u[i] - st.x) * st.y;   // uh
        put_col<128>(ta, c0, r, u, live ? 1.f : 0.f);     // uh^T
    }
    ok = operands_ready(ok);
    if (ok) {
        if (warp == 0) {
            if (elect_one()) {
                const SmemDesc dw = smem_desc_split(smem_u32(S.w), 16, 256, 6);
#pragma unroll
                for (int kk = 0; kk < 24; ++kk)
                    mma_tf32_ts(tb + 192, tb + 8 * kk, desc_at(dw, kk * 64 * 32), idesc_tf32(128, 64), kk > 0);
                mma_commit(&ctl.bar);
            }
            __syncwarp();
        }
        ok = mma_wait_cta(ctl, phase, status);
    }
    const uint32_t dxs = smem_u32(S.w);                   // dx staging (W_qkv is consumed)
    if (ok) {
        float du[kHalf];
        tld32(tl + 192 + c0, du);
        put_col<kTR>(tbb, 192 + c0, r, du, 1.f);          // du^T
        float m1 = 0.f, m2 = 0.f;
#pragma unroll
        for (int i = 0; i < kHalf; ++i) {
            du[i] *= S.g1[c0 + i];
            m1 += du[i];
            m2 = fmaf(du[i], u[i], m2);
        }
        const float2 m = xc.sum(hf, r, make_float2(m1, m2));
        m1 = m.x * (1.0f / kC);
        m2 = m.y * (1.0f / kC);
#pragma unroll
        for (int i = 0; i < kHalf; ++i) d[i] += st.y * (du[i] - m1 - u[i] * m2);
        sts_f32x32(dxs, kRow32, r, hf * kHalf * 4, d);
    }
    ok = operands_ready(ok);                              // also makes the dx tile visible to bulk stores
    if (ok) {
        if (warp == 0) {
            if (elect_one()) {
                const SmemDesc da_ = smem_desc_split(ta, 16, 256, 6), db_ = smem_desc_split(tbb, 16, 256, 6);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)            // [uh | ones]^T [dq | dk | dv | du]
                    mma_ss(tb + 0, desc_at(da_, kk * 128 * 32), desc_at(db_, kk * kTR * 32),
                           idesc_bf16(128, 256, false, false), kk > 0);
                mma_commit(&ctl.bar);
            }
            __syncwarp();
        }
        if (tid == 0) bulk_store(dx + (size_t)row0 * kC, dxs, rows * kRow32);   // while it runs
        ok = mma_wait(ctl, phase, status);
    }
    const uint32_t ps = ta, pvec = ps + 3 * kC * kC * 4;   // dW_qkv rows, then db_qkv | dLN1 gain | shift
    if (ok && (warp & 3) == 2) {                          // lane 64: the column sums, 128 columns per half
#pragma unroll 1
        for (int c = 128 * hf; c < 128 * (hf + 1); c += 32) {
            float t[32];
            tld32(tl + c, t);
            if (r == 64) sts_f32x32(smem_u32(S.vec), 0, r, 4 * c, t);
        }
    }
    ok = __syncthreads_and(ok) != 0;
    if (ok) {
        if (r < 64) {
            const float gm = S.g1[r], bm = S.b1[r];
#pragma unroll 1
            for (int c = 3 * kHalf * hf; c < 3 * kHalf * (hf + 1); c += 32) {
                float t[32];
                tld32(tl + c, t);
#pragma unroll
                for (int j = 0; j < 32; ++j) t[j] = fmaf(gm, t[j], bm * S.vec[c + j]);
                sts_f32x32(ps, 3 * kC * 4, r, 4 * c, t);
            }
            float t[32];
            tld32(tl + 192 + c0, t);
            if ((r >> 5) == hf) st_shared_f32(pvec + 4 * (3 * kC + r), pick(t, r - c0));   // gain: diag of uh^T du
        } else {
            const int f = r - 64;
            if (hf == 0) {
                st_shared_f32(pvec + 4 * f, S.vec[f]);                    // db_qkv 0..63
                st_shared_f32(pvec + 4 * (kC + f), S.vec[kC + f]);        // db_qkv 64..127
            } else {
                st_shared_f32(pvec + 4 * (2 * kC + f), S.vec[2 * kC + f]);   // db_qkv 128..191
                st_shared_f32(pvec + 4 * (4 * kC + f), S.vec[3 * kC + f]);   // dLN1 shift
            }
        }
    }
    ok = __syncthreads_and(ok) != 0;
    staged_ready();
    if (tid == 0) {
        if (ok) bulk_store(part + (size_t)blockIdx.x * kPartStride, ps, kPartStride * 4);
        bulk_store_drain();                               // the dx tile too
    }
    ctl_finish(ctl, ok, phase, kQkvBwdCols);
}

int tiles_of(int n) { return (n + kTile - 1) / kTile; }

template <typename T>
constexpr size_t smem_bytes() { return sizeof(T) + 1024; }

// layer_ln_qkv and layer_out_ffn hold 256 TMEM columns; asking for this much
// shared memory keeps at most two of their CTAs on an SM, so every allocation
// succeeds at once.
constexpr size_t kMinSmem256 = 80 * 1024;
constexpr size_t kLnQkvSmem = smem_bytes<SmemLnQkv>() > kMinSmem256 ? smem_bytes<SmemLnQkv>() : kMinSmem256;
constexpr size_t kOutFfnSmem = smem_bytes<SmemOutFfn>() > kMinSmem256 ? smem_bytes<SmemOutFfn>() : kMinSmem256;

template <typename K>
bool set_smem(K kern, size_t bytes) {
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) == cudaSuccess;
}

bool weights_ok(const gt_layer_weights* w) {
    return w && w->ln1_g && w->ln1_b && w->w_qkv && w->b_qkv && w->w_o && w->b_o && w->ln2_g && w->ln2_b &&
           w->w_1 && w->b_1 && w->w_2 && w->b_2 && aligned16(w->w_qkv) && aligned16(w->w_o) &&
           aligned16(w->w_1) && aligned16(w->w_2);
}

bool grads_ok(const gt_layer_grads* g) {
    return g && g->ln1_g && g->ln1_b && g->w_qkv && g->b_qkv && g->w_o && g->b_o && g->ln2_g && g->ln2_b &&
           g->w_1 && g->b_1 && g->w_2 && g->b_2;
}

// backward workspace: dO (bf16), d(hh) (fp32), dq, dk, dv (bf16), then the
// attention's own workspace
struct LayerBwdWs {
    __nv_bfloat16* dO;
    float* dh;
    float* part;
    __nv_bfloat16 *dq, *dk, *dv;
    void* attn;
    size_t attn_bytes;
};

size_t layer_bwd_carve(int n, void* ws, size_t bytes, LayerBwdWs* out) {
    Carve c(ws, bytes);
    const size_t e = (size_t)n * kC;
    LayerBwdWs w;
    w.dO = c.take<__nv_bfloat16>(e);
    w.dh = c.take<float>(e);
    w.part = c.take<float>((size_t)2 * tiles_of(n) * kPartStride);   // layer_ffn_bwd's rows, then layer_qkv_bwd's
    w.dq = c.take<__nv_bfloat16>(e);
    w.dk = c.take<__nv_bfloat16>(e);
    w.dv = c.take<__nv_bfloat16>(e);
    const size_t attn = gt_bias_attn_workspace_size(GT_BF16, n, 8, 8, 0);
    w.attn = c.take<char>(attn);
    w.attn_bytes = attn;
    if (out) *out = w;
    return c.off + 256;
}

}  // namespace
}  // namespace gt

extern "C" {

size_t gt_layer_workspace_size(int32_t n, int32_t h, int32_t d, int32_t f) {
    if (n < 1 || h != 8 || d != 8 || f != gt::kF) return 0;
    const size_t fwd = gt_bias_attn_workspace_size(GT_BF16, n, h, d, 0);
    const size_t bwd = gt::layer_bwd_carve(n, nullptr, 0, nullptr);
    return fwd > bwd ? fwd : bwd;
}

int gt_layer_fwd(int32_t n, int32_t h, int32_t d, int32_t f, const float* x, const gt_layer_weights* w,
                 const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb, void* q, void* k, void* v,
                 void* o, float* lse, float* y, void* workspace, size_t ws_bytes, void* stream) {
    using namespace gt;
    if (h != 8 || d != 8 || f != kF) return GT_ERR_UNSUPPORTED;
    if (n < 1 || !x || !gt::weights_ok(w) || !q || !k || !v || !o || !lse || !y) return GT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(y))
        return GT_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* status = device_status_ptr();
    if (!status) return GT_ERR_CUDA;
    if (!set_smem(layer_ln_qkv, kLnQkvSmem) || !set_smem(layer_out_ffn, kOutFfnSmem))
        return GT_ERR_CUDA;
    {
        LaunchScope ls("layer_ln_qkv", s);
        layer_ln_qkv<<<tiles_of(n), kThreads, kLnQkvSmem, s>>>(
            n, x, w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, static_cast<__nv_bfloat16*>(q),
            static_cast<__nv_bfloat16*>(k), static_cast<__nv_bfloat16*>(v), status);
    }
    if (check_launch() != GT_OK) return GT_ERR_CUDA;
    const float scale = 0.35355339059327373f;    // 1 / sqrt(8)
    int rc = gt_bias_attn_fwd(GT_BF16, n, h, d, q, k, v, spd, ld_spd, T, nb, scale, 0, o, lse, workspace,
                              ws_bytes, stream);
    if (rc != GT_OK) return rc;
    {
        LaunchScope ls("layer_out_ffn", s);
        layer_out_ffn<<<tiles_of(n), kThreads, kOutFfnSmem, s>>>(
            n, x, static_cast<const __nv_bfloat16*>(o), w->w_o, w->b_o, w->ln2_g, w->ln2_b, w->w_1, w->b_1,
            w->w_2, w->b_2, y, status);
    }
    return check_launch();
}

int gt_layer_bwd(int32_t n, int32_t h, int32_t d, int32_t f, const float* x, const gt_layer_weights* w,
                 const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb, const void* q, const void* k,
                 const void* v, const void* o, const float* lse, const float* dy, float* dx,
                 const gt_layer_grads* g, float* dT, void* workspace, size_t ws_bytes, void* stream) {
    using namespace gt;
    if (h != 8 || d != 8 || f != kF) return GT_ERR_UNSUPPORTED;
    if (n < 1 || !x || !gt::weights_ok(w) || !gt::grads_ok(g) || !q || !k || !v || !o || !lse || !dy || !dx ||
        !dT)
        return GT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dy) ||
        !aligned16(dx))
        return GT_ERR_INVALID_ARG;
    LayerBwdWs ws;
    const size_t need = layer_bwd_carve(n, workspace, ws_bytes, &ws);
    if (!workspace || ws_bytes < need) return GT_ERR_WORKSPACE;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int* status = device_status_ptr();
    if (!status) return GT_ERR_CUDA;
    if (!set_smem(layer_ffn_bwd, smem_bytes<SmemFfnBwd>()) || !set_smem(layer_qkv_bwd, smem_bytes<SmemQkvBwd>()))
        return GT_ERR_CUDA;
    const int grid = tiles_of(n);
    {
        LaunchScope ls("layer_ffn_bwd", s);
        layer_ffn_bwd<<<grid, kThreads, smem_bytes<SmemFfnBwd>(), s>>>(
            n, x, static_cast<const __nv_bfloat16*>(o), dy, w->w_o, w->b_o, w->ln2_g, w->ln2_b, w->w_1, w->b_1,
            w->w_2, ws.dO, ws.dh, ws.part, status);
    }
    if (check_launch() != GT_OK) return GT_ERR_CUDA;
    const float scale = 0.35355339059327373f;
    int rc = gt_bias_attn_bwd(GT_BF16, n, h, d, q, k, v, o, ws.dO, lse, spd, ld_spd, T, nb, scale, ws.dq, ws.dk,
                              ws.dv, dT, ws.attn, ws.attn_bytes, stream);
    if (rc != GT_OK) return rc;
    {
        LaunchScope ls("layer_qkv_bwd", s);
        layer_qkv_bwd<<<grid, kThreads, smem_bytes<SmemQkvBwd>(), s>>>(
            n, x, w->ln1_g, w->ln1_b, w->w_qkv, ws.dq, ws.dk, ws.dv, ws.dh, dx, ws.part + (size_t)grid * kPartStride,
            status);
    }
    {
        const int q0 = kPartStride;
        PartSegs sg = {{g->w_2, g->w_1, g->w_o, g->b_2, g->b_1, g->b_o, g->ln2_g, g->ln2_b, g->w_qkv, g->b_qkv,
                        g->ln1_g, g->ln1_b},
                       {0, kF * kC, 2 * kC * kC, 3 * kC * kC, 3 * kC * kC + kC, 3 * kC * kC + 2 * kC,
                        3 * kC * kC + 3 * kC, 3 * kC * kC + 4 * kC, q0, q0 + 3 * kC * kC, q0 + 3 * kC * kC + 3 * kC,
                        q0 + 3 * kC * kC + 4 * kC},
                       12};
        LaunchScope ls("layer_grad_sum", s);
        reduce_partials<<<2 * kPartStride / 32, 256, 0, s>>>(ws.part, grid, sg, 2 * kPartStride);
    }
    return check_launch();
}

}  // extern "C"

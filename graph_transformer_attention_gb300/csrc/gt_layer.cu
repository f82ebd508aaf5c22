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
// Four tile kernels, one CTA of 128 threads per 128 node rows, thread r = node
// row r of the tile = TMEM lane r.  Every product with a layer matrix is a
// tcgen05.mma (M = 128 node rows): the activation row goes into TMEM as the A
// operand (tf32, fp32 storage), the matrix sits in shared memory as the B
// operand, the fp32 accumulator comes back with tcgen05.ld, and the thread does
// the LayerNorms, GELU, residuals and the LayerNorm backward on its own row in
// registers:
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
constexpr int kThreads = kTile; // one thread per node row
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

// Weights go to shared memory with cp.async: every copy of a thread in flight at
// once (one memory latency, not one per element), overlapped with the row loads.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// B operand (n, k) = W[n][k] of a row-major [N][K] fp32 matrix (v W^T): 16-byte copies.
template <int N, int K>
__device__ __forceinline__ void load_b_rows(uint8_t* dst, const float* __restrict__ W) {
    const uint32_t d = smem_u32(dst);
#pragma unroll 4
    for (int i = threadIdx.x; i < N * K / 4; i += kThreads) {
        const int n = i / (K / 4), k = 4 * (i % (K / 4));
        cp_async16(d + sw32(N, n, 4 * k), W + 4 * i);
    }
}

// B operand (n, k) = W[k][n] of a row-major [K][N] fp32 matrix (v W): 4-byte
// copies.  A warp takes a block of 4 n x 8 k: lane (n & 3, k & 7) writes word
// (k & 7) of row n, so the 32 lanes hit 32 different banks (the 32-byte rows of
// 4 consecutive n start 8 banks apart), and reads 8 runs of 16 bytes.
template <int K, int N>
__device__ __forceinline__ void load_b_cols(uint8_t* dst, const float* __restrict__ W) {
    static_assert(N % 4 == 0 && K % 8 == 0, "4 x 8 blocks");
    const uint32_t d = smem_u32(dst);
    const int lane = threadIdx.x & 31;
#pragma unroll 4
    for (int b = threadIdx.x >> 5; b < (N / 4) * (K / 8); b += kThreads / 32) {
        const int n = 4 * (b % (N / 4)) + (lane & 3), k = 8 * (b / (N / 4)) + (lane >> 2);
        cp_async4(d + sw32(N, n, 4 * k), W + (size_t)k * N + n);
    }
}

__device__ __forceinline__ void st_shared_u16(uint32_t addr, uint16_t v) {
    asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
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
// A thread's node row is loaded into registers with all its global loads in
// flight at once, and the rows a kernel needs are all requested before the first
// of them is used.  Rows that must outlive a product wait in TMEM (the thread's
// lane).  TMEM reads take 32 or 64 columns per wait; only the GELU loops, whose
// per-element code is long, run in rolled 8-column chunks (the next chunk's read
// in flight while the current one is computed): a tile kernel runs its code once
// per CTA, so long unrolled loops spend their time fetching instructions.

__device__ __forceinline__ void ldg_row_f32(const float* __restrict__ src, int row, bool live, float (&v)[64]) {
    if (live) {
        const float4* s = reinterpret_cast<const float4*>(src + (size_t)row * kC);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float4 q = __ldg(s + i);
            v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) v[i] = 0.f;
    }
}

// bf16 row as 32 words (element 2j in the low half of word j)
__device__ __forceinline__ void ldg_row_bf16(const __nv_bfloat16* __restrict__ src, int row, bool live,
                                             uint32_t (&w)[32]) {
    if (live) {
        const uint4* s = reinterpret_cast<const uint4*>(src + (size_t)row * kC);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 q = __ldg(s + i);
            w[4 * i] = q.x; w[4 * i + 1] = q.y; w[4 * i + 2] = q.z; w[4 * i + 3] = q.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) w[i] = 0u;
    }
}

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

// a bf16 row (32 words) into 64 fp32 TMEM columns
__device__ __forceinline__ void tst_bf16(uint32_t t, const uint32_t (&w)[32]) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
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

__device__ __forceinline__ void tld64(uint32_t t, float (&v)[64]) {
    uint32_t r[64];
    tmem_ld_x32(t, *reinterpret_cast<uint32_t(*)[32]>(r));
    tmem_ld_x32(t + 32, *reinterpret_cast<uint32_t(*)[32]>(r + 32));
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// two 64-column reads behind one wait
__device__ __forceinline__ void tld64x2(uint32_t t0, float (&v0)[64], uint32_t t1, float (&v1)[64]) {
    uint32_t r0[64], r1[64];
    tmem_ld_x32(t0, *reinterpret_cast<uint32_t(*)[32]>(r0));
    tmem_ld_x32(t0 + 32, *reinterpret_cast<uint32_t(*)[32]>(r0 + 32));
    tmem_ld_x32(t1, *reinterpret_cast<uint32_t(*)[32]>(r1));
    tmem_ld_x32(t1 + 32, *reinterpret_cast<uint32_t(*)[32]>(r1 + 32));
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 64; ++i) { v0[i] = __uint_as_float(r0[i]); v1[i] = __uint_as_float(r1[i]); }
}

__device__ __forceinline__ void tst8(uint32_t t, const float (&v)[8]) {
    uint32_t r[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(v[i]);
    tmem_st_x8(t, r);
}

template <int NV>
__device__ __forceinline__ void stg_f32(float* dst, const float (&v)[NV]) {
    float4* d = reinterpret_cast<float4*>(dst);
#pragma unroll
    for (int i = 0; i < NV / 4; ++i) d[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
}

template <int NV>
__device__ __forceinline__ void stg_bf16(__nv_bfloat16* dst, const float (&v)[NV]) {
    uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int i = 0; i < NV / 8; ++i)
        d[i] = make_uint4(pack_bf16x2(v[8 * i], v[8 * i + 1]), pack_bf16x2(v[8 * i + 2], v[8 * i + 3]),
                          pack_bf16x2(v[8 * i + 4], v[8 * i + 5]), pack_bf16x2(v[8 * i + 6], v[8 * i + 7]));
}

// Column k = r of rows rho .. rho + 63 of a bf16 operand from a bf16 row held as
// 32 words (no rounding: the values are bf16 already).
template <int R>
__device__ __forceinline__ void put_col_bf16(uint32_t base, int rho, int r, const uint32_t (&w)[32]) {
    const uint32_t a = base + (uint32_t)((r >> 4) * R * 32 + rho * 32 + (r & 7) * 2);
    const uint32_t c = (uint32_t)((r >> 3) & 1);
    const uint32_t a0 = a + (c << 4), a1 = a + ((c ^ 1u) << 4);
#pragma unroll
    for (int f = 0; f < 64; ++f)
        st_shared_u16((((f >> 2) & 1) ? a1 : a0) + 32u * f,
                      (uint16_t)((f & 1) ? (w[f >> 1] >> 16) : (w[f >> 1] & 0xffffu)));
}

// Mean and 1 / std of a row (LayerNorm statistics, two passes).
__device__ __forceinline__ float2 ln_stats(const float (&v)[64]) {
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) s += v[i];
    const float mu = s * (1.0f / kC);
    float q = 0.f;
#pragma unroll
    for (int i = 0; i < 64; ++i) q = fmaf(v[i] - mu, v[i] - mu, q);
    return make_float2(mu, rsqrtf(q * (1.0f / kC) + kLnEps));
}

// v[j] by selects (no local memory)
template <int NV>
__device__ __forceinline__ float pick(const float (&v)[NV], int j) {
    float r = v[0];
#pragma unroll
    for (int i = 1; i < NV; ++i) r = j == i ? v[i] : r;
    return r;
}

// The GELU loops: for each 8-column chunk c of the 64 columns at `src`, f(c,
// v) with v the chunk's values; the next chunk's TMEM read is issued before f
// runs and waited for after it.
template <typename F>
__device__ __forceinline__ void chunks8_pipelined(uint32_t src, F&& f) {
    uint32_t cur[8], nxt[8] = {};
    tmem_ld_x8(src, cur);
    tmem_wait_ld();
#pragma unroll 1
    for (int c = 0; c < 64; c += 8) {
        if (c + 8 < 64) tmem_ld_x8(src + c + 8, nxt);
        float v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(cur[i]);
        f(c, v);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 8; ++i) cur[i] = nxt[i];
    }
}

// ------------------------------------------------------------ CTA control

struct Ctl {
    uint64_t bar;      // one arrival per committed group of MMAs
    uint32_t tbase;    // TMEM base address
    int abort;
};

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return p + ((1024u - (smem_u32(p) & 1023u)) & 1023u);
}

__device__ __forceinline__ void ctl_init(Ctl& c, uint32_t cols) {
    if (threadIdx.x == 0) {
        mbar_init(&c.bar, 1);
        c.abort = 0;
        fence_barrier_init();
    }
    if (threadIdx.x < 32) tmem_alloc(&c.tbase, cols);
}

// This thread's weight copies, TMEM stores and shared-memory operand stores are complete and
// visible to the tensor core, in every thread of the CTA; returns whether every
// thread's `ok` held (one uniform decision per phase).
__device__ __forceinline__ bool operands_ready(bool ok) {
    cp_async_wait_all();
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

// End of a tile kernel: if a wait gave up, give the last group a second bounded
// wait so that no MMA is still writing TMEM, then free the columns.
__device__ __forceinline__ void ctl_finish(Ctl& c, bool ok, uint32_t phase, uint32_t cols) {
    tc_fence_before();
    const bool all = __syncthreads_and(ok) != 0;
    if (threadIdx.x < 32) {
        if (!all) {
            int never = 0;
            mbar_wait(&c.bar, phase ^ 1u, &never, tc::kWaitNs);
        }
        tc_fence_after();
        tmem_dealloc(c.tbase, cols);
    }
}

// ------------------------------------------------------------------ forward

struct SmemLnQkv {
    uint8_t w[3 * kC * kC * 4];     // B (n, k) = W_qkv[k][n], n < 192
    float g1[kC], b1[kC], bq[3 * kC];
};
constexpr uint32_t kLnQkvCols = 256;   // u (A, 64 columns), then the q | k | v accumulator (192)

__global__ void __launch_bounds__(kThreads)
layer_ln_qkv(int n, const float* __restrict__ x, const float* __restrict__ ln_g, const float* __restrict__ ln_b,
             const float* __restrict__ w_qkv, const float* __restrict__ b_qkv, __nv_bfloat16* __restrict__ q,
             __nv_bfloat16* __restrict__ k, __nv_bfloat16* __restrict__ v, int* status) {
    extern __shared__ uint8_t smem_raw[];
    SmemLnQkv& S = *reinterpret_cast<SmemLnQkv*>(align1024(smem_raw));
    __shared__ Ctl ctl;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = blockIdx.x * kTile + tid;
    const bool live = row < n;
    ctl_init(ctl, kLnQkvCols);
    load_b_cols<kC, 3 * kC>(S.w, w_qkv);
    float u[64];
    ldg_row_f32(x, row, live, u);
    for (int i = tid; i < kC; i += kThreads) { S.g1[i] = ln_g[i]; S.b1[i] = ln_b[i]; }
    for (int i = tid; i < 3 * kC; i += kThreads) S.bq[i] = b_qkv[i];
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = ctl.tbase, tl = tb + ((uint32_t)(32 * warp) << 16);
    const float2 st = ln_stats(u);
#pragma unroll
    for (int i = 0; i < 64; ++i) u[i] = fmaf((u[i] - st.x) * st.y, S.g1[i], S.b1[i]);
    tst(tl, u);
    bool ok = operands_ready(true);
    uint32_t phase = 0;
    if (warp == 0) {
        if (elect_one()) {
            const SmemDesc dw = smem_desc_split(smem_u32(S.w), 16, 256, 6);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                mma_tf32_ts(tb + 64, tb + 8 * kk, desc_at(dw, kk * 3 * kC * 32), idesc_tf32(128, 3 * kC), kk > 0);
            mma_commit(&ctl.bar);
        }
        __syncwarp();
    }
    ok = mma_wait(ctl, phase, status);
    if (ok) {
#pragma unroll 1
        for (int c = 0; c < 3 * kC; c += 32) {
            float t[32];
            tld32(tl + 64 + c, t);
#pragma unroll
            for (int i = 0; i < 32; ++i) t[i] += S.bq[c + i];
            __nv_bfloat16* dst = c < kC ? q : c < 2 * kC ? k : v;
            if (live) stg_bf16(dst + (size_t)row * kC + (c & (kC - 1)), t);
        }
    }
    ctl_finish(ctl, ok, phase, kLnQkvCols);
}

struct SmemOutFfn {
    uint8_t wo[kC * kC * 4], w1[kC * kF * 4], w2[kF * kC * 4];   // B (n, k) = W[k][n]
    float bo[kC], b1[kF], b2[kC], g2[kC], s2[kC];
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
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = blockIdx.x * kTile + tid;
    const bool live = row < n;
    ctl_init(ctl, kOutFfnCols);
    load_b_cols<kC, kC>(S.wo, w_o);
    load_b_cols<kC, kF>(S.w1, w_1);
    load_b_cols<kF, kC>(S.w2, w_2);
    uint32_t ow[32];
    float hh[64];
    ldg_row_bf16(o, row, live, ow);
    ldg_row_f32(x, row, live, hh);
    for (int i = tid; i < kC; i += kThreads) {
        S.bo[i] = b_o[i]; S.b1[i] = b_1[i]; S.b2[i] = b_2[i]; S.g2[i] = ln_g[i]; S.s2[i] = ln_b[i];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = ctl.tbase, tl = tb + ((uint32_t)(32 * warp) << 16);
    tst_bf16(tl, ow);                                     // slot 0: o
    bool ok = operands_ready(true);
    uint32_t phase = 0;
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
    issue(64, 0, dwo);
    ok = mma_wait(ctl, phase, status);
    if (ok) {
        float t[64];
        tld64(tl + 64, t);
#pragma unroll
        for (int i = 0; i < 64; ++i) hh[i] += t[i] + S.bo[i];
        tst(tl + 128, hh);                                // hh, for the last residual
        const float2 st = ln_stats(hh);
#pragma unroll
        for (int i = 0; i < 64; ++i) t[i] = fmaf((hh[i] - st.x) * st.y, S.g2[i], S.s2[i]);
        tst(tl + 64, t);                                  // slot 1: z
    }
    ok = operands_ready(ok);
    if (ok) issue(0, 64, dw1);
    ok = ok && mma_wait(ctl, phase, status);
    if (ok) {
        chunks8_pipelined(tl, [&](int c, float (&a)[8]) {
#pragma unroll
            for (int i = 0; i < 8; ++i) a[i] = gelu(a[i] + S.b1[c + i]);
            tst8(tl + c, a);                              // slot 0: GELU(a)
        });
    }
    ok = operands_ready(ok);
    if (ok) issue(64, 0, dw2);
    ok = ok && mma_wait(ctl, phase, status);
    if (ok) {
        float f[64];
        tld64x2(tl + 64, f, tl + 128, hh);
#pragma unroll
        for (int i = 0; i < 64; ++i) f[i] += hh[i] + S.b2[i];
        if (live) stg_f32(y + (size_t)row * kC, f);
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
};
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
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = blockIdx.x * kTile + tid;
    const bool live = row < n;
    ctl_init(ctl, kFfnBwdCols);
    load_b_cols<kC, kC>(S.wo_c, w_o);
    load_b_cols<kC, kF>(S.w1_c, w_1);
    load_b_rows<kF, kC>(S.w2_r, w_2);
    load_b_rows<kC, kF>(S.w1_r, w_1);
    load_b_rows<kC, kC>(S.wo_r, w_o);
    uint32_t ow[32];
    float v[64], w[64];
    ldg_row_bf16(o, row, live, ow);
    ldg_row_f32(dy, row, live, v);
    ldg_row_f32(x, row, live, w);
    put_ones_block<kTR>(S.ta, 192);
    for (int i = tid; i < kC; i += kThreads) {
        S.bo[i] = b_o[i]; S.b1[i] = b_1[i]; S.g2[i] = ln_g[i]; S.s2[i] = ln_b[i];
    }
    const uint32_t ta = smem_u32(S.ta), tbb = smem_u32(S.tb);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = ctl.tbase, tl = tb + ((uint32_t)(32 * warp) << 16);
    // rows past the end are zeros, so their columns of the gradient operands are too
    tst_bf16(tl + 0, ow);
    tst(tl + 64, v);
    put_col_bf16<kTR>(ta, 64, tid, ow);                   // o^T
    put_col<kTR>(tbb, 64, tid, v, 1.f);                   // dy^T
    bool ok = operands_ready(true);
    uint32_t phase = 0;
    const bool issuer = warp == 0;
    auto mma64 = [&](uint32_t d, uint32_t a, const uint8_t* wm) {   // D (64 columns) = A (TMEM, K = 64) W
        const SmemDesc dw = smem_desc_split(smem_u32(wm), 16, 256, 6);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
            mma_tf32_ts(tb + d, tb + a + 8 * kk, desc_at(dw, kk * 64 * 32), idesc_tf32(128, 64), kk > 0);
    };
    if (issuer) {
        if (elect_one()) {
            mma64(128, 0, S.wo_c);                        // t
            mma64(192, 64, S.w2_r);                       // dg = dy W_2^T
            mma_commit(&ctl.bar);
        }
        __syncwarp();
    }
    ok = mma_wait(ctl, phase, status);
    float r2 = 0.f;
    if (ok) {
        tld64(tl + 128, v);
#pragma unroll
        for (int i = 0; i < 64; ++i) w[i] += v[i] + S.bo[i];   // hh
        const float2 st = ln_stats(w);
        r2 = st.y;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            w[i] = (w[i] - st.x) * st.y;                  // zh
            v[i] = fmaf(w[i], S.g2[i], S.s2[i]);          // z
        }
        tst(tl + 0, w);                                   // zh (o is consumed)
        tst(tl + 128, v);
        put_col<kTR>(ta, 128, tid, w, 1.f);               // zh^T
    }
    ok = operands_ready(ok);
    if (ok && issuer) {
        if (elect_one()) {
            mma64(256, 128, S.w1_c);                      // a = z W_1
            mma_commit(&ctl.bar);
        }
        __syncwarp();
    }
    ok = ok && mma_wait(ctl, phase, status);
    if (ok) {
        const float lm = live ? 1.f : 0.f;
        uint32_t ca[8], cg[8], na[8] = {}, ng[8] = {};
        tmem_ld_x8(tl + 256, ca);
        tmem_ld_x8(tl + 192, cg);
        tmem_wait_ld();
#pragma unroll 1
        for (int c = 0; c < 64; c += 8) {
            if (c + 8 < 64) {
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
            put_col<kTR>(ta, c, tid, g, lm);              // GELU(a)^T (a dead row's GELU(b_1) is not zero)
            put_col<kTR>(tbb, c, tid, a, 1.f);            // da^T
            tmem_wait_ld();
#pragma unroll
            for (int i = 0; i < 8; ++i) { ca[i] = na[i]; cg[i] = ng[i]; }
        }
    }
    ok = operands_ready(ok);
    if (ok && issuer) {
        if (elect_one()) {
            mma64(320, 256, S.w1_r);                      // dz = da W_1^T
            mma_commit(&ctl.bar);
        }
        __syncwarp();
    }
    ok = ok && mma_wait(ctl, phase, status);
    if (ok) {
        tld64x2(tl + 320, v, tl + 0, w);                  // dz, zh
        put_col<kTR>(tbb, 192, tid, v, 1.f);              // dz^T
        float m1 = 0.f, m2 = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            v[i] *= S.g2[i];
            m1 += v[i];
            m2 = fmaf(v[i], w[i], m2);
        }
        m1 *= 1.0f / kC;
        m2 *= 1.0f / kC;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            float d[32];
            tld32(tl + 64 + 32 * h, d);                   // dy
#pragma unroll
            for (int i = 0; i < 32; ++i) d[i] += r2 * (v[32 * h + i] - m1 - w[32 * h + i] * m2);   // dh
            if (live) stg_f32(dh + (size_t)row * kC + 32 * h, d);
            tst(tl + 384 + 32 * h, d);
            put_col<kTR>(tbb, 128 + 32 * h, tid, d, 1.f); // dh^T
        }
    }
    ok = operands_ready(ok);
    if (ok && issuer) {
        if (elect_one()) {
            mma64(448, 384, S.wo_r);                      // dO = dh W_o^T
            const SmemDesc da_ = smem_desc_split(ta, 16, 256, 6), db_ = smem_desc_split(tbb, 16, 256, 6);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)                // [GELU(a) | o]^T [dy | dh]
                mma_ss(tb + 256, desc_at(da_, kk * kTR * 32), desc_at(db_, kk * kTR * 32 + 64 * 32),
                       idesc_bf16(128, 128, false, false), kk > 0);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)                // [zh | ones]^T [da | dy | dh | dz]
                mma_ss(tb + 0, desc_at(da_, kk * kTR * 32 + 128 * 32), desc_at(db_, kk * kTR * 32),
                       idesc_bf16(128, 256, false, false), kk > 0);
            mma_commit(&ctl.bar);
        }
        __syncwarp();
    }
    ok = ok && mma_wait(ctl, phase, status);
    if (ok) {
        tld64(tl + 448, v);
        if (live) stg_bf16(dO + (size_t)row * kC, v);
        if (warp == 2) {                                  // lane 64: the column sums
#pragma unroll 1
            for (int c = 0; c < 4 * kC; c += 64) {
                tld64(tl + c, v);
                if (tid == 64) stg_f32(S.vec + c, v);
            }
        }
    }
    ok = __syncthreads_and(ok) != 0;
    float* pp = part + (size_t)blockIdx.x * kPartStride;
    if (ok) {
        // partial layout: dW_2, dW_1, dW_o (4096 each), then db_2, db_1, db_o, dLN2 gain, shift
        if (tid < 64) {
            tld64x2(tl + 256, v, tl + 0, w);
            stg_f32(pp + tid * kC, v);                    // dW_2 row j
            const float gi = S.g2[tid], si = S.s2[tid];
#pragma unroll
            for (int j = 0; j < 64; ++j) w[j] = fmaf(gi, w[j], si * S.vec[j]);
            stg_f32(pp + kF * kC + tid * kC, w);          // dW_1 row i
            tld64(tl + 192, v);
            pp[3 * kC * kC + 3 * kC + tid] = pick(v, tid);   // dLN2 gain: the diagonal of zh^T dz
        } else {
            const int f = tid - 64;
            tld64(tl + 256 + 64, v);
            stg_f32(pp + 2 * kC * kC + f * kC, v);        // dW_o row m
            pp[3 * kC * kC + f] = S.vec[64 + f];          // db_2
            pp[3 * kC * kC + kC + f] = S.vec[f];          // db_1
            pp[3 * kC * kC + 2 * kC + f] = S.vec[128 + f];   // db_o
            pp[3 * kC * kC + 4 * kC + f] = S.vec[192 + f];   // dLN2 shift
        }
    }
    ctl_finish(ctl, ok, phase, kFfnBwdCols);
}

struct SmemQkvBwd {
    uint8_t w[kC * 3 * kC * 4];  // (n = m, k = c) = W_qkv[m][c]: du = dqkv W_qkv^T (24 k-steps)
    uint8_t ta[8 * 128 * 32];    // rows: uh | ones (A of the gradient product)
    uint8_t tb[kTBytes];         // rows: dq | dk | dv | du
    float g1[kC], b1[kC];
    float vec[4 * kC];           // column sums: db_qkv | dLN1 shift
};
// TMEM columns: dq | dk | dv 0..191 (A operand), du 192, uh 256; then the
// gradient product 0..255.
constexpr uint32_t kQkvBwdCols = 512;

__global__ void __launch_bounds__(kThreads)
layer_qkv_bwd(int n, const float* __restrict__ x, const float* __restrict__ ln_g, const float* __restrict__ ln_b,
              const float* __restrict__ w_qkv, const __nv_bfloat16* __restrict__ dq,
              const __nv_bfloat16* __restrict__ dk, const __nv_bfloat16* __restrict__ dv,
              const float* __restrict__ dh, float* __restrict__ dx, float* __restrict__ part, int* status) {
    extern __shared__ uint8_t smem_raw[];
    SmemQkvBwd& S = *reinterpret_cast<SmemQkvBwd*>(align1024(smem_raw));
    __shared__ Ctl ctl;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = blockIdx.x * kTile + tid;
    const bool live = row < n;
    ctl_init(ctl, kQkvBwdCols);
    load_b_rows<kC, 3 * kC>(S.w, w_qkv);
    uint32_t gq[32], gk[32], gv[32];
    float u[64];
    ldg_row_bf16(dq, row, live, gq);
    ldg_row_bf16(dk, row, live, gk);
    ldg_row_bf16(dv, row, live, gv);
    ldg_row_f32(x, row, live, u);
    put_ones_block<128>(S.ta, 64);
    for (int i = tid; i < kC; i += kThreads) { S.g1[i] = ln_g[i]; S.b1[i] = ln_b[i]; }
    const uint32_t ta = smem_u32(S.ta), tbb = smem_u32(S.tb);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = ctl.tbase, tl = tb + ((uint32_t)(32 * warp) << 16);
    // rows past the end are zeros, so their columns of the gradient operands are too
    tst_bf16(tl + 0, gq);
    tst_bf16(tl + 64, gk);
    tst_bf16(tl + 128, gv);
    put_col_bf16<kTR>(tbb, 0, tid, gq);                   // dq^T
    put_col_bf16<kTR>(tbb, 64, tid, gk);                  // dk^T
    put_col_bf16<kTR>(tbb, 128, tid, gv);                 // dv^T
    const float2 st = ln_stats(u);
#pragma unroll
    for (int i = 0; i < 64; ++i) u[i] = (u[i] - st.x) * st.y;
    tst(tl + 256, u);                                     // uh
    put_col<128>(ta, 0, tid, u, live ? 1.f : 0.f);        // uh^T
    bool ok = operands_ready(true);
    uint32_t phase = 0;
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
    float d[64];
    ldg_row_f32(dh, row, live, d);                        // while the product runs
    ok = mma_wait(ctl, phase, status);
    if (ok) {
        float du[64];
        tld64(tl + 192, du);
        put_col<kTR>(tbb, 192, tid, du, 1.f);             // du^T
        float m1 = 0.f, m2 = 0.f;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
            du[i] *= S.g1[i];
            m1 += du[i];
            m2 = fmaf(du[i], u[i], m2);
        }
        m1 *= 1.0f / kC;
        m2 *= 1.0f / kC;
#pragma unroll
        for (int i = 0; i < 64; ++i) d[i] += st.y * (du[i] - m1 - u[i] * m2);
        if (live) stg_f32(dx + (size_t)row * kC, d);
    }
    ok = operands_ready(ok);
    if (ok && warp == 0) {
        if (elect_one()) {
            const SmemDesc da_ = smem_desc_split(ta, 16, 256, 6), db_ = smem_desc_split(tbb, 16, 256, 6);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)                // [uh | ones]^T [dq | dk | dv | du]
                mma_ss(tb + 0, desc_at(da_, kk * 128 * 32), desc_at(db_, kk * kTR * 32),
                       idesc_bf16(128, 256, false, false), kk > 0);
            mma_commit(&ctl.bar);
        }
        __syncwarp();
    }
    ok = ok && mma_wait(ctl, phase, status);
    if (ok && warp == 2) {                                // lane 64: the column sums
#pragma unroll 1
        for (int c = 0; c < 4 * kC; c += 64) {
            tld64(tl + c, d);
            if (tid == 64) stg_f32(S.vec + c, d);
        }
    }
    ok = __syncthreads_and(ok) != 0;
    float* pp = part + (size_t)blockIdx.x * kPartStride;
    if (ok) {
        // partial layout: dW_qkv (64 x 192), db_qkv (192), dLN1 gain, shift
        if (tid < 64) {
            const float gm = S.g1[tid], bm = S.b1[tid];
#pragma unroll 1
            for (int c = 0; c < 3 * kC; c += 64) {
                tld64(tl + c, d);
#pragma unroll
                for (int j = 0; j < 64; ++j) d[j] = fmaf(gm, d[j], bm * S.vec[c + j]);
                stg_f32(pp + tid * 3 * kC + c, d);
            }
            tld64(tl + 192, d);
            pp[3 * kC * kC + 3 * kC + tid] = pick(d, tid);   // dLN1 gain: the diagonal of uh^T du
        } else {
            const int f = tid - 64;
#pragma unroll
            for (int c = 0; c < 3; ++c) pp[3 * kC * kC + 64 * c + f] = S.vec[64 * c + f];   // db_qkv
            pp[3 * kC * kC + 4 * kC + f] = S.vec[192 + f];                                 // dLN1 shift
        }
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

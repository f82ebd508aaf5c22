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
// Four row kernels, one warp per node row (lane l holds features l and l + 32),
// the layer's matrices in shared memory with rows padded by one word so that both
// v W (lanes over columns) and v W^T (lanes over rows) are free of bank
// conflicts:
//   layer_ln_qkv    x -> LN1 -> q, k, v (bf16, the attention's inputs)
//   layer_out_ffn   o, x -> hh -> LN2 -> FFN -> y
//   layer_ffn_bwd   dy, and hh, z, a, GELU(a) recomputed from x and o -> dO for
//                   the attention backward (bf16) and d(hh); dW_2, dW_1, dW_o and
//                   their biases, dLN2
//   layer_qkv_bwd   dq, dk, dv, d(hh), and u recomputed from x -> dx; dW_qkv,
//                   db_qkv, dLN1
// Weight gradients: the 8 warps of a CTA each leave one row's vectors in shared
// memory; then every thread adds the 8 rows' outer products into its own
// registers (16 or 48 entries of each matrix); at the end each CTA stores its
// sums in its own row of a partials buffer, which reduce_partials adds up in a
// fixed order (deterministic, no atomics).  The attention itself is the
// library's tensor-core forward and backward.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "gt_common.cuh"
#include "gt_stats.cuh"

namespace gt {
namespace {

constexpr int kC = 64;          // width (8 heads x 8 channels)
constexpr int kF = 64;          // FFN width
constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kS = kC + 1;      // padded row stride of a 64-column matrix in shared memory
constexpr int kS3 = 3 * kC + 1; // of W_qkv
constexpr float kLnEps = 1e-5f;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// GELU(a) = a Phi(a) and its derivative Phi(a) + a phi(a)
__device__ __forceinline__ float gelu(float a) { return 0.5f * a * (1.0f + erff(a * 0.70710678118654752f)); }
__device__ __forceinline__ float gelu_grad(float a) {
    return 0.5f * (1.0f + erff(a * 0.70710678118654752f)) + a * 0.39894228040143268f * expf(-0.5f * a * a);
}

// Copy a [ROWS][COLS] fp32 matrix (16-byte aligned, COLS % 4 == 0) into shared
// memory with row stride `stride`: 16-byte loads, all of a thread's in flight
// before its stores.
template <int ROWS, int COLS>
__device__ __forceinline__ void load_mat(float* dst, const float* src, int stride) {
    constexpr int kN4 = ROWS * COLS / 4;
    constexpr int kPer = (kN4 + kThreads - 1) / kThreads;
    const float4* s4 = reinterpret_cast<const float4*>(src);
    float4 v[kPer];
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int i = threadIdx.x + u * kThreads;
        if (i < kN4) v[u] = __ldg(s4 + i);
    }
#pragma unroll
    for (int u = 0; u < kPer; ++u) {
        const int i = threadIdx.x + u * kThreads;
        if (i < kN4) {
            const int r = i / (COLS / 4), c = 4 * (i % (COLS / 4));
            float* d = dst + r * stride + c;
            d[0] = v[u].x; d[1] = v[u].y; d[2] = v[u].z; d[3] = v[u].w;
        }
    }
}

// out[j] for j = lane + 32 i (i < NO): b[j] + sum_k in[k] W[k][j]; `in` in shared memory.
template <int NO>
__device__ __forceinline__ void matvec(const float* in, const float* W, int stride, const float* b, int lane,
                                       float (&out)[NO]) {
#pragma unroll
    for (int i = 0; i < NO; ++i) out[i] = b ? b[lane + 32 * i] : 0.f;
#pragma unroll 8
    for (int k = 0; k < kC; ++k) {
        const float x = in[k];
#pragma unroll
        for (int i = 0; i < NO; ++i) out[i] = fmaf(x, W[k * stride + lane + 32 * i], out[i]);
    }
}

// out[k] for k = lane, lane + 32: sum_j in[j] W[k][j] over j < NJ (v W^T).
template <int NJ>
__device__ __forceinline__ void matvec_t(const float* in, const float* W, int stride, int lane, float (&out)[2]) {
    out[0] = out[1] = 0.f;
#pragma unroll 8
    for (int j = 0; j < NJ; ++j) {
        const float x = in[j];
        out[0] = fmaf(x, W[lane * stride + j], out[0]);
        out[1] = fmaf(x, W[(lane + 32) * stride + j], out[1]);
    }
}

// LayerNorm of the row held as (v0, v1) = features (lane, lane + 32):
// normalised values and 1/std
__device__ __forceinline__ void ln_row(float v0, float v1, float& h0, float& h1, float& r) {
    const float mu = warp_sum(v0 + v1) * (1.0f / kC);
    const float d0 = v0 - mu, d1 = v1 - mu;
    const float var = warp_sum(d0 * d0 + d1 * d1) * (1.0f / kC);
    r = rsqrtf(var + kLnEps);
    h0 = d0 * r;
    h1 = d1 * r;
}

// d(input) of a LayerNorm given dz = d(output) * gain, the normalised input vh
// and 1/std r: r (dz - mean dz - vh mean(dz vh))
__device__ __forceinline__ void ln_bwd_row(float dz0, float dz1, float vh0, float vh1, float r, float& dv0,
                                           float& dv1) {
    const float m1 = warp_sum(dz0 + dz1) * (1.0f / kC);
    const float m2 = warp_sum(dz0 * vh0 + dz1 * vh1) * (1.0f / kC);
    dv0 = r * (dz0 - m1 - vh0 * m2);
    dv1 = r * (dz1 - m1 - vh1 * m2);
}

// Accumulate the outer products of the 8 rows' vectors A (64) and B (NB) into
// this thread's entries (f, c0 .. c0 + E - 1), f = tid / 4, c0 = (tid % 4) E.
template <int E>
__device__ __forceinline__ void outer_acc(const float* A, int astride, const float* B, int bstride, int nrows,
                                          float (&acc)[E]) {
    const int f = threadIdx.x >> 2, c0 = (threadIdx.x & 3) * E;
    for (int r = 0; r < nrows; ++r) {
        const float a = A[r * astride + f];
        const float4* b4 = reinterpret_cast<const float4*>(B + r * bstride + c0);
#pragma unroll
        for (int i = 0; i < E / 4; ++i) {
            const float4 b = b4[i];
            acc[4 * i] = fmaf(a, b.x, acc[4 * i]);
            acc[4 * i + 1] = fmaf(a, b.y, acc[4 * i + 1]);
            acc[4 * i + 2] = fmaf(a, b.z, acc[4 * i + 2]);
            acc[4 * i + 3] = fmaf(a, b.w, acc[4 * i + 3]);
        }
    }
}

// This thread's entries of a [64][ncols] partial sum, stored (the CTA's own copy).
template <int E>
__device__ __forceinline__ void store_outer(float* g, int ncols, const float (&acc)[E]) {
    const int f = threadIdx.x >> 2, c0 = (threadIdx.x & 3) * E;
#pragma unroll
    for (int i = 0; i < E; i += 4)
        *reinterpret_cast<float4*>(g + f * ncols + c0 + i) = make_float4(acc[i], acc[i + 1], acc[i + 2], acc[i + 3]);
}

// Per-CTA partial weight gradients: each CTA stores its sums in its own row of
// `part` ([nparts][kPartStride]); reduce_partials adds the rows in a fixed
// order (no atomics: no contention on the few thousand gradient entries, and
// the same result on every run) into the gradient arrays.
constexpr int kPartStride = kC * 3 * kC + 5 * kC;   // the larger of the two kernels' layouts (12608)

struct PartSegs {
    float* dst[8];
    int off[8];
    int nseg;
};

// One CTA per 32 consecutive entries: warp w adds partial rows w, w + 8, ...
// (coalesced along the entries), then warp 0 adds the 8 warp sums.
__global__ void __launch_bounds__(256) reduce_partials(const float* __restrict__ part, int nparts, PartSegs sg,
                                                       int total) {
    __shared__ float red[8][33];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int i = blockIdx.x * 32 + tx;
    float acc = 0.f;
    if (i < total) {
#pragma unroll 4
        for (int p = ty; p < nparts; p += 8) acc += part[(size_t)p * kPartStride + i];
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

// ------------------------------------------------------------------ forward

struct SmemQkv {
    float w[kC * kS3];
    float b[3 * kC];
    float g1[kC], b1[kC];
    float u[kWarps][kC];
};

__global__ void __launch_bounds__(kThreads)
layer_ln_qkv(int n, const float* __restrict__ x, const float* __restrict__ ln_g, const float* __restrict__ ln_b,
             const float* __restrict__ w_qkv, const float* __restrict__ b_qkv, __nv_bfloat16* __restrict__ q,
             __nv_bfloat16* __restrict__ k, __nv_bfloat16* __restrict__ v) {
    extern __shared__ float4 smem_f4[];
    SmemQkv& S = *reinterpret_cast<SmemQkv*>(smem_f4);
    load_mat<kC, 3 * kC>(S.w, w_qkv, kS3);
    for (int i = threadIdx.x; i < 3 * kC; i += blockDim.x) S.b[i] = b_qkv[i];
    for (int i = threadIdx.x; i < kC; i += blockDim.x) { S.g1[i] = ln_g[i]; S.b1[i] = ln_b[i]; }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* ub = S.u[warp];
    for (int row = blockIdx.x * kWarps + warp; row < n; row += gridDim.x * kWarps) {
        const float* xr = x + (int64_t)row * kC;
        float h0, h1, r;
        ln_row(xr[lane], xr[lane + 32], h0, h1, r);
        ub[lane] = h0 * S.g1[lane] + S.b1[lane];
        ub[lane + 32] = h1 * S.g1[lane + 32] + S.b1[lane + 32];
        __syncwarp();
        float o[6];
        matvec<6>(ub, S.w, kS3, S.b, lane, o);
        __nv_bfloat16* dst[3] = {q + (int64_t)row * kC, k + (int64_t)row * kC, v + (int64_t)row * kC};
#pragma unroll
        for (int i = 0; i < 6; ++i) dst[i >> 1][lane + 32 * (i & 1)] = __float2bfloat16_rn(o[i]);
        __syncwarp();
    }
}

struct SmemFfn {
    float wo[kC * kS], w1[kC * kS], w2[kF * kS];
    float bo[kC], b1[kF], b2[kC], g2[kC], s2[kC];
    float v0[kWarps][kC], v1[kWarps][kC];
};

__global__ void __launch_bounds__(kThreads)
layer_out_ffn(int n, const float* __restrict__ x, const __nv_bfloat16* __restrict__ o,
              const float* __restrict__ w_o, const float* __restrict__ b_o, const float* __restrict__ ln_g,
              const float* __restrict__ ln_b, const float* __restrict__ w_1, const float* __restrict__ b_1,
              const float* __restrict__ w_2, const float* __restrict__ b_2, float* __restrict__ y) {
    extern __shared__ float4 smem_f4[];
    SmemFfn& S = *reinterpret_cast<SmemFfn*>(smem_f4);
    load_mat<kC, kC>(S.wo, w_o, kS);
    load_mat<kC, kF>(S.w1, w_1, kS);
    load_mat<kF, kC>(S.w2, w_2, kS);
    for (int i = threadIdx.x; i < kC; i += blockDim.x) {
        S.bo[i] = b_o[i]; S.b1[i] = b_1[i]; S.b2[i] = b_2[i]; S.g2[i] = ln_g[i]; S.s2[i] = ln_b[i];
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float* va = S.v0[warp];
    float* vb = S.v1[warp];
    for (int row = blockIdx.x * kWarps + warp; row < n; row += gridDim.x * kWarps) {
        const int64_t base = (int64_t)row * kC;
        va[lane] = __bfloat162float(o[base + lane]);
        va[lane + 32] = __bfloat162float(o[base + lane + 32]);
        __syncwarp();
        float t[2];
        matvec<2>(va, S.wo, kS, S.bo, lane, t);
        const float hh0 = x[base + lane] + t[0], hh1 = x[base + lane + 32] + t[1];
        float z0, z1, r;
        ln_row(hh0, hh1, z0, z1, r);
        vb[lane] = z0 * S.g2[lane] + S.s2[lane];
        vb[lane + 32] = z1 * S.g2[lane + 32] + S.s2[lane + 32];
        __syncwarp();
        float a[2];
        matvec<2>(vb, S.w1, kS, S.b1, lane, a);
        __syncwarp();
        va[lane] = gelu(a[0]);
        va[lane + 32] = gelu(a[1]);
        __syncwarp();
        float f[2];
        matvec<2>(va, S.w2, kS, S.b2, lane, f);
        y[base + lane] = hh0 + f[0];
        y[base + lane + 32] = hh1 + f[1];
        __syncwarp();
    }
}

// ----------------------------------------------------------------- backward

// per-row vectors a warp leaves for the CTA's weight-gradient pass
enum { kRg = 0, kRdy, kRz, kRda, kRo, kRdh, kRdzh, kRdz, kRvec };

struct SmemFfnBwd {
    float wo[kC * kS], w1[kC * kS], w2[kF * kS];
    float bo[kC], b1[kF], g2[kC], s2[kC];
    float rowv[kWarps][kRvec][kC];
};

__global__ void __launch_bounds__(kThreads)
layer_ffn_bwd(int n, const float* __restrict__ x, const __nv_bfloat16* __restrict__ o,
              const float* __restrict__ dy, const float* __restrict__ w_o, const float* __restrict__ b_o,
              const float* __restrict__ ln_g, const float* __restrict__ ln_b, const float* __restrict__ w_1,
              const float* __restrict__ b_1, const float* __restrict__ w_2, __nv_bfloat16* __restrict__ dO,
              float* __restrict__ dh, float* __restrict__ part) {
    extern __shared__ float4 smem_f4[];
    SmemFfnBwd& S = *reinterpret_cast<SmemFfnBwd*>(smem_f4);
    load_mat<kC, kC>(S.wo, w_o, kS);
    load_mat<kC, kF>(S.w1, w_1, kS);
    load_mat<kF, kC>(S.w2, w_2, kS);
    for (int i = threadIdx.x; i < kC; i += blockDim.x) {
        S.bo[i] = b_o[i]; S.b1[i] = b_1[i]; S.g2[i] = ln_g[i]; S.s2[i] = ln_b[i];
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    float aw2[16] = {}, aw1[16] = {}, awo[16] = {};
    float avec[5] = {};       // thread t < 64: db_2, db_1, db_o, dLN2 gain, dLN2 shift of feature t
    const int rows_per_pass = gridDim.x * kWarps;
    const int npass = (n + rows_per_pass - 1) / rows_per_pass;
    __syncthreads();
    for (int pass = 0; pass < npass; ++pass) {
        const int row = pass * rows_per_pass + blockIdx.x * kWarps + warp;
        float(*R)[kC] = S.rowv[warp];
        if (row < n) {
            const int64_t base = (int64_t)row * kC;
            R[kRo][lane] = __bfloat162float(o[base + lane]);
            R[kRo][lane + 32] = __bfloat162float(o[base + lane + 32]);
            __syncwarp();
            float t[2];
            matvec<2>(R[kRo], S.wo, kS, S.bo, lane, t);
            const float hh0 = x[base + lane] + t[0], hh1 = x[base + lane + 32] + t[1];
            float zh0, zh1, r2;
            ln_row(hh0, hh1, zh0, zh1, r2);
            R[kRz][lane] = zh0 * S.g2[lane] + S.s2[lane];
            R[kRz][lane + 32] = zh1 * S.g2[lane + 32] + S.s2[lane + 32];
            const float dy0 = dy[base + lane], dy1 = dy[base + lane + 32];
            R[kRdy][lane] = dy0;
            R[kRdy][lane + 32] = dy1;
            __syncwarp();
            float a[2];
            matvec<2>(R[kRz], S.w1, kS, S.b1, lane, a);
            R[kRg][lane] = gelu(a[0]);
            R[kRg][lane + 32] = gelu(a[1]);
            float dg[2];
            matvec_t<kC>(R[kRdy], S.w2, kS, lane, dg);          // dy W_2^T
            const float da0 = dg[0] * gelu_grad(a[0]), da1 = dg[1] * gelu_grad(a[1]);
            R[kRda][lane] = da0;
            R[kRda][lane + 32] = da1;
            __syncwarp();
            float dz[2];
            matvec_t<kF>(R[kRda], S.w1, kS, lane, dz);          // da W_1^T
            R[kRdzh][lane] = dz[0] * zh0;
            R[kRdzh][lane + 32] = dz[1] * zh1;
            R[kRdz][lane] = dz[0];
            R[kRdz][lane + 32] = dz[1];
            float dl0, dl1;
            ln_bwd_row(dz[0] * S.g2[lane], dz[1] * S.g2[lane + 32], zh0, zh1, r2, dl0, dl1);
            const float dh0 = dy0 + dl0, dh1 = dy1 + dl1;
            R[kRdh][lane] = dh0;
            R[kRdh][lane + 32] = dh1;
            dh[base + lane] = dh0;
            dh[base + lane + 32] = dh1;
            __syncwarp();
            float d_o[2];
            matvec_t<kC>(R[kRdh], S.wo, kS, lane, d_o);         // dh W_o^T
            dO[base + lane] = __float2bfloat16_rn(d_o[0]);
            dO[base + lane + 32] = __float2bfloat16_rn(d_o[1]);
        } else {
            for (int v = 0; v < kRvec; ++v) { R[v][lane] = 0.f; R[v][lane + 32] = 0.f; }
        }
        __syncthreads();
        outer_acc<16>(&S.rowv[0][kRg][0], kRvec * kC, &S.rowv[0][kRdy][0], kRvec * kC, kWarps, aw2);
        outer_acc<16>(&S.rowv[0][kRz][0], kRvec * kC, &S.rowv[0][kRda][0], kRvec * kC, kWarps, aw1);
        outer_acc<16>(&S.rowv[0][kRo][0], kRvec * kC, &S.rowv[0][kRdh][0], kRvec * kC, kWarps, awo);
        if (tid < kC) {
            for (int r = 0; r < kWarps; ++r) {
                avec[0] += S.rowv[r][kRdy][tid];
                avec[1] += S.rowv[r][kRda][tid];
                avec[2] += S.rowv[r][kRdh][tid];
                avec[3] += S.rowv[r][kRdzh][tid];
                avec[4] += S.rowv[r][kRdz][tid];
            }
        }
        __syncthreads();
    }
    // partial layout: dW_2, dW_1, dW_o (4096 each), then db_2, db_1, db_o, dLN2 gain, shift
    float* pp = part + (size_t)blockIdx.x * kPartStride;
    store_outer<16>(pp, kC, aw2);
    store_outer<16>(pp + kF * kC, kF, aw1);
    store_outer<16>(pp + 2 * kC * kC, kC, awo);
    if (tid < kC)
        for (int i = 0; i < 5; ++i) pp[3 * kC * kC + i * kC + tid] = avec[i];
}

enum { kQu = 0, kQduh = 64, kQdu = 128, kQdqkv = 192, kQvec = 384 };

struct SmemQkvBwd {
    float w[kC * kS3];
    float g1[kC], b1[kC];
    float rowv[kWarps][kQvec];
};

__global__ void __launch_bounds__(kThreads)
layer_qkv_bwd(int n, const float* __restrict__ x, const float* __restrict__ ln_g, const float* __restrict__ ln_b,
              const float* __restrict__ w_qkv, const __nv_bfloat16* __restrict__ dq,
              const __nv_bfloat16* __restrict__ dk, const __nv_bfloat16* __restrict__ dv,
              const float* __restrict__ dh, float* __restrict__ dx, float* __restrict__ part) {
    extern __shared__ float4 smem_f4[];
    SmemQkvBwd& S = *reinterpret_cast<SmemQkvBwd*>(smem_f4);
    load_mat<kC, 3 * kC>(S.w, w_qkv, kS3);
    for (int i = threadIdx.x; i < kC; i += blockDim.x) { S.g1[i] = ln_g[i]; S.b1[i] = ln_b[i]; }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, tid = threadIdx.x;
    float aw[48] = {};
    float ab = 0.f, ag = 0.f, as = 0.f;     // db_qkv (tid < 192), dLN1 gain and shift (tid < 64)
    const int rows_per_pass = gridDim.x * kWarps;
    const int npass = (n + rows_per_pass - 1) / rows_per_pass;
    __syncthreads();
    for (int pass = 0; pass < npass; ++pass) {
        const int row = pass * rows_per_pass + blockIdx.x * kWarps + warp;
        float* R = S.rowv[warp];
        if (row < n) {
            const int64_t base = (int64_t)row * kC;
            float uh0, uh1, r1;
            ln_row(x[base + lane], x[base + lane + 32], uh0, uh1, r1);
            R[kQu + lane] = uh0 * S.g1[lane] + S.b1[lane];
            R[kQu + lane + 32] = uh1 * S.g1[lane + 32] + S.b1[lane + 32];
            const __nv_bfloat16* src[3] = {dq + base, dk + base, dv + base};
#pragma unroll
            for (int i = 0; i < 6; ++i) R[kQdqkv + lane + 32 * i] = __bfloat162float(src[i >> 1][lane + 32 * (i & 1)]);
            __syncwarp();
            float du[2];
            matvec_t<3 * kC>(R + kQdqkv, S.w, kS3, lane, du);   // dqkv W_qkv^T
            R[kQduh + lane] = du[0] * uh0;
            R[kQduh + lane + 32] = du[1] * uh1;
            R[kQdu + lane] = du[0];
            R[kQdu + lane + 32] = du[1];
            float dl0, dl1;
            ln_bwd_row(du[0] * S.g1[lane], du[1] * S.g1[lane + 32], uh0, uh1, r1, dl0, dl1);
            dx[base + lane] = dh[base + lane] + dl0;
            dx[base + lane + 32] = dh[base + lane + 32] + dl1;
        } else {
            for (int i = lane; i < kQvec; i += 32) R[i] = 0.f;
        }
        __syncthreads();
        outer_acc<48>(&S.rowv[0][kQu], kQvec, &S.rowv[0][kQdqkv], kQvec, kWarps, aw);
        if (tid < 3 * kC)
            for (int r = 0; r < kWarps; ++r) ab += S.rowv[r][kQdqkv + tid];
        if (tid < kC)
            for (int r = 0; r < kWarps; ++r) { ag += S.rowv[r][kQduh + tid]; as += S.rowv[r][kQdu + tid]; }
        __syncthreads();
    }
    // partial layout: dW_qkv (64 x 192), db_qkv (192), dLN1 gain, shift
    float* pp = part + (size_t)blockIdx.x * kPartStride;
    store_outer<48>(pp, 3 * kC, aw);
    if (tid < 3 * kC) pp[3 * kC * kC + tid] = ab;
    if (tid < kC) { pp[3 * kC * kC + 3 * kC + tid] = ag; pp[3 * kC * kC + 4 * kC + tid] = as; }
}

// one row per warp while the rows last, at most `per_sm` CTAs per SM (what the
// kernel's shared memory lets an SM hold): more warps in flight hide the
// shared-memory latency of the row products
int row_grid(int n, int per_sm) {
    const int want = (n + kWarps - 1) / kWarps;
    const int cap = per_sm * num_sms();
    return want < cap ? want : cap;
}

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
    w.part = c.take<float>((size_t)row_grid(n, 2) * kPartStride);
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
    if (!set_smem(layer_ln_qkv, sizeof(SmemQkv)) || !set_smem(layer_out_ffn, sizeof(SmemFfn))) return GT_ERR_CUDA;
    {
        LaunchScope ls("layer_ln_qkv", s);
        layer_ln_qkv<<<row_grid(n, 2), kThreads, sizeof(SmemQkv), s>>>(
            n, x, w->ln1_g, w->ln1_b, w->w_qkv, w->b_qkv, static_cast<__nv_bfloat16*>(q),
            static_cast<__nv_bfloat16*>(k), static_cast<__nv_bfloat16*>(v));
    }
    if (check_launch() != GT_OK) return GT_ERR_CUDA;
    const float scale = 0.35355339059327373f;    // 1 / sqrt(8)
    int rc = gt_bias_attn_fwd(GT_BF16, n, h, d, q, k, v, spd, ld_spd, T, nb, scale, 0, o, lse, workspace,
                              ws_bytes, stream);
    if (rc != GT_OK) return rc;
    {
        LaunchScope ls("layer_out_ffn", s);
        layer_out_ffn<<<row_grid(n, 2), kThreads, sizeof(SmemFfn), s>>>(
            n, x, static_cast<const __nv_bfloat16*>(o), w->w_o, w->b_o, w->ln2_g, w->ln2_b, w->w_1, w->b_1,
            w->w_2, w->b_2, y);
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
    if (!set_smem(layer_ffn_bwd, sizeof(SmemFfnBwd)) || !set_smem(layer_qkv_bwd, sizeof(SmemQkvBwd)))
        return GT_ERR_CUDA;
    const int grid = row_grid(n, 2);
    const int rgrid = (kPartStride + 31) / 32;
    {
        LaunchScope ls("layer_ffn_bwd", s);
        layer_ffn_bwd<<<grid, kThreads, sizeof(SmemFfnBwd), s>>>(
            n, x, static_cast<const __nv_bfloat16*>(o), dy, w->w_o, w->b_o, w->ln2_g, w->ln2_b, w->w_1, w->b_1,
            w->w_2, ws.dO, ws.dh, ws.part);
    }
    {
        PartSegs sg = {{g->w_2, g->w_1, g->w_o, g->b_2, g->b_1, g->b_o, g->ln2_g, g->ln2_b},
                       {0, kF * kC, 2 * kC * kC, 3 * kC * kC, 3 * kC * kC + kC, 3 * kC * kC + 2 * kC,
                        3 * kC * kC + 3 * kC, 3 * kC * kC + 4 * kC},
                       8};
        LaunchScope ls("layer_grad_sum", s);
        reduce_partials<<<rgrid, 256, 0, s>>>(ws.part, grid, sg, 3 * kC * kC + 5 * kC);
    }
    if (check_launch() != GT_OK) return GT_ERR_CUDA;
    const float scale = 0.35355339059327373f;
    int rc = gt_bias_attn_bwd(GT_BF16, n, h, d, q, k, v, o, ws.dO, lse, spd, ld_spd, T, nb, scale, ws.dq, ws.dk,
                              ws.dv, dT, ws.attn, ws.attn_bytes, stream);
    if (rc != GT_OK) return rc;
    {
        LaunchScope ls("layer_qkv_bwd", s);
        layer_qkv_bwd<<<grid, kThreads, sizeof(SmemQkvBwd), s>>>(n, x, w->ln1_g, w->ln1_b, w->w_qkv, ws.dq, ws.dk,
                                                                 ws.dv, ws.dh, dx, ws.part);
    }
    {
        PartSegs sg = {{g->w_qkv, g->b_qkv, g->ln1_g, g->ln1_b},
                       {0, 3 * kC * kC, 3 * kC * kC + 3 * kC, 3 * kC * kC + 4 * kC},
                       4};
        LaunchScope ls("layer_grad_sum", s);
        reduce_partials<<<rgrid, 256, 0, s>>>(ws.part, grid, sg, 3 * kC * kC + 5 * kC);
    }
    return check_launch();
}

}  // extern "C"

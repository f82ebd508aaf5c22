// gt_attn_simt.cu -- CUDA-core biased attention (exact fp32 arithmetic).
//
// This is the path for fp32 storage (fp32 products and softmax statistics;
// tensor cores would round the products to tf32) and for shapes the
// tensor-core kernels do not take.  It follows the blockwise form of the
// MegaGraph paper's Fig. 4: each thread block streams KV tiles of 64 columns
// past its rows, and the bias of the current tile is formed from the int8
// bucket codes and a per-head table in shared memory.
//
// Forward: one thread per (row i, head h); online softmax in fp32 with expf.
// Backward: D_i = <dO_i, o_i> first; then a row pass (dq and dT, dS summed per
// bucket in shared memory, then added in fp64 to a global table) and a column
// pass (dk, dv), each recomputing p from lse.  No atomics touch dq, dk or dv.
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>
#include <type_traits>

#include "gt_common.cuh"
#include "gt_stats.cuh"

namespace gt {
namespace {

constexpr int kRows = 128;   // rows (or columns) per thread block, one per thread
constexpr int kTile = 64;    // streamed tile of the other dimension
constexpr int kCodes = 256;  // every byte value has a table slot
constexpr int kHCopies = 8;  // copies of each dT bin (see bwd_rows_simt)

template <typename TE, int DP>
__device__ __forceinline__ void load_vec(const TE* __restrict__ src, int d, float scale, float* dst) {
#pragma unroll
    for (int c = 0; c < DP; ++c) dst[c] = c < d ? scale * to_f32(src[c]) : 0.f;
}

// Stage a [kTile][DP] tile of x (rows r0..r0+kTile of head h) into shared fp32.
template <typename TE, int DP>
__device__ __forceinline__ void stage_tile(float (*dst)[DP], const TE* __restrict__ x, int n, int h,
                                           int d, int head, int r0) {
    for (int idx = threadIdx.x; idx < kTile * DP; idx += blockDim.x) {
        int r = idx / DP, c = idx % DP;
        int row = r0 + r;
        dst[r][c] = (row < n && c < d) ? to_f32(x[((int64_t)row * h + head) * d + c]) : 0.f;
    }
}

// Forward over the KV columns [kv_begin, kv_end), cut into nsplit splits of
// kv_block columns.  grid = (ceil(n / (128 / SPL)), h, nsplit); block = 128: SPL
// adjacent threads per query row, thread phase ph taking the columns j = ph mod
// SPL of each tile, their running (max, sum, output) merged exactly at the end.
// parts == 0: writes o (TE) and lse.  Otherwise writes fp32 partials
// o_part[z][n][h][d] and lse_part[z][h][n] for the KV columns of split z.
template <typename TE, int DP, int SPL>
__global__ void __launch_bounds__(kRows)
fwd_simt(int n, int h, int d, const TE* __restrict__ q, const TE* __restrict__ k,
         const TE* __restrict__ v, const uint8_t* __restrict__ spd, int64_t ld,
         const float* __restrict__ T, int nb, float scale, int kv_begin, int kv_end, int kv_block,
         int parts, TE* __restrict__ o, float* __restrict__ lse, float* __restrict__ o_part,
         float* __restrict__ lse_part) {
    __shared__ float sK[kTile][DP];
    __shared__ float sV[kTile][DP];
    __shared__ float sT[kCodes];
    const int head = blockIdx.y;
    const int ph = (int)threadIdx.x % SPL;
    const int i = blockIdx.x * (kRows / SPL) + (int)threadIdx.x / SPL;
    const int split = blockIdx.z;
    const int j_begin = kv_begin + (kv_block > 0 ? split * kv_block : 0);
    const int j_end = kv_block > 0 ? min(kv_end, j_begin + kv_block) : kv_end;
    for (int c = threadIdx.x; c < kCodes; c += blockDim.x) sT[c] = c < nb ? T[head * nb + c] : 0.f;

    float qi[DP], acc[DP];
    const bool live = i < n;
    load_vec<TE, DP>(q + ((int64_t)(live ? i : 0) * h + head) * d, d, scale, qi);
#pragma unroll
    for (int c = 0; c < DP; ++c) acc[c] = 0.f;
    float m = -INFINITY, l = 0.f;
    const uint8_t* row = spd + (int64_t)(live ? i : 0) * ld;

    for (int j0 = j_begin; j0 < j_end; j0 += kTile) {
        __syncthreads();
        stage_tile<TE, DP>(sK, k, n, h, d, head, j0);
        stage_tile<TE, DP>(sV, v, n, h, d, head, j0);
        __syncthreads();
        const int jn = min(kTile, j_end - j0);
#pragma unroll 1
        for (int jj = ph; jj < jn; jj += SPL) {
            float dot = 0.f;
#pragma unroll
            for (int c = 0; c < DP; ++c) dot = fmaf(qi[c], sK[jj][c], dot);
            const float x = dot + sT[row[j0 + jj]];
            if (x > m) {                          // new running max: rescale what we have
                const float corr = expf(m - x);   // 0 for the first column (m = -inf)
                l *= corr;
#pragma unroll
                for (int c = 0; c < DP; ++c) acc[c] *= corr;
                m = x;
            }
            const float p = expf(x - m);
            l += p;
#pragma unroll
            for (int c = 0; c < DP; ++c) acc[c] = fmaf(p, sV[jj][c], acc[c]);
        }
    }
    // the row's SPL phases: (m, l, acc) combined through their maxima (a phase
    // that saw no column has m = -inf and l = 0)
#pragma unroll
    for (int off = SPL / 2; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
        const float l2 = __shfl_xor_sync(0xffffffffu, l, off);
        const float mn = fmaxf(m, m2);
        const float a = mn == -INFINITY ? 0.f : expf(m - mn);
        const float b = mn == -INFINITY ? 0.f : expf(m2 - mn);
        l = l * a + l2 * b;
#pragma unroll
        for (int c = 0; c < DP; ++c) {
            const float o2 = __shfl_xor_sync(0xffffffffu, acc[c], off);
            acc[c] = acc[c] * a + o2 * b;
        }
        m = mn;
    }
    if (!live || ph != 0) return;
    const float inv = 1.f / l;
    if (!parts) {
        TE* oi = o + ((int64_t)i * h + head) * d;
#pragma unroll
        for (int c = 0; c < DP; ++c)
            if (c < d) oi[c] = from_f32<TE>(acc[c] * inv);
        lse[(int64_t)head * n + i] = m + logf(l);
    } else {
        float* oi = o_part + (((int64_t)split * n + i) * h + head) * d;
#pragma unroll
        for (int c = 0; c < DP; ++c)
            if (c < d) oi[c] = acc[c] * inv;
        lse_part[((int64_t)split * h + head) * n + i] = m + logf(l);
    }
}

// D[h][n] = <dO_i, o_i> in fp32.
template <typename TE>
__global__ void bwd_delta(int n, int h, int d, const TE* __restrict__ o, const TE* __restrict__ dO,
                          float* __restrict__ Dv) {
    const int64_t total = (int64_t)n * h;
    for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(x / h), head = (int)(x % h);
        const TE* a = o + x * d;
        const TE* b = dO + x * d;
        float acc = 0.f;
        for (int c = 0; c < d; ++c) acc = fmaf(to_f32(a[c]), to_f32(b[c]), acc);
        Dv[(int64_t)head * n + i] = acc;
    }
}

// Row pass: dq_i and dS summed per bucket.  grid = (ceil(n / (128 / SPL)), h);
// block = 128, SPL adjacent threads per query row taking every SPL-th column,
// their dq partials added at the end.
template <typename TE, int DP, int SPL>
__global__ void __launch_bounds__(kRows)
bwd_rows_simt(int n, int h, int d, const TE* __restrict__ q, const TE* __restrict__ k,
              const TE* __restrict__ v, const TE* __restrict__ dO, const float* __restrict__ lse,
              const float* __restrict__ Dv, const uint8_t* __restrict__ spd, int64_t ld,
              const float* __restrict__ T, int nb, float scale, TE* __restrict__ dq,
              double* __restrict__ dT64) {
    __shared__ float sK[kTile][DP];
    __shared__ float sV[kTile][DP];
    __shared__ float sT[kCodes];
    // dT sums: kHCopies copies per code, lane l adding into copy l % kHCopies, so
    // rows of a warp that share a code do not all contend for one address
    __shared__ float sH[kCodes][kHCopies];
    const int head = blockIdx.y;
    const int ph = (int)threadIdx.x % SPL;
    const int i = blockIdx.x * (kRows / SPL) + (int)threadIdx.x / SPL;
    for (int c = threadIdx.x; c < kCodes; c += blockDim.x) sT[c] = c < nb ? T[head * nb + c] : 0.f;
    for (int c = threadIdx.x; c < kCodes * kHCopies; c += blockDim.x) (&sH[0][0])[c] = 0.f;
    const bool live = i < n;
    const int ii = live ? i : 0;
    float qi[DP], gi[DP], acc[DP];
    load_vec<TE, DP>(q + ((int64_t)ii * h + head) * d, d, scale, qi);
    load_vec<TE, DP>(dO + ((int64_t)ii * h + head) * d, d, 1.f, gi);
#pragma unroll
    for (int c = 0; c < DP; ++c) acc[c] = 0.f;
    const float L = lse[(int64_t)head * n + ii];
    const float Di = Dv[(int64_t)head * n + ii];
    const uint8_t* row = spd + (int64_t)ii * ld;

    for (int j0 = 0; j0 < n; j0 += kTile) {
        __syncthreads();
        stage_tile<TE, DP>(sK, k, n, h, d, head, j0);
        stage_tile<TE, DP>(sV, v, n, h, d, head, j0);
        __syncthreads();
        if (!live) continue;
        const int jn = min(kTile, n - j0);
#pragma unroll 1
        for (int jj = ph; jj < jn; jj += SPL) {
            float dot = 0.f, dp = 0.f;
#pragma unroll
            for (int c = 0; c < DP; ++c) {
                dot = fmaf(qi[c], sK[jj][c], dot);
                dp = fmaf(gi[c], sV[jj][c], dp);
            }
            const int code = row[j0 + jj];
            const float p = expf(dot + sT[code] - L);
            const float ds = p * (dp - Di);
#pragma unroll
            for (int c = 0; c < DP; ++c) acc[c] = fmaf(ds, sK[jj][c], acc[c]);
            atomicAdd(&sH[code][threadIdx.x % kHCopies], ds);
        }
    }
#pragma unroll
    for (int off = SPL / 2; off > 0; off >>= 1)
#pragma unroll
        for (int c = 0; c < DP; ++c) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], off);
    if (live && ph == 0) {
        TE* out = dq + ((int64_t)i * h + head) * d;
#pragma unroll
        for (int c = 0; c < DP; ++c)
            if (c < d) out[c] = from_f32<TE>(acc[c] * scale);
    }
    __syncthreads();
    for (int c = threadIdx.x; c < nb; c += blockDim.x) {
        double sum = 0.0;
#pragma unroll
        for (int k = 0; k < kHCopies; ++k) sum += sH[c][k];
        if (sum != 0.0) atomicAdd(&dT64[head * nb + c], sum);
    }
}

// Column pass: dk_j, dv_j.  grid = (ceil(n / (128 / SPL)), h); block = 128, SPL
// adjacent threads per key column taking every SPL-th query row, their dk and
// dv partials added at the end.
template <typename TE, int DP, int SPL>
__global__ void __launch_bounds__(kRows)
bwd_cols_simt(int n, int h, int d, const TE* __restrict__ q, const TE* __restrict__ k,
              const TE* __restrict__ v, const TE* __restrict__ dO, const float* __restrict__ lse,
              const float* __restrict__ Dv, const uint8_t* __restrict__ spd, int64_t ld,
              const float* __restrict__ T, int nb, float scale, TE* __restrict__ dk,
              TE* __restrict__ dv) {
    __shared__ float sQ[kTile][DP];
    __shared__ float sG[kTile][DP];
    __shared__ float sL[kTile], sD[kTile];
    __shared__ uint8_t sS[kTile][kRows];
    __shared__ float sT[kCodes];
    constexpr int kCols = kRows / SPL;   // key columns per block
    const int head = blockIdx.y;
    const int ph = (int)threadIdx.x % SPL;
    const int jc = (int)threadIdx.x / SPL;
    const int j = blockIdx.x * kCols + jc;
    const int jbase = blockIdx.x * kCols;
    for (int c = threadIdx.x; c < kCodes; c += blockDim.x) sT[c] = c < nb ? T[head * nb + c] : 0.f;
    const bool live = j < n;
    const int jj_ = live ? j : 0;
    float kj[DP], vj[DP], ak[DP], av[DP];
    load_vec<TE, DP>(k + ((int64_t)jj_ * h + head) * d, d, scale, kj);
    load_vec<TE, DP>(v + ((int64_t)jj_ * h + head) * d, d, 1.f, vj);
#pragma unroll
    for (int c = 0; c < DP; ++c) ak[c] = av[c] = 0.f;

    for (int i0 = 0; i0 < n; i0 += kTile) {
        __syncthreads();
        stage_tile<TE, DP>(sQ, q, n, h, d, head, i0);
        stage_tile<TE, DP>(sG, dO, n, h, d, head, i0);
        for (int x = threadIdx.x; x < kTile; x += blockDim.x) {
            const int row = i0 + x;
            sL[x] = row < n ? lse[(int64_t)head * n + row] : 0.f;
            sD[x] = row < n ? Dv[(int64_t)head * n + row] : 0.f;
        }
        for (int x = threadIdx.x; x < kTile * kCols; x += blockDim.x) {
            const int r = x / kCols, c = x % kCols;
            const int row = i0 + r, col = jbase + c;
            sS[r][c] = (row < n && col < n) ? spd[(int64_t)row * ld + col] : 0;
        }
        __syncthreads();
        if (!live) continue;
        const int in_ = min(kTile, n - i0);
#pragma unroll 1
        for (int r = ph; r < in_; r += SPL) {
            float dot = 0.f, dp = 0.f;
#pragma unroll
            for (int c = 0; c < DP; ++c) {
                dot = fmaf(sQ[r][c], kj[c], dot);
                dp = fmaf(sG[r][c], vj[c], dp);
            }
            const float p = expf(dot + sT[sS[r][jc]] - sL[r]);
            const float ds = p * (dp - sD[r]);
#pragma unroll
            for (int c = 0; c < DP; ++c) {
                ak[c] = fmaf(ds, sQ[r][c], ak[c]);
                av[c] = fmaf(p, sG[r][c], av[c]);
            }
        }
    }
#pragma unroll
    for (int off = SPL / 2; off > 0; off >>= 1)
#pragma unroll
        for (int c = 0; c < DP; ++c) {
            ak[c] += __shfl_xor_sync(0xffffffffu, ak[c], off);
            av[c] += __shfl_xor_sync(0xffffffffu, av[c], off);
        }
    if (!live || ph != 0) return;
    TE* ok = dk + ((int64_t)j * h + head) * d;
    TE* ov = dv + ((int64_t)j * h + head) * d;
#pragma unroll
    for (int c = 0; c < DP; ++c)
        if (c < d) {
            ok[c] = from_f32<TE>(ak[c] * scale);
            ov[c] = from_f32<TE>(av[c]);
        }
}

__global__ void dT_finalize(int count, const double* __restrict__ dT64, float* __restrict__ dT) {
    for (int x = blockIdx.x * blockDim.x + threadIdx.x; x < count; x += gridDim.x * blockDim.x)
        dT[x] = (float)dT64[x];
}

// Exact merge of per-split partials: lse = log sum_z e^{lse_z};
// o = sum_z e^{lse_z - lse} o_z.
template <typename TE>
__global__ void merge_splits(int n, int h, int d, int nsplit, const float* __restrict__ o_part,
                             const float* __restrict__ lse_part, TE* __restrict__ o,
                             float* __restrict__ lse) {
    const int64_t total = (int64_t)n * h;
    for (int64_t x = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; x < total;
         x += (int64_t)gridDim.x * blockDim.x) {
        const int i = (int)(x / h), head = (int)(x % h);
        float mx = -INFINITY;
        for (int z = 0; z < nsplit; ++z) mx = fmaxf(mx, lse_part[((int64_t)z * h + head) * n + i]);
        float sum = 0.f;
        for (int z = 0; z < nsplit; ++z) sum += expf(lse_part[((int64_t)z * h + head) * n + i] - mx);
        const float L = mx + logf(sum);
        for (int c = 0; c < d; ++c) {
            float acc = 0.f;
            for (int z = 0; z < nsplit; ++z) {
                const float w = expf(lse_part[((int64_t)z * h + head) * n + i] - L);
                acc = fmaf(w, o_part[(((int64_t)z * n + i) * h + head) * d + c], acc);
            }
            o[x * d + c] = from_f32<TE>(acc);
        }
        lse[(int64_t)head * n + i] = L;
    }
}

int grid_for(int64_t total) {
    const int64_t b = (total + 255) / 256;
    return (int)(b < 4096 ? (b > 0 ? b : 1) : 4096);
}

// Threads per row (or column) of the fp32 kernels: 8 when one per row would not
// give every SM two blocks of 128, else 1.
int simt_spl(int n, int h, int nsplit) {
    return (int64_t)((n + kRows - 1) / kRows) * h * nsplit < 2 * num_sms() ? 8 : 1;
}

template <typename TE, int DP>
int fwd_simt_launch(int n, int h, int d, const void* q, const void* k, const void* v,
                    const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                    int kv_begin, int kv_end, int kv_block, int parts, void* o, float* lse,
                    float* o_part, float* lse_part, cudaStream_t s) {
    const int nsplit = kv_block > 0 ? (kv_end - kv_begin + kv_block - 1) / kv_block : 1;
    const int spl = simt_spl(n, h, nsplit);
    dim3 grid((n + kRows / spl - 1) / (kRows / spl), h, nsplit);
    {
        LaunchScope ls("fwd_simt", s);
        auto kern = spl == 8 ? fwd_simt<TE, DP, 8> : fwd_simt<TE, DP, 1>;
        kern<<<grid, kRows, 0, s>>>(n, h, d, (const TE*)q, (const TE*)k, (const TE*)v, (const uint8_t*)spd, ld,
                                    T, nb, scale, kv_begin, kv_end, nsplit > 1 ? kv_block : 0, parts, (TE*)o,
                                    lse, o_part, lse_part);
    }
    return check_launch();
}

template <typename TE, int DP>
int bwd_simt_launch(int n, int h, int d, const void* q, const void* k, const void* v,
                    const void* o, const void* dO, const float* lse, const int8_t* spd,
                    int64_t ld, const float* T, int nb, float scale, void* dq, void* dk, void* dv,
                    float* dT, float* Dv, double* dT64, cudaStream_t s) {
    if (cudaMemsetAsync(dT64, 0, sizeof(double) * (size_t)h * nb, s) != cudaSuccess) return GT_ERR_CUDA;
    {
        LaunchScope ls("bwd_delta", s);
        bwd_delta<TE><<<grid_for((int64_t)n * h), 256, 0, s>>>(n, h, d, (const TE*)o, (const TE*)dO, Dv);
    }
    const int spl = simt_spl(n, h, 1);
    dim3 grid((n + kRows / spl - 1) / (kRows / spl), h);
    {
        LaunchScope ls("bwd_rows_simt", s);
        auto kern = spl == 8 ? bwd_rows_simt<TE, DP, 8> : bwd_rows_simt<TE, DP, 1>;
        kern<<<grid, kRows, 0, s>>>(n, h, d, (const TE*)q, (const TE*)k, (const TE*)v, (const TE*)dO, lse, Dv,
                                    (const uint8_t*)spd, ld, T, nb, scale, (TE*)dq, dT64);
    }
    {
        LaunchScope ls("bwd_cols_simt", s);
        auto kern = spl == 8 ? bwd_cols_simt<TE, DP, 8> : bwd_cols_simt<TE, DP, 1>;
        kern<<<grid, kRows, 0, s>>>(n, h, d, (const TE*)q, (const TE*)k, (const TE*)v, (const TE*)dO, lse, Dv,
                                    (const uint8_t*)spd, ld, T, nb, scale, (TE*)dk, (TE*)dv);
    }
    {
        LaunchScope ls("bwd_dT_finalize", s);
        dT_finalize<<<1, 256, 0, s>>>(h * nb, dT64, dT);
    }
    return check_launch();
}

template <typename TE>
int fwd_simt_dispatch(int n, int h, int d, const void* q, const void* k, const void* v,
                      const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                      int kv_begin, int kv_end, int kv_block, int parts, void* o, float* lse,
                      float* o_part, float* lse_part, cudaStream_t s) {
#define GT_FWD_SIMT(DP) fwd_simt_launch<TE, DP>(n, h, d, q, k, v, spd, ld, T, nb, scale, kv_begin, kv_end, \
                                                kv_block, parts, o, lse, o_part, lse_part, s)
    if (d <= 8) return GT_FWD_SIMT(8);
    if (d <= 16) return GT_FWD_SIMT(16);
    if (d <= 32) return GT_FWD_SIMT(32);
    return GT_FWD_SIMT(64);
#undef GT_FWD_SIMT
}

template <typename TE>
int bwd_simt_dispatch(int n, int h, int d, const void* q, const void* k, const void* v,
                      const void* o, const void* dO, const float* lse, const int8_t* spd,
                      int64_t ld, const float* T, int nb, float scale, void* dq, void* dk,
                      void* dv, float* dT, float* Dv, double* dT64, cudaStream_t s) {
    if (d <= 8) return bwd_simt_launch<TE, 8>(n, h, d, q, k, v, o, dO, lse, spd, ld, T, nb, scale, dq, dk, dv, dT, Dv, dT64, s);
    if (d <= 16) return bwd_simt_launch<TE, 16>(n, h, d, q, k, v, o, dO, lse, spd, ld, T, nb, scale, dq, dk, dv, dT, Dv, dT64, s);
    if (d <= 32) return bwd_simt_launch<TE, 32>(n, h, d, q, k, v, o, dO, lse, spd, ld, T, nb, scale, dq, dk, dv, dT, Dv, dT64, s);
    return bwd_simt_launch<TE, 64>(n, h, d, q, k, v, o, dO, lse, spd, ld, T, nb, scale, dq, dk, dv, dT, Dv, dT64, s);
}

}  // namespace

int merge_partials(int dtype, int n, int h, int d, int nsplit, const float* o_part,
                   const float* lse_part, void* o, float* lse, cudaStream_t s);

int attn_fwd_simt(int dtype, int n, int h, int d, const void* q, const void* k, const void* v,
                  const int8_t* spd, int64_t ld, const float* T, int nb, float scale, int kv_block,
                  void* o, float* lse, float* o_part, float* lse_part, cudaStream_t s) {
    const int nsplit = kv_block > 0 ? (n + kv_block - 1) / kv_block : 1;
    const int parts = nsplit > 1;
    const int rc = dtype == GT_F32
        ? fwd_simt_dispatch<float>(n, h, d, q, k, v, spd, ld, T, nb, scale, 0, n, kv_block, parts, o, lse,
                                   o_part, lse_part, s)
        : fwd_simt_dispatch<__nv_bfloat16>(n, h, d, q, k, v, spd, ld, T, nb, scale, 0, n, kv_block, parts,
                                           o, lse, o_part, lse_part, s);
    if (rc != GT_OK || !parts) return rc;
    return merge_partials(dtype, n, h, d, nsplit, o_part, lse_part, o, lse, s);
}

// Attention over the KV columns [kv_begin, kv_end) only (see attn_fwd_tc_range).
int attn_fwd_simt_range(int dtype, int n, int h, int d, const void* q, const void* k, const void* v,
                        const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                        int kv_begin, int kv_end, float* o_part, float* lse_part, cudaStream_t s) {
    if (dtype == GT_F32)
        return fwd_simt_dispatch<float>(n, h, d, q, k, v, spd, ld, T, nb, scale, kv_begin, kv_end, 0, 1,
                                        nullptr, nullptr, o_part, lse_part, s);
    return fwd_simt_dispatch<__nv_bfloat16>(n, h, d, q, k, v, spd, ld, T, nb, scale, kv_begin, kv_end, 0, 1,
                                            nullptr, nullptr, o_part, lse_part, s);
}

int merge_partials(int dtype, int n, int h, int d, int nsplit, const float* o_part,
                   const float* lse_part, void* o, float* lse, cudaStream_t s) {
    if (dtype == GT_F32)
        {
            LaunchScope ls("fwd_merge", s);
            merge_splits<float><<<grid_for((int64_t)n * h), 256, 0, s>>>(n, h, d, nsplit, o_part, lse_part,
                                                                         (float*)o, lse);
        }
    else
        {
            LaunchScope ls("fwd_merge", s);
            merge_splits<__nv_bfloat16><<<grid_for((int64_t)n * h), 256, 0, s>>>(
                n, h, d, nsplit, o_part, lse_part, (__nv_bfloat16*)o, lse);
        }
    return check_launch();
}

int attn_bwd_simt(int dtype, int n, int h, int d, const void* q, const void* k, const void* v,
                  const void* o, const void* dO, const float* lse, const int8_t* spd, int64_t ld,
                  const float* T, int nb, float scale, void* dq, void* dk, void* dv, float* dT,
                  float* Dv, double* dT64, cudaStream_t s) {
    if (dtype == GT_F32)
        return bwd_simt_dispatch<float>(n, h, d, q, k, v, o, dO, lse, spd, ld, T, nb, scale, dq, dk, dv, dT, Dv, dT64, s);
    return bwd_simt_dispatch<__nv_bfloat16>(n, h, d, q, k, v, o, dO, lse, spd, ld, T, nb, scale, dq, dk, dv, dT, Dv, dT64, s);
}

}  // namespace gt

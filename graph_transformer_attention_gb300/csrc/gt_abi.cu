// gt_abi.cu -- the extern "C" entry points of libgt: argument checks,
// workspace layout and kernel dispatch.  Declarations and the contract of every
// call are in include/gt_attn.h.
#include <cuda_runtime.h>
#include <mutex>
#include <stdint.h>

#include "gt_attn.h"
#include "gt_common.cuh"

__device__ int g_gt_status = 0;

namespace gt {

// implemented in the kernel files
size_t spd_workspace_bytes(int32_t n, int64_t nnz, int32_t D, int algo);
int spd_build(const int64_t* indptr, const int32_t* indices, int32_t n, int64_t nnz, int32_t D,
              int8_t* spd, int64_t ld, void* ws, size_t ws_bytes, int algo, cudaStream_t stream);
int attn_fwd_simt(int dtype, int n, int h, int d, const void* q, const void* k, const void* v,
                  const int8_t* spd, int64_t ld, const float* T, int nb, float scale, int kv_block,
                  void* o, float* lse, float* o_part, float* lse_part, cudaStream_t s);
bool fwd_tc_supported(int h, int d);
size_t fwd_tc_piece_floats(int n, int d);
int fwd_tc_balanced_ctas(int n);
int attn_fwd_tc(int n, int d, const void* q, const void* k, const void* v, const int8_t* spd,
                int64_t ld, const float* T, int nb, float scale, int kv_block, void* o, float* lse,
                float* o_part, float* lse_part, cudaStream_t s);
int attn_fwd_tc_range(int n, int d, const void* q, const void* k, const void* v, const int8_t* spd,
                      int64_t ld, const float* T, int nb, float scale, int kv_begin, int kv_end,
                      float* o_part, float* lse_part, cudaStream_t s);
int attn_fwd_simt_range(int dtype, int n, int h, int d, const void* q, const void* k, const void* v,
                        const int8_t* spd, int64_t ld, const float* T, int nb, float scale,
                        int kv_begin, int kv_end, float* o_part, float* lse_part, cudaStream_t s);
int merge_partials(int dtype, int n, int h, int d, int nsplit, const float* o_part,
                   const float* lse_part, void* o, float* lse, cudaStream_t s);
int attn_bwd_simt(int dtype, int n, int h, int d, const void* q, const void* k, const void* v,
                  const void* o, const void* dO, const float* lse, const int8_t* spd, int64_t ld,
                  const float* T, int nb, float scale, void* dq, void* dk, void* dv, float* dT,
                  float* Dv, double* dT64, cudaStream_t s);
bool bwd_tc_supported(int h, int d, int nb);
int attn_bwd_tc(int n, int d, const void* q, const void* k, const void* v, const void* o,
                const void* dO, const float* lse, const int8_t* spd, int64_t ld, const float* T,
                int nb, float scale, void* dq, void* dk, void* dv, float* dT, float* LD, uint16_t* LB,
                float* Dv, double* dT64, float* aux, int tail, int dq_tail, float* acc,
                cudaStream_t s);
int bwd_dkdv_tail_split(int n);
int bwd_dq_tail_split(int n);

int* device_status_ptr() {
    static std::mutex mu;
    static int* ptrs[64] = {nullptr};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!ptrs[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_gt_status) != cudaSuccess) return nullptr;
        ptrs[dev] = static_cast<int*>(p);
    }
    return ptrs[dev];
}

namespace {

bool valid_dtype(int dtype) { return dtype == GT_F32 || dtype == GT_BF16; }

int check_common(int dtype, int n, int h, int d, const void* q, const void* k, const void* v,
                 const int8_t* spd, int64_t ld, const float* T, int nb) {
    if (!valid_dtype(dtype)) return GT_ERR_INVALID_ARG;
    if (n < 1 || h < 1 || d < 1 || nb < 1) return GT_ERR_INVALID_ARG;
    if (!q || !k || !v || !spd || !T) return GT_ERR_INVALID_ARG;
    if (ld < n || (ld % 16) != 0) return GT_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(spd)) return GT_ERR_INVALID_ARG;
    if (nb > 128) return GT_ERR_UNSUPPORTED;
    if (h > 16 || d > 64) return GT_ERR_UNSUPPORTED;
    return GT_OK;
}

struct FwdWs {
    float* o_part;
    float* lse_part;
};

struct BwdWs {
    float* Dv;
    double* dT64;
    float* LD;
    uint16_t* LB;   // bf16 [n][8][16]: per node and head -lse / scale and -D in three parts (dk/dv)
    float* aux;     // [16]: per head the largest row norm of v (tensor-core path)
    float* acc;     // split backward: fp32 dq, dk, dv accumulators, else null
};

size_t fwd_ws(int dtype, int n, int h, int d, int kv_block, void* base, size_t cap, FwdWs* out) {
    Carve c(base, cap);
    const int nsplit = kv_block > 0 ? (n + kv_block - 1) / kv_block : 1;
    FwdWs w{nullptr, nullptr};
    if (nsplit > 1) {
        w.o_part = c.take<float>((size_t)nsplit * n * h * d);
        w.lse_part = c.take<float>((size_t)nsplit * h * n);
    } else if (dtype == GT_BF16 && fwd_tc_supported(h, d)) {
        const size_t f = fwd_tc_piece_floats(n, d);
        if (f) w.o_part = c.take<float>(f);
    }
    if (out) *out = w;
    return c.off;
}

// Splits of the tensor-core backward kernels' work past their last full wave:
// the dq tasks (tile, head half; two CTAs per SM) along their KV blocks, the
// dk/dv groups (KV tile, head half; one CTA per SM) along their query tiles, k
// ways each (1 = none), chosen so that the last waves fill the SMs; on a graph
// too small to fill one wave every dq task is split, and dk/dv runs equal shares
// of all its (group, query tile) steps instead (bwd_tail 2).  Split or shared
// work sums into fp32 accumulators (workspace `acc`, 3 [n][h][d] arrays) turned
// into bf16 at the end.
int bwd_tail(int dtype, int n, int h, int d, int nb) {
    if (dtype != GT_BF16 || !bwd_tc_supported(h, d, nb)) return 1;
    return bwd_dkdv_tail_split(n);
}

int bwd_dq_tail(int dtype, int n, int h, int d, int nb) {
    if (dtype != GT_BF16 || !bwd_tc_supported(h, d, nb)) return 1;
    return bwd_dq_tail_split(n);
}

size_t bwd_ws(int n, int h, int d, bool with_acc, void* base, size_t cap, BwdWs* out) {
    Carve c(base, cap);
    BwdWs w;
    w.acc = with_acc ? c.take<float>((size_t)3 * n * h * d) : nullptr;
    w.Dv = c.take<float>((size_t)h * n);
    w.dT64 = c.take<double>((size_t)h * 128);
    // per-node lse log2 e (rows 0..7) and D (rows 8..15) of the 8 heads, [16][ld_ld]
    w.LD = c.take<float>((size_t)16 * bwd_ld_ld(n));
    w.LB = c.take<uint16_t>((size_t)n * 8 * 16);
    w.aux = c.take<float>(16);
    if (out) *out = w;
    return c.off;
}

}  // namespace

// Workspace of the backward run unsplit: the least a backward call accepts.
size_t bwd_ws_unsplit(int n, int h, int d) { return bwd_ws(n, h, d, false, nullptr, 0, nullptr); }

}  // namespace gt

extern "C" {

const char* gt_status_string(int status) {
    switch (status) {
        case GT_OK: return "ok";
        case GT_ERR_INVALID_ARG: return "invalid argument (NULL pointer, size, alignment or layout)";
        case GT_ERR_UNSUPPORTED: return "shape not supported by this library";
        case GT_ERR_CUDA: return "CUDA runtime error";
        case GT_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
        case GT_ERR_WORKSPACE: return "workspace missing or too small";
        default: return "unknown status";
    }
}

size_t gt_spd_workspace_size_algo(int32_t algo, int32_t n, int64_t nnz, int32_t D) {
    if (n < 1 || nnz < 0 || D < 1 || D > GT_MAX_D) return 0;
    return gt::spd_workspace_bytes(n, nnz, D, algo);
}

size_t gt_spd_workspace_size(int32_t n, int64_t nnz, int32_t D) {
    return gt_spd_workspace_size_algo(GT_SPD_AUTO, n, nnz, D);
}

int gt_spd_build_algo(int32_t algo, const int64_t* indptr, const int32_t* indices, int32_t n,
                      int64_t nnz, int32_t D, int8_t* spd, int64_t ld_spd, void* workspace,
                      size_t ws_bytes, void* stream) {
    if (!indptr || !spd || n < 1 || nnz < 0 || D < 1 || D > GT_MAX_D) return GT_ERR_INVALID_ARG;
    if (nnz > 0 && !indices) return GT_ERR_INVALID_ARG;
    if (ld_spd < n || (ld_spd % 16) != 0 || !gt::aligned16(spd)) return GT_ERR_INVALID_ARG;
    if (algo < GT_SPD_AUTO || algo > GT_SPD_GLOBAL64) return GT_ERR_INVALID_ARG;
    const size_t need = gt::spd_workspace_bytes(n, nnz, D, algo);
    if (need == 0) return GT_ERR_UNSUPPORTED;
    if (!workspace || ws_bytes < need) return GT_ERR_WORKSPACE;
    return gt::spd_build(indptr, indices, n, nnz, D, spd, ld_spd, workspace, ws_bytes, algo,
                         static_cast<cudaStream_t>(stream));
}

int gt_spd_build(const int64_t* indptr, const int32_t* indices, int32_t n, int64_t nnz, int32_t D,
                 int8_t* spd, int64_t ld_spd, void* workspace, size_t ws_bytes, void* stream) {
    return gt_spd_build_algo(GT_SPD_AUTO, indptr, indices, n, nnz, D, spd, ld_spd, workspace, ws_bytes,
                             stream);
}

size_t gt_bias_attn_workspace_size(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t kv_block) {
    if (!gt::valid_dtype(dtype) || n < 1 || h < 1 || d < 1 || kv_block < 0) return 0;
    if (kv_block >= n) kv_block = 0;
    size_t a = gt::fwd_ws(dtype, n, h, d, kv_block, nullptr, 0, nullptr);
    const bool acc = gt::bwd_tail(dtype, n, h, d, 128) > 1 || gt::bwd_dq_tail(dtype, n, h, d, 128) > 1;
    size_t b = gt::bwd_ws(n, h, d, acc, nullptr, 0, nullptr);
    return (a > b ? a : b) + 256;
}

int32_t gt_bias_attn_bwd_split(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t nb) {
    if (!gt::valid_dtype(dtype) || n < 1 || h < 1 || d < 1 || nb < 1) return -1;
    return gt::bwd_dq_tail(dtype, n, h, d, nb);
}

int32_t gt_bias_attn_fwd_kv_block(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t kv_block) {
    if (!gt::valid_dtype(dtype) || n < 1 || h < 1 || d < 1 || kv_block < 0) return -1;
    if (kv_block >= n) kv_block = 0;
    return kv_block;   // used as given; 0 (no uniform split) lets the tensor-core path balance its work
}

int32_t gt_bias_attn_fwd_ctas(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t kv_block) {
    if (!gt::valid_dtype(dtype) || n < 1 || h < 1 || d < 1 || kv_block < 0) return -1;
    if (kv_block >= n) kv_block = 0;
    if (kv_block > 0 || dtype != GT_BF16 || !gt::fwd_tc_supported(h, d)) return 0;
    return gt::fwd_tc_balanced_ctas(n);
}

int gt_bias_attn_launches(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t nb, int32_t kv_block,
                          int32_t* fwd, int32_t* bwd) {
    if (!fwd || !bwd || !gt::valid_dtype(dtype) || n < 1 || h < 1 || d < 1 || nb < 1 || kv_block < 0)
        return GT_ERR_INVALID_ARG;
    if (kv_block >= n) kv_block = 0;
    const bool tc_fwd = dtype == GT_BF16 && gt::fwd_tc_supported(h, d);
    const bool kv_split = kv_block > 0 && (n + kv_block - 1) / kv_block > 1;
    *fwd = 1 + ((kv_split || (tc_fwd && kv_block == 0 && gt::fwd_tc_balanced_ctas(n) > 0)) ? 1 : 0);
    if (!(dtype == GT_BF16 && gt::bwd_tc_supported(h, d, nb))) {
        *bwd = 4;   // D, rows, columns, dT
        return GT_OK;
    }
    // prep, dq, dk/dv, and the finish (fp32 sums and dT converted); a tail split
    // adds its second launch when whole tasks fill waves before it
    int count = 4;
    if (gt::bwd_tail(dtype, n, h, d, nb) > 1 && 2 * ((n + 127) / 128) >= gt::num_sms()) count += 1;
    if (gt::bwd_dq_tail(dtype, n, h, d, nb) > 1 && 2 * ((n + 127) / 128) >= 2 * gt::num_sms()) count += 1;
    *bwd = count;
    return GT_OK;
}

int gt_bias_attn_fwd(int32_t dtype, int32_t n, int32_t h, int32_t d, const void* q, const void* k,
                     const void* v, const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb,
                     float scale, int32_t kv_block, void* o, float* lse, void* workspace,
                     size_t ws_bytes, void* stream) {
    int rc = gt::check_common(dtype, n, h, d, q, k, v, spd, ld_spd, T, nb);
    if (rc != GT_OK) return rc;
    if (!o || !lse || !gt::aligned16(o)) return GT_ERR_INVALID_ARG;
    if (kv_block < 0 || (kv_block > 0 && kv_block % 128 != 0)) return GT_ERR_INVALID_ARG;
    if (kv_block >= n) kv_block = 0;
    const size_t need = gt::fwd_ws(dtype, n, h, d, kv_block, nullptr, 0, nullptr);
    if (need > 0 && (!workspace || ws_bytes < need)) return GT_ERR_WORKSPACE;
    gt::FwdWs w;
    gt::fwd_ws(dtype, n, h, d, kv_block, workspace, ws_bytes, &w);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == GT_BF16 && gt::fwd_tc_supported(h, d))
        return gt::attn_fwd_tc(n, d, q, k, v, spd, ld_spd, T, nb, scale, kv_block, o, lse, w.o_part,
                               w.lse_part, s);
    return gt::attn_fwd_simt(dtype, n, h, d, q, k, v, spd, ld_spd, T, nb, scale, kv_block, o, lse,
                             w.o_part, w.lse_part, s);
}

int gt_bias_attn_fwd_partial(int32_t dtype, int32_t n, int32_t h, int32_t d, const void* q,
                             const void* k, const void* v, const int8_t* spd, int64_t ld_spd,
                             const float* T, int32_t nb, float scale, int32_t kv_begin,
                             int32_t kv_end, float* o_part, float* lse_part, void* stream) {
    int rc = gt::check_common(dtype, n, h, d, q, k, v, spd, ld_spd, T, nb);
    if (rc != GT_OK) return rc;
    if (!o_part || !lse_part || !gt::aligned16(o_part)) return GT_ERR_INVALID_ARG;
    if (kv_begin < 0 || kv_begin % 128 != 0 || kv_end <= kv_begin || kv_end > n) return GT_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == GT_BF16 && gt::fwd_tc_supported(h, d))
        return gt::attn_fwd_tc_range(n, d, q, k, v, spd, ld_spd, T, nb, scale, kv_begin, kv_end, o_part,
                                     lse_part, s);
    return gt::attn_fwd_simt_range(dtype, n, h, d, q, k, v, spd, ld_spd, T, nb, scale, kv_begin, kv_end,
                                   o_part, lse_part, s);
}

int gt_bias_attn_merge(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t nparts,
                       const float* o_parts, const float* lse_parts, void* o, float* lse, void* stream) {
    if (!gt::valid_dtype(dtype) || n < 1 || h < 1 || d < 1 || nparts < 1) return GT_ERR_INVALID_ARG;
    if (h > 16 || d > 64) return GT_ERR_UNSUPPORTED;
    if (!o_parts || !lse_parts || !o || !lse) return GT_ERR_INVALID_ARG;
    return gt::merge_partials(dtype, n, h, d, nparts, o_parts, lse_parts, o, lse,
                              static_cast<cudaStream_t>(stream));
}

int gt_bias_attn_bwd(int32_t dtype, int32_t n, int32_t h, int32_t d, const void* q, const void* k,
                     const void* v, const void* o, const void* dO, const float* lse,
                     const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb, float scale,
                     void* dq, void* dk, void* dv, float* dT, void* workspace, size_t ws_bytes,
                     void* stream) {
    int rc = gt::check_common(dtype, n, h, d, q, k, v, spd, ld_spd, T, nb);
    if (rc != GT_OK) return rc;
    if (!o || !dO || !lse || !dq || !dk || !dv || !dT) return GT_ERR_INVALID_ARG;
    if (!gt::aligned16(o) || !gt::aligned16(dO) || !gt::aligned16(dq) || !gt::aligned16(dk) ||
        !gt::aligned16(dv))
        return GT_ERR_INVALID_ARG;
    // the splits need their accumulators; a workspace sized for the unsplit pass
    // (a caller's fixed scratch) runs unsplit
    int tail = gt::bwd_tail(dtype, n, h, d, nb);
    int dq_tail = gt::bwd_dq_tail(dtype, n, h, d, nb);
    bool with_acc = tail > 1 || dq_tail > 1;
    if (with_acc && ws_bytes < gt::bwd_ws(n, h, d, true, nullptr, 0, nullptr)) {
        with_acc = false;
        tail = dq_tail = 1;
    }
    const size_t need = gt::bwd_ws(n, h, d, with_acc, nullptr, 0, nullptr);
    if (!workspace || ws_bytes < need) return GT_ERR_WORKSPACE;
    gt::BwdWs w;
    gt::bwd_ws(n, h, d, with_acc, workspace, ws_bytes, &w);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (dtype == GT_BF16 && gt::bwd_tc_supported(h, d, nb))
        return gt::attn_bwd_tc(n, d, q, k, v, o, dO, lse, spd, ld_spd, T, nb, scale, dq, dk, dv, dT,
                               w.LD, w.LB, w.Dv, w.dT64, w.aux, tail, dq_tail, w.acc, s);
    return gt::attn_bwd_simt(dtype, n, h, d, q, k, v, o, dO, lse, spd, ld_spd, T, nb, scale, dq, dk,
                             dv, dT, w.Dv, w.dT64, s);
}

int gt_check_device_status(void* stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return GT_ERR_CUDA;
    int* p = gt::device_status_ptr();
    if (!p) return GT_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyAsync(&word, p, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return GT_ERR_CUDA;
    if (cudaMemsetAsync(p, 0, sizeof(int), s) != cudaSuccess) return GT_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return GT_ERR_CUDA;
    if (word & gt::kStatusTimeout) return GT_ERR_TIMEOUT;
    return GT_OK;
}

}  // extern "C"

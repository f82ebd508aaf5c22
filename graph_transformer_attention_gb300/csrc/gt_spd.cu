// gt_spd.cu -- clipped shortest-path buckets of an undirected graph.
//
// spd[i][j] = min(dist(i,j), D) for reachable pairs, D+1 otherwise (the
// topology behind the bias matrix of the MegaGraph abstract; Graphormer's
// spatial-encoding buckets).
//
// Design (one GPU, CSR in HBM):
//  1. Connected components by lock-free union-find (hook the larger root under
//     the smaller with atomicCAS, then compress).  Pairs that the breadth-first
//     search below does not reach within D-1 levels get D when they share a
//     component and D+1 when they do not.
//  2. Bit-parallel multi-source BFS: each CTA owns a batch of 32 consecutive
//     sources, one bit per source in a 32-bit word per vertex, and pushes into
//     a shared-memory word per vertex (bfs32_smem; when 4 n bytes do not fit in
//     shared memory, batches of 64 with 64-bit words pushed in global memory,
//     bfs_batches).  A level pushes
//     the frontier word of every queued vertex to its neighbours with atomicOr
//     (work is proportional to the edges of the active frontier, so a batch that
//     lives in one small component touches only that component), then keeps the
//     bits not seen before.  Distances are stored bit-sliced: slice k holds bit k
//     of the level at which each source reached the vertex.
//  3. The same CTA writes its 64 output rows, 4 bytes per store, coalesced along
//     the row, then clears only the state it touched.
// Every loop is bounded: union-find retries and the level loop have hard caps.
#include <cuda_runtime.h>
#include <stdint.h>

#include "gt_common.cuh"
#include "gt_stats.cuh"

namespace gt {
namespace {

constexpr int kSpdThreads = 1024;
constexpr int kUfRetryCap = 1 << 22;

__device__ __forceinline__ int uf_find(int* parent, int x) {
    // Path halving; parents only ever move to smaller ids, so this terminates.
    for (int it = 0; it < (1 << 30); ++it) {
        int p = __ldcg(parent + x);
        if (p == x) return x;
        int gp = __ldcg(parent + p);
        if (gp != p) atomicMin(parent + x, gp);
        x = gp;
    }
    return x;
}

__global__ void uf_init(int* parent, int n) {
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < n; v += gridDim.x * blockDim.x)
        parent[v] = v;
}

// One warp per vertex u, lanes over its neighbours; each edge (u, w) with w > u
// unites the two trees.
__global__ void uf_hook(const int64_t* __restrict__ indptr, const int32_t* __restrict__ indices,
                        int* parent, int n, int* status) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int u = warp; u < n; u += nwarps) {
        const int64_t e0 = indptr[u], e1 = indptr[u + 1];
        for (int64_t e = e0 + lane; e < e1; e += 32) {
            int w = indices[e];
            if (w <= u || w >= n) continue;
            int a = u, b = w;
            int tries = 0;
            while (true) {
                a = uf_find(parent, a);
                b = uf_find(parent, b);
                if (a == b) break;
                if (a > b) { int t = a; a = b; b = t; }
                // hook root b under the smaller root a
                if (atomicCAS(parent + b, b, a) == b) break;
                if (++tries > kUfRetryCap) { atomicOr(status, kStatusTimeout); break; }
            }
        }
    }
}

__global__ void uf_compress(int* parent, int n) {
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < n; v += gridDim.x * blockDim.x)
        parent[v] = uf_find(parent, v);
}

struct BfsState {
    uint64_t* vis;     // [n] sources that reached v
    uint64_t* fr;      // [n] bits new at v in the previous level
    uint64_t* acc;     // [n] bits pushed to v in the current level
    uint64_t* db;      // [nslices][n] bit-sliced distances
    int32_t* qa;       // [n] frontier queue
    int32_t* qb;       // [n] next frontier queue
    int32_t* cand;     // [n] vertices that received a push this level
    int32_t* touched;  // [n] vertices with vis != 0
};

__device__ __forceinline__ BfsState bfs_slice(char* base, size_t per_cta, int cta, int n, int nslices) {
    char* p = base + per_cta * (size_t)cta;
    BfsState s;
    size_t w = (size_t)n * sizeof(uint64_t);
    s.vis = reinterpret_cast<uint64_t*>(p); p += w;
    s.fr = reinterpret_cast<uint64_t*>(p); p += w;
    s.acc = reinterpret_cast<uint64_t*>(p); p += w;
    s.db = reinterpret_cast<uint64_t*>(p); p += w * (size_t)nslices;
    size_t q = (size_t)n * sizeof(int32_t);
    s.qa = reinterpret_cast<int32_t*>(p); p += q;
    s.qb = reinterpret_cast<int32_t*>(p); p += q;
    s.cand = reinterpret_cast<int32_t*>(p); p += q;
    s.touched = reinterpret_cast<int32_t*>(p);
    return s;
}

// Four codes of columns 4c..4c+3 of one output row; the ragged end of the row
// is written byte by byte so that columns >= n stay untouched.
__device__ __forceinline__ void store_codes(int8_t* row, int c, int n, uint32_t word) {
    if (4 * c + 4 <= n) {
        *reinterpret_cast<uint32_t*>(row + 4 * c) = word;
    } else {
        for (int t = 0; 4 * c + t < n; ++t) row[4 * c + t] = (int8_t)(word >> (8 * t));
    }
}

__global__ void __launch_bounds__(kSpdThreads)
bfs_batches(const int64_t* __restrict__ indptr, const int32_t* __restrict__ indices,
            const int* __restrict__ comp, int n, int D, int nslices,
            int8_t* __restrict__ spd, int64_t ld, char* ws, size_t per_cta) {
    __shared__ int s_qlen, s_nlen, s_clen, s_tlen;
    __shared__ int s_comp[64];
    BfsState st = bfs_slice(ws, per_cta, blockIdx.x, n, nslices);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int nbatches = (n + 63) / 64;

    for (int batch = blockIdx.x; batch < nbatches; batch += gridDim.x) {
        const int s0 = batch * 64;
        const int nsrc = min(64, n - s0);
        // level 0: every source reaches itself
        if (tid < nsrc) {
            int s = s0 + tid;
            st.vis[s] = 1ull << tid;
            st.fr[s] = 1ull << tid;
            st.qa[tid] = s;
            st.touched[tid] = s;
            s_comp[tid] = comp[s];
        }
        if (tid == 0) { s_qlen = nsrc; s_tlen = nsrc; }
        __syncthreads();

        int32_t* q = st.qa;
        int32_t* qn = st.qb;
        for (int level = 1; level < D; ++level) {
            const int qlen = s_qlen;
            if (qlen == 0) break;
            if (tid == 0) { s_clen = 0; s_nlen = 0; }
            __syncthreads();
            // push: one warp per queued vertex, lanes over its neighbours
            for (int qi = warp; qi < qlen; qi += nwarps) {
                const int u = q[qi];
                const uint64_t w = st.fr[u];
                const int64_t e0 = indptr[u], e1 = indptr[u + 1];
                for (int64_t e = e0 + lane; e < e1; e += 32) {
                    const int v = indices[e];
                    if ((unsigned)v >= (unsigned)n) continue;
                    unsigned long long old = atomicOr(reinterpret_cast<unsigned long long*>(st.acc + v),
                                                      (unsigned long long)w);
                    if (old == 0ull) st.cand[atomicAdd(&s_clen, 1)] = v;
                }
            }
            __syncthreads();
            const int clen = s_clen;
            // keep the bits not seen before (acc is only touched in L2)
            for (int ci = tid; ci < clen; ci += blockDim.x) {
                const int v = st.cand[ci];
                const uint64_t a = __ldcg(reinterpret_cast<const unsigned long long*>(st.acc + v));
                __stcg(reinterpret_cast<unsigned long long*>(st.acc + v), 0ull);
                const uint64_t seen = st.vis[v];
                const uint64_t nw = a & ~seen;
                if (nw) {
                    if (seen == 0) st.touched[atomicAdd(&s_tlen, 1)] = v;
                    st.vis[v] = seen | nw;
                    st.fr[v] = nw;
                    for (int k = 0; k < nslices; ++k)
                        if ((level >> k) & 1) st.db[(size_t)k * n + v] |= nw;
                    qn[atomicAdd(&s_nlen, 1)] = v;
                }
            }
            __syncthreads();
            if (tid == 0) s_qlen = s_nlen;
            int32_t* t = q; q = qn; qn = t;
            __syncthreads();
        }

        // write rows s0 .. s0+nsrc-1, four columns per store
        const int nchunks = (n + 3) / 4;
        const int8_t Dc = (int8_t)D, Dfar = (int8_t)(D + 1);
        for (int c = tid; c < nchunks; c += blockDim.x) {
            uint64_t vis4[4];
            int comp4[4];
            bool any = false;
            for (int t = 0; t < 4; ++t) {
                int v = 4 * c + t;
                vis4[t] = v < n ? st.vis[v] : 0ull;
                comp4[t] = v < n ? comp[v] : -1;
                any |= vis4[t] != 0ull;
            }
            if (!any) {
                for (int b = 0; b < nsrc; ++b) {
                    const int cs = s_comp[b];
                    uint32_t word = 0;
                    for (int t = 0; t < 4; ++t)
                        word |= (uint32_t)(uint8_t)(comp4[t] == cs ? Dc : Dfar) << (8 * t);
                    store_codes(spd + (int64_t)(s0 + b) * ld, c, n, word);
                }
            } else {
                uint64_t db4[4][7];
                for (int t = 0; t < 4; ++t) {
                    int v = 4 * c + t;
                    for (int k = 0; k < 7; ++k)
                        db4[t][k] = (v < n && k < nslices) ? st.db[(size_t)k * n + v] : 0ull;
                }
                for (int b = 0; b < nsrc; ++b) {
                    const int cs = s_comp[b];
                    uint32_t word = 0;
                    for (int t = 0; t < 4; ++t) {
                        int code;
                        if ((vis4[t] >> b) & 1ull) {
                            code = 0;
                            for (int k = 0; k < 7; ++k) code |= (int)((db4[t][k] >> b) & 1ull) << k;
                        } else {
                            code = comp4[t] == cs ? D : D + 1;
                        }
                        word |= (uint32_t)(uint8_t)code << (8 * t);
                    }
                    store_codes(spd + (int64_t)(s0 + b) * ld, c, n, word);
                }
            }
        }
        __syncthreads();
        // clear what this batch touched
        const int tlen = s_tlen;
        for (int ti = tid; ti < tlen; ti += blockDim.x) {
            const int v = st.touched[ti];
            st.vis[v] = 0;
            for (int k = 0; k < nslices; ++k) st.db[(size_t)k * n + v] = 0;
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------------------
// Batches of 32 sources with the per-level pushes into shared memory: one
// 32-bit word per vertex (acc, 4 N bytes) holds the source bits pushed to it
// in the current level, so the pushes are shared-memory atomicOr instead of
// global ones.  Used whenever 4 N bytes fit in shared memory; the queue of a
// level carries each frontier vertex with its new bits.

struct Bfs32State {
    uint32_t* vis;     // [n] sources that reached v
    uint32_t* db;      // [nslices][n] bit-sliced distances
    int32_t* qv0;      // frontier queues (two, alternating): vertex
    int32_t* qv1;
    uint32_t* qw0;     // and its bits new in the previous level
    uint32_t* qw1;
    int32_t* cand;     // [n] vertices that received a push this level
    int32_t* touched;  // [n] vertices with vis != 0
    int32_t* heavy;    // [n] queue slots of frontier vertices pushed by a whole warp
};

size_t per_cta_bytes32(int n, int nslices) {
    const size_t w = (size_t)n * 4;
    const size_t b = w * (size_t)(1 + nslices) + 7 * w;
    return (b + 255) & ~size_t(255);
}

__device__ __forceinline__ Bfs32State bfs32_slice(char* base, size_t per_cta, int cta, int n, int nslices) {
    char* p = base + per_cta * (size_t)cta;
    const size_t w = (size_t)n * 4;
    Bfs32State s;
    s.vis = reinterpret_cast<uint32_t*>(p); p += w;
    s.db = reinterpret_cast<uint32_t*>(p); p += w * (size_t)nslices;
    s.qv0 = reinterpret_cast<int32_t*>(p); p += w;
    s.qv1 = reinterpret_cast<int32_t*>(p); p += w;
    s.qw0 = reinterpret_cast<uint32_t*>(p); p += w;
    s.qw1 = reinterpret_cast<uint32_t*>(p); p += w;
    s.cand = reinterpret_cast<int32_t*>(p); p += w;
    s.touched = reinterpret_cast<int32_t*>(p); p += w;
    s.heavy = reinterpret_cast<int32_t*>(p);
    return s;
}

// Appends `val` (for lanes with `take`) to list[*counter ...] with one shared
// atomic per group of converged lanes; every active lane must call it.
__device__ __forceinline__ void warp_append(bool take, int* counter, int32_t* list, int32_t val,
                                            uint32_t* list2 = nullptr, uint32_t val2 = 0) {
    const unsigned active = __activemask();
    const unsigned mask = __ballot_sync(active, take);
    if (!mask) return;
    const int lane = threadIdx.x & 31;
    const int leader = __ffs(mask) - 1;
    int base = 0;
    if (lane == leader) base = atomicAdd(counter, __popc(mask));
    base = __shfl_sync(active, base, leader);
    if (take) {
        const int at = base + __popc(mask & ((1u << lane) - 1u));
        list[at] = val;
        if (list2) list2[at] = val2;
    }
}

constexpr int kLightDeg = 32;   // frontier vertices up to this degree: one thread each

__global__ void __launch_bounds__(kSpdThreads)
bfs32_smem(const int64_t* __restrict__ indptr, const int32_t* __restrict__ indices,
           const int* __restrict__ comp, int n, int D, int nslices, int8_t* __restrict__ spd,
           int64_t ld, char* ws, size_t per_cta) {
    extern __shared__ uint32_t acc[];          // [n], zero between levels
    __shared__ int s_qlen, s_nlen, s_clen, s_tlen, s_hlen;
    __shared__ int s_comp[32];
    Bfs32State st = bfs32_slice(ws, per_cta, blockIdx.x, n, nslices);
    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int nbatches = (n + 31) / 32;
    for (int v = tid; v < n; v += blockDim.x) acc[v] = 0u;
    __syncthreads();

    for (int batch = blockIdx.x; batch < nbatches; batch += gridDim.x) {
        const int s0 = batch * 32;
        const int nsrc = min(32, n - s0);
        if (tid < nsrc) {
            const int s = s0 + tid;
            st.vis[s] = 1u << tid;
            st.qv0[tid] = s;
            st.qw0[tid] = 1u << tid;
            st.touched[tid] = s;
            s_comp[tid] = comp[s];
        }
        if (tid == 0) { s_qlen = nsrc; s_tlen = nsrc; }
        __syncthreads();
        int cur = 0;
        for (int level = 1; level < D; ++level) {
            const int qlen = s_qlen;
            if (qlen == 0) break;
            if (tid == 0) { s_clen = 0; s_nlen = 0; s_hlen = 0; }
            __syncthreads();
            // push: one thread per queued vertex of small degree (many loads in flight);
            // vertices of larger degree are set aside for one warp each
            const int32_t* qv = cur ? st.qv1 : st.qv0;
            const uint32_t* qw = cur ? st.qw1 : st.qw0;
            int32_t* heavy = st.heavy;
            // (a short queue goes to the warps whole: lanes over the edges)
            const int light_deg = qlen <= 4 * nwarps ? 0 : kLightDeg;
            for (int qi = tid; qi < qlen; qi += blockDim.x) {
                const int u = qv[qi];
                const uint32_t w = qw[qi];
                const int64_t e0 = indptr[u], e1 = indptr[u + 1];
                if (e1 - e0 > light_deg) {
                    heavy[atomicAdd(&s_hlen, 1)] = qi;
                    continue;
                }
                // four neighbour loads in flight at a time, then their pushes
                for (int64_t e = e0; e < e1; e += 4) {
                    int vv[4];
#pragma unroll
                    for (int k = 0; k < 4; ++k) vv[k] = e + k < e1 ? __ldg(indices + e + k) : -1;
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        bool fresh = false;
                        if ((unsigned)vv[k] < (unsigned)n) fresh = atomicOr(&acc[vv[k]], w) == 0u;
                        warp_append(fresh, &s_clen, st.cand, vv[k]);
                    }
                }
            }
            __syncthreads();
            const int hlen = s_hlen;
            for (int hi = warp; hi < hlen; hi += nwarps) {
                const int qi = heavy[hi];
                const int u = qv[qi];
                const uint32_t w = qw[qi];
                const int64_t e0 = indptr[u], e1 = indptr[u + 1];
                for (int64_t e0l = e0; e0l < e1; e0l += 32) {
                    const int64_t e = e0l + lane;
                    bool fresh = false;
                    int v = -1;
                    if (e < e1) {
                        v = indices[e];
                        if ((unsigned)v < (unsigned)n) fresh = atomicOr(&acc[v], w) == 0u;
                    }
                    warp_append(fresh, &s_clen, st.cand, v);
                }
            }
            __syncthreads();
            const int clen = s_clen;
            // keep the bits not seen before
            int32_t* nqv = cur ? st.qv0 : st.qv1;
            uint32_t* nqw = cur ? st.qw0 : st.qw1;
            for (int c0 = 0; c0 < clen; c0 += blockDim.x) {
                const int ci = c0 + tid;
                int v = -1;
                uint32_t nw = 0, seen = 0;
                if (ci < clen) {
                    v = st.cand[ci];
                    const uint32_t a = acc[v];
                    acc[v] = 0u;
                    seen = st.vis[v];
                    nw = a & ~seen;
                    if (nw) {
                        st.vis[v] = seen | nw;
                        for (int k = 0; k < nslices; ++k)
                            if ((level >> k) & 1) st.db[(size_t)k * n + v] |= nw;
                    }
                }
                warp_append(nw != 0u && seen == 0u, &s_tlen, st.touched, v);
                warp_append(nw != 0u, &s_nlen, nqv, v, nqw, nw);
            }
            __syncthreads();
            if (tid == 0) s_qlen = s_nlen;
            cur ^= 1;
            __syncthreads();
        }

        // write rows s0 .. s0+nsrc-1, four columns per store
        const int nchunks = (n + 3) / 4;
        const int8_t Dc = (int8_t)D, Dfar = (int8_t)(D + 1);
        for (int c = tid; c < nchunks; c += blockDim.x) {
            uint32_t vis4[4];
            int comp4[4];
            bool any = false;
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int v = 4 * c + t;
                vis4[t] = v < n ? st.vis[v] : 0u;
                comp4[t] = v < n ? comp[v] : -1;
                any |= vis4[t] != 0u;
            }
            if (!any) {
                for (int b = 0; b < nsrc; ++b) {
                    const int cs = s_comp[b];
                    uint32_t word = 0;
#pragma unroll
                    for (int t = 0; t < 4; ++t)
                        word |= (uint32_t)(uint8_t)(comp4[t] == cs ? Dc : Dfar) << (8 * t);
                    store_codes(spd + (int64_t)(s0 + b) * ld, c, n, word);
                }
            } else {
                uint32_t db4[4][7];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int v = 4 * c + t;
#pragma unroll
                    for (int k = 0; k < 7; ++k)
                        db4[t][k] = (v < n && k < nslices) ? st.db[(size_t)k * n + v] : 0u;
                }
                for (int b = 0; b < nsrc; ++b) {
                    const int cs = s_comp[b];
                    uint32_t word = 0;
#pragma unroll
                    for (int t = 0; t < 4; ++t) {
                        int code;
                        if ((vis4[t] >> b) & 1u) {
                            code = 0;
#pragma unroll
                            for (int k = 0; k < 7; ++k) code |= (int)((db4[t][k] >> b) & 1u) << k;
                        } else {
                            code = comp4[t] == cs ? D : D + 1;
                        }
                        word |= (uint32_t)(uint8_t)code << (8 * t);
                    }
                    store_codes(spd + (int64_t)(s0 + b) * ld, c, n, word);
                }
            }
        }
        __syncthreads();
        // clear what this batch touched
        const int tlen = s_tlen;
        for (int ti = tid; ti < tlen; ti += blockDim.x) {
            const int v = st.touched[ti];
            st.vis[v] = 0u;
            for (int k = 0; k < nslices; ++k) st.db[(size_t)k * n + v] = 0u;
        }
        __syncthreads();
    }
}

// Largest n whose 4 n-byte push words fit the shared memory of one CTA.
int bfs32_max_n() {
    static int cached = -1;
    if (cached < 0) {
        int dev = 0, optin = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cached = (optin - 1024) / 4;
    }
    return cached;
}

int slices_for(int D) {
    int s = 0;
    while ((1 << s) <= D - 1) ++s;   // levels recorded are 1 .. D-1
    return s;
}

size_t per_cta_bytes(int n, int nslices) {
    size_t b = (size_t)n * sizeof(uint64_t) * (size_t)(3 + nslices) + (size_t)n * sizeof(int32_t) * 4;
    return (b + 255) & ~size_t(255);
}

int spd_ctas(int n) {
    int nb = (n + 63) / 64;
    int sms = num_sms();
    return nb < sms ? nb : sms;
}

}  // namespace

// The BFS runs in batches of 32 sources with shared-memory pushes when 4 n
// bytes fit in shared memory, else in batches of 64 with global pushes.
bool use_bfs32(int n) { return n <= bfs32_max_n(); }

int spd_ctas32(int n) {
    int nb = (n + 31) / 32;
    int sms = num_sms();
    return nb < sms ? nb : sms;
}

size_t bfs_state_bytes(int n, int nslices, size_t* per, int* nctas) {
    if (use_bfs32(n)) {
        *per = per_cta_bytes32(n, nslices);
        *nctas = spd_ctas32(n);
    } else {
        *per = per_cta_bytes(n, nslices);
        *nctas = spd_ctas(n);
    }
    return *per * (size_t)*nctas;
}

size_t spd_workspace_bytes(int32_t n, int32_t D) {
    Carve c(nullptr, 0);
    c.take<int>((size_t)n);
    size_t per = 0;
    int nctas = 0;
    c.take<char>(bfs_state_bytes(n, slices_for(D), &per, &nctas));
    return c.off + 256;
}

int spd_build(const int64_t* indptr, const int32_t* indices, int32_t n, int32_t D,
              int8_t* spd, int64_t ld, void* ws, size_t ws_bytes, cudaStream_t stream) {
    Carve c(ws, ws_bytes);
    int* comp = c.take<int>((size_t)n);
    const int nslices = slices_for(D);
    size_t per = 0;
    int nctas = 0;
    char* bfs_ws = c.take<char>(bfs_state_bytes(n, nslices, &per, &nctas));
    if (!c.fits()) return GT_ERR_WORKSPACE;
    int* status = device_status_ptr();
    if (!status) return GT_ERR_CUDA;
    const int sms = num_sms();
    {
        LaunchScope ls("spd_uf_init", stream);
        uf_init<<<sms * 4, 256, 0, stream>>>(comp, n);
    }
    {
        LaunchScope ls("spd_uf_hook", stream);
        uf_hook<<<sms * 8, 256, 0, stream>>>(indptr, indices, comp, n, status);
    }
    {
        LaunchScope ls("spd_uf_compress", stream);
        uf_compress<<<sms * 4, 256, 0, stream>>>(comp, n);
    }
    // the BFS keeps vis / acc / db zero between batches; start from zero
    if (cudaMemsetAsync(bfs_ws, 0, per * (size_t)nctas, stream) != cudaSuccess) return GT_ERR_CUDA;
    if (use_bfs32(n)) {
        const size_t smem = (size_t)n * 4;
        if (cudaFuncSetAttribute(bfs32_smem, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) !=
            cudaSuccess)
            return GT_ERR_CUDA;
        LaunchScope ls("spd_bfs", stream);
        bfs32_smem<<<nctas, kSpdThreads, smem, stream>>>(indptr, indices, comp, n, D, nslices, spd, ld,
                                                         bfs_ws, per);
    } else {
        LaunchScope ls("spd_bfs", stream);
        bfs_batches<<<nctas, kSpdThreads, 0, stream>>>(indptr, indices, comp, n, D, nslices, spd, ld,
                                                       bfs_ws, per);
    }
    return check_launch();
}

}  // namespace gt

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
//  3. The same CTA writes its output rows, coalesced along the row, then clears
//     only the state it touched.
//  The default search (bfs_scan, below) keeps all per-vertex words of a batch of
//  32 or 16 sources in shared memory and works on the range of vertex ids the
//  batch has touched; bfs32_smem and bfs_batches take graphs too large for it.
// Every loop is bounded: union-find retries and the level loop have hard caps.
#include <cuda_runtime.h>
#include <climits>
#include <stdint.h>

#include "gt_common.cuh"
#include "gt_stats.cuh"
#include "gt_sm100.cuh"

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

// The same union over the packed edge list (`target | source << 16` per CSR
// entry, csr_pairs): one thread per entry, so a vertex's few edges do not leave
// the rest of a warp idle behind its dependent loads.
__global__ void uf_hook_pairs(const uint32_t* __restrict__ pairs, int64_t nnz, int* parent, int n, int* status) {
    sm100::pdl_wait();      // launched to overlap csr_pairs, which writes the pairs and the roots
    sm100::pdl_trigger();
    for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < nnz; e += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t pr = pairs[e];
        const int w = (int)(pr & 0xffffu), u = (int)(pr >> 16);
        if (w <= u || w >= n) continue;
        // link root b under the smaller root a with an atomic min; if b had
        // already been linked (to c), the min keeps the smaller of a and c, and
        // the larger of the two still has to be joined to it: continue with that
        // pair (parents only move to smaller ids, so this ends)
        int a = uf_find(parent, u), b = uf_find(parent, w);
        int tries = 0;
        while (a != b) {
            if (a > b) { int t = a; a = b; b = t; }
            const int c = atomicMin(parent + b, a);
            if (c == b) break;                     // b was a root: linked
            b = uf_find(parent, c);                // c or a is now b's parent: join the other
            a = uf_find(parent, a);
            if (++tries > kUfRetryCap) { atomicOr(status, kStatusTimeout); break; }
        }
    }
}

__global__ void uf_compress(int* parent, int n) {
    sm100::pdl_wait();      // may be launched to overlap the hook kernel
    sm100::pdl_trigger();
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
// Bits 0..3 of x to the low bit of bytes 0..3 (the four shifted copies of x
// occupy disjoint bit ranges, so the product has no carries).
__device__ __forceinline__ uint32_t spread4(uint32_t x) { return (x * 0x00204081u) & 0x01010101u; }

// store_codes with an evict-first store: the N^2 output streams through L2
// without displacing the graph and the search state.
__device__ __forceinline__ void store_codes_cs(int8_t* row, int c, int n, uint32_t word) {
    if (4 * c + 4 <= n) {
        __stcs(reinterpret_cast<unsigned int*>(row + 4 * c), word);
    } else {
        for (int t = 0; 4 * c + t < n; ++t) row[4 * c + t] = (int8_t)(word >> (8 * t));
    }
}

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

// ---------------------------------------------------------------------------
// Batches of W sources with every per-vertex word in shared memory: acc (the
// bits pushed to a vertex in the current level), vis (the bits that reached it)
// and fr (the bits new at it in the previous level).  W = 32 keeps one 32-bit
// word per vertex (12 n bytes of shared memory); W = 16 packs two vertices per
// word (6 n bytes), for graphs too large for the first.  Only the bit-sliced
// distances are in global memory: nslices words per vertex word per CTA, small
// enough to stay in L2.  A level works on the range of vertex ids the batch has
// touched so far ([s_lo, s_hi]) and is a push or a pull, then an update:
//   push, flat   (frontier at least 1/8 of the range) the range's CSR entries,
//                as 32-bit pairs target | source << 16, split evenly over the
//                warps; frontier bits of the source from shared memory, atomicOr
//                into the target's acc; eight 32-entry chunks of loads in flight.
//   push, block  (small frontier) one warp per block of 32 consecutive vertices
//                that holds a frontier vertex: a mostly active block walks its
//                whole CSR segment; a sparse one walks only the edges of its
//                frontier vertices as one virtual segment (lane l's edges at
//                pre_l .. pre_l + len_l - 1), each lane finding its position's
//                vertex by a binary search over the lanes' pre values; the next
//                active block's row starts are loaded while one is walked.
//   pull         (the range is the whole graph and fewer vertices are open than
//                in the frontier) each open vertex ORs its neighbours' frontier
//                bits and stops once it has every bit it lacks; no atomics.
//   update       one thread per word keeps the bits not seen before, records them
//                in the slices of the level, makes them the next frontier, and
//                counts frontier and open vertices for the next level's choice.
// The search ends when an update finds no new bit, or at level D - 1.  The batch's
// rows then go out: 16-column groups outside the touched range by component only,
// 16-byte evict-first stores; the others four rows at a time from the slices.
// One CTA of 1024 threads per SM, or two of 512 when two fit the SM's shared
// memory and the batches outnumber the SMs (a level ends at a CTA-wide barrier, and
// the other CTA's output pass fills that wait).

constexpr int kScanThreads = 1024;
constexpr int kPushChunks = 4;     // 32-edge chunks whose index loads a lane has in flight
constexpr int kFlatChunks = 8;     // the same for the flat push
constexpr int kUpdateWords = 4;    // words per thread whose slice updates overlap

template <int W>
struct ScanWords {
    static constexpr int VPW = 32 / W;                       // vertices per 32-bit word
    static constexpr uint32_t MASK = W == 32 ? 0xffffffffu : 0xffffu;
    __device__ static __forceinline__ int word(int v) { return VPW == 1 ? v : v >> 1; }
    __device__ static __forceinline__ int shift(int v) { return VPW == 1 ? 0 : (v & 1) << 4; }
};

// words per shared array (and per distance slice): the vertex words rounded up
// so that the output pass's last group of four columns stays inside
__host__ __device__ inline int scan_nwp(int n, int W) {
    const int vpw = 32 / W;
    const int nwords = (n + vpw - 1) / vpw;
    return (nwords + 2 + 3) & ~3;
}

// pairs[e] = indices[e] | (the vertex whose adjacency list holds CSR entry e) << 16:
// one 4-byte load gives a push's target and source (vertex ids of the
// shared-memory searches fit 16 bits; an entry outside 0..n-1 is stored as
// 0xffff, which is >= n and so never pushed).  One warp per vertex; entries
// outside [0, nnz) are never written.
__global__ void csr_pairs(const int64_t* __restrict__ indptr, const int32_t* __restrict__ indices, int n,
                          int64_t nnz, uint32_t* __restrict__ pairs, int* __restrict__ parent) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    sm100::pdl_trigger();   // the hook kernel may launch meanwhile; it waits for this grid
    for (int v = warp; v < n; v += nwarps) {
        if (lane == 0) parent[v] = v;   // union-find roots, for uf_hook_pairs
        const int64_t e0 = max(indptr[v], (int64_t)0), e1 = min(indptr[v + 1], nnz);
        for (int64_t e = e0 + lane; e < e1; e += 32) {
            const int u = indices[e];
            const uint32_t uu = (unsigned)u < (unsigned)n ? (uint32_t)u : 0xffffu;
            pairs[e] = uu | ((uint32_t)v << 16);
        }
    }
}

template <int W>
__global__ void __launch_bounds__(kScanThreads)
bfs_scan(const int64_t* __restrict__ indptr, const int32_t* __restrict__ indices,
         const uint32_t* __restrict__ pairs, const int* __restrict__ comp, int n, int D, int nslices,
         int8_t* __restrict__ spd, int64_t ld, uint32_t* __restrict__ db_all) {
    using SW = ScanWords<W>;
    extern __shared__ uint32_t sw[];
    __shared__ int s_comp[32];
    __shared__ int s_csrc;
    __shared__ int s_lo, s_hi;     // the vertex ids the batch has pushed to lie in [s_lo, s_hi]
    __shared__ int s_nfront[2];    // frontier vertices after the update pass of an odd / even level
    __shared__ int s_nopen[2];     // vertices not reached by every source, the same way
    const int nwp = scan_nwp(n, W);
    uint32_t* acc = sw;
    uint32_t* vis = sw + nwp;
    uint32_t* fr = sw + 2 * nwp;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int nbatches = (n + W - 1) / W;
    uint32_t* db = db_all + (size_t)blockIdx.x * nslices * nwp;
    const unsigned full = 0xffffffffu;
    const bool comp16 = (reinterpret_cast<uintptr_t>(comp) & 15u) == 0;
    for (int p = tid; p < 3 * nwp; p += blockDim.x) sw[p] = 0u;
    // launched to overlap the components kernel: the shared state above is this
    // CTA's own; the components, pairs and global state are read only after it
    sm100::pdl_wait();
    __syncthreads();

    for (int batch = blockIdx.x; batch < nbatches; batch += gridDim.x) {
        const int s0 = batch * W;
        const int nsrc = min(W, n - s0);
        if (tid < nsrc) {
            const int s = s0 + tid;
            const uint32_t bit = 1u << (SW::shift(s) + tid);
            atomicOr(&vis[SW::word(s)], bit);
            atomicOr(&fr[SW::word(s)], bit);
            s_comp[tid] = comp[s];
        }
        if (tid == 0) {
            s_lo = s0;
            s_hi = s0 + nsrc - 1;
            s_nfront[0] = nsrc;
            s_nopen[0] = n;
        }
        __syncthreads();
        if (warp == 0) {
            const int c0 = s_comp[0];
            const bool same = __all_sync(full, lane >= nsrc || s_comp[lane] == c0);
            if (lane == 0) s_csrc = same ? c0 : -1;
        }
        __syncthreads();

        // a vertex is open while some source of the batch has not reached it
        const uint32_t fmask = nsrc == 32 ? 0xffffffffu : (1u << nsrc) - 1u;
        for (int level = 1; level < D; ++level) {
            const int lo = s_lo, hi = s_hi;
            const int nfront = s_nfront[(level - 1) & 1];
            const int nopen = s_nopen[(level - 1) & 1];
            if (tid == 0) {
                s_nfront[level & 1] = 0;
                s_nopen[level & 1] = 0;
            }
            const bool whole = lo == 0 && hi == n - 1;
            int umin = INT_MAX, umax = -1;     // this lane's pushed vertex ids
            if (whole && level > 1 && nopen < nfront) {
            // ---- pull, few open vertices left (the batch has reached every vertex
            // id, so no vertex outside the scanned range can gain bits): each open
            // vertex ORs the frontier bits of its neighbours, stopping once it has
            // every bit it lacks; a thread owns its words, so no atomics
            for (int p = tid; p < (n + SW::VPW - 1) / SW::VPW; p += blockDim.x) {
                const uint32_t seen = vis[p];
                uint32_t got = 0u;
#pragma unroll
                for (int h = 0; h < SW::VPW; ++h) {
                    const int v = p * SW::VPW + h;
                    const uint32_t miss = v < n ? fmask & ~((seen >> SW::shift(v)) & SW::MASK) : 0u;
                    if (!miss) continue;
                    uint32_t g = 0u;
                    const int64_t e1 = __ldg(indptr + v + 1);
                    for (int64_t e = __ldg(indptr + v); e < e1 && (g & miss) != miss; e += 4) {
                        int uu[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) uu[k] = e + k < e1 ? __ldg(indices + e + k) : -1;
#pragma unroll
                        for (int k = 0; k < 4; ++k)
                            if ((unsigned)uu[k] < (unsigned)n) g |= (fr[SW::word(uu[k])] >> SW::shift(uu[k])) & SW::MASK;
                    }
                    got |= (g & miss) << SW::shift(v);
                }
                if (got) acc[p] = got;
            }
            } else if (8 * nfront >= hi - lo + 1) {
            // ---- push, large frontier: the edges of the touched range split evenly
            // over the warps; each edge's source is checked against the frontier
            const int64_t Elo = __ldg(indptr + lo), Ehi = __ldg(indptr + hi + 1);
            const int64_t per = ((Ehi - Elo + nwarps - 1) / nwarps + 31) & ~(int64_t)31;
            const int64_t my0 = min(Elo + warp * per, Ehi);
            const int seg = (int)(min(my0 + per, Ehi) - my0);
            const uint32_t* pr = pairs + my0;
            for (int x = 0; x < seg; x += 32 * kFlatChunks) {
                uint32_t ed[kFlatChunks];
#pragma unroll
                for (int q = 0; q < kFlatChunks; ++q) {
                    const int off = x + 32 * q + lane;
                    ed[q] = off < seg ? __ldg(pr + off) : 0xffffffffu;
                }
#pragma unroll
                for (int q = 0; q < kFlatChunks; ++q) {
                    const int u = (int)(ed[q] & 0xffffu), r = (int)(ed[q] >> 16);
                    if (u < n && r < n) {
                        const uint32_t ww = (fr[SW::word(r)] >> SW::shift(r)) & SW::MASK;
                        if (ww) {
                            atomicOr(&acc[SW::word(u)], ww << SW::shift(u));
                            if (!whole) {                 // the range can still grow
                                umin = min(umin, u);
                                umax = max(umax, u);
                            }
                        }
                    }
                }
            }
            } else {
            // ---- push, small frontier: each warp walks the active blocks of the
            // touched range; the row starts of its next active block are loaded
            // before the current one is walked
            const int blo = lo >> 5, bhi = hi >> 5;
            auto next_block = [&](int b, uint32_t& w, int64_t& st, int64_t& en) -> int {
                for (; b <= bhi; b += nwarps) {
                    const int v = b * 32 + lane;
                    w = v < n ? (fr[SW::word(v)] >> SW::shift(v)) & SW::MASK : 0u;
                    if (__ballot_sync(full, w != 0u)) {
                        st = __ldg(indptr + min(v, n));
                        en = v < n ? __ldg(indptr + v + 1) : st;
                        return b;
                    }
                }
                w = 0u;
                return bhi + 1;
            };
            uint32_t w = 0u;
            int64_t st = 0, en = 0;
            int blk = next_block(blo + warp, w, st, en);
            while (blk <= bhi) {
                uint32_t w2 = 0u;
                int64_t st2 = 0, en2 = 0;
                const int blk2 = next_block(blk + nwarps, w2, st2, en2);
                // the block's active edges as one virtual segment: lane l's edges
                // (if its vertex is active) at positions pre_l .. pre_l + len_l - 1
                const int len = w ? (int)(en - st) : 0;
                int pre = len;
#pragma unroll
                for (int dd = 1; dd < 32; dd <<= 1) {
                    const int t = __shfl_up_sync(full, pre, dd);
                    if (lane >= dd) pre += t;
                }
                const int total = __shfl_sync(full, pre, 31);
                pre -= len;
                const int64_t E0 = __shfl_sync(full, st, 0), E1 = __shfl_sync(full, en, 31);
                if (5 * (int64_t)total >= 2 * (E1 - E0)) {
                    // mostly active: walk all the block's edges, the owner of each
                    // from the row array (inactive owners push nothing)
                    const int vb = blk * 32;
                    const int seg = (int)(E1 - E0);
                    const uint32_t* pr0 = pairs + E0;
                    for (int x = 0; x < seg; x += 32 * kPushChunks) {
                        int u[kPushChunks], o[kPushChunks];
#pragma unroll
                        for (int q = 0; q < kPushChunks; ++q) {
                            const int off = x + 32 * q + lane;
                            u[q] = -1;
                            o[q] = 0;
                            if (off < seg) {
                                const uint32_t ed = __ldg(pr0 + off);
                                u[q] = (int)(ed & 0xffffu);
                                o[q] = (int)(ed >> 16) - vb;
                            }
                        }
#pragma unroll
                        for (int q = 0; q < kPushChunks; ++q) {
                            const uint32_t ww = __shfl_sync(full, w, o[q] & 31);
                            if (ww && (unsigned)u[q] < (unsigned)n) {
                                atomicOr(&acc[SW::word(u[q])], ww << SW::shift(u[q]));
                                umin = min(umin, u[q]);
                                umax = max(umax, u[q]);
                            }
                        }
                    }
                } else {
                    // sparse: only the active edges, each lane finding its position's
                    // vertex by a binary search over the lanes' pre values
                    for (int x = 0; x < total; x += 32 * kPushChunks) {
                        int u[kPushChunks];
                        uint32_t ww[kPushChunks];
#pragma unroll
                        for (int q = 0; q < kPushChunks; ++q) {
                            const int pos = x + 32 * q + lane;
                            int lo = 0;
#pragma unroll
                            for (int step = 16; step > 0; step >>= 1) {
                                const int c = lo + step;
                                if (__shfl_sync(full, pre, c) <= pos) lo = c;
                            }
                            ww[q] = __shfl_sync(full, w, lo);
                            const int64_t so = __shfl_sync(full, st, lo);
                            const int po = __shfl_sync(full, pre, lo);
                            u[q] = pos < total ? __ldg(indices + so + (pos - po)) : -1;
                        }
#pragma unroll
                        for (int q = 0; q < kPushChunks; ++q)
                            if ((unsigned)u[q] < (unsigned)n) {
                                atomicOr(&acc[SW::word(u[q])], ww[q] << SW::shift(u[q]));
                                umin = min(umin, u[q]);
                                umax = max(umax, u[q]);
                            }
                    }
                }
                blk = blk2;
                w = w2;
                st = st2;
                en = en2;
            }
            }
            umin = __reduce_min_sync(full, umin);
            umax = __reduce_max_sync(full, umax);
            if (lane == 0 && umax >= 0) {
                atomicMin(&s_lo, umin);
                atomicMax(&s_hi, umax);
            }
            __syncthreads();
            // ---- update over the touched words, four per thread at a time so that
            // their slice read-modify-writes overlap
            const int wlo = SW::word(s_lo), whi = SW::word(s_hi);
            uint32_t any = 0u;
            int nfv = 0, nov = 0;     // this thread's frontier and open vertices
            for (int p0 = wlo + tid; p0 <= whi; p0 += kUpdateWords * blockDim.x) {
                uint32_t nw[kUpdateWords];
#pragma unroll
                for (int r = 0; r < kUpdateWords; ++r) {
                    const int p = p0 + r * blockDim.x;
                    nw[r] = 0u;
                    if (p <= whi) {
                        const uint32_t a = acc[p];
                        uint32_t seen = vis[p];
                        if (a) {
                            acc[p] = 0u;
                            nw[r] = a & ~seen;
                            seen |= nw[r];
                            vis[p] = seen;
                        }
                        fr[p] = nw[r];
#pragma unroll
                        for (int h = 0; h < SW::VPW; ++h) {
                            const int v = p * SW::VPW + h;
                            if (v < n) {
                                nfv += ((nw[r] >> SW::shift(v)) & SW::MASK) != 0u;
                                nov += ((seen >> SW::shift(v)) & SW::MASK) != fmask;
                            }
                        }
                    }
                    any |= nw[r];
                }
                if (nw[0] | nw[1] | nw[2] | nw[3]) {
                    // the level's bits are new, so the slices take them with
                    // reductions (no read, no wait on L2); the output pass reads
                    // the slices at L2
                    for (int k = 0; k < nslices; ++k) {
                        if (!((level >> k) & 1)) continue;
                        uint32_t* dk = db + (size_t)k * nwp;
#pragma unroll
                        for (int r = 0; r < kUpdateWords; ++r)
                            if (nw[r]) atomicOr(dk + p0 + r * blockDim.x, nw[r]);
                    }
                }
            }
            nfv = __reduce_add_sync(full, nfv);
            nov = __reduce_add_sync(full, nov);
            if (lane == 0) {
                if (nfv) atomicAdd(&s_nfront[level & 1], nfv);
                if (nov) atomicAdd(&s_nopen[level & 1], nov);
            }
            if (!__syncthreads_or(any != 0u)) break;
        }

        // ---- rows s0 .. s0+nsrc-1.  Columns outside the touched range (in
        // 16-column groups) were reached by no source: their codes depend on the
        // component only and go out as 16-byte stores.  The rest, in groups of four
        // columns, build codes four rows at a time: each slice's four row bits of a
        // column are spread to the low bits of four bytes, and a 4 x 4 byte
        // transpose turns the four columns' words into four rows' words; the same
        // thread then clears the words of its columns for the next batch.
        const int csrc = s_csrc;
        const uint32_t Dc = (uint32_t)D, Dfar = (uint32_t)(D + 1);
        const int n16 = n >> 4;                     // full 16-column groups
        const bool fast16 = csrc >= 0 && comp16;
        const int glo = fast16 ? (s_lo >> 4) : 0;
        const int ghi = fast16 ? (s_hi >> 4) : n16;
        if (fast16) {
            for (int g = tid; g < n16; g += blockDim.x) {
                if (g >= glo && g <= ghi) continue;
                const int v0 = 16 * g;
                uint32_t wd[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int4 c4 = __ldg(reinterpret_cast<const int4*>(comp + v0 + 4 * q));
                    wd[q] = (c4.x == csrc ? Dc : Dfar) | (c4.y == csrc ? Dc : Dfar) << 8 |
                            (c4.z == csrc ? Dc : Dfar) << 16 | (c4.w == csrc ? Dc : Dfar) << 24;
                }
                const uint4 wv = make_uint4(wd[0], wd[1], wd[2], wd[3]);
                for (int b = 0; b < nsrc; ++b)
                    __stcs(reinterpret_cast<uint4*>(spd + (int64_t)(s0 + b) * ld + v0), wv);
            }
        }
        // 4-column groups: those of 16-groups glo..ghi, and the ragged tail
        const int c_lo = 4 * glo, c_hi = min(4 * ghi + 3, (n + 3) / 4 - 1);
        const int c_tail = 4 * n16;
        const int nmid = c_hi >= c_lo ? c_hi - c_lo + 1 : 0;
        const int ntail = max(0, (n + 3) / 4 - max(c_tail, c_hi + 1));
        for (int i = tid; i < nmid + ntail; i += blockDim.x) {
            const int c = i < nmid ? c_lo + i : max(c_tail, c_hi + 1) + (i - nmid);
            const int v0 = 4 * c;
            uint32_t vw[4];
            int cp[4];
            uint32_t anyv = 0u;
            if (v0 + 4 <= n && comp16) {
                const int4 c4 = __ldg(reinterpret_cast<const int4*>(comp + v0));
                cp[0] = c4.x; cp[1] = c4.y; cp[2] = c4.z; cp[3] = c4.w;
            } else {
#pragma unroll
                for (int t = 0; t < 4; ++t) cp[t] = v0 + t < n ? comp[v0 + t] : -1;
            }
#pragma unroll
            for (int t = 0; t < 4; ++t) {
                const int v = v0 + t;
                vw[t] = v < n ? (vis[SW::word(v)] >> SW::shift(v)) & SW::MASK : 0u;
                anyv |= vw[t];
            }
            if (!anyv && csrc >= 0) {
                uint32_t word = 0;
#pragma unroll
                for (int t = 0; t < 4; ++t) word |= (cp[t] == csrc ? Dc : Dfar) << (8 * t);
                for (int b = 0; b < nsrc; ++b) store_codes_cs(spd + (int64_t)(s0 + b) * ld, c, n, word);
                continue;
            }
            uint32_t dw[4][7];
#pragma unroll
            for (int k = 0; k < 7; ++k) {
#pragma unroll
                for (int t = 0; t < 4; ++t) dw[t][k] = 0u;
                if (k >= nslices) continue;              // uniform: the slices past the count cost nothing
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    const int v = v0 + t;
                    dw[t][k] = (__ldcg(db + (size_t)k * nwp + SW::word(v)) >> SW::shift(v)) & SW::MASK;
                }
            }
            for (int b0 = 0; b0 < nsrc; b0 += 4) {
                uint32_t col[4];
#pragma unroll
                for (int t = 0; t < 4; ++t) {
                    uint32_t code4 = 0u;
#pragma unroll
                    for (int k = 0; k < 7; ++k) {
                        if (k >= nslices) break;                 // uniform
                        code4 |= spread4((dw[t][k] >> b0) & 0xfu) << k;
                    }
                    const uint32_t m = spread4((vw[t] >> b0) & 0xfu) * 0xffu;
                    uint32_t fill4;
                    if (csrc >= 0) {
                        fill4 = (cp[t] == csrc ? Dc : Dfar) * 0x01010101u;
                    } else {
                        fill4 = 0u;
#pragma unroll
                        for (int r = 0; r < 4; ++r)
                            fill4 |= (cp[t] == s_comp[min(b0 + r, nsrc - 1)] ? Dc : Dfar) << (8 * r);
                    }
                    col[t] = code4 | (fill4 & ~m);
                }
                const uint32_t lo01 = __byte_perm(col[0], col[1], 0x5140), lo23 = __byte_perm(col[2], col[3], 0x5140);
                const uint32_t hi01 = __byte_perm(col[0], col[1], 0x7362), hi23 = __byte_perm(col[2], col[3], 0x7362);
                const uint32_t rw[4] = {__byte_perm(lo01, lo23, 0x5410), __byte_perm(lo01, lo23, 0x7632),
                                        __byte_perm(hi01, hi23, 0x5410), __byte_perm(hi01, hi23, 0x7632)};
#pragma unroll
                for (int r = 0; r < 4; ++r)
                    if (b0 + r < nsrc) store_codes_cs(spd + (int64_t)(s0 + b0 + r) * ld, c, n, rw[r]);
            }
            // clear: the words of columns v0 .. v0+3 (inside nwp by construction)
            const int w0 = SW::word(v0), w1 = SW::word(v0 + 3);
            for (int p = w0; p <= w1; ++p) {
                vis[p] = 0u;
                fr[p] = 0u;
                for (int k = 0; k < nslices; ++k) db[(size_t)k * nwp + p] = 0u;
            }
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

int scan_smem_bytes(int n, int W) { return 3 * scan_nwp(n, W) * 4; }

int optin_smem() {
    static int cached = -1;
    if (cached < 0) {
        int dev = 0, optin = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        cached = optin;
    }
    return cached;
}

// static shared memory of bfs_scan and some slack
constexpr int kScanStaticSmem = 1024;

// (vertex ids of the scan searches travel as 16-bit fields of the edge pairs)
bool scan_fits(int n, int W) { return n < 65535 && scan_smem_bytes(n, W) + kScanStaticSmem <= optin_smem(); }

// CTAs of the search per SM: two of half the threads when two fit the SM's shared
// memory and there are more batches than SMs (one CTA's output pass then runs
// while the other waits at its per-level barriers), else one.
int scan_per_sm(int n, int W) {
    static int per_sm_smem = -1;
    if (per_sm_smem < 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&per_sm_smem, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
    }
    const int nb = (n + W - 1) / W;
    return 2 * (scan_smem_bytes(n, W) + kScanStaticSmem + 1024) <= per_sm_smem && nb > num_sms() ? 2 : 1;
}

// The algorithm used for a graph of n vertices: the first that fits of
// shared-memory words with 32 sources, with 16, the queue-based search with
// shared-memory pushes, the global-memory search.  -1: the requested one
// does not fit.
int resolve_algo(int algo, int n) {
    switch (algo) {
        case GT_SPD_AUTO:
            // two CTAs per SM when they fit, with 16 sources per batch if 32 do not fit
            // twice and 32-source batches would fill the SMs anyway
            if (scan_fits(n, 32) && scan_per_sm(n, 32) == 2) return GT_SPD_SCAN32;
            if (scan_fits(n, 16) && scan_per_sm(n, 16) == 2 && (n + 31) / 32 >= num_sms())
                return GT_SPD_SCAN16;
            if (scan_fits(n, 32)) return GT_SPD_SCAN32;
            if (scan_fits(n, 16)) return GT_SPD_SCAN16;
            if (n <= bfs32_max_n()) return GT_SPD_QUEUE32;
            return GT_SPD_GLOBAL64;
        case GT_SPD_SCAN32: return scan_fits(n, 32) ? algo : -1;
        case GT_SPD_SCAN16: return scan_fits(n, 16) ? algo : -1;
        case GT_SPD_QUEUE32: return n <= bfs32_max_n() ? algo : -1;
        case GT_SPD_GLOBAL64: return algo;
        default: return -1;
    }
}

int nctas_for(int n, int per_batch) {
    const int nb = (n + per_batch - 1) / per_batch;
    const int sms = num_sms();
    return nb < sms ? nb : sms;
}

// Bytes of the search state for a resolved algorithm.
size_t bfs_state_bytes(int algo, int n, int nslices, size_t* per, int* nctas) {
    switch (algo) {
        case GT_SPD_SCAN32:
        case GT_SPD_SCAN16: {
            const int W = algo == GT_SPD_SCAN32 ? 32 : 16;
            *per = (size_t)nslices * scan_nwp(n, W) * 4;
            *nctas = nctas_for(n, W);
            if (scan_per_sm(n, W) == 2) {
                const int nb = (n + W - 1) / W;
                *nctas = nb < 2 * num_sms() ? nb : 2 * num_sms();
            }
            break;
        }
        case GT_SPD_QUEUE32:
            *per = per_cta_bytes32(n, nslices);
            *nctas = nctas_for(n, 32);
            break;
        default:
            *per = per_cta_bytes(n, nslices);
            *nctas = spd_ctas(n);
            break;
    }
    return *per * (size_t)*nctas;
}

}  // namespace

bool is_scan(int a) { return a == GT_SPD_SCAN32 || a == GT_SPD_SCAN16; }

size_t spd_workspace_bytes(int32_t n, int64_t nnz, int32_t D, int algo) {
    const int a = resolve_algo(algo, n);
    if (a < 0) return 0;
    Carve c(nullptr, 0);
    c.take<int>((size_t)n);
    if (is_scan(a)) c.take<uint32_t>((size_t)(nnz > 0 ? nnz : 1));
    size_t per = 0;
    int nctas = 0;
    c.take<char>(bfs_state_bytes(a, n, slices_for(D), &per, &nctas));
    return c.off + 256;
}

int spd_build(const int64_t* indptr, const int32_t* indices, int32_t n, int64_t nnz, int32_t D,
              int8_t* spd, int64_t ld, void* ws, size_t ws_bytes, int algo, cudaStream_t stream) {
    const int a = resolve_algo(algo, n);
    if (a < 0) return GT_ERR_UNSUPPORTED;
    Carve c(ws, ws_bytes);
    int* comp = c.take<int>((size_t)n);
    uint32_t* pairs = is_scan(a) ? c.take<uint32_t>((size_t)(nnz > 0 ? nnz : 1)) : nullptr;
    const int nslices = slices_for(D);
    size_t per = 0;
    int nctas = 0;
    char* bfs_ws = c.take<char>(bfs_state_bytes(a, n, nslices, &per, &nctas));
    if (!c.fits()) return GT_ERR_WORKSPACE;
    int* status = device_status_ptr();
    if (!status) return GT_ERR_CUDA;
    const int sms = num_sms();
    // every search keeps its global state zero between batches; start from zero
    if (per * (size_t)nctas > 0 && cudaMemsetAsync(bfs_ws, 0, per * (size_t)nctas, stream) != cudaSuccess)
        return GT_ERR_CUDA;
    // components: union-find over the edges (the scan searches first pack the edge
    // list, with the roots set alongside, and hook over it one thread per entry)
    if (is_scan(a)) {
        {
            LaunchScope ls("spd_pairs", stream);
            csr_pairs<<<sms * 8, 256, 0, stream>>>(indptr, indices, n, nnz, pairs, comp);
        }
        if (nnz > 0) {
            LaunchScope ls("spd_uf_hook", stream);
            const int64_t blocks = (nnz + 255) / 256;
            if (launch_overlapped(uf_hook_pairs, dim3((unsigned)(blocks < sms * 16 ? blocks : sms * 16)), dim3(256), 0,
                                  stream, (const uint32_t*)pairs, nnz, comp, n, status) != cudaSuccess)
                return GT_ERR_CUDA;
        }
    } else {
        {
            LaunchScope ls("spd_uf_init", stream);
            uf_init<<<sms * 4, 256, 0, stream>>>(comp, n);
        }
        LaunchScope ls("spd_uf_hook", stream);
        uf_hook<<<sms * 8, 256, 0, stream>>>(indptr, indices, comp, n, status);
    }
    {
        LaunchScope ls("spd_uf_compress", stream);
        if (launch_overlapped(uf_compress, dim3(sms * 4), dim3(256), 0, stream, comp, n) != cudaSuccess)
            return GT_ERR_CUDA;
    }
    if (is_scan(a)) {
        const int W = a == GT_SPD_SCAN32 ? 32 : 16;
        const int smem = scan_smem_bytes(n, W);
        auto kern = W == 32 ? bfs_scan<32> : bfs_scan<16>;
        if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
            return GT_ERR_CUDA;
        LaunchScope ls("spd_bfs", stream);
        if (launch_overlapped(kern, dim3(nctas), dim3(kScanThreads / scan_per_sm(n, W)), (size_t)smem, stream, indptr,
                              indices, (const uint32_t*)pairs, (const int*)comp, n, D, nslices, spd, ld,
                              reinterpret_cast<uint32_t*>(bfs_ws)) != cudaSuccess)
            return GT_ERR_CUDA;
    } else if (a == GT_SPD_QUEUE32) {
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

/*
 * gt_attn.h -- C ABI of libgt: topology-biased graph attention on one GB300.
 *
 * The operation (MegaGraph, "Towards Efficient Training of Large-Scale Graph
 * Transformers with Automated Hybrid Parallelism"):
 *   - abstract: a Graph Transformer layer carries, besides the attention score
 *     matrix, a topology-aware bias matrix of the same N x N shape per head;
 *   - Fig. 4: attention is computed KV block by KV block, and the bias columns
 *     that go with each incoming KV block are sliced on the fly.
 * The bias is the Graphormer spatial encoding over clipped shortest-path
 * distances:  b[h][i][j] = T[h][ spd[i][j] ],  spd[i][j] = min(dist(i,j), D) for
 * reachable pairs and D+1 otherwise, so T has nb = D+2 columns.  Per head h:
 *   s_ij = scale * <q_i, k_j> + b[h][i][j],   o_i = sum_j softmax_j(s_i) v_j,
 *   lse_i = log sum_j exp(s_ij)  (natural log),
 * and the backward pass returns dq, dk, dv and dT[h][c] = sum over pairs with
 * spd[i][j] = c of dS_ij, where dS_ij = p_ij (<dO_i, v_j> - <dO_i, o_i>).
 * Neither the N x N scores nor the N x N x H bias is ever stored.
 *
 * Conventions for every call below
 *   - Pointers named as device buffers must be device memory of the current
 *     CUDA device.  The caller owns and allocates every buffer, including the
 *     workspace; the library allocates no device memory and keeps no state
 *     between calls apart from one device status word per device (see
 *     gt_check_device_status) and the launch statistics at the end of this
 *     header.  Every kernel runs on the caller's stream.
 *   - The library caches per-device addresses (the status word; the scratch
 *     array of gt_bias_attn_bwd_noalloc).  Do not reset a device
 *     (cudaDeviceReset) while the library is loaded in the process: the cached
 *     addresses would outlive the context they belong to.
 *   - Layouts are dense row-major: q, k, v, o, dO, dq, dk, dv are [n][h][d]
 *     (node, head, channel); lse is [h][n] fp32; T and dT are [h][nb] fp32;
 *     spd is int8 [n][ld_spd] (row i holds the bucket codes of pairs (i, *)).
 *   - `dtype` selects the element type of q, k, v, o, dO, dq, dk, dv:
 *     GT_F32 (exact fp32 arithmetic) or GT_BF16 (bf16 storage, tensor-core
 *     products with fp32 accumulation, fp32 softmax statistics).
 *   - All calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *     default stream).  They check their arguments on the host before any
 *     launch and return a negative gt_status without launching if a check
 *     fails.  GT_OK means the work was enqueued.  Within a call, a kernel may
 *     be scheduled while the one before it finishes (programmatic dependent
 *     launch); each such kernel waits for its predecessor before reading that
 *     one's output and before it completes, so what the caller's later work
 *     on the stream sees is the same as with plain stream order.
 *   - Bucket codes are read as unsigned bytes; codes >= nb select a zero bias
 *     in the forward and are dropped from dT (they never occur in the output of
 *     gt_spd_build).
 */
#ifndef GT_ATTN_H
#define GT_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    GT_OK = 0,
    GT_ERR_INVALID_ARG = -1,  /* NULL, size, alignment or layout check failed */
    GT_ERR_UNSUPPORTED = -2,  /* shape valid but not handled by this library */
    GT_ERR_CUDA = -3,         /* a CUDA runtime call or launch failed */
    GT_ERR_TIMEOUT = -4,      /* a kernel gave up a bounded wait (see below) */
    GT_ERR_WORKSPACE = -5     /* workspace NULL or smaller than the size query */
} gt_status;

typedef enum { GT_F32 = 0, GT_BF16 = 1 } gt_dtype;

/* Largest clip distance: codes 0..D+1 must fit a signed byte. */
#define GT_MAX_D 126

/*
 * Bytes of device workspace gt_spd_build needs for this graph size on the
 * current device.
 */
size_t gt_spd_workspace_size(int32_t n, int64_t nnz, int32_t D);

/*
 * gt_spd_build: clipped shortest-path bucket matrix of an undirected graph
 * (the topology the bias of the MegaGraph abstract is built from).
 *   indptr  device int64[n+1], indices device int32[nnz]: CSR adjacency with
 *           both directions of every edge stored (self-loops and repeated
 *           entries are harmless).
 *   n >= 1, 1 <= D <= GT_MAX_D.
 *   spd     device int8 [n][ld_spd], written for columns 0..n-1 of every row:
 *           spd[i][j] = min(dist(i,j), D) if j is reachable from i, D+1 if not,
 *           0 on the diagonal.  ld_spd >= n and ld_spd % 16 == 0; spd 16-byte
 *           aligned.  Columns n..ld_spd-1 are not written.
 *   workspace/ws_bytes: device scratch of at least gt_spd_workspace_size().
 * Errors: GT_ERR_INVALID_ARG for NULL pointers, n < 1, nnz < 0, D out of range,
 * bad ld_spd or alignment; GT_ERR_WORKSPACE for a short workspace.
 */
int gt_spd_build(const int64_t* indptr, const int32_t* indices, int32_t n, int64_t nnz,
                 int32_t D, int8_t* spd, int64_t ld_spd,
                 void* workspace, size_t ws_bytes, void* stream);

/*
 * Search algorithms of gt_spd_build.  All give the same codes; they differ in
 * where the per-vertex state lives, which bounds the graph size they take:
 *   GT_SPD_SCAN32    32 sources per batch, every per-vertex word in shared
 *                    memory (12 bytes per vertex), n up to ~18.8K on a GB300.
 *   GT_SPD_SCAN16    16 sources per batch, two vertices per word (6 bytes per
 *                    vertex), n up to ~37K.
 *   GT_SPD_QUEUE32   32 sources per batch, frontier queues in global memory,
 *                    pushes into shared memory (4 bytes per vertex), n up to ~58K.
 *   GT_SPD_GLOBAL64  64 sources per batch, all state in global memory: any n.
 *   GT_SPD_AUTO      what gt_spd_build uses: a scan search that runs two CTAs
 *                    per SM when its state fits twice in an SM's shared memory
 *                    and the batches outnumber the SMs (SCAN32 if it does so,
 *                    else SCAN16 when 32-source batches would fill the SMs
 *                    anyway), otherwise the first of these that fits.
 * The scan searches run one CTA of 1024 threads per SM, or two of 512 under the
 * condition above.
 */
enum { GT_SPD_AUTO = 0, GT_SPD_SCAN32 = 1, GT_SPD_SCAN16 = 2, GT_SPD_QUEUE32 = 3, GT_SPD_GLOBAL64 = 4 };

/*
 * Workspace bytes of gt_spd_build_algo for this algorithm, or 0 when the
 * algorithm cannot take n vertices on the current device (or the arguments are
 * out of range).
 */
size_t gt_spd_workspace_size_algo(int32_t algo, int32_t n, int64_t nnz, int32_t D);

/*
 * gt_spd_build with an explicit search algorithm (same arguments and result).
 * Errors as gt_spd_build, plus GT_ERR_INVALID_ARG for an unknown algo and
 * GT_ERR_UNSUPPORTED when the algorithm cannot take n vertices on this device.
 */
int gt_spd_build_algo(int32_t algo, const int64_t* indptr, const int32_t* indices, int32_t n,
                      int64_t nnz, int32_t D, int8_t* spd, int64_t ld_spd,
                      void* workspace, size_t ws_bytes, void* stream);

/*
 * The uniform KV block gt_bias_attn_fwd uses for these arguments (0 = none;
 * -1 for invalid arguments): an explicit kv_block (< n) is used as given.  With
 * kv_block = 0 no uniform split is made; the bf16 tensor-core path instead
 * deals its (query tile, head half, KV block) work out in equal contiguous
 * shares to a whole number of waves of two CTAs per SM, whenever one CTA per
 * tile and head half would leave part of the last wave idle.  A share covers
 * the end of one tile's KV range and the start of the next; rows whose range
 * more than one CTA covered are merged exactly through their lse (the same
 * merge as for KV blocks, Fig. 4), the others are written directly.
 */
int32_t gt_bias_attn_fwd_kv_block(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t kv_block);

/*
 * CTAs of that balanced tensor-core forward for these arguments on the current
 * device (-1 for invalid arguments): 0 when the forward runs one CTA per 128-row
 * tile and head half (an explicit kv_block, another dtype or shape, or a grid
 * whose waves are full already).  A balanced forward launches one merge kernel
 * after the attention kernel.
 */
int32_t gt_bias_attn_fwd_ctas(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t kv_block);

/*
 * How many CTAs share each dq task (a 128-row query tile and a head half) of
 * the bf16 tensor-core backward for these sizes on the current device (1 = none;
 * -1 for invalid arguments).  The dq tasks that do not fill a whole wave of two
 * CTAs per SM (all of them on a graph too small to fill one) are split along
 * their KV blocks, k ways with k in 2..8 chosen so that the last waves fill the
 * SMs.  The dk/dv groups (a 128-row KV tile and a head half) past the last full
 * wave of one CTA per SM are split along their query tiles the same way; fewer
 * groups than SMs run instead as equal shares of all (group, query tile) steps,
 * one CTA per SM.  Split or shared work sums in fp32 (workspace included in
 * gt_bias_attn_workspace_size; a workspace too small for the sums runs
 * unsplit).
 */
int32_t gt_bias_attn_bwd_split(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t nb);

/*
 * Kernel launches of one gt_bias_attn_fwd call (*fwd, with this kv_block) and of
 * one gt_bias_attn_bwd call (*bwd, with these nb buckets) on the current device,
 * given a workspace of gt_bias_attn_workspace_size bytes; memsets are not
 * counted.  A split of the tasks past the last full wave (see
 * gt_bias_attn_bwd_split) adds the split tasks' own launch when whole tasks
 * fill waves before them; the backward's last launch converts every split's
 * fp32 sums and the bucket sums at once.  Returns GT_OK, or
 * GT_ERR_INVALID_ARG for invalid arguments or NULL outputs.
 */
int gt_bias_attn_launches(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t nb, int32_t kv_block,
                          int32_t* fwd, int32_t* bwd);

/*
 * Bytes of device workspace needed by gt_bias_attn_fwd (with this kv_block)
 * and by gt_bias_attn_bwd for these sizes; one buffer of this size serves both.
 */
size_t gt_bias_attn_workspace_size(int32_t dtype, int32_t n, int32_t h, int32_t d,
                                   int32_t kv_block);

/*
 * gt_bias_attn_fwd: o = softmax(scale * q k^T + T[h][spd]) v per head, plus lse.
 *   q, k, v  device [n][h][d] of `dtype`, 16-byte aligned.
 *   spd      device int8 [n][ld_spd] bucket codes (ld_spd >= n, % 16 == 0,
 *            16-byte aligned).
 *   T        device fp32 [h][nb], nb <= 128.
 *   scale    multiplies q.k before the bias is added (1/sqrt(d) is usual).
 *   kv_block 0: every Q tile streams all n KV columns (in at most a few
 *            balanced pieces: see gt_bias_attn_fwd_kv_block).
 *            > 0 (a multiple of 128): the columns are cut into blocks of
 *            kv_block (the KV blocks of Fig. 4); each block yields a partial
 *            (o, lse) and the partials are merged exactly through their lse.
 *   o        device [n][h][d] of `dtype` (output); lse device fp32 [h][n].
 *   workspace/ws_bytes: at least gt_bias_attn_workspace_size(...).
 * Supported: n >= 1, 1 <= h <= 16, 1 <= d <= 64.  GT_BF16 with h = 8 and
 * d in {8, 16} runs on the tensor cores; other shapes run on a CUDA-core kernel.
 */
int gt_bias_attn_fwd(int32_t dtype, int32_t n, int32_t h, int32_t d,
                     const void* q, const void* k, const void* v,
                     const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb,
                     float scale, int32_t kv_block,
                     void* o, float* lse, void* workspace, size_t ws_bytes, void* stream);

/*
 * The forward over one range of KV columns, and the exact merge of such
 * partials: Fig. 4's ring step on one GPU.  A caller that holds KV blocks
 * [a_0, a_1), [a_1, a_2), ... in turn (a ring across GPUs, or blocks streamed
 * from host memory) computes each block's partial with gt_bias_attn_fwd_partial
 * and combines them with gt_bias_attn_merge; the result equals
 * gt_bias_attn_fwd over all columns up to rounding.
 *
 * gt_bias_attn_fwd_partial: every query row attends only to KV columns
 * [kv_begin, kv_end), with the bias columns of that range.
 *   q, k, v, spd, ld_spd, T, nb, scale: as for gt_bias_attn_fwd (k and v hold
 *            all n rows; only the range's rows are read).
 *   kv_begin a multiple of 128, 0 <= kv_begin < kv_end <= n.
 *   o_part   device fp32 [n][h][d] (output, 16-byte aligned): the output
 *            normalised over the range's columns.
 *   lse_part device fp32 [h][n] (output): log of the range's softmax
 *            denominator (natural log, scores include the bias).
 * Needs no workspace.  Errors as for gt_bias_attn_fwd, plus GT_ERR_INVALID_ARG
 * for a bad range.
 *
 * gt_bias_attn_merge: o = sum_p exp(lse_p - lse) o_p with lse = log sum_p
 * exp(lse_p), per (node, head).
 *   o_parts  device fp32 [nparts][n][h][d]; lse_parts device fp32 [nparts][h][n].
 *   o        device [n][h][d] of `dtype` (output); lse device fp32 [h][n].
 * Errors: GT_ERR_INVALID_ARG for NULL pointers, n, h, d or nparts < 1;
 * GT_ERR_UNSUPPORTED for h > 16 or d > 64.
 */
int gt_bias_attn_fwd_partial(int32_t dtype, int32_t n, int32_t h, int32_t d,
                             const void* q, const void* k, const void* v,
                             const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb,
                             float scale, int32_t kv_begin, int32_t kv_end,
                             float* o_part, float* lse_part, void* stream);
int gt_bias_attn_merge(int32_t dtype, int32_t n, int32_t h, int32_t d, int32_t nparts,
                       const float* o_parts, const float* lse_parts, void* o, float* lse,
                       void* stream);

/*
 * gt_bias_attn_bwd: gradients of sum(o * dO) with respect to q, k, v and T.
 *   o, lse   the forward's outputs for the same inputs.
 *   dO       device [n][h][d] of `dtype`, the upstream gradient.
 *   dq, dk, dv device [n][h][d] of `dtype` (outputs, overwritten).
 *   dT       device fp32 [h][nb] (output, overwritten).
 * Other arguments and the supported shapes are as for gt_bias_attn_fwd.
 */
int gt_bias_attn_bwd(int32_t dtype, int32_t n, int32_t h, int32_t d,
                     const void* q, const void* k, const void* v, const void* o,
                     const void* dO, const float* lse,
                     const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb,
                     float scale, void* dq, void* dk, void* dv, float* dT,
                     void* workspace, size_t ws_bytes, void* stream);

/*
 * gt_bias_attn_bwd_noalloc: gt_bias_attn_bwd for callers that cannot allocate.
 * The paper has no counterpart; this is a library convenience.
 *
 * Some callers cannot call cudaMalloc or any allocator (a host framework that
 * owns all device memory, a real-time or embedded host that forbids allocation
 * after start-up, a plain C host with no caching allocator).  This variant takes
 * no workspace: it runs the same backward pass with its scratch in an array of
 * GT_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that loads
 * the library holds until the process exits.  Inputs and outputs are passed and
 * owned by the caller exactly as for gt_bias_attn_bwd, and the results match it.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, once per device, with that device current); make
 *     that first call before any stream capture.  No call allocates or frees
 *     device memory.
 *   - Every call shares the one array and leaves its contents behind (the pass
 *     clears what must start at zero).  Calls whose GPU work overlaps, on
 *     different streams or host threads of one device, race on the array and
 *     corrupt each other's results: serialise them.
 *   - Returns GT_ERR_WORKSPACE, with nothing launched, when the backward run
 *     without its split (the split's fp32 sums are left out when they do not
 *     fit) needs more than GT_NOALLOC_SCRATCH_BYTES.  That scratch is, in bytes,
 *     with 256-byte alignment of each part: 4 h n (D) + 1024 (dT sums)
 *     + 64 * ((n + 3) / 4 * 4) (per-node lse and D rows) + 256 n (the bf16 lse / D
 *     operand of the dk/dv products) + 64; with H = 8 about 352 bytes per node,
 *     so N up to about 11,900 nodes.  gt_bias_attn_workspace_size may report
 *     more than this for small graphs (it includes the split's sums); such calls
 *     still succeed, unsplit.
 */
#define GT_NOALLOC_SCRATCH_BYTES (4u << 20)
int gt_bias_attn_bwd_noalloc(int32_t dtype, int32_t n, int32_t h, int32_t d,
                             const void* q, const void* k, const void* v, const void* o,
                             const void* dO, const float* lse,
                             const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb,
                             float scale, void* dq, void* dk, void* dv, float* dT, void* stream);

/*
 * The GT encoder layer around the biased attention (MegaGraph, Fig. 8: 8 heads,
 * hidden and FFN width 64).  The pages give the widths, not the order of the
 * steps; this is the pre-LayerNorm (Graphormer) encoder layer:
 *
 *   u = LN1(x); [q|k|v] = u W_qkv + b_qkv; o = biased attention(q, k, v);
 *   hh = x + o W_o + b_o; z = LN2(hh); y = hh + GELU(z W_1 + b_1) W_2 + b_2
 *
 * with LN(v) = gain (v - mean v) / sqrt(var v + 1e-5) + shift over the 64
 * features of a node, GELU(a) = a Phi(a) (Phi the normal CDF), the attention
 * scale 1/sqrt(8), and q, k, v split into heads as [n][8][8] (feature = head * 8
 * + channel).  Supported: h = 8, d = 8, f = 64 (else GT_ERR_UNSUPPORTED); the
 * attention runs in bf16 on the tensor cores, and so do the layer's products:
 * tf32 (fp32 storage) for the projections and the FFN, bf16 for the products
 * over node rows that form the weight gradients, fp32 accumulation in both.
 *
 * All weights are device fp32, row-major: ln*_g / ln*_b [64]; w_qkv [64][192]
 * (columns q | k | v); b_qkv [192]; w_o [64][64]; b_o [64]; w_1 [64][64] (in x
 * out); b_1 [64]; w_2 [64][64]; b_2 [64]; the four matrices 16-byte aligned,
 * and so every node-row array (x, y, dy, dx, q, k, v, o): the layer kernels move
 * whole rows with bulk copies.
 * gt_layer_grads has the same shapes and receives dL/d(weight) (overwritten).
 */
typedef struct {
    const float *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_o, *b_o, *ln2_g, *ln2_b, *w_1, *b_1, *w_2, *b_2;
} gt_layer_weights;

typedef struct {
    float *ln1_g, *ln1_b, *w_qkv, *b_qkv, *w_o, *b_o, *ln2_g, *ln2_b, *w_1, *b_1, *w_2, *b_2;
} gt_layer_grads;

/* Workspace bytes of gt_layer_fwd and gt_layer_bwd (one buffer serves both);
 * 0 for unsupported sizes. */
size_t gt_layer_workspace_size(int32_t n, int32_t h, int32_t d, int32_t f);

/*
 * gt_layer_fwd: y (device fp32 [n][64]) from x (device fp32 [n][64]).  Also
 * writes what the backward needs: q, k, v, o (device bf16 [n][8][8]) and lse
 * (fp32 [8][n]).  spd, ld_spd, T, nb as for gt_bias_attn_fwd.
 * Errors: GT_ERR_UNSUPPORTED for other sizes, GT_ERR_INVALID_ARG for NULL
 * pointers (any weight included) or unaligned matrices, the attention's own
 * checks, GT_ERR_WORKSPACE.
 */
int gt_layer_fwd(int32_t n, int32_t h, int32_t d, int32_t f, const float* x, const gt_layer_weights* w,
                 const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb,
                 void* q, void* k, void* v, void* o, float* lse, float* y,
                 void* workspace, size_t ws_bytes, void* stream);

/*
 * gt_layer_bwd: given dy = dL/dy (device fp32 [n][64]) and the forward's x, q,
 * k, v, o, lse: dx (device fp32 [n][64], overwritten), every weight gradient
 * (overwritten) and dT (fp32 [8][nb], overwritten).  Errors as gt_layer_fwd.
 */
int gt_layer_bwd(int32_t n, int32_t h, int32_t d, int32_t f, const float* x, const gt_layer_weights* w,
                 const int8_t* spd, int64_t ld_spd, const float* T, int32_t nb,
                 const void* q, const void* k, const void* v, const void* o, const float* lse,
                 const float* dy, float* dx, const gt_layer_grads* g, float* dT,
                 void* workspace, size_t ws_bytes, void* stream);

/* Static English text for a gt_status value. */
const char* gt_status_string(int status);

/*
 * Synchronises `stream`, then reports GT_ERR_TIMEOUT if any kernel of this
 * library gave up a bounded wait since the last check (kernels never spin
 * without a limit; on giving up they record it in a device status word and
 * return), GT_ERR_CUDA if the stream reports an error, else GT_OK.  The status
 * word is cleared by the call.
 */
int gt_check_device_status(void* stream);

/*
 * Self-test of the bounded waits (no counterpart in the method): launches one
 * CTA on `stream` whose wait on a barrier that nothing arrives at gives up after
 * limit_ns nanoseconds of wall time, exactly as a kernel's wait would; the next
 * gt_check_device_status then reports GT_ERR_TIMEOUT and the context stays
 * usable.  1e6 <= limit_ns <= 1e9, else GT_ERR_INVALID_ARG.
 */
int gt_selftest_wait_timeout(int64_t limit_ns, void* stream);

/*
 * Launch statistics (a measurement aid; no counterpart in the method).
 *
 * The library counts, per kernel name, every kernel it launches.  With timing
 * on, each launch is also bracketed by two CUDA events recorded on the
 * launching stream (events come from a pool the library creates on demand and
 * keeps), so the sum of (end - start) per name is the device time of that
 * kernel's launches, queueing behind earlier work on the stream excluded.
 * Timing adds two event records per launch; leave it off while timing whole
 * steps.  The table is process-wide and guarded by a mutex; with timing on,
 * use one CUDA device per process.
 *
 *   gt_kernel_stats_reset(timing)  clears the table (waiting for events still
 *       pending) and sets timing on (non-zero) or off.  Returns GT_OK or
 *       GT_ERR_CUDA.
 *   gt_kernel_stats_read(out, cap, count)  waits for the recorded events, sets
 *       *count to the number of distinct kernel names seen since the reset and
 *       fills min(cap, *count) entries of out (host memory, caller-owned) in
 *       first-launch order; total_ms is -1 when timing is off.  Returns
 *       GT_ERR_INVALID_ARG for count == NULL, cap < 0 or out == NULL with
 *       cap > 0, GT_ERR_CUDA if an event query fails, else GT_OK.
 */
typedef struct {
    char name[40];      /* NUL-terminated kernel name, e.g. "bwd_dq" */
    int64_t launches;   /* launches since the last reset */
    double total_ms;    /* summed device time of those launches (timing on) */
} gt_kernel_stat;

int gt_kernel_stats_reset(int32_t timing);
int gt_kernel_stats_read(gt_kernel_stat* out, int32_t cap, int32_t* count);

#ifdef __cplusplus
}
#endif
#endif /* GT_ATTN_H */

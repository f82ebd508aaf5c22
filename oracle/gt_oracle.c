/*
 * gt_oracle.c -- plain fp64 CPU oracle for topology-biased graph attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call this code:
 * only the tests, the package smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no source, header, table or helper with the CUDA library.
 *
 * What it computes (MegaGraph, "Towards Efficient Training of Large-Scale Graph
 * Transformers with Automated Hybrid Parallelism", abstract: attention scores
 * plus a topology-aware bias matrix per layer; Fig. 4: the bias column slice that
 * goes with each KV block).  The bias is the Graphormer-style spatial encoding
 *     b[h][i][j] = T[h][ spd[i][j] ],
 *     spd[i][j]  = min(dist(i,j), D) if j is reachable from i, else D+1,
 * and one layer of biased multi-head attention is, per head h and row i,
 *     s_ij  = scale * <q_i, k_j> + b[h][i][j]
 *     p_ij  = exp(s_ij - lse_i),   lse_i = log sum_j exp(s_ij)
 *     o_i   = sum_j p_ij v_j
 * with its backward for an upstream gradient dO:
 *     D_i   = <dO_i, o_i>
 *     dS_ij = p_ij (<dO_i, v_j> - D_i)
 *     dq_i  = scale sum_j dS_ij k_j,  dk_j = scale sum_i dS_ij q_i
 *     dv_j  = sum_i p_ij dO_i,        dT[h][c] = sum_{(i,j): spd[i][j]=c} dS_ij
 * Every sum is taken densely over all N columns (or rows); there is no blocking
 * over KV, no fusion and no reordering beyond splitting independent rows or
 * columns over threads.
 *
 * Bucket bytes are read as unsigned codes 0..255.  The pages define only the
 * codes a shortest-path build produces (0..D+1, i.e. below nb); a byte at or
 * above nb is read as "no bias": it adds 0 to the score and belongs to no
 * column of T, so it adds nothing to dT.
 *
 * Layouts (row-major): q, k, v, o, dO, dq, dk, dv are [n][h][d] doubles;
 * lse and D are [h][n]; T and dT are [h][nb]; spd is int8 [n][ld].
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- threads */

typedef void (*range_fn)(void* ctx, int64_t lo, int64_t hi, int tid);

typedef struct {
    range_fn fn;
    void* ctx;
    int64_t lo, hi;
    int tid;
} job_t;

static void* job_main(void* arg) {
    job_t* j = (job_t*)arg;
    j->fn(j->ctx, j->lo, j->hi, j->tid);
    return NULL;
}

/* Runs fn over [0, count) split into nthreads contiguous ranges. */
static int parallel_for(int64_t count, int nthreads, range_fn fn, void* ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > count) nthreads = (int)(count > 0 ? count : 1);
    pthread_t th[256];
    int spawned[256];
    job_t jobs[256];
    int64_t per = (count + nthreads - 1) / nthreads;
    for (int t = 0; t < nthreads; ++t) {
        int64_t lo = (int64_t)t * per, hi = lo + per;
        if (hi > count) hi = count;
        if (lo > hi) lo = hi;
        jobs[t] = (job_t){fn, ctx, lo, hi, t};
        spawned[t] = 0;
        if (t < nthreads - 1 && pthread_create(&th[t], NULL, job_main, &jobs[t]) == 0)
            spawned[t] = 1;
        else
            job_main(&jobs[t]);   /* the last range, or a failed spawn, runs here */
    }
    for (int t = 0; t < nthreads; ++t)
        if (spawned[t]) pthread_join(th[t], NULL);
    return 0;
}

/* ------------------------------------------------------- shortest paths */

typedef struct {
    int32_t n;
    const int64_t* indptr;
    const int32_t* indices;
    int32_t D;
    int8_t* spd;
    int64_t ld;
} spd_ctx;

/* One FIFO breadth-first search per source row; unreached pairs get D+1,
 * distances beyond D are clipped to D. */
static void spd_rows(void* vctx, int64_t lo, int64_t hi, int tid) {
    (void)tid;
    spd_ctx* c = (spd_ctx*)vctx;
    int32_t n = c->n;
    int32_t* dist = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
    int32_t* queue = (int32_t*)malloc(sizeof(int32_t) * (size_t)n);
    for (int64_t s = lo; s < hi; ++s) {
        for (int32_t v = 0; v < n; ++v) dist[v] = -1;
        int32_t head = 0, tail = 0;
        dist[s] = 0;
        queue[tail++] = (int32_t)s;
        while (head < tail) {
            int32_t u = queue[head++];
            for (int64_t e = c->indptr[u]; e < c->indptr[u + 1]; ++e) {
                int32_t w = c->indices[e];
                if (dist[w] < 0) {
                    dist[w] = dist[u] + 1;
                    queue[tail++] = w;
                }
            }
        }
        int8_t* row = c->spd + s * c->ld;
        for (int32_t v = 0; v < n; ++v) {
            int32_t code = dist[v] < 0 ? c->D + 1 : (dist[v] < c->D ? dist[v] : c->D);
            row[v] = (int8_t)code;
        }
    }
    free(dist);
    free(queue);
}

int gto_spd(int32_t n, const int64_t* indptr, const int32_t* indices, int32_t D,
            int8_t* spd, int64_t ld, int32_t nthreads) {
    if (n < 0 || D < 1 || D > 126 || ld < n) return -1;
    spd_ctx c = {n, indptr, indices, D, spd, ld};
    parallel_for(n, nthreads, spd_rows, &c);
    return 0;
}

/* ------------------------------------------------------------ attention */

typedef struct {
    int32_t n, h, d, nb;
    const double *q, *k, *v, *T;
    const int8_t* spd;
    int64_t ld;
    double scale;
    const int32_t* rows;   /* rows handled (forward / dq) */
    int32_t nrows;
    const int32_t* cols;   /* columns handled (dk / dv) */
    int32_t ncols;
    const double *dO, *lse, *Dv;  /* lse, Dv: [h][n], full */
    double *o, *lse_out;          /* forward outputs: [nrows][h][d], [h][nrows] */
    double *dq;                   /* [nrows][h][d] */
    double *dk, *dv;              /* [ncols][h][d] */
    double* dT_part;              /* [nthreads][h][nb] */
} attn_ctx;

/* score s_ij for head hh, bias included */
static double score(const attn_ctx* c, int32_t i, int32_t j, int32_t hh) {
    const double* qi = c->q + ((int64_t)i * c->h + hh) * c->d;
    const double* kj = c->k + ((int64_t)j * c->h + hh) * c->d;
    double dot = 0.0;
    for (int32_t t = 0; t < c->d; ++t) dot += qi[t] * kj[t];
    int code = (int)(uint8_t)c->spd[(int64_t)i * c->ld + j];
    double bias = code < c->nb ? c->T[(int64_t)hh * c->nb + code] : 0.0;
    return c->scale * dot + bias;
}

static void fwd_rows(void* vctx, int64_t lo, int64_t hi, int tid) {
    (void)tid;
    attn_ctx* c = (attn_ctx*)vctx;
    double* s = (double*)malloc(sizeof(double) * (size_t)c->n);
    for (int64_t r = lo; r < hi; ++r) {
        int32_t i = c->rows[r];
        for (int32_t hh = 0; hh < c->h; ++hh) {
            double m = -INFINITY;
            for (int32_t j = 0; j < c->n; ++j) {
                s[j] = score(c, i, j, hh);
                if (s[j] > m) m = s[j];
            }
            double l = 0.0;
            for (int32_t j = 0; j < c->n; ++j) {
                s[j] = exp(s[j] - m);   /* s now holds e^{s_ij - m} */
                l += s[j];
            }
            double* oi = c->o + (r * c->h + hh) * c->d;
            for (int32_t t = 0; t < c->d; ++t) oi[t] = 0.0;
            for (int32_t j = 0; j < c->n; ++j) {
                double p = s[j] / l;
                const double* vj = c->v + ((int64_t)j * c->h + hh) * c->d;
                for (int32_t t = 0; t < c->d; ++t) oi[t] += p * vj[t];
            }
            c->lse_out[(int64_t)hh * c->nrows + r] = m + log(l);
        }
    }
    free(s);
}

/* Forward for the listed rows: o [nrows][h][d], lse [h][nrows] (natural log). */
int gto_attn_fwd_rows(int32_t n, int32_t h, int32_t d,
                      const double* q, const double* k, const double* v,
                      const int8_t* spd, int64_t ld, const double* T, int32_t nb,
                      double scale, const int32_t* rows, int32_t nrows,
                      double* o, double* lse, int32_t nthreads) {
    if (n < 1 || h < 1 || d < 1 || nb < 1 || ld < n || nrows < 0) return -1;
    attn_ctx c;
    memset(&c, 0, sizeof c);
    c.n = n; c.h = h; c.d = d; c.nb = nb;
    c.q = q; c.k = k; c.v = v; c.T = T; c.spd = spd; c.ld = ld; c.scale = scale;
    c.rows = rows; c.nrows = nrows; c.o = o; c.lse_out = lse;
    parallel_for(nrows, nthreads, fwd_rows, &c);
    return 0;
}

/* D_i = <dO_i, o_i> per head, for all n rows: Dv [h][n]. */
int gto_attn_bwd_delta(int32_t n, int32_t h, int32_t d, const double* o, const double* dO,
                       double* Dv) {
    for (int32_t i = 0; i < n; ++i)
        for (int32_t hh = 0; hh < h; ++hh) {
            const double* a = o + ((int64_t)i * h + hh) * d;
            const double* b = dO + ((int64_t)i * h + hh) * d;
            double acc = 0.0;
            for (int32_t t = 0; t < d; ++t) acc += a[t] * b[t];
            Dv[(int64_t)hh * n + i] = acc;
        }
    return 0;
}

static double prob(const attn_ctx* c, int32_t i, int32_t j, int32_t hh) {
    return exp(score(c, i, j, hh) - c->lse[(int64_t)hh * c->n + i]);
}

static double dprob(const attn_ctx* c, int32_t i, int32_t j, int32_t hh) {
    const double* g = c->dO + ((int64_t)i * c->h + hh) * c->d;
    const double* vj = c->v + ((int64_t)j * c->h + hh) * c->d;
    double acc = 0.0;
    for (int32_t t = 0; t < c->d; ++t) acc += g[t] * vj[t];
    return acc;
}

/* dq for the listed rows, and this thread's share of dT over those rows. */
static void bwd_rows(void* vctx, int64_t lo, int64_t hi, int tid) {
    attn_ctx* c = (attn_ctx*)vctx;
    double* dT = c->dT_part ? c->dT_part + (int64_t)tid * c->h * c->nb : NULL;
    for (int64_t r = lo; r < hi; ++r) {
        int32_t i = c->rows[r];
        for (int32_t hh = 0; hh < c->h; ++hh) {
            double* dqi = c->dq ? c->dq + (r * c->h + hh) * c->d : NULL;
            if (dqi) for (int32_t t = 0; t < c->d; ++t) dqi[t] = 0.0;
            double Di = c->Dv[(int64_t)hh * c->n + i];
            for (int32_t j = 0; j < c->n; ++j) {
                double p = prob(c, i, j, hh);
                double ds = p * (dprob(c, i, j, hh) - Di);
                if (dqi) {
                    const double* kj = c->k + ((int64_t)j * c->h + hh) * c->d;
                    for (int32_t t = 0; t < c->d; ++t) dqi[t] += c->scale * ds * kj[t];
                }
                int code = (int)(uint8_t)c->spd[(int64_t)i * c->ld + j];
                if (dT && code < c->nb) dT[(int64_t)hh * c->nb + code] += ds;
            }
        }
    }
}

/* dk and dv for the listed columns. */
static void bwd_cols(void* vctx, int64_t lo, int64_t hi, int tid) {
    (void)tid;
    attn_ctx* c = (attn_ctx*)vctx;
    for (int64_t r = lo; r < hi; ++r) {
        int32_t j = c->cols[r];
        for (int32_t hh = 0; hh < c->h; ++hh) {
            double* dkj = c->dk + (r * c->h + hh) * c->d;
            double* dvj = c->dv + (r * c->h + hh) * c->d;
            for (int32_t t = 0; t < c->d; ++t) dkj[t] = dvj[t] = 0.0;
            for (int32_t i = 0; i < c->n; ++i) {
                double p = prob(c, i, j, hh);
                double ds = p * (dprob(c, i, j, hh) - c->Dv[(int64_t)hh * c->n + i]);
                const double* qi = c->q + ((int64_t)i * c->h + hh) * c->d;
                const double* gi = c->dO + ((int64_t)i * c->h + hh) * c->d;
                for (int32_t t = 0; t < c->d; ++t) {
                    dkj[t] += c->scale * ds * qi[t];
                    dvj[t] += p * gi[t];
                }
            }
        }
    }
}

/*
 * Backward.  lse and Dv are the full [h][n] arrays (from the forward over all
 * rows).  dq is produced for `rows` (NULL: skip), dk/dv for `cols` (ncols may be
 * 0), and dT (NULL: skip) sums dS over the listed rows only -- pass all rows for
 * the full table gradient.
 */
int gto_attn_bwd(int32_t n, int32_t h, int32_t d,
                 const double* q, const double* k, const double* v, const double* dO,
                 const double* lse, const double* Dv,
                 const int8_t* spd, int64_t ld, const double* T, int32_t nb, double scale,
                 const int32_t* rows, int32_t nrows, double* dq, double* dT,
                 const int32_t* cols, int32_t ncols, double* dk, double* dv,
                 int32_t nthreads) {
    if (n < 1 || h < 1 || d < 1 || nb < 1 || ld < n) return -1;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    attn_ctx c;
    memset(&c, 0, sizeof c);
    c.n = n; c.h = h; c.d = d; c.nb = nb;
    c.q = q; c.k = k; c.v = v; c.T = T; c.spd = spd; c.ld = ld; c.scale = scale;
    c.dO = dO; c.lse = lse; c.Dv = Dv;
    c.rows = rows; c.nrows = nrows; c.dq = dq;
    c.cols = cols; c.ncols = ncols; c.dk = dk; c.dv = dv;
    if (nrows > 0 && (dq || dT)) {
        if (dT) {
            c.dT_part = (double*)calloc((size_t)nthreads * h * nb, sizeof(double));
            if (!c.dT_part) return -2;
        }
        parallel_for(nrows, nthreads, bwd_rows, &c);
        if (dT) {
            for (int64_t x = 0; x < (int64_t)h * nb; ++x) {
                double acc = 0.0;
                for (int t = 0; t < nthreads; ++t) acc += c.dT_part[(int64_t)t * h * nb + x];
                dT[x] = acc;
            }
            free(c.dT_part);
            c.dT_part = NULL;
        }
    }
    if (ncols > 0 && dk && dv) parallel_for(ncols, nthreads, bwd_cols, &c);
    return 0;
}

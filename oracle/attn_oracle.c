/*
 * attn_oracle.c -- plain fp64 CPU oracle for exact attention forward.
 *
 * TEST INFRASTRUCTURE ONLY (see attn_oracle.h): used by the tests, the smoke
 * check and the benchmark's CPU-baseline leg, never by the product path.
 *
 * Written for a reader to check by eye against the definition: one query row
 * at a time, the score row s is materialised in full, the max-subtracted
 * softmax is taken over it, then P.V.  Compiled with -O2 and without
 * -ffast-math so that exp/log and the summation order are the plain ones.
 * Threads only split independent rows (or Q tiles); no arithmetic is shared
 * between threads.
 */
#define _GNU_SOURCE
#include "attn_oracle.h"

#include <math.h>
#include <pthread.h>
#include <sched.h>
#include <stdlib.h>
#include <string.h>

int attn_oracle_default_threads(void)
{
    cpu_set_t set;
    CPU_ZERO(&set);
    if (sched_getaffinity(0, sizeof(set), &set) == 0) {
        int n = CPU_COUNT(&set);
        if (n > 0) return n;
    }
    return 1;
}

static int resolve_threads(int nthreads)
{
    return nthreads > 0 ? nthreads : attn_oracle_default_threads();
}

/* ---------------------------------------------------------------------------
 * One query row from the definition.
 * "1 朴素的Attention" §1.1.2 of the cishoon.github.io page:
 *   s_ij = q_i . k_j * scale; safe softmax alpha_ij = exp(s_ij - m_i) / sum;
 *   o_i = sum_j alpha_ij v_j.
 * Causal visibility j <= i: §3.4 of the dandandamowang.xyz v2 page.
 * s is caller scratch of N doubles.
 * ------------------------------------------------------------------------- */
static void one_row(const double* qh, const double* kh, const double* vh,
                    int64_t N, int64_t D, double scale, int causal, int64_t i,
                    double* s, double* o_row, double* lse_out)
{
    const double* qi = qh + i * D;
    int64_t nvis = causal ? (i + 1) : N; /* keys 0 .. nvis-1 are visible */
    if (nvis > N) nvis = N;

    /* S row: s_ij = scale * (q_i . k_j) */
    for (int64_t j = 0; j < nvis; ++j) {
        const double* kj = kh + j * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += qi[d] * kj[d];
        s[j] = scale * dot;
    }

    /* m_i = max_j s_ij */
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j)
        if (s[j] > m) m = s[j];

    /* Z = sum_j exp(s_ij - m_i);  overwrite s with the unnormalised weights */
    double z = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        s[j] = exp(s[j] - m);
        z += s[j];
    }

    /* o_ic = sum_j (e_ij / Z) v_jc */
    for (int64_t c = 0; c < D; ++c) o_row[c] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        double p = s[j] / z;
        const double* vj = vh + j * D;
        for (int64_t c = 0; c < D; ++c) o_row[c] += p * vj[c];
    }

    if (lse_out) *lse_out = m + log(z);
}

/* ---------------------------------------------------------------------------
 * Thread plumbing: a flat list of (bh, row) work items split into contiguous
 * chunks, one chunk per thread.
 * ------------------------------------------------------------------------- */
typedef struct {
    const double *q, *k, *v;
    double *o, *lse;                 /* full-tensor outputs (fwd) */
    double *o_rows, *lse_rows;       /* per-request outputs (rows) */
    const int64_t *bh_idx, *row_idx; /* requests (rows); NULL for fwd */
    int64_t H, Hkv;                  /* query heads, key/value heads */
    int64_t N, D;
    double scale;
    int causal;
    int64_t begin, end;              /* item range of this thread */
    int failed;
} row_job;

static void* row_worker(void* arg)
{
    row_job* jb = (row_job*)arg;
    double* s = (double*)malloc(sizeof(double) * (size_t)(jb->N > 0 ? jb->N : 1));
    if (!s) { jb->failed = 1; return NULL; }
    const int64_t N = jb->N, D = jb->D;
    for (int64_t it = jb->begin; it < jb->end; ++it) {
        int64_t bh, i;
        double *o_row, *lse_out;
        if (jb->bh_idx) {            /* selected rows */
            bh = jb->bh_idx[it];
            i = jb->row_idx[it];
            o_row = jb->o_rows + it * D;
            lse_out = jb->lse_rows ? jb->lse_rows + it : NULL;
        } else {                     /* every row: item = bh*N + i */
            bh = it / N;
            i = it % N;
            o_row = jb->o + it * D;
            lse_out = jb->lse ? jb->lse + it : NULL;
        }
        /* query head bh = b*H + h reads key/value head b*Hkv + h/(H/Hkv) */
        const int64_t b = bh / jb->H, h = bh % jb->H;
        const int64_t kvh = b * jb->Hkv + h / (jb->H / jb->Hkv);
        const int64_t head = bh * N * D, kvhead = kvh * N * D;
        one_row(jb->q + head, jb->k + kvhead, jb->v + kvhead, N, D, jb->scale,
                jb->causal, i, s, o_row, lse_out);
    }
    free(s);
    return NULL;
}

static int run_rows(row_job proto, int64_t nitems, int nthreads)
{
    int nt = resolve_threads(nthreads);
    if (nt > nitems) nt = (int)(nitems > 0 ? nitems : 1);
    pthread_t* tid = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    row_job* jobs = (row_job*)calloc((size_t)nt, sizeof(row_job));
    int* started = (int*)calloc((size_t)nt, sizeof(int));
    if (!tid || !jobs || !started) { free(tid); free(jobs); free(started); return -3; }
    int rc = 0;
    for (int t = 0; t < nt; ++t) {
        jobs[t] = proto;
        jobs[t].begin = nitems * t / nt;
        jobs[t].end = nitems * (t + 1) / nt;
        jobs[t].failed = 0;
        if (nt == 1) {
            row_worker(&jobs[t]);
        } else if (pthread_create(&tid[t], NULL, row_worker, &jobs[t]) == 0) {
            started[t] = 1;
        } else {
            row_worker(&jobs[t]); /* could not spawn: do the chunk here */
        }
    }
    for (int t = 0; t < nt; ++t) {
        if (started[t]) pthread_join(tid[t], NULL);
        if (jobs[t].failed) rc = -3;
    }
    free(tid); free(jobs); free(started);
    return rc;
}

static int check_shape(int64_t B, int64_t H, int64_t N, int64_t D)
{
    return (B < 0 || H < 0 || N < 0 || D <= 0) ? -1 : 0;
}

static int check_heads(int64_t H, int64_t Hkv)
{
    return (Hkv <= 0 && H > 0) || Hkv < 0 || (Hkv > 0 && H % Hkv != 0) ? -1 : 0;
}

int attn_oracle_fwd_gqa(const double* q, const double* k, const double* v,
                        double* o, double* lse,
                        int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                        double scale, int causal, int nthreads)
{
    if (check_shape(B, H, N, D) || check_heads(H, Hkv)) return -1;
    int64_t nitems = B * H * N;
    if (nitems == 0) return 0;
    if (!q || !k || !v || !o) return -2;
    row_job p;
    memset(&p, 0, sizeof(p));
    p.q = q; p.k = k; p.v = v; p.o = o; p.lse = lse;
    p.H = H; p.Hkv = Hkv;
    p.N = N; p.D = D; p.scale = scale; p.causal = causal;
    return run_rows(p, nitems, nthreads);
}

int attn_oracle_fwd(const double* q, const double* k, const double* v,
                    double* o, double* lse,
                    int64_t B, int64_t H, int64_t N, int64_t D,
                    double scale, int causal, int nthreads)
{
    return attn_oracle_fwd_gqa(q, k, v, o, lse, B, H, H, N, D, scale, causal, nthreads);
}

int attn_oracle_rows_gqa(const double* q, const double* k, const double* v,
                         int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                         double scale, int causal,
                         const int64_t* bh_idx, const int64_t* row_idx, int64_t nrows,
                         double* o_rows, double* lse_rows, int nthreads)
{
    if (check_shape(B, H, N, D) || check_heads(H, Hkv) || nrows < 0) return -1;
    if (nrows == 0) return 0;
    if (!q || !k || !v || !bh_idx || !row_idx || !o_rows) return -2;
    for (int64_t r = 0; r < nrows; ++r)
        if (bh_idx[r] < 0 || bh_idx[r] >= B * H || row_idx[r] < 0 || row_idx[r] >= N)
            return -1;
    row_job p;
    memset(&p, 0, sizeof(p));
    p.q = q; p.k = k; p.v = v;
    p.o_rows = o_rows; p.lse_rows = lse_rows;
    p.bh_idx = bh_idx; p.row_idx = row_idx;
    p.H = H; p.Hkv = Hkv;
    p.N = N; p.D = D; p.scale = scale; p.causal = causal;
    return run_rows(p, nrows, nthreads);
}

int attn_oracle_rows(const double* q, const double* k, const double* v,
                     int64_t B, int64_t H, int64_t N, int64_t D,
                     double scale, int causal,
                     const int64_t* bh_idx, const int64_t* row_idx, int64_t nrows,
                     double* o_rows, double* lse_rows, int nthreads)
{
    return attn_oracle_rows_gqa(q, k, v, B, H, H, N, D, scale, causal, bh_idx, row_idx,
                                nrows, o_rows, lse_rows, nthreads);
}

int attn_oracle_probs(const double* q, const double* k,
                      int64_t B, int64_t H, int64_t N, int64_t D, int64_t bh,
                      double scale, int causal, double* p)
{
    if (check_shape(B, H, N, D) || bh < 0 || bh >= B * H) return -1;
    if (N == 0) return 0;
    if (!q || !k || !p) return -2;
    const double* qh = q + bh * N * D;
    const double* kh = k + bh * N * D;
    for (int64_t i = 0; i < N; ++i) {
        double* row = p + i * N;
        int64_t nvis = causal ? (i + 1) : N;
        const double* qi = qh + i * D;
        for (int64_t j = 0; j < N; ++j) row[j] = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += qi[d] * kh[j * D + d];
            row[j] = scale * dot;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < nvis; ++j) if (row[j] > m) m = row[j];
        double z = 0.0;
        for (int64_t j = 0; j < nvis; ++j) { row[j] = exp(row[j] - m); z += row[j]; }
        for (int64_t j = 0; j < nvis; ++j) row[j] /= z;
    }
    return 0;
}

/* ---------------------------------------------------------------------------
 * The tiled online-softmax method in the pages' order (fp64).
 *
 * Q tile [q_start, q_start+Br) outer; for each K/V tile [kv_start, kv_start+Bc):
 *   m_new  = max(m, rowmax(S_tile))                  running max
 *   corr   = exp(m_old - m_new)                      rescale factor
 *   l      = corr * l + sum_c exp(S_c - m_new)        running sum
 *   O~     = corr * O~ + exp(S_tile - m_new) @ V_tile unnormalised output
 * and O = O~ / l once at the end  (chang-wenbin.github.io report §2 "在线
 * Softmax"; deferred normalisation: dandandamowang.xyz v2 page §1.3).
 * Causal: kv_limit = min(q_start + Br, N) bounds the KV loop (tiles wholly
 * above the diagonal are never visited); tiles with kv_start + Bc - 1 >
 * q_start get the per-element mask key > row -> -inf; keys >= N -> -inf
 * (dandandamowang.xyz v2 page §3.2, §3.4).
 * ------------------------------------------------------------------------- */
typedef struct {
    const double *q, *k, *v;
    double *o, *lse;
    int64_t N, D, Br, Bc, ntiles_q;
    double scale;
    int causal;
    int64_t begin, end;   /* range of (bh, q_tile) items */
    int failed;
} tile_job;

static void* tile_worker(void* arg)
{
    tile_job* jb = (tile_job*)arg;
    const int64_t N = jb->N, D = jb->D, Br = jb->Br, Bc = jb->Bc;
    double* m = (double*)malloc(sizeof(double) * (size_t)Br);
    double* l = (double*)malloc(sizeof(double) * (size_t)Br);
    double* acc = (double*)malloc(sizeof(double) * (size_t)(Br * D));
    double* st = (double*)malloc(sizeof(double) * (size_t)Bc);
    if (!m || !l || !acc || !st) { jb->failed = 1; free(m); free(l); free(acc); free(st); return NULL; }

    for (int64_t it = jb->begin; it < jb->end; ++it) {
        int64_t bh = it / jb->ntiles_q;
        int64_t q_start = (it % jb->ntiles_q) * Br;
        const double* qh = jb->q + bh * N * D;
        const double* kh = jb->k + bh * N * D;
        const double* vh = jb->v + bh * N * D;

        for (int64_t r = 0; r < Br; ++r) {
            m[r] = -INFINITY;
            l[r] = 0.0;
            for (int64_t c = 0; c < D; ++c) acc[r * D + c] = 0.0;
        }

        int64_t kv_limit = N;
        if (jb->causal) kv_limit = (q_start + Br < N) ? q_start + Br : N;
        int64_t Tc = (kv_limit + Bc - 1) / Bc;

        for (int64_t t = 0; t < Tc; ++t) {
            int64_t kv_start = t * Bc;
            int diag = jb->causal && (kv_start + Bc - 1 > q_start);
            for (int64_t r = 0; r < Br; ++r) {
                int64_t row = q_start + r;
                if (row >= N) continue;  /* out-of-range rows are never written */
                /* S tile row with masks */
                double mt = -INFINITY;
                for (int64_t c = 0; c < Bc; ++c) {
                    int64_t key = kv_start + c;
                    if (key >= N || (diag && key > row)) { st[c] = -INFINITY; continue; }
                    double dot = 0.0;
                    for (int64_t d = 0; d < D; ++d) dot += qh[row * D + d] * kh[key * D + d];
                    st[c] = jb->scale * dot;
                    if (st[c] > mt) mt = st[c];
                }
                double m_new = m[r] > mt ? m[r] : mt;
                if (m_new == -INFINITY) continue;   /* nothing visible yet */
                double corr = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);
                double lsum = 0.0;
                for (int64_t c = 0; c < Bc; ++c) {
                    st[c] = (st[c] == -INFINITY) ? 0.0 : exp(st[c] - m_new);
                    lsum += st[c];
                }
                l[r] = corr * l[r] + lsum;
                for (int64_t d = 0; d < D; ++d) {
                    double pv = 0.0;
                    for (int64_t c = 0; c < Bc; ++c) {
                        int64_t key = kv_start + c;
                        if (key < N) pv += st[c] * vh[key * D + d];
                    }
                    acc[r * D + d] = corr * acc[r * D + d] + pv;
                }
                m[r] = m_new;
            }
        }

        for (int64_t r = 0; r < Br; ++r) {
            int64_t row = q_start + r;
            if (row >= N) continue;
            double inv_l = 1.0 / l[r];
            for (int64_t d = 0; d < D; ++d)
                jb->o[(bh * N + row) * D + d] = acc[r * D + d] * inv_l;
            if (jb->lse) jb->lse[bh * N + row] = m[r] + log(l[r]);
        }
    }
    free(m); free(l); free(acc); free(st);
    return NULL;
}

int attn_oracle_online_fwd(const double* q, const double* k, const double* v,
                           double* o, double* lse,
                           int64_t B, int64_t H, int64_t N, int64_t D,
                           double scale, int causal, int64_t Br, int64_t Bc,
                           int nthreads)
{
    if (check_shape(B, H, N, D) || Br <= 0 || Bc <= 0) return -1;
    if (B * H * N == 0) return 0;
    if (!q || !k || !v || !o) return -2;
    int64_t ntq = (N + Br - 1) / Br;
    int64_t nitems = B * H * ntq;
    int nt = resolve_threads(nthreads);
    if (nt > nitems) nt = (int)nitems;
    pthread_t* tid = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    tile_job* jobs = (tile_job*)calloc((size_t)nt, sizeof(tile_job));
    int* started = (int*)calloc((size_t)nt, sizeof(int));
    if (!tid || !jobs || !started) { free(tid); free(jobs); free(started); return -3; }
    int rc = 0;
    for (int t = 0; t < nt; ++t) {
        tile_job* jb = &jobs[t];
        jb->q = q; jb->k = k; jb->v = v; jb->o = o; jb->lse = lse;
        jb->N = N; jb->D = D; jb->Br = Br; jb->Bc = Bc; jb->ntiles_q = ntq;
        jb->scale = scale; jb->causal = causal;
        jb->begin = nitems * t / nt;
        jb->end = nitems * (t + 1) / nt;
        if (nt == 1) tile_worker(jb);
        else if (pthread_create(&tid[t], NULL, tile_worker, jb) == 0) started[t] = 1;
        else tile_worker(jb);
    }
    for (int t = 0; t < nt; ++t) {
        if (started[t]) pthread_join(tid[t], NULL);
        if (jobs[t].failed) rc = -3;
    }
    free(tid); free(jobs); free(started);
    return rc;
}

/* ===========================================================================
 * Backward pass: the gradients of L = sum_{i,c} dO_ic * O_ic with respect to
 * Q, K and V, for a given upstream gradient dO.
 *
 * The chang-wenbin.github.io FA2 report (section "反向传播性能分析") only
 * sketches the backward kernel (the forward's tiling, gradient buffers
 * updated in place with atomics).  The gradients themselves are the chain
 * rule through the definition used by one_row above, written out per
 * element:
 *   P_ij    = exp(s_ij - LSE_i)            for visible j, s_ij = scale q_i.k_j
 *   dV_j    = sum_i P_ij dO_i
 *   dP_ij   = dO_i . v_j
 *   Delta_i = sum_j P_ij dP_ij              (= dO_i . O_i)
 *   dS_ij   = P_ij (dP_ij - Delta_i)       (softmax Jacobian)
 *   dQ_i    = scale sum_j dS_ij k_j
 *   dK_j    = scale sum_i dS_ij q_i
 * Sums run over the visible pairs only (j <= i under causal masking).
 * ========================================================================= */

/* LSE_i and Delta_i of row i of one head.  s: scratch of N doubles. */
static void bwd_row_stats(const double* qh, const double* kh, const double* vh,
                          const double* doh, int64_t N, int64_t D, double scale,
                          int causal, int64_t i, double* s,
                          double* lse_out, double* delta_out)
{
    const double* qi = qh + i * D;
    const double* doi = doh + i * D;
    int64_t nvis = causal ? (i + 1) : N;
    if (nvis > N) nvis = N;
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        const double* kj = kh + j * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += qi[d] * kj[d];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (int64_t j = 0; j < nvis; ++j) z += exp(s[j] - m);
    const double lse = m + log(z);
    double delta = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        const double* vj = vh + j * D;
        double dp = 0.0;
        for (int64_t c = 0; c < D; ++c) dp += doi[c] * vj[c];
        delta += exp(s[j] - lse) * dp;
    }
    *lse_out = lse;
    *delta_out = delta;
}

/* dQ_i = scale sum_j P_ij (dP_ij - Delta_i) k_j */
static void bwd_dq_row(const double* qh, const double* kh, const double* vh,
                       const double* doh, int64_t N, int64_t D, double scale,
                       int causal, int64_t i, double lse_i, double delta_i,
                       double* dq_row)
{
    const double* qi = qh + i * D;
    const double* doi = doh + i * D;
    int64_t nvis = causal ? (i + 1) : N;
    if (nvis > N) nvis = N;
    for (int64_t c = 0; c < D; ++c) dq_row[c] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        const double* kj = kh + j * D;
        const double* vj = vh + j * D;
        double dot = 0.0, dp = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += qi[d] * kj[d];
        for (int64_t c = 0; c < D; ++c) dp += doi[c] * vj[c];
        const double p = exp(scale * dot - lse_i);
        const double ds = p * (dp - delta_i);
        for (int64_t c = 0; c < D; ++c) dq_row[c] += scale * ds * kj[c];
    }
}

/* dK_j = scale sum_i P_ij (dP_ij - Delta_i) q_i and dV_j = sum_i P_ij dO_i,
 * over the rows i that see key j (i >= j under causal masking). */
static void bwd_dkdv_row(const double* qh, const double* kh, const double* vh,
                         const double* doh, int64_t N, int64_t D, double scale,
                         int causal, int64_t j, const double* lse_h,
                         const double* delta_h, double* dk_row, double* dv_row)
{
    const double* kj = kh + j * D;
    const double* vj = vh + j * D;
    for (int64_t c = 0; c < D; ++c) { dk_row[c] = 0.0; dv_row[c] = 0.0; }
    for (int64_t i = causal ? j : 0; i < N; ++i) {
        const double* qi = qh + i * D;
        const double* doi = doh + i * D;
        double dot = 0.0, dp = 0.0;
        for (int64_t d = 0; d < D; ++d) dot += qi[d] * kj[d];
        for (int64_t c = 0; c < D; ++c) dp += doi[c] * vj[c];
        const double p = exp(scale * dot - lse_h[i]);
        const double ds = p * (dp - delta_h[i]);
        for (int64_t c = 0; c < D; ++c) {
            dv_row[c] += p * doi[c];
            dk_row[c] += scale * ds * qi[c];
        }
    }
}

/* Generic split of nitems independent items over threads (contiguous chunks),
 * each thread with its own scratch of `scratch_len` doubles. */
typedef void (*item_fn)(const void* ctx, int64_t item, double* scratch);

typedef struct {
    item_fn fn;
    const void* ctx;
    int64_t begin, end, scratch_len;
    int failed;
} item_job;

static void* item_worker(void* arg)
{
    item_job* jb = (item_job*)arg;
    double* s = (double*)malloc(sizeof(double) * (size_t)(jb->scratch_len > 0 ? jb->scratch_len : 1));
    if (!s) { jb->failed = 1; return NULL; }
    for (int64_t it = jb->begin; it < jb->end; ++it) jb->fn(jb->ctx, it, s);
    free(s);
    return NULL;
}

static int parallel_items(item_fn fn, const void* ctx, int64_t nitems, int64_t scratch_len,
                          int nthreads)
{
    if (nitems <= 0) return 0;
    int nt = resolve_threads(nthreads);
    if (nt > nitems) nt = (int)nitems;
    pthread_t* tid = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
    item_job* jobs = (item_job*)calloc((size_t)nt, sizeof(item_job));
    int* started = (int*)calloc((size_t)nt, sizeof(int));
    if (!tid || !jobs || !started) { free(tid); free(jobs); free(started); return -3; }
    int rc = 0;
    for (int t = 0; t < nt; ++t) {
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].begin = nitems * t / nt;
        jobs[t].end = nitems * (t + 1) / nt;
        jobs[t].scratch_len = scratch_len;
        if (nt == 1) {
            item_worker(&jobs[t]);
        } else if (pthread_create(&tid[t], NULL, item_worker, &jobs[t]) == 0) {
            started[t] = 1;
        } else {
            item_worker(&jobs[t]);
        }
    }
    for (int t = 0; t < nt; ++t) {
        if (started[t]) pthread_join(tid[t], NULL);
        if (jobs[t].failed) rc = -3;
    }
    free(tid); free(jobs); free(started);
    return rc;
}

typedef struct {
    const double *q, *k, *v, *dout;
    int64_t N, D;
    double scale;
    int causal;
    const int64_t* heads;            /* head (b*H + h) of each slot */
    double *lse, *delta;             /* [nslots][N] */
    const double *lse_c, *delta_c;   /* read-only views of the same */
    const int64_t *slot_idx, *idx;   /* requests: slot and row (or key) */
    double *out0, *out1;             /* dq rows, or dk and dv rows */
} bwd_ctx;

static void stats_item(const void* vctx, int64_t it, double* s)
{
    const bwd_ctx* c = (const bwd_ctx*)vctx;
    const int64_t slot = it / c->N, i = it % c->N;
    const int64_t head = c->heads[slot] * c->N * c->D;
    bwd_row_stats(c->q + head, c->k + head, c->v + head, c->dout + head, c->N, c->D,
                  c->scale, c->causal, i, s, c->lse + it, c->delta + it);
}

static void dq_item(const void* vctx, int64_t it, double* s)
{
    const bwd_ctx* c = (const bwd_ctx*)vctx;
    (void)s;
    const int64_t slot = c->slot_idx[it], i = c->idx[it];
    const int64_t head = c->heads[slot] * c->N * c->D;
    bwd_dq_row(c->q + head, c->k + head, c->v + head, c->dout + head, c->N, c->D,
               c->scale, c->causal, i, c->lse_c[slot * c->N + i],
               c->delta_c[slot * c->N + i], c->out0 + it * c->D);
}

static void dkdv_item(const void* vctx, int64_t it, double* s)
{
    const bwd_ctx* c = (const bwd_ctx*)vctx;
    (void)s;
    const int64_t slot = c->slot_idx[it], j = c->idx[it];
    const int64_t head = c->heads[slot] * c->N * c->D;
    bwd_dkdv_row(c->q + head, c->k + head, c->v + head, c->dout + head, c->N, c->D,
                 c->scale, c->causal, j, c->lse_c + slot * c->N, c->delta_c + slot * c->N,
                 c->out0 + it * c->D, c->out1 + it * c->D);
}

int attn_oracle_bwd_stats(const double* q, const double* k, const double* v,
                          const double* dout, int64_t B, int64_t H, int64_t N, int64_t D,
                          double scale, int causal, const int64_t* heads, int64_t nheads,
                          double* lse, double* delta, int nthreads)
{
    if (check_shape(B, H, N, D) || nheads < 0) return -1;
    if (nheads == 0 || N == 0) return 0;
    if (!q || !k || !v || !dout || !heads || !lse || !delta) return -2;
    for (int64_t t = 0; t < nheads; ++t)
        if (heads[t] < 0 || heads[t] >= B * H) return -1;
    bwd_ctx c;
    memset(&c, 0, sizeof(c));
    c.q = q; c.k = k; c.v = v; c.dout = dout;
    c.N = N; c.D = D; c.scale = scale; c.causal = causal;
    c.heads = heads; c.lse = lse; c.delta = delta;
    return parallel_items(stats_item, &c, nheads * N, N, nthreads);
}

int attn_oracle_bwd_dq_rows(const double* q, const double* k, const double* v,
                            const double* dout, int64_t B, int64_t H, int64_t N, int64_t D,
                            double scale, int causal, const int64_t* heads, int64_t nheads,
                            const double* lse, const double* delta,
                            const int64_t* slot_idx, const int64_t* row_idx, int64_t nrows,
                            double* dq_rows, int nthreads)
{
    if (check_shape(B, H, N, D) || nheads < 0 || nrows < 0) return -1;
    if (nrows == 0) return 0;
    if (!q || !k || !v || !dout || !heads || !lse || !delta || !slot_idx || !row_idx || !dq_rows)
        return -2;
    for (int64_t r = 0; r < nrows; ++r)
        if (slot_idx[r] < 0 || slot_idx[r] >= nheads || row_idx[r] < 0 || row_idx[r] >= N) return -1;
    for (int64_t t = 0; t < nheads; ++t)
        if (heads[t] < 0 || heads[t] >= B * H) return -1;
    bwd_ctx c;
    memset(&c, 0, sizeof(c));
    c.q = q; c.k = k; c.v = v; c.dout = dout;
    c.N = N; c.D = D; c.scale = scale; c.causal = causal;
    c.heads = heads; c.lse_c = lse; c.delta_c = delta;
    c.slot_idx = slot_idx; c.idx = row_idx; c.out0 = dq_rows;
    return parallel_items(dq_item, &c, nrows, 1, nthreads);
}

int attn_oracle_bwd_dkdv_rows(const double* q, const double* k, const double* v,
                              const double* dout, int64_t B, int64_t H, int64_t N, int64_t D,
                              double scale, int causal, const int64_t* heads, int64_t nheads,
                              const double* lse, const double* delta,
                              const int64_t* slot_idx, const int64_t* key_idx, int64_t nkeys,
                              double* dk_rows, double* dv_rows, int nthreads)
{
    if (check_shape(B, H, N, D) || nheads < 0 || nkeys < 0) return -1;
    if (nkeys == 0) return 0;
    if (!q || !k || !v || !dout || !heads || !lse || !delta || !slot_idx || !key_idx ||
        !dk_rows || !dv_rows)
        return -2;
    for (int64_t r = 0; r < nkeys; ++r)
        if (slot_idx[r] < 0 || slot_idx[r] >= nheads || key_idx[r] < 0 || key_idx[r] >= N) return -1;
    for (int64_t t = 0; t < nheads; ++t)
        if (heads[t] < 0 || heads[t] >= B * H) return -1;
    bwd_ctx c;
    memset(&c, 0, sizeof(c));
    c.q = q; c.k = k; c.v = v; c.dout = dout;
    c.N = N; c.D = D; c.scale = scale; c.causal = causal;
    c.heads = heads; c.lse_c = lse; c.delta_c = delta;
    c.slot_idx = slot_idx; c.idx = key_idx; c.out0 = dk_rows; c.out1 = dv_rows;
    return parallel_items(dkdv_item, &c, nkeys, 1, nthreads);
}

int attn_oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv,
                    int64_t B, int64_t H, int64_t N, int64_t D,
                    double scale, int causal, int nthreads)
{
    if (check_shape(B, H, N, D)) return -1;
    const int64_t BH = B * H;
    if (BH * N == 0) return 0;
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return -2;
    int64_t* heads = (int64_t*)malloc(sizeof(int64_t) * (size_t)BH);
    int64_t* slot = (int64_t*)malloc(sizeof(int64_t) * (size_t)(BH * N));
    int64_t* idx = (int64_t*)malloc(sizeof(int64_t) * (size_t)(BH * N));
    double* lse = (double*)malloc(sizeof(double) * (size_t)(BH * N));
    double* delta = (double*)malloc(sizeof(double) * (size_t)(BH * N));
    int rc = -3;
    if (heads && slot && idx && lse && delta) {
        for (int64_t t = 0; t < BH; ++t) heads[t] = t;
        for (int64_t it = 0; it < BH * N; ++it) { slot[it] = it / N; idx[it] = it % N; }
        rc = attn_oracle_bwd_stats(q, k, v, dout, B, H, N, D, scale, causal, heads, BH,
                                   lse, delta, nthreads);
        if (rc == 0)
            rc = attn_oracle_bwd_dq_rows(q, k, v, dout, B, H, N, D, scale, causal, heads, BH,
                                         lse, delta, slot, idx, BH * N, dq, nthreads);
        if (rc == 0)
            rc = attn_oracle_bwd_dkdv_rows(q, k, v, dout, B, H, N, D, scale, causal, heads, BH,
                                           lse, delta, slot, idx, BH * N, dk, dv, nthreads);
    }
    free(heads); free(slot); free(idx); free(lse); free(delta);
    return rc;
}

/* ---------------------------------------------------------------------------
 * Backward of grouped-query attention: query head h of batch b reads key/value
 * head b*Hkv + h/(H/Hkv), so by the chain rule the gradient of a shared key or
 * value row is the sum of the per-query-head gradients over the H/Hkv query
 * heads that read it; dQ is per query head as before.
 * ------------------------------------------------------------------------- */
typedef struct {
    const double *q, *k, *v, *dout;
    int64_t H, Hkv, N, D;
    double scale;
    int causal;
    double *lse, *delta;   /* [B*H][N] */
    double *dq, *dk, *dv;  /* dq [B,H,N,D]; dk, dv [B,Hkv,N,D] */
} gqa_bwd_ctx;

static int64_t gqa_kv_head(const gqa_bwd_ctx* c, int64_t bh)
{
    const int64_t b = bh / c->H, h = bh % c->H;
    return b * c->Hkv + h / (c->H / c->Hkv);
}

static void gqa_stats_item(const void* vctx, int64_t it, double* s)
{
    const gqa_bwd_ctx* c = (const gqa_bwd_ctx*)vctx;
    const int64_t bh = it / c->N, i = it % c->N;
    const int64_t qo = bh * c->N * c->D, ko = gqa_kv_head(c, bh) * c->N * c->D;
    bwd_row_stats(c->q + qo, c->k + ko, c->v + ko, c->dout + qo, c->N, c->D, c->scale, c->causal,
                  i, s, c->lse + it, c->delta + it);
}

static void gqa_dq_item(const void* vctx, int64_t it, double* s)
{
    const gqa_bwd_ctx* c = (const gqa_bwd_ctx*)vctx;
    (void)s;
    const int64_t bh = it / c->N, i = it % c->N;
    const int64_t qo = bh * c->N * c->D, ko = gqa_kv_head(c, bh) * c->N * c->D;
    bwd_dq_row(c->q + qo, c->k + ko, c->v + ko, c->dout + qo, c->N, c->D, c->scale, c->causal, i,
               c->lse[it], c->delta[it], c->dq + it * c->D);
}

/* item = (kv head, key j): sum over the query heads of the group; scratch
 * holds one dK row and one dV row of a single query head. */
static void gqa_dkdv_item(const void* vctx, int64_t it, double* s)
{
    const gqa_bwd_ctx* c = (const gqa_bwd_ctx*)vctx;
    const int64_t kvh = it / c->N, j = it % c->N;
    const int64_t b = kvh / c->Hkv, hk = kvh % c->Hkv, G = c->H / c->Hkv;
    const int64_t ko = kvh * c->N * c->D;
    double* dk_row = c->dk + it * c->D;
    double* dv_row = c->dv + it * c->D;
    for (int64_t d = 0; d < c->D; ++d) { dk_row[d] = 0.0; dv_row[d] = 0.0; }
    for (int64_t g = 0; g < G; ++g) {
        const int64_t bh = b * c->H + hk * G + g;
        const int64_t qo = bh * c->N * c->D;
        bwd_dkdv_row(c->q + qo, c->k + ko, c->v + ko, c->dout + qo, c->N, c->D, c->scale, c->causal,
                     j, c->lse + bh * c->N, c->delta + bh * c->N, s, s + c->D);
        for (int64_t d = 0; d < c->D; ++d) { dk_row[d] += s[d]; dv_row[d] += s[c->D + d]; }
    }
}

int attn_oracle_bwd_gqa(const double* q, const double* k, const double* v, const double* dout,
                        double* dq, double* dk, double* dv,
                        int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                        double scale, int causal, int nthreads)
{
    if (check_shape(B, H, N, D) || check_heads(H, Hkv)) return -1;
    if (B * H * N == 0) return 0;
    if (!q || !k || !v || !dout || !dq || !dk || !dv) return -2;
    double* lse = (double*)malloc(sizeof(double) * (size_t)(B * H * N));
    double* delta = (double*)malloc(sizeof(double) * (size_t)(B * H * N));
    int rc = -3;
    if (lse && delta) {
        gqa_bwd_ctx c;
        memset(&c, 0, sizeof(c));
        c.q = q; c.k = k; c.v = v; c.dout = dout;
        c.H = H; c.Hkv = Hkv; c.N = N; c.D = D; c.scale = scale; c.causal = causal;
        c.lse = lse; c.delta = delta; c.dq = dq; c.dk = dk; c.dv = dv;
        rc = parallel_items(gqa_stats_item, &c, B * H * N, N, nthreads);
        if (rc == 0) rc = parallel_items(gqa_dq_item, &c, B * H * N, 1, nthreads);
        if (rc == 0) rc = parallel_items(gqa_dkdv_item, &c, B * Hkv * N, 2 * D, nthreads);
    }
    free(lse); free(delta);
    return rc;
}

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

/*
 * attn_oracle.h -- slow, plain fp64 CPU oracle for exact scaled-dot-product
 * attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this library: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library.
 *
 * What it computes (the plain definition; the tiled GPU method reaches the
 * same result up to rounding order):
 *
 *   For every (b, h) and query row i of an [B,H,N,D] row-major tensor set,
 *     visible(i) = { j : 0 <= j < N }            (non-causal)
 *                = { j : 0 <= j <= i }           (causal, top-left aligned)
 *     s_ij   = scale * sum_d q_id * k_jd                  j in visible(i)
 *     m_i    = max_j s_ij
 *     p_ij   = exp(s_ij - m_i) / sum_j' exp(s_ij' - m_i)
 *     o_ic   = sum_j p_ij * v_jc
 *     lse_i  = m_i + ln sum_j exp(s_ij - m_i)     (natural log, scaled scores)
 *
 * Sources:
 *   - "1 朴素的Attention", §1.1.2 "Attention公式拆解" of the cishoon.github.io
 *     flashattention page: Attention(Q,K,V) = softmax(QK^T/sqrt(d)) V, the
 *     safe (max-subtracted) softmax and o_i = sum_j alpha_ij v_j; its §2
 *     "编写朴素Attention的 cuda 算子" (S, then row softmax, then P V).
 *   - Causal visibility (key j visible to row i iff j <= i): §1.4 and §3.4 of
 *     the dandandamowang.xyz "Flash Attention (二) v2" page.
 *   - Online-softmax recurrence used by attn_oracle_online_fwd: §2 "在线
 *     Softmax 的数值稳定性" of the chang-wenbin.github.io FA2 report; the
 *     Br/Bc tiling with causal block skip and diagonal element mask: §3.4 of
 *     the dandandamowang.xyz page.
 *
 * Every function returns 0 on success and a negative value on a bad argument.
 * All arrays are caller-owned host memory; nothing is retained after return.
 * nthreads <= 0 means "one thread per CPU in this process's affinity mask".
 */
#ifndef ATTN_ORACLE_H
#define ATTN_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Full forward.  q,k,v: [B,H,N,D] fp64.  o: [B,H,N,D].  lse: [B,H,N] or NULL. */
int attn_oracle_fwd(const double* q, const double* k, const double* v,
                    double* o, double* lse,
                    int64_t B, int64_t H, int64_t N, int64_t D,
                    double scale, int causal, int nthreads);

/* Selected rows only.  Row r of the request is (bh_idx[r], row_idx[r]) with
 * bh_idx = b*H + h.  o_rows: [nrows, D].  lse_rows: [nrows] or NULL. */
int attn_oracle_rows(const double* q, const double* k, const double* v,
                     int64_t B, int64_t H, int64_t N, int64_t D,
                     double scale, int causal,
                     const int64_t* bh_idx, const int64_t* row_idx, int64_t nrows,
                     double* o_rows, double* lse_rows, int nthreads);

/* Attention probabilities of one head (b*H+h = bh): p: [N, N], row i holds
 * p_ij for every key j (0 where j is not visible to i). */
int attn_oracle_probs(const double* q, const double* k,
                      int64_t B, int64_t H, int64_t N, int64_t D, int64_t bh,
                      double scale, int causal, double* p);

/* The tiled method itself, restated on the CPU in fp64 in the pages' order:
 * Q tiles of Br rows outer, K/V tiles of Bc keys inner, running row max m and
 * sum l, unnormalised accumulator O~ rescaled by exp(m_old - m_new), one
 * division by l at the end, KV loop cut at min(q_start + Br, N) under causal
 * masking and the element mask applied on tiles that cross the diagonal.
 * It exists to pin the tiling algebra (masks, skip bounds, tails) against the
 * definition above, independently of any GPU code. */
int attn_oracle_online_fwd(const double* q, const double* k, const double* v,
                           double* o, double* lse,
                           int64_t B, int64_t H, int64_t N, int64_t D,
                           double scale, int causal, int64_t Br, int64_t Bc,
                           int nthreads);

/* Grouped-query attention: q and o are [B,H,N,D], k and v are [B,Hkv,N,D]
 * with H a multiple of Hkv; query head h reads key/value head
 * h / (H/Hkv) of the same batch (consecutive query heads share a K/V head).
 * Hkv == H is ordinary multi-head attention; Hkv == 1 is multi-query.
 * Source: the GQA entry (Ainslie et al.) among the references of the
 * chang-wenbin.github.io FA2 report; the head mapping itself is not on the
 * pages and is the usual consecutive grouping. */
int attn_oracle_fwd_gqa(const double* q, const double* k, const double* v,
                        double* o, double* lse,
                        int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                        double scale, int causal, int nthreads);

/* Selected rows of the grouped-query forward; bh_idx indexes query heads
 * (b*H + h). */
int attn_oracle_rows_gqa(const double* q, const double* k, const double* v,
                         int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                         double scale, int causal,
                         const int64_t* bh_idx, const int64_t* row_idx, int64_t nrows,
                         double* o_rows, double* lse_rows, int nthreads);

/* ---- backward pass ------------------------------------------------------
 * Gradients of L = sum dO * O with respect to Q, K, V for the upstream
 * gradient dout ([B,H,N,D]), from the chain rule through the definition:
 * dV_j = sum_i P_ij dO_i; dP_ij = dO_i.v_j; Delta_i = sum_j P_ij dP_ij;
 * dS_ij = P_ij (dP_ij - Delta_i); dQ_i = scale sum_j dS_ij k_j;
 * dK_j = scale sum_i dS_ij q_i (visible pairs only).  The FA2 report of
 * chang-wenbin.github.io sketches the backward kernel without formulas.
 * Multi-head only (k and v have q's shape). */
int attn_oracle_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv,
                    int64_t B, int64_t H, int64_t N, int64_t D,
                    double scale, int causal, int nthreads);

/* Per-row LSE_i and Delta_i of the heads listed in heads[0..nheads) (each a
 * b*H + h index); lse and delta are [nheads][N]. */
int attn_oracle_bwd_stats(const double* q, const double* k, const double* v,
                          const double* dout, int64_t B, int64_t H, int64_t N, int64_t D,
                          double scale, int causal, const int64_t* heads, int64_t nheads,
                          double* lse, double* delta, int nthreads);

/* Selected rows of dQ: request r is row row_idx[r] of head heads[slot_idx[r]];
 * lse / delta as returned by attn_oracle_bwd_stats for the same heads list. */
int attn_oracle_bwd_dq_rows(const double* q, const double* k, const double* v,
                            const double* dout, int64_t B, int64_t H, int64_t N, int64_t D,
                            double scale, int causal, const int64_t* heads, int64_t nheads,
                            const double* lse, const double* delta,
                            const int64_t* slot_idx, const int64_t* row_idx, int64_t nrows,
                            double* dq_rows, int nthreads);

/* Selected rows of dK and dV (key key_idx[r] of head heads[slot_idx[r]]). */
int attn_oracle_bwd_dkdv_rows(const double* q, const double* k, const double* v,
                              const double* dout, int64_t B, int64_t H, int64_t N, int64_t D,
                              double scale, int causal, const int64_t* heads, int64_t nheads,
                              const double* lse, const double* delta,
                              const int64_t* slot_idx, const int64_t* key_idx, int64_t nkeys,
                              double* dk_rows, double* dv_rows, int nthreads);

/* Backward of grouped-query attention (k, v, dk, dv are [B,Hkv,N,D]): dQ per
 * query head; the dK and dV rows of a shared key/value head are the sums of
 * the per-query-head gradients over the H/Hkv query heads that read it. */
int attn_oracle_bwd_gqa(const double* q, const double* k, const double* v, const double* dout,
                        double* dq, double* dk, double* dv,
                        int64_t B, int64_t H, int64_t Hkv, int64_t N, int64_t D,
                        double scale, int causal, int nthreads);

/* Number of threads nthreads<=0 resolves to (CPUs in the affinity mask). */
int attn_oracle_default_threads(void);

#ifdef __cplusplus
}
#endif
#endif

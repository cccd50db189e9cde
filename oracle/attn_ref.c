/*
 * attn_ref.c -- float64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library calls this file: only the
 * test suite, the smoke check and the benchmark's CPU-baseline leg load it.
 * It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes is the plain definition, written out one query row at a
 * time, because the tiled method reaches exactly the standard result up to
 * floating-point evaluation order ("FlashAttention: GPU 메모리 계층을 활용한
 * 어텐션 최적화 분석", youngju.dev, sections 2.1 and 6.2):
 *
 *     s_j = scale * sum_c q[i,c] * k[j,c]        (j visible to i)
 *     m   = max_j s_j                            (safe softmax, eq. (1) of
 *     p_j = exp(s_j - m)                          "Flash Attention",
 *     l   = sum_j p_j                             suniverse77.github.io)
 *     O_i = sum_j p_j v[j,:] / l
 *     LSE_i = m + ln l
 *
 * Causal visibility: key j is visible to query i iff j <= i (top-left
 * aligned; section 11.3 of the youngju.dev page fuses this mask in the
 * kernel).  A row with no visible key yields O = 0 and LSE = -inf.
 *
 * The paged decode oracle first gathers each sequence's keys and values out
 * of the paged cache through the block table, using the cache layouts of
 * "PagedAttention" (data-sketchers.com, sections "Inputs", "Key" and
 * "Value"), and then applies the same single-row definition with one query
 * token and every context token visible.
 *
 * Every array is float64 and C-contiguous.  Parallelism is OpenMP over
 * independent rows only; each row is evaluated sequentially, so the result
 * does not depend on the thread count.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* One query row against n_keys contiguous key/value rows of width d.
 * scores is caller scratch of n_keys doubles.  Writes d outputs and the LSE;
 * if probs is non-NULL it also receives the normalised row of P. */
static void attend_row(const double *qi, const double *kk, const double *vv,
                       long n_keys, long d, double scale, double *scores,
                       double *oi, double *lse_i, double *probs)
{
    if (n_keys <= 0) {
        for (long c = 0; c < d; ++c) oi[c] = 0.0;
        *lse_i = -INFINITY;
        return;
    }
    /* S row: scaled dot products. */
    for (long j = 0; j < n_keys; ++j) {
        const double *kj = kk + j * d;
        double acc = 0.0;
        for (long c = 0; c < d; ++c) acc += qi[c] * kj[c];
        scores[j] = scale * acc;
    }
    /* Safe softmax: row max, exponentials, row sum. */
    double m = scores[0];
    for (long j = 1; j < n_keys; ++j)
        if (scores[j] > m) m = scores[j];
    double l = 0.0;
    for (long j = 0; j < n_keys; ++j) {
        scores[j] = exp(scores[j] - m);
        l += scores[j];
    }
    /* O row = P V with P = p / l. */
    for (long c = 0; c < d; ++c) oi[c] = 0.0;
    for (long j = 0; j < n_keys; ++j) {
        const double pj = scores[j] / l;
        const double *vj = vv + j * d;
        for (long c = 0; c < d; ++c) oi[c] += pj * vj[c];
        if (probs) probs[j] = pj;
    }
    *lse_i = m + log(l);
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward over [B,H,N,d] tensors for the query rows listed in rows[0..nrows)
 * of every (b,h).  o_rows is [B,H,nrows,d], lse_rows is [B,H,nrows].
 * Returns 0, or -1 on a bad argument / allocation failure. */
int oracle_forward_rows(const double *q, const double *k, const double *v,
                        const long *rows, long nrows, double *o_rows,
                        double *lse_rows, long B, long H, long N, long d,
                        double scale, int causal, int nthreads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || nrows < 0) return -1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -1;
    set_threads(nthreads);
    const long BH = B * H;
    int failed = 0;
#pragma omp parallel
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
        if (!scores) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long t = 0; t < BH * nrows; ++t) {
                const long bh = t / nrows, r = t % nrows;
                const long i = rows[r];
                const double *qh = q + bh * N * d, *kh = k + bh * N * d, *vh = v + bh * N * d;
                const long n_keys = causal ? i + 1 : N;
                attend_row(qh + i * d, kh, vh, n_keys, d, scale, scores,
                           o_rows + (bh * nrows + r) * d, lse_rows + bh * nrows + r, NULL);
            }
            free(scores);
        }
    }
    return failed ? -1 : 0;
}

/* Full forward: every query row.  o is [B,H,N,d], lse is [B,H,N]. */
int oracle_forward(const double *q, const double *k, const double *v, double *o,
                   double *lse, long B, long H, long N, long d, double scale,
                   int causal, int nthreads)
{
    if (N <= 0) return (B < 0 || H < 0 || N < 0 || d <= 0) ? -1 : 0;
    long *rows = (long *)malloc(sizeof(long) * (size_t)N);
    if (!rows) return -1;
    for (long i = 0; i < N; ++i) rows[i] = i;
    const int rc = oracle_forward_rows(q, k, v, rows, N, o, lse, B, H, N, d, scale,
                                       causal, nthreads);
    free(rows);
    return rc;
}

/* Forward with a boolean attention mask ("FlashAttention: GPU 메모리 계층을
 * 활용한 어텐션 최적화 분석", youngju.dev, section 11.3: a custom boolean
 * attn_mask, True = the key takes part): for row i of head bh the visible keys
 * are the j with mask[bh * mask_bh_stride + i * N + j] != 0 (mask_bh_stride = 0
 * shares one [N, N] mask across heads).  The visible keys and values are
 * gathered in order and the row definition applied to them; a row with no
 * visible key gives O = 0 and LSE = -inf. */
int oracle_forward_masked_rows(const double *q, const double *k, const double *v,
                               const unsigned char *mask, long mask_bh_stride,
                               const long *rows, long nrows, double *o_rows,
                               double *lse_rows, long B, long H, long N, long d,
                               double scale, int nthreads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0 || nrows < 0 || mask_bh_stride < 0) return -1;
    for (long r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= N) return -1;
    set_threads(nthreads);
    const long BH = B * H;
    int failed = 0;
#pragma omp parallel
    {
        const size_t n1 = (size_t)(N > 0 ? N : 1);
        double *scores = (double *)malloc(sizeof(double) * n1);
        double *kv = (double *)malloc(sizeof(double) * n1 * (size_t)d);
        double *vv = (double *)malloc(sizeof(double) * n1 * (size_t)d);
        if (!scores || !kv || !vv) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (long t = 0; t < BH * nrows; ++t) {
                const long bh = t / nrows, r = t % nrows;
                const long i = rows[r];
                const double *qh = q + bh * N * d, *kh = k + bh * N * d, *vh = v + bh * N * d;
                const unsigned char *mrow = mask + bh * mask_bh_stride + i * N;
                long n_vis = 0;
                for (long j = 0; j < N; ++j) {
                    if (mrow[j] != 0) {
                        for (long c = 0; c < d; ++c) {
                            kv[n_vis * d + c] = kh[j * d + c];
                            vv[n_vis * d + c] = vh[j * d + c];
                        }
                        ++n_vis;
                    }
                }
                attend_row(qh + i * d, kv, vv, n_vis, d, scale, scores,
                           o_rows + (bh * nrows + r) * d, lse_rows + bh * nrows + r, NULL);
            }
        }
        free(scores); free(kv); free(vv);
    }
    return failed ? -1 : 0;
}

/* The normalised softmax row P[i, 0..N) of one head (q,k are [N,d]); entries
 * of masked keys are written as 0.  Used to check that rows sum to one. */
int oracle_probs_row(const double *q, const double *k, long N, long d, long i,
                     double scale, int causal, double *p_out)
{
    if (N <= 0 || d <= 0 || i < 0 || i >= N) return -1;
    double *scores = (double *)malloc(sizeof(double) * (size_t)N);
    double *o_tmp = (double *)calloc((size_t)d, sizeof(double));
    double *v_zero = (double *)calloc((size_t)(N * d), sizeof(double));
    if (!scores || !o_tmp || !v_zero) {
        free(scores); free(o_tmp); free(v_zero);
        return -1;
    }
    const long n_keys = causal ? i + 1 : N;
    double lse;
    for (long j = 0; j < N; ++j) p_out[j] = 0.0;
    attend_row(q + i * d, k, v_zero, n_keys, d, scale, scores, o_tmp, &lse, p_out);
    free(scores); free(o_tmp); free(v_zero);
    return 0;
}

/* Single-query paged decode with grouped key/value heads.
 *   q            [num_seqs, num_heads, head_size]
 *   k_cache      [num_blocks, num_kv_heads, head_size/x, block_size, x]
 *   v_cache      [num_blocks, num_kv_heads, head_size, block_size]
 *   block_tables [num_seqs, max_blocks]  (logical block -> physical block)
 *   context_lens [num_seqs]
 *   out          [num_seqs, num_heads, head_size], lse [num_seqs, num_heads]
 * ("PagedAttention", data-sketchers.com, sections "Inputs", "Concepts",
 * "Key", "Value".)  Token t of sequence s lives in physical block
 * block_tables[s][t / block_size] at offset t % block_size.  Query head h
 * reads key/value head kvh = h / (num_heads / num_kv_heads): the page indexes
 * the caches by a kv_head_idx without showing how it is derived; consecutive
 * query heads sharing one key/value head is the reading taken.  Element c of
 * the key is k_cache[pb][kvh][c / x][t % block_size][c % x] and element c of
 * the value is v_cache[pb][kvh][c][t % block_size]. */
int oracle_paged_decode_gqa(const double *q, const double *k_cache, const double *v_cache,
                            const int *block_tables, const int *context_lens,
                            double *out, double *lse, long num_seqs, long num_heads,
                            long num_kv_heads, long head_size, long block_size, long x,
                            long max_blocks, long num_blocks, double scale, int nthreads)
{
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || num_heads % num_kv_heads != 0 ||
        head_size <= 0 || block_size <= 0 || x <= 0 || head_size % x != 0 || max_blocks <= 0 ||
        num_blocks <= 0)
        return -1;
    for (long s = 0; s < num_seqs; ++s) {
        const long ctx = context_lens[s];
        if (ctx < 0 || ctx > max_blocks * block_size) return -1;
        for (long b = 0; b < (ctx + block_size - 1) / block_size; ++b) {
            const long pb = block_tables[s * max_blocks + b];
            if (pb < 0 || pb >= num_blocks) return -1;
        }
    }
    set_threads(nthreads);
    const long D = head_size;
    const long group = num_heads / num_kv_heads;
    const long kv_block_stride = num_kv_heads * D * block_size;  /* same for K and V */
    const long kv_head_stride = D * block_size;
    int failed = 0;
#pragma omp parallel
    {
        const long cap = max_blocks * block_size;
        double *K = (double *)malloc(sizeof(double) * (size_t)(cap * D));
        double *V = (double *)malloc(sizeof(double) * (size_t)(cap * D));
        double *scores = (double *)malloc(sizeof(double) * (size_t)cap);
        if (!K || !V || !scores) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long t = 0; t < num_seqs * num_heads; ++t) {
                const long s = t / num_heads, h = t % num_heads;
                const long kvh = h / group;
                const long ctx = context_lens[s];
                /* Gather this (sequence, head)'s keys and values. */
                for (long tok = 0; tok < ctx; ++tok) {
                    const long pb = block_tables[s * max_blocks + tok / block_size];
                    const long off = tok % block_size;
                    const double *kb = k_cache + pb * kv_block_stride + kvh * kv_head_stride;
                    const double *vb = v_cache + pb * kv_block_stride + kvh * kv_head_stride;
                    for (long c = 0; c < D; ++c) {
                        K[tok * D + c] = kb[((c / x) * block_size + off) * x + (c % x)];
                        V[tok * D + c] = vb[c * block_size + off];
                    }
                }
                attend_row(q + (s * num_heads + h) * D, K, V, ctx, D, scale, scores,
                           out + (s * num_heads + h) * D, lse + s * num_heads + h, NULL);
            }
        }
        free(K); free(V); free(scores);
    }
    return failed ? -1 : 0;
}

/* Single-query paged decode with one key/value head per query head
 * (num_kv_heads = num_heads): the caches are [num_blocks, num_heads, ...]. */
int oracle_paged_decode(const double *q, const double *k_cache, const double *v_cache,
                        const int *block_tables, const int *context_lens,
                        double *out, double *lse, long num_seqs, long num_heads,
                        long head_size, long block_size, long x, long max_blocks,
                        long num_blocks, double scale, int nthreads)
{
    return oracle_paged_decode_gqa(q, k_cache, v_cache, block_tables, context_lens, out, lse,
                                   num_seqs, num_heads, num_heads, head_size, block_size, x,
                                   max_blocks, num_blocks, scale, nthreads);
}

/* Backward pass of the same attention: given dO = dLoss/dO, the gradients
 * of the loss with respect to Q, K and V, obtained by differentiating the
 * forward definition above ("FlashAttention: GPU 메모리 계층을 활용한 어텐션
 * 최적화 분석", youngju.dev, section 7 describes the backward as recomputing
 * S and P from Q, K and the saved row statistics; the gradient formulas are
 * the chain rule through O = P V, P = softmax(S), S = scale * Q K^T):
 *
 *     dV_j  = sum_i P_ij dO_i
 *     dP_ij = dO_i . V_j
 *     D_i   = sum_j P_ij dP_ij
 *     dS_ij = P_ij (dP_ij - D_i)
 *     dQ_i  = scale * sum_j dS_ij K_j
 *     dK_j  = scale * sum_i dS_ij Q_i
 *
 * over visible pairs only (causal: j <= i).  Each row's P is materialised
 * from scratch exactly as in the forward.  Heads are independent and run in
 * parallel; inside a head the rows are visited in order, so the sums into
 * dK and dV have a fixed order.  All of dq, dk, dv are [B,H,N,d] and are
 * overwritten.  Returns 0, or -1 on a bad argument / allocation failure. */
int oracle_backward(const double *q, const double *k, const double *v, const double *dout,
                    double *dq, double *dk, double *dv, long B, long H, long N, long d,
                    double scale, int causal, int nthreads)
{
    if (B < 0 || H < 0 || N < 0 || d <= 0) return -1;
    if (N == 0) return 0;
    set_threads(nthreads);
    const long BH = B * H;
    int failed = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)N);
        double *dp = (double *)malloc(sizeof(double) * (size_t)N);
        if (!p || !dp) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 1)
            for (long bh = 0; bh < BH; ++bh) {
                const long base = bh * N * d;
                const double *qh = q + base, *kh = k + base, *vh = v + base, *doh = dout + base;
                double *dqh = dq + base, *dkh = dk + base, *dvh = dv + base;
                for (long x = 0; x < N * d; ++x) dqh[x] = dkh[x] = dvh[x] = 0.0;
                for (long i = 0; i < N; ++i) {
                    const long n_keys = causal ? i + 1 : N;
                    const double *qi = qh + i * d, *doi = doh + i * d;
                    /* P row (safe softmax of the scaled scores). */
                    double m = -INFINITY;
                    for (long j = 0; j < n_keys; ++j) {
                        double acc = 0.0;
                        for (long c = 0; c < d; ++c) acc += qi[c] * kh[j * d + c];
                        p[j] = scale * acc;
                        if (p[j] > m) m = p[j];
                    }
                    double l = 0.0;
                    for (long j = 0; j < n_keys; ++j) {
                        p[j] = exp(p[j] - m);
                        l += p[j];
                    }
                    for (long j = 0; j < n_keys; ++j) p[j] /= l;
                    /* dP row and D_i. */
                    double D = 0.0;
                    for (long j = 0; j < n_keys; ++j) {
                        double acc = 0.0;
                        for (long c = 0; c < d; ++c) acc += doi[c] * vh[j * d + c];
                        dp[j] = acc;
                        D += p[j] * acc;
                    }
                    /* Accumulate the three gradients. */
                    for (long j = 0; j < n_keys; ++j) {
                        const double ds = p[j] * (dp[j] - D);
                        for (long c = 0; c < d; ++c) {
                            dqh[i * d + c] += scale * ds * kh[j * d + c];
                            dkh[j * d + c] += scale * ds * qi[c];
                            dvh[j * d + c] += p[j] * doi[c];
                        }
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return failed ? -1 : 0;
}

/*
 * fmha_oracle.c -- plain, slow, fp64 CPU oracle for the fused attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the test suite, the smoke check and the CPU-baseline leg of
 * the benchmark do.  It shares no code, header or constant with the CUDA path.
 *
 * What it computes (the definition, written out with no blocking or fusion):
 * for every sequence b, head h and query row i of that sequence,
 *
 *   visible(i) = { j in [0, Lk) : not causal  or  j <= i + Lk - Lq }
 *   s_ij       = scale * sum_d q[i,d] * k[j,d]            (all j, then masked)
 *   s_ij       = -inf for j not in visible(i)             (explicit mask row)
 *   M_i        = max_j s_ij
 *   p_ij       = exp(s_ij - M_i)
 *   O_i        = sum_j p_ij v_j / sum_j p_ij
 *   LSE_i      = M_i + log(sum_j p_ij)                    (natural log)
 *
 * Sources: "[BUG] Unexpected Slower Performance in C++ CuTe (77_blackwell_fmha)
 * vs Python CuTe DSL (fmha.py) on Jetson Thor", section "Implementation
 * Differences in softmax_step" (scores scaled, shifted by the row max and
 * exponentiated, then used as the PV operand); "[BUG] CuTe DSL 4.7/4.8
 * regression: FlashAttention-4 SM100 forward kernel spills registers",
 * section "Steps/Code to reproduce bug" (packed [tokens, heads, head_dim]
 * tensors, cu_seqlens prefix offsets, causal varlen forward).  The pages do
 * not print the log-sum-exp or the causal alignment for Lq != Lk; this file
 * reads LSE as the natural log of sum_j exp(s_ij) and aligns the causal
 * diagonal to the bottom-right (j <= i + Lk - Lq).  A row with no visible key
 * gets O = 0 and LSE = -inf.
 *
 * Grouped K/V heads (not on the pages; the plainest extension): with kv_heads
 * K/V heads for heads query heads (heads a multiple of kv_heads), query head h
 * reads K/V head h / (heads / kv_heads), i.e. consecutive query heads share
 * one K/V head.  kv_heads == heads is ordinary multi-head attention.
 *
 * Inputs are bf16 bit patterns (uint16), upcast exactly to double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Sequence bounds of doc b: [*q0, *q0 + *lq) and [*k0, *k0 + *lk). */
static void doc_bounds(const int32_t *cu_q, const int32_t *cu_k, int b,
                       int max_seqlen_q, int max_seqlen_k,
                       int64_t *q0, int64_t *lq, int64_t *k0, int64_t *lk)
{
    if (cu_q) {
        *q0 = cu_q[b];
        *lq = (int64_t)cu_q[b + 1] - cu_q[b];
        *k0 = cu_k[b];
        *lk = (int64_t)cu_k[b + 1] - cu_k[b];
    } else {
        *q0 = (int64_t)b * max_seqlen_q;
        *lq = max_seqlen_q;
        *k0 = (int64_t)b * max_seqlen_k;
        *lk = max_seqlen_k;
    }
}

/*
 * One output row: query token (doc-local index i) of doc b, head h.
 * s_buf has room for lk doubles, mask_buf for lk chars.
 */
static void oracle_row(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                       int64_t q0, int64_t lq, int64_t k0, int64_t lk,
                       int64_t i, int h, int heads, int kv_heads, int head_dim,
                       double scale, int causal, double *s_buf, char *mask_buf,
                       double *o_row, double *lse_out)
{
    const int64_t row_stride = (int64_t)heads * head_dim;
    const int64_t kv_stride = (int64_t)kv_heads * head_dim;
    const int hk = h / (heads / kv_heads); /* this query head's K/V head */
    const uint16_t *qi = q + (q0 + i) * row_stride + (int64_t)h * head_dim;

    /* explicit mask row */
    for (int64_t j = 0; j < lk; ++j)
        mask_buf[j] = (!causal) || (j <= i + lk - lq);

    /* all scores, then the mask */
    for (int64_t j = 0; j < lk; ++j) {
        const uint16_t *kj = k + (k0 + j) * kv_stride + (int64_t)hk * head_dim;
        double dot = 0.0;
        for (int d = 0; d < head_dim; ++d)
            dot += bf16_bits_to_double(qi[d]) * bf16_bits_to_double(kj[d]);
        s_buf[j] = scale * dot;
    }
    for (int64_t j = 0; j < lk; ++j)
        if (!mask_buf[j])
            s_buf[j] = -INFINITY;

    double m = -INFINITY;
    for (int64_t j = 0; j < lk; ++j)
        if (s_buf[j] > m)
            m = s_buf[j];

    for (int d = 0; d < head_dim; ++d)
        o_row[d] = 0.0;
    if (m == -INFINITY) { /* no visible key */
        *lse_out = -INFINITY;
        return;
    }

    double z = 0.0;
    for (int64_t j = 0; j < lk; ++j) {
        double p = exp(s_buf[j] - m);
        s_buf[j] = p;
        z += p;
    }
    for (int64_t j = 0; j < lk; ++j) {
        if (s_buf[j] == 0.0)
            continue;
        const uint16_t *vj = v + (k0 + j) * kv_stride + (int64_t)hk * head_dim;
        for (int d = 0; d < head_dim; ++d)
            o_row[d] += s_buf[j] * bf16_bits_to_double(vj[d]);
    }
    for (int d = 0; d < head_dim; ++d)
        o_row[d] /= z;
    *lse_out = m + log(z);
}

/* Doc index holding packed query token tok (cu_q non-NULL), by linear scan. */
static int doc_of_token(const int32_t *cu_q, int batch, int64_t tok)
{
    for (int b = 0; b < batch; ++b)
        if (tok >= cu_q[b] && tok < cu_q[b + 1])
            return b;
    return -1;
}

/*
 * oracle_fmha_fwd
 *
 * q       : bf16 bits, [total_q, heads, head_dim] contiguous.
 * k, v    : bf16 bits, [total_k, kv_heads, head_dim] contiguous.
 * cu_q/cu_k : int32 prefix offsets [batch + 1], or both NULL for dense
 *             batches of max_seqlen_q / max_seqlen_k rows each.
 * rows == NULL : full output.  out is [total_q, heads, head_dim] double and
 *             lse is [heads, total_q] double.
 * rows != NULL : n_rows flattened indices (token * heads + head); out is
 *             [n_rows, head_dim] and lse is [n_rows].
 * n_threads <= 0 uses the OpenMP default.
 * Returns 0, or -1 on a bad argument (nothing written).
 */
int oracle_fmha_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    double *out, double *lse,
                    const int32_t *cu_q, const int32_t *cu_k, int batch,
                    int64_t total_q, int64_t total_k,
                    int max_seqlen_q, int max_seqlen_k,
                    int heads, int kv_heads, int head_dim, double scale, int causal,
                    const int64_t *rows, int64_t n_rows, int n_threads)
{
    (void)total_k;
    if (!q || !k || !v || !out || !lse || batch < 0 || heads < 1 || head_dim < 1)
        return -1;
    if (kv_heads < 1 || heads % kv_heads != 0)
        return -1;
    if ((cu_q == NULL) != (cu_k == NULL))
        return -1;
    int64_t lk_max = 0;
    for (int b = 0; b < batch; ++b) {
        int64_t q0, lq, k0, lk;
        doc_bounds(cu_q, cu_k, b, max_seqlen_q, max_seqlen_k, &q0, &lq, &k0, &lk);
        if (lq < 0 || lk < 0)
            return -1;
        if (lk > lk_max)
            lk_max = lk;
    }
    const int64_t n_items = rows ? n_rows : total_q * heads;
    int bad = 0;

#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif

#pragma omp parallel reduction(| : bad)
    {
        double *s_buf = (double *)malloc(sizeof(double) * (size_t)(lk_max > 0 ? lk_max : 1));
        char *mask_buf = (char *)malloc((size_t)(lk_max > 0 ? lk_max : 1));
        double *o_row = (double *)malloc(sizeof(double) * (size_t)head_dim);
        if (!s_buf || !mask_buf || !o_row)
            bad = 1;
#pragma omp for schedule(dynamic, 4)
        for (int64_t it = 0; it < n_items; ++it) {
            if (bad)
                continue;
            const int64_t flat = rows ? rows[it] : it;
            const int64_t tok = flat / heads;
            const int h = (int)(flat % heads);
            if (tok < 0 || tok >= total_q) {
                bad = 1;
                continue;
            }
            const int b = cu_q ? doc_of_token(cu_q, batch, tok)
                               : (int)(tok / (max_seqlen_q > 0 ? max_seqlen_q : 1));
            if (b < 0 || b >= batch) {
                bad = 1;
                continue;
            }
            int64_t q0, lq, k0, lk;
            doc_bounds(cu_q, cu_k, b, max_seqlen_q, max_seqlen_k, &q0, &lq, &k0, &lk);
            double lse_val;
            oracle_row(q, k, v, q0, lq, k0, lk, tok - q0, h, heads, kv_heads, head_dim,
                       scale, causal, s_buf, mask_buf, o_row, &lse_val);
            double *dst = rows ? out + it * head_dim
                               : out + (tok * heads + h) * (int64_t)head_dim;
            memcpy(dst, o_row, sizeof(double) * (size_t)head_dim);
            if (rows)
                lse[it] = lse_val;
            else
                lse[(int64_t)h * total_q + tok] = lse_val;
        }
        free(s_buf);
        free(mask_buf);
        free(o_row);
    }
    return bad ? -1 : 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

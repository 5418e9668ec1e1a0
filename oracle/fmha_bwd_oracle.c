/*
 * fmha_bwd_oracle.c -- plain, slow, fp64 CPU oracle for the backward pass of
 * the fused attention forward (the gradients dQ, dK, dV).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the test suite and the benchmark's CPU-baseline leg do.  It
 * shares no code, header or constant with the CUDA path, nor with the forward
 * oracle (fmha_oracle.c).
 *
 * The forward is, for every sequence b, head h and query row i:
 *   visible(i) = { j in [0, Lk) : not causal  or  j <= i + Lk - Lq }
 *   s_ij = scale * q_i . k_j,  P_ij = softmax over visible(i) of s_ij (0 elsewhere),
 *   O_i  = sum_j P_ij v_j.
 * The backward pass takes an upstream gradient dO (same layout as O) and
 * returns the gradients of L = sum_i dO_i . O_i with respect to q, k, v.
 * Written out by the chain rule through the softmax, with no blocking or
 * fusion:
 *   dV_j  = sum_i P_ij dO_i                   (over every query row and every
 *                                             query head that reads this K/V head)
 *   dP_ij = dO_i . v_j
 *   D_i   = sum_j P_ij dP_ij                  (the softmax Jacobian's row term)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale * sum_j dS_ij k_j
 *   dK_j  = scale * sum_i dS_ij q_i
 * Rows with no visible key have P = 0 and get dQ = 0.  With grouped K/V heads
 * (query head h reads K/V head h / (heads / kv_heads)), dK and dV of a K/V head
 * sum the contributions of all its query heads.
 *
 * Sources: the forward pass is the one of "[BUG] Unexpected Slower Performance
 * in C++ CuTe (77_blackwell_fmha) vs Python CuTe DSL (fmha.py) on Jetson
 * Thor" (section "Implementation Differences in softmax_step") and "[BUG] CuTe
 * DSL 4.7/4.8 regression: FlashAttention-4 SM100 forward kernel spills
 * registers" (section "Steps/Code to reproduce bug"), whose benchmark step
 * runs this backward pass after the varlen causal forward (a mean-square loss
 * of the output, then .backward()).  The pages print no backward formula;
 * the gradient of the forward's definition is the plainest reading.
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

static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

typedef struct {
    const uint16_t *q, *k, *v, *dout;
    const int32_t *cu_q, *cu_k;
    int batch, max_seqlen_q, max_seqlen_k;
    int heads, kv_heads, head_dim;
    double scale;
    int causal;
} problem_t;

static void bounds(const problem_t *pr, int b, int64_t *q0, int64_t *lq, int64_t *k0, int64_t *lk)
{
    if (pr->cu_q) {
        *q0 = pr->cu_q[b];
        *lq = (int64_t)pr->cu_q[b + 1] - pr->cu_q[b];
        *k0 = pr->cu_k[b];
        *lk = (int64_t)pr->cu_k[b + 1] - pr->cu_k[b];
    } else {
        *q0 = (int64_t)b * pr->max_seqlen_q;
        *lq = pr->max_seqlen_q;
        *k0 = (int64_t)b * pr->max_seqlen_k;
        *lk = pr->max_seqlen_k;
    }
}

/* Is key j visible to query row i of a sequence with lq queries and lk keys? */
static int visible(const problem_t *pr, int64_t i, int64_t j, int64_t lq, int64_t lk)
{
    return !pr->causal || j <= i + lk - lq;
}

static const uint16_t *qrow(const problem_t *pr, int64_t tok, int h)
{
    return pr->q + (tok * pr->heads + h) * (int64_t)pr->head_dim;
}
static const uint16_t *dorow(const problem_t *pr, int64_t tok, int h)
{
    return pr->dout + (tok * pr->heads + h) * (int64_t)pr->head_dim;
}
static const uint16_t *krow(const problem_t *pr, int64_t tok, int hk)
{
    return pr->k + (tok * pr->kv_heads + hk) * (int64_t)pr->head_dim;
}
static const uint16_t *vrow(const problem_t *pr, int64_t tok, int hk)
{
    return pr->v + (tok * pr->kv_heads + hk) * (int64_t)pr->head_dim;
}

static double dot_bf16(const uint16_t *a, const uint16_t *b, int n)
{
    double s = 0.0;
    for (int d = 0; d < n; ++d)
        s += bf16_to_double(a[d]) * bf16_to_double(b[d]);
    return s;
}

/*
 * Softmax statistics of query row i (sequence-local) of head h: the row max
 * m_i and normaliser z_i = sum_j exp(s_ij - m_i) over the visible keys, so
 * that P_ij = exp(s_ij - m_i) / z_i, and D_i = sum_j P_ij dP_ij with
 * dP_ij = dO_i . v_j.  A row with no visible key gets z_i = 0 (and P = 0).
 * p is scratch for lk doubles.
 */
typedef struct {
    double m, z, d;
} rowstat_t;

static double score(const problem_t *pr, int64_t qtok, int h, int64_t ktok, int hk)
{
    return pr->scale * dot_bf16(qrow(pr, qtok, h), krow(pr, ktok, hk), pr->head_dim);
}

static rowstat_t row_stats(const problem_t *pr, int64_t q0, int64_t lq, int64_t k0, int64_t lk,
                           int64_t i, int h, double *p)
{
    const int hk = h / (pr->heads / pr->kv_heads);
    rowstat_t st = {-INFINITY, 0.0, 0.0};
    for (int64_t j = 0; j < lk; ++j) {
        p[j] = visible(pr, i, j, lq, lk) ? score(pr, q0 + i, h, k0 + j, hk) : -INFINITY;
        if (p[j] > st.m)
            st.m = p[j];
    }
    if (st.m == -INFINITY)
        return st;
    for (int64_t j = 0; j < lk; ++j)
        st.z += exp(p[j] - st.m); /* masked: exp(-inf) = 0 */
    const uint16_t *doi = dorow(pr, q0 + i, h);
    for (int64_t j = 0; j < lk; ++j) {
        const double pij = exp(p[j] - st.m) / st.z;
        if (pij != 0.0)
            st.d += pij * dot_bf16(doi, vrow(pr, k0 + j, hk), pr->head_dim);
    }
    return st;
}

/* P_ij from the row's statistics (0 for a masked key or an empty row). */
static double prob(const problem_t *pr, const rowstat_t *st, int64_t q0, int64_t lq, int64_t k0,
                   int64_t lk, int64_t i, int h, int64_t j)
{
    if (st->z == 0.0 || !visible(pr, i, j, lq, lk))
        return 0.0;
    const int hk = h / (pr->heads / pr->kv_heads);
    return exp(score(pr, q0 + i, h, k0 + j, hk) - st->m) / st->z;
}

/* dQ of sequence-local query row i, head h (sequence b). */
static void dq_row(const problem_t *pr, int b, int64_t i, int h, double *p, double *out)
{
    int64_t q0, lq, k0, lk;
    bounds(pr, b, &q0, &lq, &k0, &lk);
    const int hk = h / (pr->heads / pr->kv_heads);
    const rowstat_t st = row_stats(pr, q0, lq, k0, lk, i, h, p);
    for (int d = 0; d < pr->head_dim; ++d)
        out[d] = 0.0;
    for (int64_t j = 0; j < lk; ++j) {
        const double pij = prob(pr, &st, q0, lq, k0, lk, i, h, j);
        if (pij == 0.0)
            continue;
        const double dpij = dot_bf16(dorow(pr, q0 + i, h), vrow(pr, k0 + j, hk), pr->head_dim);
        const double ds = pij * (dpij - st.d);
        const uint16_t *kj = krow(pr, k0 + j, hk);
        for (int d = 0; d < pr->head_dim; ++d)
            out[d] += pr->scale * ds * bf16_to_double(kj[d]);
    }
}

/*
 * dK and dV of sequence-local key j, K/V head hk (sequence b): sums over every
 * query head h of the group and every query row i that sees key j.  stats
 * holds the row statistics of the sequence's rows for the group's heads,
 * [group][lq].
 */
static void dkdv_row(const problem_t *pr, int b, int64_t j, int hk, const rowstat_t *stats,
                     double *dk, double *dv)
{
    int64_t q0, lq, k0, lk;
    bounds(pr, b, &q0, &lq, &k0, &lk);
    const int group = pr->heads / pr->kv_heads;
    for (int d = 0; d < pr->head_dim; ++d)
        dk[d] = dv[d] = 0.0;
    for (int g = 0; g < group; ++g) {
        const int h = hk * group + g;
        for (int64_t i = 0; i < lq; ++i) {
            const rowstat_t *st = &stats[(int64_t)g * lq + i];
            const double pij = prob(pr, st, q0, lq, k0, lk, i, h, j);
            if (pij == 0.0)
                continue;
            const uint16_t *doi = dorow(pr, q0 + i, h);
            const double dpij = dot_bf16(doi, vrow(pr, k0 + j, hk), pr->head_dim);
            const double ds = pij * (dpij - st->d);
            const uint16_t *qi = qrow(pr, q0 + i, h);
            for (int d = 0; d < pr->head_dim; ++d) {
                dv[d] += pij * bf16_to_double(doi[d]);
                dk[d] += pr->scale * ds * bf16_to_double(qi[d]);
            }
        }
    }
}

static int doc_of(const int32_t *cu, int batch, int64_t tok, int max_seqlen)
{
    if (!cu)
        return (max_seqlen > 0 && tok >= 0 && tok / max_seqlen < batch) ? (int)(tok / max_seqlen) : -1;
    for (int b = 0; b < batch; ++b)
        if (tok >= cu[b] && tok < cu[b + 1])
            return b;
    return -1;
}

/*
 * oracle_fmha_bwd
 *
 * q, dout : bf16 bits [total_q, heads, head_dim];  k, v : [total_k, kv_heads, head_dim].
 * cu_q/cu_k : int32 prefix offsets [batch + 1], or both NULL for dense batches.
 * rows    : NULL, or n_rows flattened query indices (token * heads + head):
 *           dq is then [n_rows, head_dim], else [total_q, heads, head_dim].
 * keys    : NULL, or n_keys flattened key indices (token * kv_heads + kv_head):
 *           dk, dv are then [n_keys, head_dim], else [total_k, kv_heads, head_dim].
 * dq or dk/dv may be NULL to skip that part.  Tokens outside every sequence
 * get zero gradients in full mode and are rejected in sample mode.
 * Returns 0, or -1 on a bad argument.
 */
int oracle_fmha_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v, const uint16_t *dout,
                    double *dq, double *dk, double *dv,
                    const int32_t *cu_q, const int32_t *cu_k, int batch,
                    int64_t total_q, int64_t total_k, int max_seqlen_q, int max_seqlen_k,
                    int heads, int kv_heads, int head_dim, double scale, int causal,
                    const int64_t *rows, int64_t n_rows, const int64_t *keys, int64_t n_keys,
                    int n_threads)
{
    if (!q || !k || !v || !dout || batch < 0 || heads < 1 || head_dim < 1)
        return -1;
    if (kv_heads < 1 || heads % kv_heads != 0 || (cu_q == NULL) != (cu_k == NULL))
        return -1;
    if ((dk == NULL) != (dv == NULL))
        return -1;
    problem_t pr = {q, k, v, dout, cu_q, cu_k, batch, max_seqlen_q, max_seqlen_k,
                    heads, kv_heads, head_dim, scale, causal};
    int64_t lk_max = 1;
    for (int b = 0; b < batch; ++b) {
        int64_t q0, lq, k0, lk;
        bounds(&pr, b, &q0, &lq, &k0, &lk);
        if (lq < 0 || lk < 0)
            return -1;
        if (lk > lk_max)
            lk_max = lk;
    }
#ifdef _OPENMP
    if (n_threads > 0)
        omp_set_num_threads(n_threads);
#else
    (void)n_threads;
#endif
    int bad = 0;
    const int64_t nq = rows ? n_rows : total_q * heads;
    const int64_t nk = keys ? n_keys : total_k * kv_heads;
    /* every requested row and key must name a token of some sequence */
    for (int64_t it = 0; rows && it < n_rows; ++it)
        if (rows[it] < 0 || rows[it] >= total_q * heads ||
            doc_of(cu_q, batch, rows[it] / heads, max_seqlen_q) < 0)
            return -1;
    for (int64_t it = 0; keys && it < n_keys; ++it)
        if (keys[it] < 0 || keys[it] >= total_k * kv_heads ||
            doc_of(cu_k, batch, keys[it] / kv_heads, max_seqlen_k) < 0)
            return -1;
    if (!rows && dq)
        memset(dq, 0, sizeof(double) * (size_t)(total_q * heads * head_dim));
    if (!keys && dk) {
        memset(dk, 0, sizeof(double) * (size_t)(total_k * kv_heads * head_dim));
        memset(dv, 0, sizeof(double) * (size_t)(total_k * kv_heads * head_dim));
    }

    /* dQ: one row at a time */
    if (dq) {
#pragma omp parallel reduction(| : bad)
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)lk_max);
            if (!p)
                bad = 1;
#pragma omp for schedule(dynamic, 4)
            for (int64_t it = 0; it < nq; ++it) {
                if (bad)
                    continue;
                const int64_t flat = rows ? rows[it] : it;
                const int64_t tok = flat / heads;
                const int h = (int)(flat % heads);
                const int b = (tok >= 0 && tok < total_q) ? doc_of(cu_q, batch, tok, max_seqlen_q) : -1;
                if (b < 0 || b >= batch) {
                    if (rows)
                        bad = 1;
                    continue;
                }
                int64_t q0, lq, k0, lk;
                bounds(&pr, b, &q0, &lq, &k0, &lk);
                double *dst = rows ? dq + it * head_dim : dq + (tok * heads + h) * (int64_t)head_dim;
                dq_row(&pr, b, tok - q0, h, p, dst);
            }
            free(p);
        }
    }
    if (bad || !dk)
        return bad ? -1 : 0;

    /* dK, dV: per (sequence, K/V head) with a requested key, the row
     * statistics of that sequence's rows for the group's query heads, then
     * the requested keys */
    const int group = heads / kv_heads;
    for (int b = 0; b < batch && !bad; ++b) {
        int64_t q0, lq, k0, lk;
        bounds(&pr, b, &q0, &lq, &k0, &lk);
        for (int hk = 0; hk < kv_heads && !bad; ++hk) {
            /* the requested keys of this (sequence, K/V head): indices into keys, or
             * the flat indices themselves in full mode */
            int64_t *mine = (int64_t *)malloc(sizeof(int64_t) * (size_t)(keys ? (n_keys > 0 ? n_keys : 1)
                                                                              : (lk > 0 ? lk : 1)));
            if (!mine) {
                bad = 1;
                break;
            }
            int64_t n_here = 0;
            if (keys) {
                for (int64_t it = 0; it < nk; ++it) {
                    const int64_t tok = keys[it] / kv_heads;
                    if ((int)(keys[it] % kv_heads) == hk && tok >= k0 && tok < k0 + lk)
                        mine[n_here++] = it;
                }
            } else {
                for (int64_t tok = k0; tok < k0 + lk; ++tok)
                    mine[n_here++] = tok * kv_heads + hk;
            }
            if (n_here == 0) {
                free(mine);
                continue;
            }
            rowstat_t *stats = (rowstat_t *)malloc(sizeof(rowstat_t) * (size_t)(group * (lq > 0 ? lq : 1)));
            if (!stats) {
                free(mine);
                bad = 1;
                break;
            }
#pragma omp parallel reduction(| : bad)
            {
                double *p = (double *)malloc(sizeof(double) * (size_t)lk_max);
                if (!p)
                    bad = 1;
#pragma omp for schedule(dynamic, 8)
                for (int64_t gi = 0; gi < (int64_t)group * lq; ++gi) {
                    if (bad)
                        continue;
                    const int g = (int)(gi / lq);
                    stats[gi] = row_stats(&pr, q0, lq, k0, lk, gi % lq, hk * group + g, p);
                }
                free(p);
            }
#pragma omp parallel for schedule(dynamic, 1)
            for (int64_t n = 0; n < n_here; ++n) {
                const int64_t it = mine[n];
                const int64_t flat = keys ? keys[it] : it;
                const int64_t tok = flat / kv_heads;
                const int64_t off = keys ? it * head_dim : flat * (int64_t)head_dim;
                dkdv_row(&pr, b, tok - k0, hk, stats, dk + off, dv + off);
            }
            free(stats);
            free(mine);
        }
    }
    return bad ? -1 : 0;
}

/*
 * Exact softmax attention and its analytic gradient, in fp64, on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the GPU kernels
 * are checked against.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load it.  It shares no code, header or
 * constant with the CUDA library, and the library never calls it.
 *
 * What it computes is the plain definition of the operation, not the tiled
 * method: the whole score row of one query is formed, the two-pass stable
 * softmax is taken over it, and the products are plain sums.  Loops run in
 * the order of the formulas; nothing is blocked, fused or reordered.
 *
 * Sources (page title, then the place on the page):
 *  - "FlashAttention-2: Faster Attention with Better Parallelism and Work
 *    Partitioning" (paper digest), section 3 "Target operation":
 *    O = softmax(Q K^T) V with an optional causal mask, fp16/bf16 inputs.
 *    The scale factor the configurations use (1/sqrt(d)) multiplies Q K^T.
 *  - same digest, section 4 notation table: L = m + log(l), the logsumexp
 *    of a score row, and D = rowsum(dO o O), the backward auxiliary.
 *  - same digest, section 4 "logsumexp fusion": P = exp(S - L).
 *  - same digest, section 3 "FLOPs": the backward pass is five matrix
 *    products; below they are S = Q K^T, dV = P^T dO, dP = dO V^T,
 *    dQ = dS K and dK = dS^T Q with dS = P o (dP - D), the gradient of the
 *    scalar sum(O o dO) through the softmax.
 *  - same digest, section 4 "six checks", GQA/MQA: several query heads share
 *    one key/value head by index, and dK, dV sum over the sharing heads.
 *
 * Readings where the pages are silent:
 *  - the mask keeps key k for query i when k <= i + (Nk - Nq) (aligned to
 *    the bottom-right corner; with Nq == Nk this is k <= i);
 *  - L is the natural logarithm, of the scaled scores;
 *  - a query row with no allowed key (only possible when Nq > Nk under the
 *    mask) has O = 0, L = -inf and zero gradients;
 *  - query head h reads key/value head h / G, G = H / Hkv;
 *  - block-sparse attention ("FlashAttention: Fast and Memory-Efficient
 *    Exact Attention with IO-Awareness", abstract and "Key contributions") is
 *    exact attention restricted to the kept blocks of a given pattern: the
 *    block mask and the causal mask both apply, and a row they empty is
 *    treated as above.
 *
 * Layout: every array is row-major.  One call works on one "group": the G
 * query heads that share one key/value head.
 *   q, o, dout, dq : [G][Nq][d]      k, v, dk, dv : [Nk][d]
 *   lse            : [G][Nq]
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/*
 * Which keys a query row may see.  causal: key k for query i when
 * k <= i + (Nk - Nq).  block (optional): query block i / bs sees key block
 * k / bs only where block[g * head_stride + (i / bs) * nbc + k / bs] != 0, g
 * the query head within the group ("FlashAttention: Fast and Memory-Efficient
 * Exact Attention with IO-Awareness", abstract and "Key contributions": block-sparse
 * FlashAttention skips the zero blocks of a given block pattern; here it is
 * exact attention restricted to that pattern).
 */
struct mask_spec {
    int causal;
    const unsigned char *block; /* NULL: no block mask */
    long bs, nbc, head_stride;
};

static int allowed(const struct mask_spec *m, long g, long i, long k, long Nq, long Nk)
{
    if (m->block && !m->block[g * m->head_stride + (i / m->bs) * m->nbc + k / m->bs])
        return 0;
    if (!m->causal)
        return 1;
    return k <= i + (Nk - Nq);
}

static double dot(const double *x, const double *y, long d)
{
    double acc = 0.0;
    for (long c = 0; c < d; ++c)
        acc += x[c] * y[c];
    return acc;
}

/*
 * Scores of one query row: s[k] = scale * q_i . k_k for allowed keys,
 * -inf elsewhere.  Returns the row logsumexp L = m + ln(sum_k exp(s_k - m))
 * (two passes: max, then the shifted sum), or -inf for an empty row.
 */
static double score_row(const double *qi, const double *k, long g, long i, long Nq,
                        long Nk, long d, const struct mask_spec *ms, double scale, double *s)
{
    double m = -INFINITY;
    for (long kk = 0; kk < Nk; ++kk) {
        if (allowed(ms, g, i, kk, Nq, Nk)) {
            s[kk] = scale * dot(qi, k + kk * d, d);
            if (s[kk] > m)
                m = s[kk];
        } else {
            s[kk] = -INFINITY;
        }
    }
    if (m == -INFINITY)
        return -INFINITY;
    double l = 0.0;
    for (long kk = 0; kk < Nk; ++kk)
        if (allowed(ms, g, i, kk, Nq, Nk))
            l += exp(s[kk] - m);
    return m + log(l);
}

/* Softmax weight of one score given the row logsumexp: P = exp(S - L). */
static double weight(double s, double lse)
{
    if (lse == -INFINITY || s == -INFINITY)
        return 0.0;
    return exp(s - lse);
}

/* One query row of the forward pass: O_i = sum_k P_ik V_k, and L_i. */
static void forward_row(const double *qi, const double *k, const double *v,
                        long g, long i, long Nq, long Nk, long d,
                        const struct mask_spec *ms, double scale, double *s,
                        double *oi, double *lse_i)
{
    double L = score_row(qi, k, g, i, Nq, Nk, d, ms, scale, s);
    for (long c = 0; c < d; ++c)
        oi[c] = 0.0;
    for (long kk = 0; kk < Nk; ++kk) {
        double p = weight(s[kk], L);
        if (p == 0.0)
            continue;
        for (long c = 0; c < d; ++c)
            oi[c] += p * v[kk * d + c];
    }
    *lse_i = L;
}

/*
 * Forward pass for one group of G query heads.
 * q [G][Nq][d], k/v [Nk][d] -> o [G][Nq][d], lse [G][Nq].
 */
static void fwd_group(const double *q, const double *k, const double *v, long G, long Nq,
                      long Nk, long d, const struct mask_spec *ms, double scale, double *o,
                      double *lse)
{
    long rows = G * Nq;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < rows; ++r) {
            long g = r / Nq, i = r % Nq;
            forward_row(q + r * d, k, v, g, i, Nq, Nk, d, ms, scale, s, o + r * d,
                        lse + r);
        }
        free(s);
    }
}

void oracle_fwd_group(const double *q, const double *k, const double *v,
                      long G, long Nq, long Nk, long d, int causal,
                      double scale, double *o, double *lse)
{
    struct mask_spec ms = {causal, NULL, 1, 1, 0};
    fwd_group(q, k, v, G, Nq, Nk, d, &ms, scale, o, lse);
}

/*
 * As oracle_fwd_group with a block mask: block [G or 1][ceil(Nq/bs)][nbc]
 * bytes, head_stride = bytes between the heads' masks (0: one mask shared by
 * the group's heads).
 */
void oracle_fwd_group_blockmask(const double *q, const double *k, const double *v, long G,
                                long Nq, long Nk, long d, int causal,
                                const unsigned char *block, long bs, long nbc,
                                long head_stride, double scale, double *o, double *lse)
{
    struct mask_spec ms = {causal, block, bs, nbc, head_stride};
    fwd_group(q, k, v, G, Nq, Nk, d, &ms, scale, o, lse);
}

/*
 * Forward pass for a list of query rows of one group (used to check single
 * outputs of very large problems).  rows[2*t] = head within the group,
 * rows[2*t+1] = query index.  o [n][d], lse [n].
 */
void oracle_fwd_rows(const double *q, const double *k, const double *v,
                     long G, long Nq, long Nk, long d, int causal,
                     double scale, long n, const long *rows, double *o,
                     double *lse)
{
    (void)G;
    struct mask_spec ms = {causal, NULL, 1, 1, 0};
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 1)
        for (long t = 0; t < n; ++t) {
            long g = rows[2 * t], i = rows[2 * t + 1];
            forward_row(q + (g * Nq + i) * d, k, v, g, i, Nq, Nk, d, &ms, scale, s,
                        o + t * d, lse + t);
        }
        free(s);
    }
}

/*
 * Backward pass for one group, given the upstream gradient dO of the scalar
 * sum(O o dO).  The oracle recomputes its own fp64 O and L first.
 *   dV_k = sum_{g,i} P_ik dO_i
 *   dP_ik = dO_i . V_k,   D_i = dO_i . O_i,   dS_ik = P_ik (dP_ik - D_i)
 *   dQ_i = scale * sum_k dS_ik K_k
 *   dK_k = scale * sum_{g,i} dS_ik Q_i
 * Optional outputs o_out / lse_out / delta_out receive O, L and D (may be
 * NULL).
 */
static void bwd_group(const double *q, const double *k, const double *v,
                      const double *dout, long G, long Nq, long Nk, long d,
                      const struct mask_spec *ms, double scale, double *dq, double *dk,
                      double *dv, double *o_out, double *lse_out,
                      double *delta_out)
{
    long rows = G * Nq;
    double *o = (double *)malloc(sizeof(double) * (size_t)(rows * d + 1));
    double *L = (double *)malloc(sizeof(double) * (size_t)(rows + 1));
    double *D = (double *)malloc(sizeof(double) * (size_t)(rows + 1));

    /* Pass 1: O, L and D = rowsum(dO o O) for every query row. */
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < rows; ++r) {
            long g = r / Nq, i = r % Nq;
            forward_row(q + r * d, k, v, g, i, Nq, Nk, d, ms, scale, s,
                        o + r * d, L + r);
            D[r] = dot(dout + r * d, o + r * d, d);
        }
        free(s);
    }

    /* Pass 2: dQ_i = scale * sum_k P_ik (dP_ik - D_i) K_k, row by row. */
#pragma omp parallel for schedule(dynamic, 4)
    for (long r = 0; r < rows; ++r) {
        long g = r / Nq, i = r % Nq;
        const double *qi = q + r * d, *doi = dout + r * d;
        double *dqi = dq + r * d;
        for (long c = 0; c < d; ++c)
            dqi[c] = 0.0;
        for (long kk = 0; kk < Nk; ++kk) {
            if (!allowed(ms, g, i, kk, Nq, Nk))
                continue;
            double sik = scale * dot(qi, k + kk * d, d);
            double p = weight(sik, L[r]);
            double dp = dot(doi, v + kk * d, d);
            double ds = p * (dp - D[r]);
            for (long c = 0; c < d; ++c)
                dqi[c] += scale * ds * k[kk * d + c];
        }
    }

    /* Pass 3: dK_k and dV_k, key by key, summed over the G heads. */
#pragma omp parallel for schedule(dynamic, 4)
    for (long kk = 0; kk < Nk; ++kk) {
        double *dkk = dk + kk * d, *dvk = dv + kk * d;
        for (long c = 0; c < d; ++c) {
            dkk[c] = 0.0;
            dvk[c] = 0.0;
        }
        for (long r = 0; r < rows; ++r) {
            long g = r / Nq, i = r % Nq;
            if (!allowed(ms, g, i, kk, Nq, Nk))
                continue;
            const double *qi = q + r * d, *doi = dout + r * d;
            double sik = scale * dot(qi, k + kk * d, d);
            double p = weight(sik, L[r]);
            double dp = dot(doi, v + kk * d, d);
            double ds = p * (dp - D[r]);
            for (long c = 0; c < d; ++c) {
                dvk[c] += p * doi[c];
                dkk[c] += scale * ds * qi[c];
            }
        }
    }

    if (o_out)
        memcpy(o_out, o, sizeof(double) * (size_t)(rows * d));
    if (lse_out)
        memcpy(lse_out, L, sizeof(double) * (size_t)rows);
    if (delta_out)
        memcpy(delta_out, D, sizeof(double) * (size_t)rows);
    free(o);
    free(L);
    free(D);
}

/* Backward pass for one group (see bwd_group); causal or dense mask. */
void oracle_bwd_group(const double *q, const double *k, const double *v,
                      const double *dout, long G, long Nq, long Nk, long d,
                      int causal, double scale, double *dq, double *dk,
                      double *dv, double *o_out, double *lse_out,
                      double *delta_out)
{
    struct mask_spec ms = {causal, NULL, 1, 1, 0};
    bwd_group(q, k, v, dout, G, Nq, Nk, d, &ms, scale, dq, dk, dv, o_out, lse_out,
              delta_out);
}

/* As oracle_bwd_group with the block mask of oracle_fwd_group_blockmask. */
void oracle_bwd_group_blockmask(const double *q, const double *k, const double *v,
                                const double *dout, long G, long Nq, long Nk, long d,
                                int causal, const unsigned char *block, long bs, long nbc,
                                long head_stride, double scale, double *dq, double *dk,
                                double *dv)
{
    struct mask_spec ms = {causal, block, bs, nbc, head_stride};
    bwd_group(q, k, v, dout, G, Nq, Nk, d, &ms, scale, dq, dk, dv, NULL, NULL, NULL);
}

/*
 * The backward sums run over query rows, so they split by rows.  For the
 * flattened rows r = g * Nq + i in [r0, r1) of one group, this writes dQ of
 * those rows into dq [(r - r0)][d] and ADDS their contributions to dk and dv
 * ([Nk][d], zeroed by the caller).  Summing the calls over any partition of
 * the G * Nq rows gives oracle_bwd_group's dK and dV.  (Used to time a
 * bounded sample of a large problem.)
 */
void oracle_bwd_rows(const double *q, const double *k, const double *v,
                     const double *dout, long G, long Nq, long Nk, long d,
                     int causal, double scale, long r0, long r1, double *dq,
                     double *dk, double *dv)
{
    (void)G;
    struct mask_spec ms = {causal, NULL, 1, 1, 0};
    long n = r1 - r0;
    if (n <= 0)
        return;
    double *o = (double *)malloc(sizeof(double) * (size_t)(n * d));
    double *L = (double *)malloc(sizeof(double) * (size_t)n);
    double *D = (double *)malloc(sizeof(double) * (size_t)n);

#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < n; ++t) {
            long r = r0 + t, g = r / Nq, i = r % Nq;
            forward_row(q + r * d, k, v, g, i, Nq, Nk, d, &ms, scale, s,
                        o + t * d, L + t);
            D[t] = dot(dout + r * d, o + t * d, d);
        }
        free(s);
    }

#pragma omp parallel for schedule(dynamic, 4)
    for (long t = 0; t < n; ++t) {
        long r = r0 + t, g = r / Nq, i = r % Nq;
        const double *qi = q + r * d, *doi = dout + r * d;
        double *dqi = dq + t * d;
        for (long c = 0; c < d; ++c)
            dqi[c] = 0.0;
        for (long kk = 0; kk < Nk; ++kk) {
            if (!allowed(&ms, g, i, kk, Nq, Nk))
                continue;
            double sik = scale * dot(qi, k + kk * d, d);
            double p = weight(sik, L[t]);
            double dp = dot(doi, v + kk * d, d);
            double ds = p * (dp - D[t]);
            for (long c = 0; c < d; ++c)
                dqi[c] += scale * ds * k[kk * d + c];
        }
    }

#pragma omp parallel for schedule(dynamic, 4)
    for (long kk = 0; kk < Nk; ++kk) {
        double *dkk = dk + kk * d, *dvk = dv + kk * d;
        for (long t = 0; t < n; ++t) {
            long r = r0 + t, g = r / Nq, i = r % Nq;
            if (!allowed(&ms, g, i, kk, Nq, Nk))
                continue;
            const double *qi = q + r * d, *doi = dout + r * d;
            double sik = scale * dot(qi, k + kk * d, d);
            double p = weight(sik, L[t]);
            double dp = dot(doi, v + kk * d, d);
            double ds = p * (dp - D[t]);
            for (long c = 0; c < d; ++c) {
                dvk[c] += p * doi[c];
                dkk[c] += scale * ds * qi[c];
            }
        }
    }
    free(o);
    free(L);
    free(D);
}

/* Number of threads the parallel loops above use. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

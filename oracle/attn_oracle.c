/*
 * attn_oracle.c — fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package smoke check and the bench's
 * CPU-baseline leg use it.  It shares no code, header, table or helper with
 * the CUDA library under exact_attention_tma_gb300/csrc.
 *
 * What it computes is the plain definition of attention given in
 * "Why Fast GPUs Still Wait for Memory" (srini-anirudh.github.io), section
 * "Attention from first principles" (the "core of attention" display):
 *     S = Q K^T,  P = softmax(S),  O = P V
 * and restated in "Warmup Guide — C++/CUDA & GPU Performance Engineering" (ai-engineer-zt0.pages.dev), chapter 7, Operator Fusion
 * (FlashAttention paragraph).  Decode is the same definition with a single
 * query row against the whole KV cache ("Attention III · KV cache, GQA, MLA"
 * on the roofline page).
 *
 * Readings where the pages leave a step open (each also listed in the design
 * notes):
 *   - scale: S is multiplied by the caller's `scale` before mask and softmax
 *     (the pages print softmax(QK^T) with no scale);
 *   - causal mask: with as many queries as keys, key j is visible to query i
 *     iff j <= i; masked scores are -inf, so their P entry is exactly 0;
 *   - LSE: natural log of sum_j exp(s_ij) over visible j, scale included;
 *   - split-KV (decode): chunk c = ceil(L / nsplit) keys, split s covers
 *     [s*c, min(L, (s+1)*c)); an empty split has lse = -inf and O_s = 0; the
 *     combine weights each normalised partial by exp(lse_s - max lse).
 *
 * Everything is single threaded, fp64, with no blocking or reordering beyond
 * the definition: S and P are materialised as full (rows x keys) matrices.
 * Subtracting the row maximum before exp() does not change P (it cancels in
 * the ratio) and only keeps exp() finite.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_ERR_ARG 1
#define ORACLE_ERR_NOMEM 2

/*
 * One head.  Q is nq x d, K and V are nk x d, all row-major.  `rows` lists the
 * query rows to compute (NULL means all nq, in order); `nrows` is its length.
 * Outputs: O (nrows x d), LSE (nrows), and optionally P (nrows x nk).
 * If `rowsum_err` is non-NULL it receives max_r |sum_j P[r][j] - 1|.
 */
int oracle_attention(const double *Q, long nq, const double *K, const double *V,
                     long nk, long d, double scale, int causal, const long *rows,
                     long nrows, double *O, double *LSE, double *P_out,
                     double *rowsum_err)
{
    if (!Q || !K || !V || !O || !LSE || nq < 1 || nk < 1 || d < 1 || nrows < 1)
        return ORACLE_ERR_ARG;
    if (causal && nq != nk)
        return ORACLE_ERR_ARG;

    double *S = (double *)malloc(sizeof(double) * (size_t)nrows * (size_t)nk);
    double *P = (double *)malloc(sizeof(double) * (size_t)nrows * (size_t)nk);
    if (!S || !P) {
        free(S);
        free(P);
        return ORACLE_ERR_NOMEM;
    }
    double worst = 0.0;

    /* Step 1: S = scale * Q K^T, with the causal mask applied as -inf. */
    for (long r = 0; r < nrows; ++r) {
        long i = rows ? rows[r] : r;
        if (i < 0 || i >= nq) {
            free(S);
            free(P);
            return ORACLE_ERR_ARG;
        }
        for (long j = 0; j < nk; ++j) {
            double acc = 0.0;
            for (long k = 0; k < d; ++k)
                acc += Q[i * d + k] * K[j * d + k];
            S[r * nk + j] = (causal && j > i) ? -INFINITY : scale * acc;
        }
    }

    /* Step 2: P = softmax(S) row by row; LSE = log of the row's exp-sum. */
    for (long r = 0; r < nrows; ++r) {
        double m = -INFINITY;
        for (long j = 0; j < nk; ++j)
            if (S[r * nk + j] > m)
                m = S[r * nk + j];
        double z = 0.0;
        for (long j = 0; j < nk; ++j) {
            double e = (S[r * nk + j] == -INFINITY) ? 0.0 : exp(S[r * nk + j] - m);
            P[r * nk + j] = e;
            z += e;
        }
        double sum = 0.0;
        for (long j = 0; j < nk; ++j) {
            P[r * nk + j] /= z;
            sum += P[r * nk + j];
        }
        LSE[r] = m + log(z);
        if (fabs(sum - 1.0) > worst)
            worst = fabs(sum - 1.0);
    }

    /* Step 3: O = P V. */
    for (long r = 0; r < nrows; ++r) {
        for (long k = 0; k < d; ++k) {
            double acc = 0.0;
            for (long j = 0; j < nk; ++j)
                acc += P[r * nk + j] * V[j * d + k];
            O[r * d + k] = acc;
        }
    }

    if (P_out)
        memcpy(P_out, P, sizeof(double) * (size_t)nrows * (size_t)nk);
    if (rowsum_err)
        *rowsum_err = worst;
    free(S);
    free(P);
    return ORACLE_OK;
}

/*
 * Decode for one head: the single query q (d) attends to all L cached keys;
 * the new token sits after the cache, so no key is masked.
 */
int oracle_decode(const double *q, const double *K, const double *V, long L, long d,
                  double scale, double *O, double *LSE)
{
    return oracle_attention(q, 1, K, V, L, d, scale, 0, NULL, 1, O, LSE, NULL, NULL);
}

/*
 * Split-KV decode partials for one head: split s attends only to its own
 * chunk of keys and returns its normalised output O_s (d) and its log-sum-exp
 * lse_s.  Empty splits get lse = -inf and O_s = 0.
 */
int oracle_decode_split(const double *q, const double *K, const double *V, long L,
                        long d, double scale, long nsplit, double *O_s, double *lse_s)
{
    if (nsplit < 1 || L < 1)
        return ORACLE_ERR_ARG;
    long chunk = (L + nsplit - 1) / nsplit;
    for (long s = 0; s < nsplit; ++s) {
        long lo = s * chunk;
        long hi = lo + chunk < L ? lo + chunk : L;
        if (lo >= hi) {
            lse_s[s] = -INFINITY;
            for (long k = 0; k < d; ++k)
                O_s[s * d + k] = 0.0;
            continue;
        }
        int rc = oracle_attention(q, 1, K + lo * d, V + lo * d, hi - lo, d, scale, 0,
                                  NULL, 1, O_s + s * d, lse_s + s, NULL, NULL);
        if (rc)
            return rc;
    }
    return ORACLE_OK;
}

/*
 * Log-sum-exp combine of nsplit normalised partials: with m = max_s lse_s and
 * w_s = exp(lse_s - m), O = sum_s w_s O_s / sum_s w_s and
 * LSE = m + log(sum_s w_s).
 */
int oracle_lse_combine(const double *O_s, const double *lse_s, long nsplit, long d,
                       double *O, double *LSE)
{
    if (nsplit < 1)
        return ORACLE_ERR_ARG;
    double m = -INFINITY;
    for (long s = 0; s < nsplit; ++s)
        if (lse_s[s] > m)
            m = lse_s[s];
    if (m == -INFINITY)
        return ORACLE_ERR_ARG;
    double wsum = 0.0;
    for (long k = 0; k < d; ++k)
        O[k] = 0.0;
    for (long s = 0; s < nsplit; ++s) {
        double w = (lse_s[s] == -INFINITY) ? 0.0 : exp(lse_s[s] - m);
        wsum += w;
        for (long k = 0; k < d; ++k)
            O[k] += w * O_s[s * d + k];
    }
    for (long k = 0; k < d; ++k)
        O[k] /= wsum;
    *LSE = m + log(wsum);
    return ORACLE_OK;
}

/*
 * Gradients of one head's attention with respect to Q, K and V, given the
 * upstream gradient dO (n x d) of the output.  "Why Fast GPUs Still Wait for
 * Memory", section "FlashAttention is an IO algorithm", notes that the
 * backward pass recomputes S instead of storing it; the pages print no
 * formula for it, so this is the chain rule through the definition above,
 * written out with S and P materialised:
 *     dV = P^T dO
 *     dP = dO V^T
 *     dS_ij = P_ij (dP_ij - sum_k P_ik dP_ik)     (Jacobian of the row softmax)
 *     dQ = scale * dS K,   dK = scale * dS^T Q
 * Masked entries have P = 0 and so dS = 0.  Q, K, V, dO, dQ, dK, dV are n x d.
 */
int oracle_attention_backward(const double *Q, const double *K, const double *V,
                              const double *dO, long n, long d, double scale, int causal,
                              double *dQ, double *dK, double *dV)
{
    if (!Q || !K || !V || !dO || !dQ || !dK || !dV || n < 1 || d < 1)
        return ORACLE_ERR_ARG;
    double *P = (double *)malloc(sizeof(double) * (size_t)n * (size_t)n);
    double *dS = (double *)malloc(sizeof(double) * (size_t)n * (size_t)n);
    double *O = (double *)malloc(sizeof(double) * (size_t)n * (size_t)d);
    double *LSE = (double *)malloc(sizeof(double) * (size_t)n);
    if (!P || !dS || !O || !LSE) {
        free(P);
        free(dS);
        free(O);
        free(LSE);
        return ORACLE_ERR_NOMEM;
    }
    int rc = oracle_attention(Q, n, K, V, n, d, scale, causal, NULL, n, O, LSE, P, NULL);
    if (rc) {
        free(P);
        free(dS);
        free(O);
        free(LSE);
        return rc;
    }

    /* dV = P^T dO. */
    for (long j = 0; j < n; ++j)
        for (long k = 0; k < d; ++k) {
            double acc = 0.0;
            for (long i = 0; i < n; ++i)
                acc += P[i * n + j] * dO[i * d + k];
            dV[j * d + k] = acc;
        }

    /* dP = dO V^T, then dS = P * (dP - rowsum(P * dP)). */
    for (long i = 0; i < n; ++i) {
        double dot = 0.0;
        for (long j = 0; j < n; ++j) {
            double acc = 0.0;
            for (long k = 0; k < d; ++k)
                acc += dO[i * d + k] * V[j * d + k];
            dS[i * n + j] = acc; /* dP for now */
            dot += P[i * n + j] * acc;
        }
        for (long j = 0; j < n; ++j)
            dS[i * n + j] = P[i * n + j] * (dS[i * n + j] - dot);
    }

    /* dQ = scale * dS K;  dK = scale * dS^T Q. */
    for (long i = 0; i < n; ++i)
        for (long k = 0; k < d; ++k) {
            double acc = 0.0;
            for (long j = 0; j < n; ++j)
                acc += dS[i * n + j] * K[j * d + k];
            dQ[i * d + k] = scale * acc;
        }
    for (long j = 0; j < n; ++j)
        for (long k = 0; k < d; ++k) {
            double acc = 0.0;
            for (long i = 0; i < n; ++i)
                acc += dS[i * n + j] * Q[i * d + k];
            dK[j * d + k] = scale * acc;
        }

    free(P);
    free(dS);
    free(O);
    free(LSE);
    return ORACLE_OK;
}

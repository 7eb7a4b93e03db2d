/*
 * plx_oracle.c -- fp64 CPU oracle for Parallax (PLX) attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file or the library built from it: only the test suite, the
 * smoke check and the benchmark's CPU-baseline leg use it.  It shares no code
 * with the CUDA path.
 *
 * What it computes, for one query q (with probe rho) over n keys/values
 * K[j], V[j] (j = 0..n-1), every step in double precision:
 *
 *   s_j   = scale * (q . k_j)
 *   w_j   = exp(s_j - m) / sum_t exp(s_t - m),   m = max_t s_t
 *   lse   = m + ln sum_t exp(s_t - m)                 (natural log)
 *   vbar  = sum_j w_j v_j          (= o^SA, the softmax-attention output)
 *   kbar  = sum_j w_j k_j
 *
 * and the PLX output
 *
 *   o = o^SA - Sigma_KV rho,   Sigma_KV = sum_j w_j (v_j - vbar)(k_j - kbar)^T
 *
 * Sources ("Parallax: Parameterized Local Linear Attention for Language
 * Modeling", arXiv:2605.29157):
 *   - zhichai.net, section 1.3: o_i^PLX = o_i^SA - Sigma_KV^(i) rho_i, with
 *     Sigma_KV^(i) the weighted KV covariance and rho_i = W_R x_i; section 1.1
 *     for softmax(QK^T / sqrt(d)) V.
 *   - gist.science, "Meccanismo Principale": the same output formula, the
 *     boundary term eta_i set to zero and no conjugate-gradient solve.
 *   - gist.science, "Algoritmo Consapevole dell'Hardware": a streaming form
 *     that reuses the K/V stream; the identity used here is
 *     Sigma_KV rho = sum_j w_j (k_j . rho) v_j - vbar (kbar . rho).
 *
 * Readings taken where the pages are silent: Sigma_KV is d_v x d_k (rho lives
 * in key space, since it replaces the solved probe Sigma_KK^{-1} mu); the
 * weights sum to one and the covariance has no Bessel correction; the scale
 * multiplies q.k only (rho.k is not scaled); the causal prefix includes the
 * diagonal; an empty key set gives o = 0 and lse = -inf.
 *
 * Three independent forms are provided:
 *   PLX_ORACLE_SA        textbook softmax attention (o^SA only)
 *   PLX_ORACLE_EXPLICIT  builds Sigma_KV as a d x d matrix, two-pass centred
 *   PLX_ORACLE_STREAM    c = sum w r, u = sum w r v, o = (1 + c) vbar - u,
 *                        r_j = rho . k_j
 * and one member of the attention family the pages place PLX in (zhichai.net,
 * the family taxonomy of section 2: bandwidth x probe x affine term):
 *   PLX_ORACLE_NOINT     "no intercept": vbar = kbar = 0 inside Sigma_KV, so
 *                        o = -M rho with the raw second moment
 *                        M = sum_j w_j v_j k_j^T built as a d x d matrix; with
 *                        uniform weights (scale = 0) it is linear attention
 *                        with probe -rho.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

enum { PLX_ORACLE_SA = 0, PLX_ORACLE_EXPLICIT = 1, PLX_ORACLE_STREAM = 2, PLX_ORACLE_NOINT = 3 };

/* Softmax weights of q over K[0..n): fills w[0..n), returns the natural-log
 * sum-exp of the scaled scores.  n >= 1. */
static double softmax_weights(const double *q, const double *K, long n, int d,
                              double scale, double *w)
{
    double m = -INFINITY;
    for (long j = 0; j < n; ++j) {
        const double *kj = K + (size_t)j * d;
        double dot = 0.0;
        for (int t = 0; t < d; ++t)
            dot += q[t] * kj[t];
        w[j] = scale * dot;
        if (w[j] > m)
            m = w[j];
    }
    double l = 0.0;
    for (long j = 0; j < n; ++j) {
        w[j] = exp(w[j] - m);
        l += w[j];
    }
    for (long j = 0; j < n; ++j)
        w[j] /= l;
    return m + log(l);
}

static void empty_result(int d, double *out, double *lse)
{
    for (int t = 0; t < d; ++t)
        out[t] = 0.0;
    *lse = -INFINITY;
}

/* Weighted mean sum_j w_j X[j] into mean[0..d). */
static void weighted_mean(const double *w, const double *X, long n, int d,
                          double *mean)
{
    for (int t = 0; t < d; ++t)
        mean[t] = 0.0;
    for (long j = 0; j < n; ++j) {
        const double *xj = X + (size_t)j * d;
        for (int t = 0; t < d; ++t)
            mean[t] += w[j] * xj[t];
    }
}

/* Textbook softmax attention: out = sum_j w_j v_j. */
int plx_oracle_sa(const double *q, const double *K, const double *V, long n,
                  int d, double scale, double *out, double *lse)
{
    if (n <= 0) {
        empty_result(d, out, lse);
        return 0;
    }
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    if (!w)
        return -1;
    *lse = softmax_weights(q, K, n, d, scale, w);
    weighted_mean(w, V, n, d, out);
    free(w);
    return 0;
}

/* Explicit covariance form: o = vbar - Sigma_KV rho with
 * Sigma_KV[a][b] = sum_j w_j (v_j[a] - vbar[a]) (k_j[b] - kbar[b]). */
int plx_oracle_explicit(const double *q, const double *rho, const double *K,
                        const double *V, long n, int d, double scale,
                        double *out, double *lse)
{
    if (n <= 0) {
        empty_result(d, out, lse);
        return 0;
    }
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    double *vbar = (double *)malloc(sizeof(double) * (size_t)d);
    double *kbar = (double *)malloc(sizeof(double) * (size_t)d);
    double *sigma = (double *)calloc((size_t)d * (size_t)d, sizeof(double));
    if (!w || !vbar || !kbar || !sigma) {
        free(w); free(vbar); free(kbar); free(sigma);
        return -1;
    }
    *lse = softmax_weights(q, K, n, d, scale, w);
    weighted_mean(w, V, n, d, vbar);
    weighted_mean(w, K, n, d, kbar);
    for (long j = 0; j < n; ++j) {
        const double *vj = V + (size_t)j * d;
        const double *kj = K + (size_t)j * d;
        for (int a = 0; a < d; ++a) {
            double dv = w[j] * (vj[a] - vbar[a]);
            double *row = sigma + (size_t)a * d;
            for (int b = 0; b < d; ++b)
                row[b] += dv * (kj[b] - kbar[b]);
        }
    }
    for (int a = 0; a < d; ++a) {
        const double *row = sigma + (size_t)a * d;
        double corr = 0.0;
        for (int b = 0; b < d; ++b)
            corr += row[b] * rho[b];
        out[a] = vbar[a] - corr;
    }
    free(w); free(vbar); free(kbar); free(sigma);
    return 0;
}

/* Streaming-identity form: r_j = rho . k_j, c = sum w r, u = sum w r v,
 * o = (1 + c) vbar - u. */
int plx_oracle_stream(const double *q, const double *rho, const double *K,
                      const double *V, long n, int d, double scale,
                      double *out, double *lse)
{
    if (n <= 0) {
        empty_result(d, out, lse);
        return 0;
    }
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    double *u = (double *)calloc((size_t)d, sizeof(double));
    double *vbar = (double *)malloc(sizeof(double) * (size_t)d);
    if (!w || !u || !vbar) {
        free(w); free(u); free(vbar);
        return -1;
    }
    *lse = softmax_weights(q, K, n, d, scale, w);
    weighted_mean(w, V, n, d, vbar);
    double c = 0.0;
    for (long j = 0; j < n; ++j) {
        const double *kj = K + (size_t)j * d;
        const double *vj = V + (size_t)j * d;
        double r = 0.0;
        for (int t = 0; t < d; ++t)
            r += rho[t] * kj[t];
        c += w[j] * r;
        for (int t = 0; t < d; ++t)
            u[t] += w[j] * r * vj[t];
    }
    for (int t = 0; t < d; ++t)
        out[t] = (1.0 + c) * vbar[t] - u[t];
    free(w); free(u); free(vbar);
    return 0;
}

/* No-intercept member of the family: o = -(sum_j w_j v_j k_j^T) rho, the
 * d x d raw second moment built explicitly. */
int plx_oracle_noint(const double *q, const double *rho, const double *K,
                     const double *V, long n, int d, double scale,
                     double *out, double *lse)
{
    if (n <= 0) {
        empty_result(d, out, lse);
        return 0;
    }
    double *w = (double *)malloc(sizeof(double) * (size_t)n);
    double *mom = (double *)calloc((size_t)d * (size_t)d, sizeof(double));
    if (!w || !mom) {
        free(w); free(mom);
        return -1;
    }
    *lse = softmax_weights(q, K, n, d, scale, w);
    for (long j = 0; j < n; ++j) {
        const double *vj = V + (size_t)j * d;
        const double *kj = K + (size_t)j * d;
        for (int a = 0; a < d; ++a) {
            double wv = w[j] * vj[a];
            double *row = mom + (size_t)a * d;
            for (int b = 0; b < d; ++b)
                row[b] += wv * kj[b];
        }
    }
    for (int a = 0; a < d; ++a) {
        const double *row = mom + (size_t)a * d;
        double acc = 0.0;
        for (int b = 0; b < d; ++b)
            acc += row[b] * rho[b];
        out[a] = -acc;
    }
    free(w); free(mom);
    return 0;
}

/* One query, chosen form.  rho is ignored for PLX_ORACLE_SA. */
int plx_oracle_query(int form, const double *q, const double *rho,
                     const double *K, const double *V, long n, int d,
                     double scale, double *out, double *lse)
{
    switch (form) {
    case PLX_ORACLE_SA:
        return plx_oracle_sa(q, K, V, n, d, scale, out, lse);
    case PLX_ORACLE_EXPLICIT:
        return plx_oracle_explicit(q, rho, K, V, n, d, scale, out, lse);
    case PLX_ORACLE_STREAM:
        return plx_oracle_stream(q, rho, K, V, n, d, scale, out, lse);
    case PLX_ORACLE_NOINT:
        return plx_oracle_noint(q, rho, K, V, n, d, scale, out, lse);
    default:
        return -2;
    }
}

/* Causal prefill rows of one head: for each listed row i (0 <= i < N), the
 * query Q[i] with probe RHO[i] attends to keys/values 0..i.  Q, K, V, RHO are
 * [N][d]; OUT is [nrows][d], LSE is [nrows]. */
int plx_oracle_prefill_rows(int form, const double *Q, const double *K,
                            const double *V, const double *RHO, long N, int d,
                            double scale, const long *rows, long nrows,
                            double *OUT, double *LSE)
{
    for (long r = 0; r < nrows; ++r) {
        long i = rows[r];
        if (i < 0 || i >= N)
            return -3;
        int rc = plx_oracle_query(form, Q + (size_t)i * d, RHO + (size_t)i * d,
                                  K, V, i + 1, d, scale, OUT + (size_t)r * d,
                                  LSE + r);
        if (rc)
            return rc;
    }
    return 0;
}

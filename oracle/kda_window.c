/*
 * CPU oracle of the KDA gated delta-rule recurrence, in double precision.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the tests, the package's smoke check and the CPU
 * baseline leg of the benchmark use it.  It shares no code, header or
 * constant with the CUDA library.
 *
 * What it computes is the plain definition of one KDA window, written out
 * step by step in the order of the per-token loop of `_verify_kernel` in
 * "recipes/docker-images/glm53-kindling/experimental/fixes/recoverssm.py"
 * (GLM-5.3-Flash KDA speculative verify), for one (request, head) state tile
 * H (V rows by K columns, row v, column k):
 *
 *   q^ = q / sqrt(sum q^2 + 1e-6) * scale        (L2 norm, then the scale)
 *   k^ = k / sqrt(sum k^2 + 1e-6)
 *   x  = g_raw + g_bias                           (per K channel)
 *   g  = lb * sigmoid(exp(A_log) * x)             bounded gate (kda.py)
 *        -exp(A_log) * softplus(x)                 default gate
 *   H  = H * diag(exp(g))                          decay along K
 *   beta = sigmoid(beta_raw)
 *   v' = beta * (v - H k^)                         delta
 *   H  = H + v' k^T                                rank-one update
 *   o  = H q^                                      output, after the update
 *
 * Readings of points the pages leave open:
 *   - softplus(x) = log1p(exp(x)), and x itself for x > 20 (the usual
 *     threshold; the difference there is below 1e-8 relative);
 *   - the bounded gate is used exactly when a lower bound is given, the
 *     softplus gate otherwise (no clamp of the softplus gate);
 *   - every step is done in double precision on the exact inputs.
 *
 * K and V are run-time sizes so that tiny tiles can be checked by brute
 * force; the library itself only supports K = V = 128.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* Arithmetic type of the window loops.  The oracle is the double build.  The
 * benchmark's CPU baseline also times a float build of this same file
 * (-DKDA_ORACLE_FP32, libkda_oracle_fp32.so); no test uses that build. */
#ifdef KDA_ORACLE_FP32
typedef float real;
#define R_EXP expf
#define R_LOG1P log1pf
#define R_SQRT sqrtf
#else
typedef double real;
#define R_EXP exp
#define R_LOG1P log1p
#define R_SQRT sqrt
#endif

static real oracle_softplus(real x)
{
    if (x > (real)20.0)
        return x;
    return R_LOG1P(R_EXP(x));
}

static real oracle_sigmoid(real x)
{
    return (real)1.0 / ((real)1.0 + R_EXP(-x));
}

static real oracle_gate(real x, real a_log, int bounded, real lower_bound)
{
    real a = R_EXP(a_log);
    if (bounded)
        return lower_bound * oracle_sigmoid(a * x);
    return -a * oracle_softplus(x);
}

/* Gate of one channel: x = g_raw + g_bias.  The bounded form is the one
 * kda.py describes for its FlashKDA prefill and the one the verify kernel of
 * recoverssm.py evaluates with its LOWER_BOUND constant: the lower bound
 * times the logistic of exp(A_log) * x.  The unbounded form is the softplus
 * gate that kda.py names as the layer's default. */
double kda_oracle_gate(double x, double a_log, int bounded, double lower_bound)
{
    return (double)oracle_gate((real)x, (real)a_log, bounded, (real)lower_bound);
}

/* One window of T tokens from the state h0 (V x K, row-major, k fastest).
 *
 * Token t reads q[t*K..], k[t*K..], v[t*V..], g_raw[t*K..], beta_raw[t];
 * g_bias has K entries.  q may be NULL (no outputs: the commit replay),
 * in which case out must be NULL too.
 * out:     T x V, the output of each token (may be NULL);
 * traj:    T x V x K, the state after each token (may be NULL);
 * h_final: V x K, the state after the last token (T == 0: h0);
 * delta:   T x V, each token's delta v' = beta (v - H k^) (may be NULL).
 * Returns 0, or -1 if a size is out of range or memory runs out. */
int kda_oracle_window(int K, int V, int T,
                      const double *h0,
                      const double *q, const double *k, const double *v,
                      const double *g_raw, const double *beta_raw,
                      double a_log, const double *g_bias,
                      int bounded, double lower_bound, double scale,
                      double *out, double *traj, double *h_final,
                      double *delta)
{
    if (K <= 0 || V <= 0 || T < 0)
        return -1;
    if (q == NULL && out != NULL)
        return -1;

    size_t nvk = (size_t)V * (size_t)K;
    real *H = (real *)malloc(sizeof(real) * nvk);
    real *kh = (real *)malloc(sizeof(real) * (size_t)K);
    real *qh = (real *)malloc(sizeof(real) * (size_t)K);
    real *decay = (real *)malloc(sizeof(real) * (size_t)K);
    if (H == NULL || kh == NULL || qh == NULL || decay == NULL) {
        free(H);
        free(kh);
        free(qh);
        free(decay);
        return -1;
    }
    for (size_t i = 0; i < nvk; ++i)
        H[i] = (real)h0[i];

    for (int t = 0; t < T; ++t) {
        const double *kt = k + (size_t)t * K;
        const double *vt = v + (size_t)t * V;
        const double *gt = g_raw + (size_t)t * K;

        /* L2 norm of k, eps inside the square root. */
        real sk = 0;
        for (int c = 0; c < K; ++c)
            sk += (real)kt[c] * (real)kt[c];
        real nk = R_SQRT(sk + (real)1e-6);
        for (int c = 0; c < K; ++c)
            kh[c] = (real)kt[c] / nk;

        /* L2 norm of q, then the scale. */
        if (q != NULL) {
            const double *qt = q + (size_t)t * K;
            real sq = 0;
            for (int c = 0; c < K; ++c)
                sq += (real)qt[c] * (real)qt[c];
            real nq = R_SQRT(sq + (real)1e-6);
            for (int c = 0; c < K; ++c)
                qh[c] = (real)qt[c] / nq * (real)scale;
        }

        /* Per-channel decay factor exp(g). */
        for (int c = 0; c < K; ++c)
            decay[c] = R_EXP(oracle_gate((real)gt[c] + (real)g_bias[c], (real)a_log, bounded,
                                         (real)lower_bound));

        real beta = oracle_sigmoid((real)beta_raw[t]);

        /* Decay: every row scales column c by the same factor. */
        for (int r = 0; r < V; ++r)
            for (int c = 0; c < K; ++c)
                H[(size_t)r * K + c] *= decay[c];

        /* Delta and rank-one update, one row at a time: the row's own
         * prediction H[r,:] . k^ only involves that row. */
        for (int r = 0; r < V; ++r) {
            real *row = H + (size_t)r * K;
            real u = 0;
            for (int c = 0; c < K; ++c)
                u += row[c] * kh[c];
            real vp = beta * ((real)vt[r] - u);
            for (int c = 0; c < K; ++c)
                row[c] += vp * kh[c];
            if (delta != NULL)
                delta[(size_t)t * V + r] = (double)vp;
        }

        /* Output after the update. */
        if (out != NULL) {
            for (int r = 0; r < V; ++r) {
                const real *row = H + (size_t)r * K;
                real o = 0;
                for (int c = 0; c < K; ++c)
                    o += row[c] * qh[c];
                out[(size_t)t * V + r] = (double)o;
            }
        }

        if (traj != NULL)
            for (size_t i = 0; i < nvk; ++i)
                traj[(size_t)t * nvk + i] = (double)H[i];
    }

    for (size_t i = 0; i < nvk; ++i)
        h_final[i] = (double)H[i];
    free(H);
    free(kh);
    free(qh);
    free(decay);
    return 0;
}

/* The closed form of n tokens whose deltas are known (the fp32-correction
 * commit of the Kimi-K3 deferred context: the verify stores each token's
 * delta, and the commit folds the deltas into the checkpoint without the
 * state-dependent prediction H k^).  Unrolling the per-token update
 * H <- H diag(e_t) + d_t k^_t^T over t = 1..n gives
 *
 *   H_n = H_0 diag(P_0) + sum_t d_t (k^_t * P_t)^T,
 *   P_t[c] = prod_{s = t+1..n} e_s[c]          (P_n = 1),
 *
 * with e_t = exp(g_t) the gate of token t and k^_t its normalised key.  It
 * is evaluated here term by term, as written, not as the recurrence.
 *
 * k, g_raw: n x K; delta: n x V; g_bias: K; h0, h_final: V x K (they may
 * be the same buffer).  Returns 0, or -1 on bad sizes or no memory. */
int kda_oracle_fold_deltas(int K, int V, int n,
                           const double *h0,
                           const double *k, const double *g_raw,
                           const double *delta,
                           double a_log, const double *g_bias,
                           int bounded, double lower_bound,
                           double *h_final)
{
    if (K <= 0 || V <= 0 || n < 0)
        return -1;
    size_t nk = (size_t)(n > 0 ? n : 1) * (size_t)K;
    real *kh = (real *)malloc(sizeof(real) * nk);
    real *e = (real *)malloc(sizeof(real) * nk);
    real *coef = (real *)malloc(sizeof(real) * nk);
    real *P = (real *)malloc(sizeof(real) * (size_t)K);
    real *acc = (real *)malloc(sizeof(real) * (size_t)V * (size_t)K);
    if (kh == NULL || e == NULL || coef == NULL || P == NULL || acc == NULL) {
        free(kh);
        free(e);
        free(coef);
        free(P);
        free(acc);
        return -1;
    }
    for (int t = 0; t < n; ++t) {
        const double *kt = k + (size_t)t * K;
        const double *gt = g_raw + (size_t)t * K;
        real sk = 0;
        for (int c = 0; c < K; ++c)
            sk += (real)kt[c] * (real)kt[c];
        real nrm = R_SQRT(sk + (real)1e-6);
        for (int c = 0; c < K; ++c) {
            kh[(size_t)t * K + c] = (real)kt[c] / nrm;
            e[(size_t)t * K + c] = R_EXP(oracle_gate((real)gt[c] + (real)g_bias[c], (real)a_log,
                                                     bounded, (real)lower_bound));
        }
    }
    /* P runs from P_n = 1 down to P_0; coef_t = k^_t * P_t. */
    for (int c = 0; c < K; ++c)
        P[c] = 1;
    for (int t = n - 1; t >= 0; --t) {
        for (int c = 0; c < K; ++c) {
            coef[(size_t)t * K + c] = kh[(size_t)t * K + c] * P[c];
            P[c] *= e[(size_t)t * K + c];
        }
    }
    for (int r = 0; r < V; ++r)
        for (int c = 0; c < K; ++c) {
            real s = (real)h0[(size_t)r * K + c] * P[c];
            for (int t = 0; t < n; ++t)
                s += (real)delta[(size_t)t * V + r] * coef[(size_t)t * K + c];
            acc[(size_t)r * K + c] = s;
        }
    for (size_t i = 0; i < (size_t)V * (size_t)K; ++i)
        h_final[i] = (double)acc[i];
    free(kh);
    free(e);
    free(coef);
    free(P);
    free(acc);
    return 0;
}

/* Round a double to the nearest bfloat16 value (8 significant bits, ties
 * to even), returned as a double.  Direct from the double, so there is no
 * double rounding through float.  Values below bfloat16's normal range are
 * not expected here and are rounded on the same 8-bit grid. */
double kda_oracle_round_bf16(double x)
{
    if (x == 0.0 || isnan(x) || isinf(x))
        return x;
    int e;
    double m = frexp(x, &e);          /* x = m * 2^e, 0.5 <= |m| < 1 */
    double scaled = ldexp(m, 8);      /* 8 significant bits to the left */
    double r = nearbyint(scaled);     /* default mode: nearest, ties to even */
    return ldexp(r, e - 8);
}

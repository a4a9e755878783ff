/*
 * la_variants.c - plain fp64 CPU oracle for the variants of kernelised
 * linear attention: other feature maps, sum normalisation and the delta
 * update rule.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only tests/ and bench.py's CPU-baseline leg do.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * Sources:
 *  [TaR] "Transformers are RNNs: Fast Autoregressive Transformers with Linear
 *        Attention" (Katharopoulos et al.), read in its Chinese translation.
 *  [FWP] "Linear Transformers Are Secretly Fast Weight Programmers" (Schlag,
 *        Irie, Schmidhuber), read in a Chinese news summary whose equations
 *        were lost in extraction; each step below is the plainest reading of
 *        the summary's prose, listed in the design notes.
 *
 * Feature maps phi: R^D -> R^F (applied to each row of Q and K):
 *   FM_ELU1   [TaR sec. 3.2.1 eq. (7)] phi(x)_i = elu(x_i) + 1, F = D.
 *   FM_DPFP   [FWP "DPFP"] deterministic parameter-free projection with nu
 *             shifts: r = [relu(x), relu(-x)] in R^{2D}; for shift s = 1..nu
 *             and i = 0..2D-1, phi(x)_{(s-1)*2D + i} = r_i * r_{(i+s) mod 2D}.
 *             F = 2*D*nu.  (For D = 2, nu = 1 every input has a single non-zero
 *             feature and the four quadrants map to four orthogonal
 *             directions: the summary's figure.)
 *   FM_POLY2  [TaR sec. 3.2.1] the degree-2 polynomial kernel (q^T k)^2 through
 *             its exact finite feature map phi(x)_{a*D + b} = x_a x_b, F = D^2
 *             (cost O(N D^2 M), as that section states).
 *
 * Normalisation of the read-out:
 *   NORM_DEN  [TaR eq. (12); FWP's "accumulator" variant] z_i = z_{i-1} + phi(k_i),
 *             y_i = phi(q_i)^T S_i / phi(q_i)^T z_i.
 *   NORM_SUM  [FWP "normalisation"] phi(k) and phi(q) are divided by the sum
 *             of their components; y_i = phi(q_i)^T S_i with no denominator.
 *   NORM_NONE the raw fast-weight read-out y_i = phi(q_i)^T S_i.
 *
 * Update rule of the state S (F x M; S[f][m], retrieval of key k is S^T phi(k)):
 *   UPD_SUM   [TaR eq. (10); FWP eq. (17)] S_i = S_{i-1} + phi(k_i) v_i^T.
 *   UPD_DELTA [FWP "improved update rule"] retrieve vbar_i = S_{i-1}^T phi(k_i),
 *             store the convex combination beta_i v_i + (1 - beta_i) vbar_i in
 *             place of vbar_i: S_i = S_{i-1} + phi(k_i) (beta_i (v_i - vbar_i))^T,
 *             beta_i in [0, 1] given per token.
 * The read-out always follows the update of the same token (TaR sec. 3.4
 * eqs. (18)-(20)); the start state is zero unless the caller passes one.
 *
 * Inputs fp32 (bf16 widened exactly), every operation in fp64, plain loops,
 * OpenMP over independent heads (no effect on the arithmetic).  `mutant`
 * plants one mistake for the tests; the plain entry points pass 0.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { FM_ELU1 = 0, FM_DPFP = 1, FM_POLY2 = 2 };
enum { NORM_DEN = 0, NORM_SUM = 1, NORM_NONE = 2 };
enum { UPD_SUM = 0, UPD_DELTA = 1 };

/* Planted mistakes (test use only). */
enum {
    MUTV_NONE = 0,
    MUTV_DPFP_POS_ONLY = 21,   /* r = [relu(x), relu(x)]: the negative half lost      */
    MUTV_POLY_UPPER = 22,      /* only the a <= b products of the polynomial map      */
    MUTV_SUMNORM_K_ONLY = 23,  /* sum normalisation applied to phi(k) only            */
    MUTV_DELTA_AFTER = 24,     /* retrieval from the already updated state            */
    MUTV_DELTA_SIGN = 25,      /* S += phi(k) beta (vbar - v)^T                        */
    MUTV_DELTA_BETA_V = 26     /* S += phi(k) (beta v - vbar)^T                        */
};

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

long lav_feature_dim(int fm, long D, int nu)
{
    if (D <= 0) return 0;
    if (fm == FM_ELU1) return D;
    if (fm == FM_DPFP) return (nu >= 1 && nu < 2 * D) ? 2 * D * nu : 0;
    if (fm == FM_POLY2) return D * D;
    return 0;
}

/* r_i of DPFP: relu(x_i) for i < D, relu(-x_{i-D}) for D <= i < 2D. */
static double dpfp_r(const float *x, long D, long i, int mutant)
{
    double t = (double)x[i < D ? i : i - D];
    if (i >= D && mutant != MUTV_DPFP_POS_ONLY) t = -t;
    return t > 0.0 ? t : 0.0;
}

/* phi(x) of one row into f[0..F); divided by its component sum if sumnorm. */
static void features(const float *x, long D, int fm, int nu, int sumnorm, int mutant, double *f)
{
    const long F = lav_feature_dim(fm, D, nu);
    if (fm == FM_ELU1) {
        for (long i = 0; i < D; ++i) {
            double t = (double)x[i];
            f[i] = t > 0.0 ? t + 1.0 : exp(t);
        }
    } else if (fm == FM_DPFP) {
        for (long s = 1; s <= nu; ++s)
            for (long i = 0; i < 2 * D; ++i)
                f[(s - 1) * 2 * D + i] = dpfp_r(x, D, i, mutant) * dpfp_r(x, D, (i + s) % (2 * D), mutant);
    } else {
        for (long a = 0; a < D; ++a)
            for (long b = 0; b < D; ++b)
                f[a * D + b] = (mutant == MUTV_POLY_UPPER && b < a) ? 0.0 : (double)x[a] * (double)x[b];
    }
    if (sumnorm) {
        double s = 0.0;
        for (long i = 0; i < F; ++i) s += f[i];
        for (long i = 0; i < F; ++i) f[i] /= s;
    }
}

/* phi of R rows x [R, D] into out [R, F]; returns 0, or 1 on a bad argument. */
int lav_features(const float *x, long R, long D, int fm, int nu, int sumnorm, double *out)
{
    const long F = lav_feature_dim(fm, D, nu);
    if (F == 0 || R < 0) return 1;
    for (long r = 0; r < R; ++r) features(x + r * D, D, fm, nu, sumnorm, MUTV_NONE, out + r * F);
    return 0;
}

/*
 * Causal variant.  q, k: [BH, N, D]; v: [BH, N, M]; beta: [BH, N] (UPD_DELTA
 * only, else NULL).  S0 [BH, F, M], z0 [BH, F] or NULL (zero start; z only
 * for NORM_DEN).  out [BH, N, M] or NULL; S_out, z_out or NULL.
 */
int lav_causal_mut(const float *q, const float *k, const float *v, const float *beta,
                   long BH, long N, long D, long M, int fm, int nu, int norm, int upd,
                   const double *S0, const double *z0, double *out, double *S_out, double *z_out,
                   int nthreads, int mutant)
{
    const long F = lav_feature_dim(fm, D, nu);
    if (BH < 0 || N < 0 || F == 0 || M <= 0) return 1;
    if (upd == UPD_DELTA && !beta) return 1;
    set_threads(nthreads);
    const int sum_q = (norm == NORM_SUM && mutant != MUTV_SUMNORM_K_ONLY);
    const int sum_k = (norm == NORM_SUM);
    long h;
#pragma omp parallel for schedule(dynamic, 1)
    for (h = 0; h < BH; ++h) {
        double *S = calloc((size_t)(F * M), sizeof(double));
        double *z = calloc((size_t)F, sizeof(double));
        double *fq = malloc(sizeof(double) * (size_t)F);
        double *fk = malloc(sizeof(double) * (size_t)F);
        double *u = malloc(sizeof(double) * (size_t)M);
        if (S0) memcpy(S, S0 + h * F * M, sizeof(double) * (size_t)(F * M));
        if (z0) memcpy(z, z0 + h * F, sizeof(double) * (size_t)F);
        const float *qh = q + h * N * D, *kh = k + h * N * D, *vh = v + h * N * M;
        for (long i = 0; i < N; ++i) {
            features(qh + i * D, D, fm, nu, sum_q, mutant, fq);
            features(kh + i * D, D, fm, nu, sum_k, mutant, fk);
            const float *vi = vh + i * M;
            if (upd == UPD_SUM) {
                for (long f = 0; f < F; ++f)
                    for (long m = 0; m < M; ++m) S[f * M + m] += fk[f] * (double)vi[m];
            } else {
                const double b = (double)beta[h * N + i];
                if (mutant == MUTV_DELTA_AFTER)
                    for (long f = 0; f < F; ++f)
                        for (long m = 0; m < M; ++m) S[f * M + m] += fk[f] * b * (double)vi[m];
                for (long m = 0; m < M; ++m) {
                    double vbar = 0.0;   /* the value currently paired with k_i */
                    for (long f = 0; f < F; ++f) vbar += S[f * M + m] * fk[f];
                    if (mutant == MUTV_DELTA_AFTER) u[m] = -b * vbar;
                    else if (mutant == MUTV_DELTA_SIGN) u[m] = b * (vbar - (double)vi[m]);
                    else if (mutant == MUTV_DELTA_BETA_V) u[m] = b * (double)vi[m] - vbar;
                    else u[m] = b * ((double)vi[m] - vbar);
                }
                for (long f = 0; f < F; ++f)
                    for (long m = 0; m < M; ++m) S[f * M + m] += fk[f] * u[m];
            }
            if (norm == NORM_DEN)
                for (long f = 0; f < F; ++f) z[f] += fk[f];
            if (out) {
                double den = 1.0;
                if (norm == NORM_DEN) {
                    den = 0.0;
                    for (long f = 0; f < F; ++f) den += fq[f] * z[f];
                }
                for (long m = 0; m < M; ++m) {
                    double num = 0.0;
                    for (long f = 0; f < F; ++f) num += fq[f] * S[f * M + m];
                    out[(h * N + i) * M + m] = num / den;
                }
            }
        }
        if (S_out) memcpy(S_out + h * F * M, S, sizeof(double) * (size_t)(F * M));
        if (z_out) memcpy(z_out + h * F, z, sizeof(double) * (size_t)F);
        free(S); free(z); free(fq); free(fk); free(u);
    }
    return 0;
}

/*
 * Non-causal variant ([TaR] eq. (5) with the variant's phi and read-out):
 * KV = sum_j phi(K_j) V_j^T and ksum = sum_j phi(K_j) over all N keys, then
 * y_i = phi(Q_i)^T KV (/ phi(Q_i)^T ksum for NORM_DEN).  Sum update only.
 */
int lav_noncausal(const float *q, const float *k, const float *v,
                  long BH, long N, long D, long M, int fm, int nu, int norm,
                  double *out, int nthreads)
{
    const long F = lav_feature_dim(fm, D, nu);
    if (BH < 0 || N < 0 || F == 0 || M <= 0) return 1;
    set_threads(nthreads);
    const int sn = (norm == NORM_SUM);
    long h;
#pragma omp parallel for schedule(dynamic, 1)
    for (h = 0; h < BH; ++h) {
        double *KV = calloc((size_t)(F * M), sizeof(double));
        double *ks = calloc((size_t)F, sizeof(double));
        double *f = malloc(sizeof(double) * (size_t)F);
        const float *qh = q + h * N * D, *kh = k + h * N * D, *vh = v + h * N * M;
        for (long j = 0; j < N; ++j) {
            features(kh + j * D, D, fm, nu, sn, MUTV_NONE, f);
            for (long a = 0; a < F; ++a) {
                for (long m = 0; m < M; ++m) KV[a * M + m] += f[a] * (double)vh[j * M + m];
                ks[a] += f[a];
            }
        }
        for (long i = 0; i < N; ++i) {
            features(qh + i * D, D, fm, nu, sn, MUTV_NONE, f);
            double den = 1.0;
            if (norm == NORM_DEN) {
                den = 0.0;
                for (long a = 0; a < F; ++a) den += f[a] * ks[a];
            }
            for (long m = 0; m < M; ++m) {
                double num = 0.0;
                for (long a = 0; a < F; ++a) num += f[a] * KV[a * M + m];
                out[(h * N + i) * M + m] = num / den;
            }
        }
        free(KV); free(ks); free(f);
    }
    return 0;
}

/*
 * la_oracle.c - plain fp64 CPU oracle for kernelised linear attention with
 * the feature map phi(x) = elu(x) + 1.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only tests/, the smoke check and the CPU-baseline leg of
 * bench.py do.  It shares no code, header, table or helper with the CUDA
 * library.
 *
 * Source: "Transformers are RNNs: Fast Autoregressive Transformers with
 * Linear Attention" (Katharopoulos et al.), read in its Chinese translation.
 * Every function below restates one passage of it:
 *
 *   phi            sec. 3.2.1, eq. (7): phi(x) = elu(x) + 1, elu with alpha = 1
 *                  (Clevert et al.), so phi(x) = x + 1 for x > 0, exp(x) else.
 *   lao_noncausal  sec. 3.2, eq. (5): V'_i = phi(Q_i)^T sum_j phi(K_j) V_j^T
 *                  / phi(Q_i)^T sum_j phi(K_j); both sums are formed once and
 *                  reused for every query (the paragraph after eq. (6)).
 *   lao_causal     sec. 3.3, eqs. (10)-(12): S_i = S_{i-1} + phi(K_i) V_i^T,
 *                  Z_i = Z_{i-1} + phi(K_i), V'_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i,
 *                  walked i = 1..N exactly as sec. 3.4, eqs. (16)-(20) write the
 *                  RNN: the state is updated first, then read out.  The start
 *                  state is s_0 = 0, z_0 = 0 (eqs. (16), (17)) unless the caller
 *                  passes one (the state carried between calls, sec. 3.3.2).
 *   lao_decode     sec. 3.4, eqs. (18)-(20) for one time step; the residual and
 *                  f_l of eq. (20) belong to the surrounding layer and are left
 *                  out (the attention fraction only).
 *   lao_causal_backward, lao_noncausal_backward
 *                  gradients of a loss L through eqs. (9)-(12) (resp. eq. (5)),
 *                  given G_i = dL/dV'_i.  Sec. 3.3.1 states that the gradient of
 *                  the causal numerator is a cumulative sum computable with
 *                  constant extra memory, but its equations (13)-(15) and its
 *                  Algorithm 1 are not printed on the page; the steps below are
 *                  the chain rule applied to eqs. (10)-(12), in their order:
 *                    g_i = G_i / den_i,  e_i = -(g_i . num_i) / den_i
 *                    dphi(Q_i) = S_i g_i + e_i Z_i             (forward sweep)
 *                    R_i = sum_{j>=i} phi(Q_j) g_j^T, r_i = sum_{j>=i} e_j phi(Q_j)
 *                    dphi(K_i) = R_i V_i + r_i,  dV_i = R_i^T phi(K_i)   (reverse sweep)
 *                  and dQ = dphi(Q) * phi'(Q), dK = dphi(K) * phi'(K) with
 *                  phi'(x) = 1 for x > 0, exp(x) else.  A carried-in state
 *                  (S_0, Z_0) enters as in the forward; dL/dS_N, dL/dZ_N (the
 *                  gradient arriving through the final state) start R and r,
 *                  and R_1, r_1 are dL/dS_0, dL/dZ_0.
 *
 * Readings where the page is silent (each listed in the design notes):
 *   - no epsilon in any denominator (none of eqs. (4), (5), (9), (12) has one);
 *   - no 1/sqrt(D) inside phi (eqs. (4)-(5) have none; only softmax, eq. (2));
 *   - the causal sum includes j = i (sec. 3.3, eq. (8): j <= i).
 *
 * Inputs are fp32 (bf16 tensors are widened exactly before the call); all
 * arithmetic is fp64 in plain loops, one head at a time.  OpenMP spreads the
 * independent heads over cores; it changes no arithmetic.
 *
 * The `mutant` argument of the *_mut entry points plants one deliberate
 * mistake (tests use it to show that the pins catch such mistakes); the
 * plain entry points always pass 0.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Planted mistakes (test use only). */
enum {
    MUT_NONE = 0,
    MUT_RELU = 1,          /* phi = relu(x) + 1 instead of elu(x) + 1        */
    MUT_NO_Z_UPDATE = 2,   /* forget eq. (11)/(19): z never grows             */
    MUT_READ_BEFORE = 3,   /* read out before the update (sum over j < i)     */
    MUT_TRANSPOSE_S = 4,   /* num_m = sum_d phi(q)_d S[m][d] (S transposed)    */
    MUT_PHI_NEG = 5,       /* phi(x) = exp(-x) for x <= 0 (sign slip)         */
    MUT_NO_DIAG_V = 6,     /* use V_{i-1} in place of V_i in the update       */
    MUT_DEN_Q_OF_K = 7,    /* denominator phi(K_i)^T Z_i instead of phi(Q_i)  */
    /* backward */
    MUT_B_NO_E = 11,       /* drop the denominator's term e_i                 */
    MUT_B_DPHI_IS_PHI = 12,/* chain rule through phi instead of phi'          */
    MUT_B_EXCL_DIAG = 13,  /* reverse sums over j > i instead of j >= i       */
    MUT_B_DV_USES_Q = 14   /* dV_i = R_i^T phi(Q_i) instead of phi(K_i)       */
};

static double phi_m(double x, int mutant)
{
    if (mutant == MUT_RELU) return (x > 0.0 ? x : 0.0) + 1.0;
    if (mutant == MUT_PHI_NEG) return x > 0.0 ? x + 1.0 : exp(-x);
    return x > 0.0 ? x + 1.0 : exp(x);
}

double lao_phi(double x) { return phi_m(x, MUT_NONE); }

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int lao_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Causal form.  q, k: [BH, N, D]; v: [BH, N, M] (row-major, fp32).
 * S0: [BH, D, M], z0: [BH, D] or NULL (zero start).  out: [BH, N, M] or NULL.
 * S_out: [BH, D, M], z_out: [BH, D] or NULL.  All state and output in fp64.
 */
int lao_causal_mut(const float *q, const float *k, const float *v,
                   long BH, long N, long D, long M,
                   const double *S0, const double *z0,
                   double *out, double *S_out, double *z_out,
                   int nthreads, int mutant)
{
    if (BH < 0 || N < 0 || D <= 0 || M <= 0) return 1;
    set_threads(nthreads);
    long h;
#pragma omp parallel for schedule(dynamic, 1)
    for (h = 0; h < BH; ++h) {
        double *S = (double *)calloc((size_t)(D * M), sizeof(double));
        double *z = (double *)calloc((size_t)D, sizeof(double));
        double *fq = (double *)malloc((size_t)D * sizeof(double));
        double *fk = (double *)malloc((size_t)D * sizeof(double));
        double *vprev = (double *)calloc((size_t)M, sizeof(double));
        if (S0) memcpy(S, S0 + h * D * M, (size_t)(D * M) * sizeof(double));
        if (z0) memcpy(z, z0 + h * D, (size_t)D * sizeof(double));
        const float *qh = q + h * N * D, *kh = k + h * N * D, *vh = v + h * N * M;
        for (long i = 0; i < N; ++i) {
            const float *qi = qh + i * D, *ki = kh + i * D, *vi = vh + i * M;
            for (long d = 0; d < D; ++d) {
                fq[d] = phi_m((double)qi[d], mutant);
                fk[d] = phi_m((double)ki[d], mutant);
            }
            if (mutant == MUT_READ_BEFORE && out) {
                /* planted: read out S_{i-1}, Z_{i-1} */
                double den = 0.0;
                for (long d = 0; d < D; ++d) den += fq[d] * z[d];
                for (long m = 0; m < M; ++m) {
                    double num = 0.0;
                    for (long d = 0; d < D; ++d) num += fq[d] * S[d * M + m];
                    out[(h * N + i) * M + m] = num / den;
                }
            }
            /* eq. (10)/(18): S_i = S_{i-1} + phi(K_i) V_i^T */
            for (long d = 0; d < D; ++d)
                for (long m = 0; m < M; ++m) {
                    double vm = (mutant == MUT_NO_DIAG_V) ? vprev[m] : (double)vi[m];
                    S[d * M + m] += fk[d] * vm;
                }
            for (long m = 0; m < M; ++m) vprev[m] = (double)vi[m];
            /* eq. (11)/(19): Z_i = Z_{i-1} + phi(K_i) */
            if (mutant != MUT_NO_Z_UPDATE)
                for (long d = 0; d < D; ++d) z[d] += fk[d];
            if (out && mutant != MUT_READ_BEFORE) {
                /* eq. (12)/(20): V'_i = phi(Q_i)^T S_i / phi(Q_i)^T Z_i */
                double den = 0.0;
                const double *fden = (mutant == MUT_DEN_Q_OF_K) ? fk : fq;
                for (long d = 0; d < D; ++d) den += fden[d] * z[d];
                for (long m = 0; m < M; ++m) {
                    double num = 0.0;
                    if (mutant == MUT_TRANSPOSE_S && D == M)
                        for (long d = 0; d < D; ++d) num += fq[d] * S[m * M + d];
                    else
                        for (long d = 0; d < D; ++d) num += fq[d] * S[d * M + m];
                    out[(h * N + i) * M + m] = num / den;
                }
            }
        }
        if (S_out) memcpy(S_out + h * D * M, S, (size_t)(D * M) * sizeof(double));
        if (z_out) memcpy(z_out + h * D, z, (size_t)D * sizeof(double));
        free(S); free(z); free(fq); free(fk); free(vprev);
    }
    return 0;
}

int lao_causal(const float *q, const float *k, const float *v,
               long BH, long N, long D, long M,
               const double *S0, const double *z0,
               double *out, double *S_out, double *z_out, int nthreads)
{
    return lao_causal_mut(q, k, v, BH, N, D, M, S0, z0, out, S_out, z_out,
                          nthreads, MUT_NONE);
}

/*
 * Non-causal form, eq. (5).  Shapes as lao_causal; kv_out [BH, D, M] and
 * ksum_out [BH, D] (may be NULL) receive sum_j phi(K_j) V_j^T and
 * sum_j phi(K_j).
 */
int lao_noncausal_mut(const float *q, const float *k, const float *v,
                      long BH, long N, long D, long M,
                      double *out, double *kv_out, double *ksum_out,
                      int nthreads, int mutant)
{
    if (BH < 0 || N < 0 || D <= 0 || M <= 0) return 1;
    set_threads(nthreads);
    long h;
#pragma omp parallel for schedule(dynamic, 1)
    for (h = 0; h < BH; ++h) {
        double *KV = (double *)calloc((size_t)(D * M), sizeof(double));
        double *ks = (double *)calloc((size_t)D, sizeof(double));
        double *f = (double *)malloc((size_t)D * sizeof(double));
        const float *qh = q + h * N * D, *kh = k + h * N * D, *vh = v + h * N * M;
        /* sum_j phi(K_j) V_j^T and sum_j phi(K_j), computed once */
        for (long j = 0; j < N; ++j) {
            for (long d = 0; d < D; ++d) f[d] = phi_m((double)kh[j * D + d], mutant);
            for (long d = 0; d < D; ++d) {
                for (long m = 0; m < M; ++m) KV[d * M + m] += f[d] * (double)vh[j * M + m];
                if (mutant != MUT_NO_Z_UPDATE) ks[d] += f[d];
            }
        }
        if (out) {
            for (long i = 0; i < N; ++i) {
                for (long d = 0; d < D; ++d) f[d] = phi_m((double)qh[i * D + d], mutant);
                double den = 0.0;
                for (long d = 0; d < D; ++d) den += f[d] * ks[d];
                for (long m = 0; m < M; ++m) {
                    double num = 0.0;
                    if (mutant == MUT_TRANSPOSE_S && D == M)
                        for (long d = 0; d < D; ++d) num += f[d] * KV[m * M + d];
                    else
                        for (long d = 0; d < D; ++d) num += f[d] * KV[d * M + m];
                    out[(h * N + i) * M + m] = num / den;
                }
            }
        }
        if (kv_out) memcpy(kv_out + h * D * M, KV, (size_t)(D * M) * sizeof(double));
        if (ksum_out) memcpy(ksum_out + h * D, ks, (size_t)D * sizeof(double));
        free(KV); free(ks); free(f);
    }
    return 0;
}

int lao_noncausal(const float *q, const float *k, const float *v,
                  long BH, long N, long D, long M,
                  double *out, double *kv_out, double *ksum_out, int nthreads)
{
    return lao_noncausal_mut(q, k, v, BH, N, D, M, out, kv_out, ksum_out,
                             nthreads, MUT_NONE);
}

/*
 * One recurrent step, eqs. (18)-(20).  q, k: [BH, D]; v: [BH, M];
 * S: [BH, D, M] and z: [BH, D] fp64, updated in place; y: [BH, M].
 */
int lao_decode(const float *q, const float *k, const float *v,
               long BH, long D, long M, double *S, double *z, double *y,
               int nthreads)
{
    if (BH < 0 || D <= 0 || M <= 0) return 1;
    set_threads(nthreads);
    long h;
#pragma omp parallel for schedule(static)
    for (h = 0; h < BH; ++h) {
        double *Sh = S + h * D * M, *zh = z + h * D;
        const float *qh = q + h * D, *kh = k + h * D, *vh = v + h * M;
        for (long d = 0; d < D; ++d) {
            double fk = lao_phi((double)kh[d]);
            for (long m = 0; m < M; ++m) Sh[d * M + m] += fk * (double)vh[m];
            zh[d] += fk;
        }
        double den = 0.0;
        for (long d = 0; d < D; ++d) den += lao_phi((double)qh[d]) * zh[d];
        for (long m = 0; m < M; ++m) {
            double num = 0.0;
            for (long d = 0; d < D; ++d) num += lao_phi((double)qh[d]) * Sh[d * M + m];
            y[h * M + m] = num / den;
        }
    }
    return 0;
}


/* phi'(x): 1 for x > 0, exp(x) for x <= 0 (elu with alpha = 1, plus one). */
static double dphi_m(double x, int mutant)
{
    if (mutant == MUT_B_DPHI_IS_PHI) return lao_phi(x);
    return x > 0.0 ? 1.0 : exp(x);
}

/*
 * Backward of the causal form.  q, k, G (=dL/dout): [BH, N, D] / [BH, N, M];
 * v: [BH, N, M].  S0 [BH, D, M], z0 [BH, D]: carried-in state or NULL (zero).
 * dSN [BH, D, M], dzN [BH, D]: gradient reaching the final state or NULL.
 * Outputs dq, dk [BH, N, D], dv [BH, N, M] (fp64) and, if non-NULL,
 * dS0 [BH, D, M], dz0 [BH, D] (fp64).
 */
int lao_causal_backward_mut(const float *q, const float *k, const float *v, const float *G,
                            long BH, long N, long D, long M,
                            const double *S0, const double *z0, const double *dSN, const double *dzN,
                            double *dq, double *dk, double *dv, double *dS0, double *dz0,
                            int nthreads, int mutant)
{
    if (BH < 0 || N < 0 || D <= 0 || M <= 0) return 1;
    set_threads(nthreads);
    long h;
#pragma omp parallel for schedule(static)
    for (h = 0; h < BH; ++h) {
        double *S = calloc((size_t)(D * M), sizeof(double));
        double *z = calloc((size_t)D, sizeof(double));
        double *g = malloc(sizeof(double) * (size_t)(N * M + 1));
        double *e = malloc(sizeof(double) * (size_t)(N + 1));
        double *fq = malloc(sizeof(double) * (size_t)D);
        double *fk = malloc(sizeof(double) * (size_t)D);
        double *num = malloc(sizeof(double) * (size_t)M);
        const float *qh = q + h * N * D, *kh = k + h * N * D, *vh = v + h * N * M, *Gh = G + h * N * M;
        if (S0) memcpy(S, S0 + h * D * M, sizeof(double) * (size_t)(D * M));
        if (z0) memcpy(z, z0 + h * D, sizeof(double) * (size_t)D);
        /* forward sweep: eqs. (10)-(12), then g_i, e_i and dphi(Q_i) */
        for (long i = 0; i < N; ++i) {
            for (long d = 0; d < D; ++d) {
                fq[d] = lao_phi((double)qh[i * D + d]);
                fk[d] = lao_phi((double)kh[i * D + d]);
            }
            for (long d = 0; d < D; ++d) {
                for (long m = 0; m < M; ++m) S[d * M + m] += fk[d] * (double)vh[i * M + m];
                z[d] += fk[d];
            }
            double den = 0.0;
            for (long d = 0; d < D; ++d) den += fq[d] * z[d];
            double gn = 0.0;
            for (long m = 0; m < M; ++m) {
                double t = 0.0;
                for (long d = 0; d < D; ++d) t += fq[d] * S[d * M + m];
                num[m] = t;
                g[i * M + m] = (double)Gh[i * M + m] / den;
                gn += g[i * M + m] * t;
            }
            e[i] = mutant == MUT_B_NO_E ? 0.0 : -gn / den;
            for (long d = 0; d < D; ++d) {
                double t = e[i] * z[d];
                for (long m = 0; m < M; ++m) t += S[d * M + m] * g[i * M + m];
                dq[(h * N + i) * D + d] = t * dphi_m((double)qh[i * D + d], mutant);
            }
        }
        /* reverse sweep: R and r accumulate phi(Q_j) g_j^T and e_j phi(Q_j), j >= i */
        double *R = S, *r = z;   /* reuse the buffers */
        if (dSN) memcpy(R, dSN + h * D * M, sizeof(double) * (size_t)(D * M));
        else memset(R, 0, sizeof(double) * (size_t)(D * M));
        if (dzN) memcpy(r, dzN + h * D, sizeof(double) * (size_t)D);
        else memset(r, 0, sizeof(double) * (size_t)D);
        for (long i = N - 1; i >= 0; --i) {
            for (long d = 0; d < D; ++d) {
                fq[d] = lao_phi((double)qh[i * D + d]);
                fk[d] = lao_phi((double)kh[i * D + d]);
            }
            if (mutant != MUT_B_EXCL_DIAG)
                for (long d = 0; d < D; ++d) {
                    for (long m = 0; m < M; ++m) R[d * M + m] += fq[d] * g[i * M + m];
                    r[d] += e[i] * fq[d];
                }
            for (long d = 0; d < D; ++d) {
                double t = r[d];
                for (long m = 0; m < M; ++m) t += R[d * M + m] * (double)vh[i * M + m];
                dk[(h * N + i) * D + d] = t * dphi_m((double)kh[i * D + d], mutant);
            }
            for (long m = 0; m < M; ++m) {
                double t = 0.0;
                for (long d = 0; d < D; ++d) t += R[d * M + m] * (mutant == MUT_B_DV_USES_Q ? fq[d] : fk[d]);
                dv[(h * N + i) * M + m] = t;
            }
            if (mutant == MUT_B_EXCL_DIAG)
                for (long d = 0; d < D; ++d) {
                    for (long m = 0; m < M; ++m) R[d * M + m] += fq[d] * g[i * M + m];
                    r[d] += e[i] * fq[d];
                }
        }
        if (dS0) memcpy(dS0 + h * D * M, R, sizeof(double) * (size_t)(D * M));
        if (dz0) memcpy(dz0 + h * D, r, sizeof(double) * (size_t)D);
        free(S); free(z); free(g); free(e); free(fq); free(fk); free(num);
    }
    return 0;
}

/*
 * Backward of the non-causal form, eq. (5): the same steps with every sum
 * over all N keys: S, z are the full sums; R = sum_j phi(Q_j) g_j^T and
 * r = sum_j e_j phi(Q_j) over all queries.
 */
int lao_noncausal_backward_mut(const float *q, const float *k, const float *v, const float *G,
                               long BH, long N, long D, long M,
                               double *dq, double *dk, double *dv, int nthreads, int mutant)
{
    if (BH < 0 || N < 0 || D <= 0 || M <= 0) return 1;
    set_threads(nthreads);
    long h;
#pragma omp parallel for schedule(static)
    for (h = 0; h < BH; ++h) {
        double *S = calloc((size_t)(D * M), sizeof(double));
        double *z = calloc((size_t)D, sizeof(double));
        double *R = calloc((size_t)(D * M), sizeof(double));
        double *r = calloc((size_t)D, sizeof(double));
        double *fq = malloc(sizeof(double) * (size_t)D);
        double *fk = malloc(sizeof(double) * (size_t)D);
        double *g = malloc(sizeof(double) * (size_t)M);
        const float *qh = q + h * N * D, *kh = k + h * N * D, *vh = v + h * N * M, *Gh = G + h * N * M;
        for (long j = 0; j < N; ++j)
            for (long d = 0; d < D; ++d) {
                double f = lao_phi((double)kh[j * D + d]);
                for (long m = 0; m < M; ++m) S[d * M + m] += f * (double)vh[j * M + m];
                z[d] += f;
            }
        for (long i = 0; i < N; ++i) {
            for (long d = 0; d < D; ++d) fq[d] = lao_phi((double)qh[i * D + d]);
            double den = 0.0;
            for (long d = 0; d < D; ++d) den += fq[d] * z[d];
            double gn = 0.0;
            for (long m = 0; m < M; ++m) {
                double t = 0.0;
                for (long d = 0; d < D; ++d) t += fq[d] * S[d * M + m];
                g[m] = (double)Gh[i * M + m] / den;
                gn += g[m] * t;
            }
            const double e = mutant == MUT_B_NO_E ? 0.0 : -gn / den;
            for (long d = 0; d < D; ++d) {
                double t = e * z[d];
                for (long m = 0; m < M; ++m) t += S[d * M + m] * g[m];
                dq[(h * N + i) * D + d] = t * dphi_m((double)qh[i * D + d], mutant);
                for (long m = 0; m < M; ++m) R[d * M + m] += fq[d] * g[m];
                r[d] += e * fq[d];
            }
        }
        for (long j = 0; j < N; ++j) {
            for (long d = 0; d < D; ++d) {
                fk[d] = lao_phi((double)kh[j * D + d]);
                fq[d] = lao_phi((double)qh[j * D + d]);
            }
            for (long d = 0; d < D; ++d) {
                double t = r[d];
                for (long m = 0; m < M; ++m) t += R[d * M + m] * (double)vh[j * M + m];
                dk[(h * N + j) * D + d] = t * dphi_m((double)kh[j * D + d], mutant);
            }
            for (long m = 0; m < M; ++m) {
                double t = 0.0;
                for (long d = 0; d < D; ++d) t += R[d * M + m] * (mutant == MUT_B_DV_USES_Q ? fq[d] : fk[d]);
                dv[(h * N + j) * M + m] = t;
            }
        }
        free(S); free(z); free(R); free(r); free(fq); free(fk); free(g);
    }
    return 0;
}

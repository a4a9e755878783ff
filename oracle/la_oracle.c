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
    MUT_DEN_Q_OF_K = 7     /* denominator phi(K_i)^T Z_i instead of phi(Q_i)  */
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

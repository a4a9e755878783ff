// la_bwd.cu - backward pass (gradients) of kernelised linear attention on
// CUDA cores, fp32 arithmetic, for fp32 or bf16 tensors and D, M in
// {16, 32, 64, 128}.
//
// "Transformers are RNNs" sec. 3.3.1 computes the gradient of the causal
// form as cumulative sums with constant extra memory; its equations
// (13)-(15) are not printed on the page, so these kernels follow the chain
// rule through eqs. (10)-(12).  With num_i = phi(Q_i)^T S_i, den_i =
// phi(Q_i)^T Z_i and G_i = dL/dV'_i:
//   g_i = G_i / den_i,  e_i = -(g_i . num_i) / den_i
//   dphi(Q_i) = S_i g_i + e_i Z_i                                  (pass 1)
//   R_i = sum_{j>=i} phi(Q_j) g_j^T,  r_i = sum_{j>=i} e_j phi(Q_j)
//   dphi(K_i) = R_i V_i + r_i,  dV_i = R_i^T phi(K_i)               (pass 2)
//   dQ = dphi(Q) * phi'(Q), dK = dphi(K) * phi'(K),  phi'(x) = min(phi(x), 1)
// (phi(x) = x + 1 > 1 exactly when x > 0, where phi' = 1; else phi' = e^x = phi).
// Both passes walk a head in chunks of kCs rows; inside a chunk the sums
// over j <= i become masked products with
//   A_ij = g_i . V_j + e_i,  P_ij = phi(Q_i) . phi(K_j)   (j <= i)
// so that, with S, Z the state before the chunk and R, r the sums after it,
//   dphi(Q_i) = sum_{j<=i} A_ij phi(K_j) + S g_i + e_i Z
//   dphi(K_j) = sum_{i>=j} A_ij phi(Q_i) + R V_j + r
//   dV_j      = sum_{i>=j} P_ij g_i + R^T phi(K_j).
// Pass 1 stores g and e (N (M + 1) floats per head: the O(N max(D, M))
// memory the page allows; no per-token D x M state is ever stored).
#include <algorithm>

#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kCs = 32;   // chunk rows

__device__ __forceinline__ float dphi_from_phi(float f) { return fminf(f, 1.f); }

// Shared memory of either causal pass: the D x M state and D vector, the
// chunk's phi(Q), phi(K) (padded rows), V, g (or G), e, den, and the masked
// A and P blocks.
size_t bwd_smem_bytes(int D, int M) {
    const int ldq = D + 1, lda = kCs + 1;
    return sizeof(float) * ((size_t)D * M + D + 2 * kCs * ldq + 2 * (size_t)kCs * M + 3 * kCs + 2 * kCs * lda);
}

struct BwdSmem {
    float *S, *z, *fq, *fk, *vv, *gg, *ee, *den, *es, *A, *P;
    int ldq, lda;
    __device__ BwdSmem(float *sm, int D, int M) {
        ldq = D + 1;
        lda = kCs + 1;
        S = sm;
        z = S + D * M;
        fq = z + D;
        fk = fq + kCs * ldq;
        vv = fk + kCs * ldq;
        gg = vv + kCs * M;
        ee = gg + kCs * M;
        den = ee + kCs;
        es = den + kCs;
        A = es + kCs;
        P = A + kCs * lda;
    }
};

// Pass 1, forward over the chunks of one segment of a head (one CTA per
// segment): recomputes the forward from the state entering the segment (the
// carried-in state plus the earlier segments' sums phi(K)^T V, phi(K) from
// seg_s), writes dQ and keeps g, e.
template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_causal_pass1_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                        const T *__restrict__ G, T *__restrict__ dq, float *__restrict__ g_ws,
                        float *__restrict__ e_ws, const float *__restrict__ S0, const float *__restrict__ z0,
                        const float *__restrict__ seg_s, int N, int D, int M, int nseg, int L)
{
    extern __shared__ float sm[];
    BwdSmem s(sm, D, M);
    const int ldq = s.ldq, lda = s.lda;
    const long long h = blockIdx.x / nseg;
    const int seg = blockIdx.x % nseg;
    const int tid = threadIdx.x;
    const int W = D * M + D;
    const int t_begin = seg * L, t_end = min(N, t_begin + L);
    const T *qh = q + h * N * D, *kh = k + h * N * D, *vh = v + h * N * M, *Gh = G + h * N * M;
    T *dqh = dq + h * N * D;
    float *gh = g_ws + h * N * M, *eh = e_ws + h * N;

    const float *segh = seg_s + h * nseg * (long long)W;
    for (int i = tid; i < W; i += kThreads) {
        float a = i < D * M ? (S0 ? S0[h * D * M + i] : 0.f) : (z0 ? z0[h * D + (i - D * M)] : 0.f);
        for (int g = 0; g < seg; ++g) a += segh[g * (long long)W + i];
        s.S[i] = a;   // S then z (contiguous)
    }

    for (int t0 = t_begin; t0 < t_end; t0 += kCs) {
        const int rows = min(kCs, t_end - t0);
        __syncthreads();
        for (int idx = tid; idx < kCs * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            float a = 0.f, b = 0.f;
            if (i < rows) {
                a = phi_accurate(to_f32(qh[(long long)(t0 + i) * D + d]));
                b = phi_accurate(to_f32(kh[(long long)(t0 + i) * D + d]));
            }
            s.fq[i * ldq + d] = a;
            s.fk[i * ldq + d] = b;
        }
        for (int idx = tid; idx < kCs * M; idx += kThreads) {
            const int i = idx / M, m = idx - i * M;
            const bool in = i < rows;
            s.vv[idx] = in ? to_f32(vh[(long long)(t0 + i) * M + m]) : 0.f;
            s.gg[idx] = in ? to_f32(Gh[(long long)(t0 + i) * M + m]) : 0.f;
        }
        for (int i = tid; i < kCs; i += kThreads) s.es[i] = 0.f;
        __syncthreads();
        // P_ij = phi(Q_i) . phi(K_j), j <= i
        for (int idx = tid; idx < kCs * kCs; idx += kThreads) {
            const int i = idx / kCs, j = idx - i * kCs;
            float acc = 0.f;
            if (j <= i && i < rows)
                for (int d = 0; d < D; ++d) acc += s.fq[i * ldq + d] * s.fk[j * ldq + d];
            s.P[i * lda + j] = acc;
        }
        __syncthreads();
        // den_i = sum_{j<=i} P_ij + phi(Q_i) . Z  (eq. (12) denominator, Z before the chunk)
        for (int i = tid; i < rows; i += kThreads) {
            float a = 0.f, b = 0.f;
            for (int j = 0; j <= i; ++j) a += s.P[i * lda + j];
            for (int d = 0; d < D; ++d) b += s.fq[i * ldq + d] * s.z[d];
            s.den[i] = a + b;
        }
        __syncthreads();
        // num_im, then g_im = G_im / den_i in place of G, and sum_m g_im num_im
        for (int idx = tid; idx < rows * M; idx += kThreads) {
            const int i = idx / M, m = idx - i * M;
            float intra = 0.f, inter = 0.f;
            for (int j = 0; j <= i; ++j) intra += s.P[i * lda + j] * s.vv[j * M + m];
            for (int d = 0; d < D; ++d) inter += s.fq[i * ldq + d] * s.S[d * M + m];
            const float g = s.gg[idx] / s.den[i];
            s.gg[idx] = g;
            atomicAdd(&s.es[i], g * (intra + inter));
        }
        __syncthreads();
        for (int i = tid; i < kCs; i += kThreads) {
            const float e = i < rows ? -s.es[i] / s.den[i] : 0.f;
            s.ee[i] = e;
            if (i < rows) eh[t0 + i] = e;
        }
        for (int idx = tid; idx < rows * M; idx += kThreads) gh[(long long)t0 * M + idx] = s.gg[idx];
        __syncthreads();
        // A_ij = g_i . V_j + e_i, j <= i
        for (int idx = tid; idx < kCs * kCs; idx += kThreads) {
            const int i = idx / kCs, j = idx - i * kCs;
            float acc = 0.f;
            if (j <= i && i < rows) {
                for (int m = 0; m < M; ++m) acc += s.gg[i * M + m] * s.vv[j * M + m];
                acc += s.ee[i];
            }
            s.A[i * lda + j] = acc;
        }
        __syncthreads();
        // dphi(Q_i) = sum_{j<=i} A_ij phi(K_j) + S g_i + e_i Z;  dQ = dphi(Q) phi'(Q)
        for (int idx = tid; idx < rows * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            float acc = s.ee[i] * s.z[d];
            for (int j = 0; j <= i; ++j) acc += s.A[i * lda + j] * s.fk[j * ldq + d];
            for (int m = 0; m < M; ++m) acc += s.S[d * M + m] * s.gg[i * M + m];
            dqh[(long long)(t0 + i) * D + d] = from_f32<T>(acc * dphi_from_phi(s.fq[i * ldq + d]));
        }
        __syncthreads();
        // the state after the chunk: S += phi(K)^T V, Z += sum phi(K)  (eqs. (10), (11))
        for (int idx = tid; idx < D * M; idx += kThreads) {
            const int d = idx / M, m = idx - d * M;
            float acc = 0.f;
            for (int j = 0; j < rows; ++j) acc += s.fk[j * ldq + d] * s.vv[j * M + m];
            s.S[idx] += acc;
        }
        for (int d = tid; d < D; d += kThreads) {
            float acc = 0.f;
            for (int j = 0; j < rows; ++j) acc += s.fk[j * ldq + d];
            s.z[d] += acc;
        }
    }
}

// Pass 2, backward over the chunks of one segment of a head: R, r start from
// the gradient reaching the final state (or 0) plus the later segments' sums
// phi(Q)^T g, e phi(Q) (seg_r), and take in each chunk after its dK, dV.
template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_causal_pass2_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                        const float *__restrict__ g_ws, const float *__restrict__ e_ws, T *__restrict__ dk,
                        T *__restrict__ dv, const float *__restrict__ dSN, const float *__restrict__ dzN,
                        float *__restrict__ dS0, float *__restrict__ dz0, const float *__restrict__ seg_r,
                        int N, int D, int M, int nseg, int L)
{
    extern __shared__ float sm[];
    BwdSmem s(sm, D, M);
    float *R = s.S, *r = s.z;
    const int ldq = s.ldq, lda = s.lda;
    const long long h = blockIdx.x / nseg;
    const int seg = blockIdx.x % nseg;
    const int tid = threadIdx.x;
    const int W = D * M + D;
    const int t_begin = seg * L, t_end = min(N, t_begin + L);
    const T *qh = q + h * N * D, *kh = k + h * N * D, *vh = v + h * N * M;
    T *dkh = dk + h * N * D, *dvh = dv + h * N * M;
    const float *gh = g_ws + h * N * M, *eh = e_ws + h * N;

    const float *segh = seg_r + h * nseg * (long long)W;
    for (int i = tid; i < W; i += kThreads) {
        float a = i < D * M ? (dSN ? dSN[h * D * M + i] : 0.f) : (dzN ? dzN[h * D + (i - D * M)] : 0.f);
        for (int g = seg + 1; g < nseg; ++g) a += segh[g * (long long)W + i];
        R[i] = a;     // R then r (contiguous)
    }

    const int nch = (t_end - t_begin + kCs - 1) / kCs;
    for (int c = nch - 1; c >= 0; --c) {
        const int t0 = t_begin + c * kCs, rows = min(kCs, t_end - t0);
        __syncthreads();
        for (int idx = tid; idx < kCs * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            float a = 0.f, b = 0.f;
            if (i < rows) {
                a = phi_accurate(to_f32(qh[(long long)(t0 + i) * D + d]));
                b = phi_accurate(to_f32(kh[(long long)(t0 + i) * D + d]));
            }
            s.fq[i * ldq + d] = a;
            s.fk[i * ldq + d] = b;
        }
        for (int idx = tid; idx < kCs * M; idx += kThreads) {
            const int i = idx / M, m = idx - i * M;
            const bool in = i < rows;
            s.vv[idx] = in ? to_f32(vh[(long long)(t0 + i) * M + m]) : 0.f;
            s.gg[idx] = in ? gh[(long long)(t0 + i) * M + m] : 0.f;
        }
        for (int i = tid; i < kCs; i += kThreads) s.ee[i] = i < rows ? eh[t0 + i] : 0.f;
        __syncthreads();
        for (int idx = tid; idx < kCs * kCs; idx += kThreads) {
            const int i = idx / kCs, j = idx - i * kCs;
            float p = 0.f, a = 0.f;
            if (j <= i && i < rows) {
                for (int d = 0; d < D; ++d) p += s.fq[i * ldq + d] * s.fk[j * ldq + d];
                for (int m = 0; m < M; ++m) a += s.gg[i * M + m] * s.vv[j * M + m];
                a += s.ee[i];
            }
            s.P[i * lda + j] = p;
            s.A[i * lda + j] = a;
        }
        __syncthreads();
        // dphi(K_j) = sum_{i>=j} A_ij phi(Q_i) + R V_j + r;  dK = dphi(K) phi'(K)
        for (int idx = tid; idx < rows * D; idx += kThreads) {
            const int j = idx / D, d = idx - j * D;
            float acc = r[d];
            for (int i = j; i < rows; ++i) acc += s.A[i * lda + j] * s.fq[i * ldq + d];
            for (int m = 0; m < M; ++m) acc += R[d * M + m] * s.vv[j * M + m];
            dkh[(long long)(t0 + j) * D + d] = from_f32<T>(acc * dphi_from_phi(s.fk[j * ldq + d]));
        }
        // dV_j = sum_{i>=j} P_ij g_i + R^T phi(K_j)
        for (int idx = tid; idx < rows * M; idx += kThreads) {
            const int j = idx / M, m = idx - j * M;
            float acc = 0.f;
            for (int i = j; i < rows; ++i) acc += s.P[i * lda + j] * s.gg[i * M + m];
            for (int d = 0; d < D; ++d) acc += R[d * M + m] * s.fk[j * ldq + d];
            dvh[(long long)(t0 + j) * M + m] = from_f32<T>(acc);
        }
        __syncthreads();
        // R += phi(Q_c)^T g_c, r += sum_i e_i phi(Q_i)
        for (int idx = tid; idx < D * M; idx += kThreads) {
            const int d = idx / M, m = idx - d * M;
            float acc = 0.f;
            for (int i = 0; i < rows; ++i) acc += s.fq[i * ldq + d] * s.gg[i * M + m];
            R[idx] += acc;
        }
        for (int d = tid; d < D; d += kThreads) {
            float acc = 0.f;
            for (int i = 0; i < rows; ++i) acc += s.ee[i] * s.fq[i * ldq + d];
            r[d] += acc;
        }
    }
    __syncthreads();
    if (dS0 && seg == 0)
        for (int i = tid; i < D * M; i += kThreads) dS0[h * D * M + i] = R[i];
    if (dz0 && seg == 0)
        for (int i = tid; i < D; i += kThreads) dz0[h * D + i] = r[i];
}

// Per (head, segment): sum_i phi(Q_i) g_i^T and sum_i e_i phi(Q_i) over the
// segment's rows, the part of R, r that pass 2 carries into earlier segments.
template <typename T>
__global__ void __launch_bounds__(kThreads)
bwd_qg_sums_kernel(const T *__restrict__ q, const float *__restrict__ g_ws, const float *__restrict__ e_ws,
                   float *__restrict__ seg_r, int N, int D, int M, int nseg, int L)
{
    extern __shared__ float sm[];
    const int ldq = D + 1, W = D * M + D;
    float *acc = sm;                  // [W]
    float *fq = acc + W;              // [kCs][ldq]
    float *gg = fq + kCs * ldq;       // [kCs][M]
    float *ee = gg + kCs * M;         // [kCs]
    const long long h = blockIdx.x / nseg;
    const int seg = blockIdx.x % nseg, tid = threadIdx.x;
    const int t_begin = seg * L, t_end = min(N, t_begin + L);
    const T *qh = q + h * N * D;
    const float *gh = g_ws + h * N * M, *eh = e_ws + h * N;
    for (int i = tid; i < W; i += kThreads) acc[i] = 0.f;
    for (int t0 = t_begin; t0 < t_end; t0 += kCs) {
        const int rows = min(kCs, t_end - t0);
        __syncthreads();
        for (int idx = tid; idx < kCs * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            fq[i * ldq + d] = i < rows ? phi_accurate(to_f32(qh[(long long)(t0 + i) * D + d])) : 0.f;
        }
        for (int idx = tid; idx < kCs * M; idx += kThreads) {
            const int i = idx / M;
            gg[idx] = i < rows ? gh[(long long)t0 * M + idx] : 0.f;
        }
        for (int i = tid; i < kCs; i += kThreads) ee[i] = i < rows ? eh[t0 + i] : 0.f;
        __syncthreads();
        for (int idx = tid; idx < D * M; idx += kThreads) {
            const int d = idx / M, m = idx - d * M;
            float a = 0.f;
            for (int i = 0; i < rows; ++i) a += fq[i * ldq + d] * gg[i * M + m];
            acc[idx] += a;
        }
        for (int d = tid; d < D; d += kThreads) {
            float a = 0.f;
            for (int i = 0; i < rows; ++i) a += ee[i] * fq[i * ldq + d];
            acc[D * M + d] += a;
        }
    }
    __syncthreads();
    float *dst = seg_r + (h * nseg + seg) * (long long)W;
    for (int i = tid; i < W; i += kThreads) dst[i] = acc[i];
}

// ------------------------------------------------------------- non-causal
// Same steps with every sum over all N keys (eq. (5)).
//   phase 1: S, Z per (head, split of keys) - partial sums into ws_s;
//   phase 2 (per head, block of query rows): S, Z summed from the partials;
//            per row g, e, dQ; the block's partial R = sum phi(Q_i) g_i^T and
//            r = sum e_i phi(Q_i) into ws_r;
//   phase 3 (per head, block of key rows): R, r summed; dK, dV per row.

size_t nc_bwd_smem_bytes(int D, int M) {
    const int ldq = D + 1;
    return sizeof(float) * (2 * ((size_t)D * M + D) + kCs * ldq + 2 * (size_t)kCs * M + 2 * kCs);
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
nc_bwd_sums_kernel(const T *__restrict__ k, const T *__restrict__ v, float *__restrict__ ws_s,
                   int N, int D, int M, int nsplit, int L)
{
    extern __shared__ float sm[];
    const int ldq = D + 1, W = D * M + D;
    float *acc = sm;                  // [W]
    float *fk = acc + W;              // [kCs][ldq]
    float *vv = fk + kCs * ldq;       // [kCs][M]
    const long long h = blockIdx.x;
    const int sp = blockIdx.y, tid = threadIdx.x;
    const int t_begin = sp * L, t_end = min(N, t_begin + L);
    const T *kh = k + h * N * D, *vh = v + h * N * M;
    for (int i = tid; i < W; i += kThreads) acc[i] = 0.f;
    for (int t0 = t_begin; t0 < t_end; t0 += kCs) {
        const int rows = min(kCs, t_end - t0);
        __syncthreads();
        for (int idx = tid; idx < kCs * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            fk[i * ldq + d] = i < rows ? phi_accurate(to_f32(kh[(long long)(t0 + i) * D + d])) : 0.f;
        }
        for (int idx = tid; idx < kCs * M; idx += kThreads) {
            const int i = idx / M, m = idx - i * M;
            vv[idx] = i < rows ? to_f32(vh[(long long)(t0 + i) * M + m]) : 0.f;
        }
        __syncthreads();
        for (int idx = tid; idx < D * M; idx += kThreads) {
            const int d = idx / M, m = idx - d * M;
            float a = 0.f;
            for (int j = 0; j < rows; ++j) a += fk[j * ldq + d] * vv[j * M + m];
            acc[idx] += a;
        }
        for (int d = tid; d < D; d += kThreads) {
            float a = 0.f;
            for (int j = 0; j < rows; ++j) a += fk[j * ldq + d];
            acc[D * M + d] += a;
        }
    }
    __syncthreads();
    float *dst = ws_s + (h * nsplit + sp) * (long long)W;
    for (int i = tid; i < W; i += kThreads) dst[i] = acc[i];
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
nc_bwd_q_kernel(const T *__restrict__ q, const T *__restrict__ G, const float *__restrict__ ws_s,
                T *__restrict__ dq, float *__restrict__ ws_r, int N, int D, int M, int nsplit, int nrb, int RB)
{
    extern __shared__ float sm[];
    const int ldq = D + 1, W = D * M + D;
    float *Sz = sm;                   // [W]: S then Z
    float *Rr = Sz + W;               // [W]: this block's R then r
    float *fq = Rr + W;               // [kCs][ldq]
    float *gg = fq + kCs * ldq;       // [kCs][M]: G, then g
    float *nm = gg + kCs * M;         // [kCs][M]: num
    float *den = nm + kCs * M;        // [kCs]
    float *ee = den + kCs;            // [kCs]
    const long long h = blockIdx.x;
    const int rb = blockIdx.y, tid = threadIdx.x;
    const int r0 = rb * RB, r1 = min(N, r0 + RB);
    const float *src = ws_s + h * nsplit * (long long)W;
    for (int i = tid; i < W; i += kThreads) {
        float a = 0.f;
        for (int sp = 0; sp < nsplit; ++sp) a += src[sp * (long long)W + i];
        Sz[i] = a;
        Rr[i] = 0.f;
    }
    const float *S = Sz, *z = Sz + D * M;
    const T *qh = q + h * N * D, *Gh = G + h * N * M;
    T *dqh = dq + h * N * D;
    for (int t0 = r0; t0 < r1; t0 += kCs) {
        const int rows = min(kCs, r1 - t0);
        __syncthreads();
        for (int idx = tid; idx < kCs * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            fq[i * ldq + d] = i < rows ? phi_accurate(to_f32(qh[(long long)(t0 + i) * D + d])) : 0.f;
        }
        for (int idx = tid; idx < kCs * M; idx += kThreads) {
            const int i = idx / M, m = idx - i * M;
            gg[idx] = i < rows ? to_f32(Gh[(long long)(t0 + i) * M + m]) : 0.f;
        }
        __syncthreads();
        for (int i = tid; i < kCs; i += kThreads) {
            float a = 0.f;
            if (i < rows)
                for (int d = 0; d < D; ++d) a += fq[i * ldq + d] * z[d];
            den[i] = i < rows ? a : 1.f;
        }
        for (int idx = tid; idx < kCs * M; idx += kThreads) {
            const int i = idx / M, m = idx - i * M;
            float a = 0.f;
            if (i < rows)
                for (int d = 0; d < D; ++d) a += fq[i * ldq + d] * S[d * M + m];
            nm[idx] = a;
        }
        __syncthreads();
        for (int idx = tid; idx < kCs * M; idx += kThreads) gg[idx] /= den[idx / M];
        __syncthreads();
        for (int i = tid; i < kCs; i += kThreads) {
            float a = 0.f;
            for (int m = 0; m < M; ++m) a += gg[i * M + m] * nm[i * M + m];
            ee[i] = -a / den[i];
        }
        __syncthreads();
        // dphi(Q_i) = S g_i + e_i Z;  dQ = dphi(Q) phi'(Q)
        for (int idx = tid; idx < rows * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            float a = ee[i] * z[d];
            for (int m = 0; m < M; ++m) a += S[d * M + m] * gg[i * M + m];
            dqh[(long long)(t0 + i) * D + d] = from_f32<T>(a * dphi_from_phi(fq[i * ldq + d]));
        }
        // the block's R += phi(Q)^T g, r += sum e_i phi(Q_i)
        for (int idx = tid; idx < D * M; idx += kThreads) {
            const int d = idx / M, m = idx - d * M;
            float a = 0.f;
            for (int i = 0; i < rows; ++i) a += fq[i * ldq + d] * gg[i * M + m];
            Rr[idx] += a;
        }
        for (int d = tid; d < D; d += kThreads) {
            float a = 0.f;
            for (int i = 0; i < rows; ++i) a += ee[i] * fq[i * ldq + d];
            Rr[D * M + d] += a;
        }
    }
    __syncthreads();
    float *dst = ws_r + (h * nrb + rb) * (long long)W;
    for (int i = tid; i < W; i += kThreads) dst[i] = Rr[i];
}

template <typename T>
__global__ void __launch_bounds__(kThreads)
nc_bwd_kv_kernel(const T *__restrict__ k, const T *__restrict__ v, const float *__restrict__ ws_r,
                 T *__restrict__ dk, T *__restrict__ dv, int N, int D, int M, int nrb, int RB)
{
    extern __shared__ float sm[];
    const int ldq = D + 1, W = D * M + D;
    float *Rr = sm;                   // [W]
    float *fk = Rr + W;               // [kCs][ldq]
    float *vv = fk + kCs * ldq;       // [kCs][M]
    const long long h = blockIdx.x;
    const int rb = blockIdx.y, tid = threadIdx.x;
    const int r0 = rb * RB, r1 = min(N, r0 + RB);
    const float *src = ws_r + h * nrb * (long long)W;
    for (int i = tid; i < W; i += kThreads) {
        float a = 0.f;
        for (int b = 0; b < nrb; ++b) a += src[b * (long long)W + i];
        Rr[i] = a;
    }
    const float *R = Rr, *r = Rr + D * M;
    const T *kh = k + h * N * D, *vh = v + h * N * M;
    T *dkh = dk + h * N * D, *dvh = dv + h * N * M;
    for (int t0 = r0; t0 < r1; t0 += kCs) {
        const int rows = min(kCs, r1 - t0);
        __syncthreads();
        for (int idx = tid; idx < kCs * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            fk[i * ldq + d] = i < rows ? phi_accurate(to_f32(kh[(long long)(t0 + i) * D + d])) : 0.f;
        }
        for (int idx = tid; idx < kCs * M; idx += kThreads) {
            const int i = idx / M, m = idx - i * M;
            vv[idx] = i < rows ? to_f32(vh[(long long)(t0 + i) * M + m]) : 0.f;
        }
        __syncthreads();
        // dphi(K_j) = R V_j + r;  dK = dphi(K) phi'(K)
        for (int idx = tid; idx < rows * D; idx += kThreads) {
            const int j = idx / D, d = idx - j * D;
            float a = r[d];
            for (int m = 0; m < M; ++m) a += R[d * M + m] * vv[j * M + m];
            dkh[(long long)(t0 + j) * D + d] = from_f32<T>(a * dphi_from_phi(fk[j * ldq + d]));
        }
        // dV_j = R^T phi(K_j)
        for (int idx = tid; idx < rows * M; idx += kThreads) {
            const int j = idx / M, m = idx - j * M;
            float a = 0.f;
            for (int d = 0; d < D; ++d) a += R[d * M + m] * fk[j * ldq + d];
            dvh[(long long)(t0 + j) * M + m] = from_f32<T>(a);
        }
    }
}

// Key splits of phase 1 and row blocks of phases 2 and 3: about two CTAs per
// SM over the whole grid, at least one chunk each, at most 16 per head.
void nc_bwd_grid(long long BH, int N, int sm_count, int &nsplit, int &L) {
    const long long want = (2LL * std::max(sm_count, 1) + BH - 1) / BH;
    const long long most = (N + kCs - 1) / kCs;
    nsplit = (int)std::max(1LL, std::min(want, std::min(most, 16LL)));
    L = (N + nsplit - 1) / nsplit;
    L = (L + kCs - 1) / kCs * kCs;
    nsplit = (N + L - 1) / L;
}

template <typename T>
cudaError_t set_bwd_smem(size_t bytes) {
    cudaError_t e;
    for (const void *f : {(const void *)bwd_causal_pass1_kernel<T>, (const void *)bwd_causal_pass2_kernel<T>,
                          (const void *)nc_bwd_sums_kernel<T>, (const void *)nc_bwd_q_kernel<T>,
                          (const void *)nc_bwd_kv_kernel<T>, (const void *)bwd_qg_sums_kernel<T>})
        if ((e = cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes)) != cudaSuccess)
            return e;
    return cudaSuccess;
}

size_t bwd_max_smem(int D, int M) { return std::max(bwd_smem_bytes(D, M), nc_bwd_smem_bytes(D, M)); }

// Segments per head of the causal backward: about four CTAs per SM over the
// grid, at least four chunks per segment, rows a multiple of the chunk.
void bwd_seg_grid(long long BH, int N, int sm_count, int &nseg, int &L) {
    const long long nch = (N + kCs - 1) / kCs;
    const long long want = (4LL * std::max(sm_count, 1) + BH - 1) / std::max(1LL, BH);
    nseg = (int)std::max(1LL, std::min(std::min(want, std::max(1LL, nch / 4)), 64LL));
    L = (N + nseg - 1) / nseg;
    L = (L + kCs - 1) / kCs * kCs;
    nseg = (N + L - 1) / L;
}

// The causal backward in four launches: segment sums of phi(K)^T V (the state
// entering each segment), pass 1 per segment, segment sums of phi(Q)^T g and
// e phi(Q) (the reverse sums entering each segment from the right), pass 2.
template <typename T>
cudaError_t causal_bwd_t(const BwdProblem &p, const DeviceInfo &dev) {
    int nseg, L;
    bwd_seg_grid(p.BH, p.N, dev.sm_count, nseg, L);
    const long long W = (long long)p.D * p.M + p.D;
    if (p.ws_bytes < (size_t)(p.BH * ((long long)p.N * (p.M + 1) + 2 * nseg * W)) * sizeof(float))
        return cudaErrorInvalidValue;
    const size_t sm = bwd_smem_bytes(p.D, p.M), smn = nc_bwd_smem_bytes(p.D, p.M);
    cudaError_t e = set_bwd_smem<T>(bwd_max_smem(p.D, p.M));
    if (e != cudaSuccess) return e;
    float *g_ws = (float *)p.ws;
    float *e_ws = g_ws + p.BH * (long long)p.N * p.M;
    float *seg_s = e_ws + p.BH * (long long)p.N;
    float *seg_r = seg_s + p.BH * nseg * W;
    const unsigned grid = (unsigned)(p.BH * nseg);
    nc_bwd_sums_kernel<T><<<dim3((unsigned)p.BH, (unsigned)nseg), kThreads, smn, p.stream>>>(
        (const T *)p.k, (const T *)p.v, seg_s, p.N, p.D, p.M, nseg, L);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_causal_pass1_kernel<T><<<grid, kThreads, sm, p.stream>>>(
        (const T *)p.q, (const T *)p.k, (const T *)p.v, (const T *)p.dout, (T *)p.dq, g_ws, e_ws, p.S0, p.z0,
        seg_s, p.N, p.D, p.M, nseg, L);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_qg_sums_kernel<T><<<grid, kThreads, smn, p.stream>>>((const T *)p.q, g_ws, e_ws, seg_r, p.N, p.D, p.M,
                                                             nseg, L);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_causal_pass2_kernel<T><<<grid, kThreads, sm, p.stream>>>(
        (const T *)p.q, (const T *)p.k, (const T *)p.v, g_ws, e_ws, (T *)p.dk, (T *)p.dv, p.dSN, p.dzN,
        p.dS0, p.dz0, seg_r, p.N, p.D, p.M, nseg, L);
    count_launches(1);
    return cudaGetLastError();
}

template <typename T>
cudaError_t noncausal_bwd_t(const BwdProblem &p, const DeviceInfo &dev) {
    int nsplit, L;
    nc_bwd_grid(p.BH, p.N, dev.sm_count, nsplit, L);
    const size_t sm = nc_bwd_smem_bytes(p.D, p.M);
    cudaError_t e = set_bwd_smem<T>(bwd_max_smem(p.D, p.M));
    if (e != cudaSuccess) return e;
    const long long W = (long long)p.D * p.M + p.D;
    float *ws_s = (float *)p.ws;
    float *ws_r = ws_s + p.BH * nsplit * W;
    const dim3 grid((unsigned)p.BH, (unsigned)nsplit);
    nc_bwd_sums_kernel<T><<<grid, kThreads, sm, p.stream>>>((const T *)p.k, (const T *)p.v, ws_s, p.N, p.D,
                                                           p.M, nsplit, L);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    nc_bwd_q_kernel<T><<<grid, kThreads, sm, p.stream>>>((const T *)p.q, (const T *)p.dout, ws_s, (T *)p.dq,
                                                        ws_r, p.N, p.D, p.M, nsplit, nsplit, L);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    nc_bwd_kv_kernel<T><<<grid, kThreads, sm, p.stream>>>((const T *)p.k, (const T *)p.v, ws_r, (T *)p.dk,
                                                         (T *)p.dv, p.N, p.D, p.M, nsplit, L);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

size_t causal_bwd_ws_bytes(const la_shape &s) {
    // g and e of every token, and two segment sums per (head, segment) for the
    // most segments any device picks (up to 192 SMs)
    const long long BH = (long long)s.B * s.H;
    if (BH <= 0 || s.N <= 0) return 0;
    int nseg, L;
    bwd_seg_grid(BH, s.N, 192, nseg, L);
    const size_t simt = (size_t)BH * ((size_t)s.N * ((size_t)s.M + 1) + 2 * (size_t)nseg * ((size_t)s.D * s.M + s.D)) *
                        sizeof(float);
    return tc_chunk_backward_supported(s) ? std::max(simt, tc_chunk_backward_ws_bytes(s)) : simt;
}

size_t noncausal_bwd_ws_bytes(const la_shape &s) {
    // sized for the most splits any device picks (up to 192 SMs)
    const long long BH = (long long)s.B * s.H;
    if (BH <= 0 || s.N <= 0) return 0;
    int nsplit, L;
    nc_bwd_grid(BH, s.N, 192, nsplit, L);
    const size_t simt = (size_t)2 * BH * nsplit * ((size_t)s.D * s.M + s.D) * sizeof(float);
    return tc_nc_backward_supported(s) ? std::max(simt, tc_nc_backward_ws_bytes(s)) : simt;
}

cudaError_t causal_backward(const BwdProblem &p, const DeviceInfo &dev) {
    return p.dtype == LA_DTYPE_F32 ? causal_bwd_t<float>(p, dev) : causal_bwd_t<__nv_bfloat16>(p, dev);
}

cudaError_t noncausal_backward(const BwdProblem &p, const DeviceInfo &dev) {
    return p.dtype == LA_DTYPE_F32 ? noncausal_bwd_t<float>(p, dev) : noncausal_bwd_t<__nv_bfloat16>(p, dev);
}

}  // namespace la

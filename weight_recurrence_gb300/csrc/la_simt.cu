// la_simt.cu - CUDA-core (SIMT, fp32 FFMA) kernels of liblinattn.so.
//
// * causal_simt_kernel / nc_*_simt_kernel: the fp32 path (inputs fp32 or
//   bf16, every product and sum in fp32) for any D, M in {16, 32, 64, 128}.
//   They compute the same chunked regrouping as the tensor-core path with a
//   32-row chunk, one CTA walking one head; they are the exact-arithmetic
//   workhorse for fp32 inputs (1e-4 tolerance rules out tf32/bf16 operands).
// * decode_kernel: the recurrent step, sec. 3.4 eqs. (18)-(20) of "Transformers
//   are RNNs".  It is bandwidth-bound (each head's D x M fp32 state is read
//   and written once per step) and runs on CUDA cores for every dtype.
#include <algorithm>

#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kThreads = 256;
constexpr int kCs = 32;  // SIMT chunk length

size_t causal_smem_bytes(int D, int M) {
    const int ldq = D + 1, lda = kCs + 1;
    return sizeof(float) * ((size_t)D * M + D + 2 * kCs * ldq + (size_t)kCs * M + kCs * lda + kCs);
}

// Causal form, "Transformers are RNNs" sec. 3.3 eqs. (9)-(12), regrouped by
// chunks of kCs rows: for the rows i of a chunk,
//   num_i = sum_{j in chunk, j <= i} (phi(Q_i).phi(K_j)) V_j + phi(Q_i)^T S_prev
//   den_i = sum_{j in chunk, j <= i}  phi(Q_i).phi(K_j)      + phi(Q_i)^T z_prev
// then S_prev += phi(K_c)^T V_c and z_prev += sum_rows phi(K_c) (eqs. (10), (11)).
// One CTA per (b, h); the state lives in shared memory in fp32.
template <typename T>
__global__ void __launch_bounds__(kThreads)
causal_simt_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                   T *__restrict__ out, float *__restrict__ S_io, float *__restrict__ z_io,
                   int N, int D, int M, const int *__restrict__ lens, int H)
{
    extern __shared__ float sm[];
    const int ldq = D + 1, lda = kCs + 1;
    float *S = sm;                  // [D][M]
    float *z = S + D * M;           // [D]
    float *fq = z + D;              // [kCs][ldq]  phi(Q) of the chunk
    float *fk = fq + kCs * ldq;     // [kCs][ldq]  phi(K) of the chunk (0 past N)
    float *vv = fk + kCs * ldq;     // [kCs][M]
    float *A = vv + kCs * M;        // [kCs][lda]  masked phi(Q) phi(K)^T
    float *den = A + kCs * lda;     // [kCs]
    const long long h = blockIdx.x;
    const int tid = threadIdx.x;
    const T *qh = q + h * N * D, *kh = k + h * N * D, *vh = v + h * N * M;
    T *oh = out ? out + h * N * M : nullptr;

    for (int i = tid; i < D * M; i += kThreads) S[i] = S_io ? S_io[h * D * M + i] : 0.f;
    for (int i = tid; i < D; i += kThreads) z[i] = z_io ? z_io[h * D + i] : 0.f;
    __syncthreads();

    // this head's sequence length (rows past it are ignored)
    const int Nh = lens ? max(0, min(N, lens[h / H])) : N;
    for (int t0 = 0; t0 < Nh; t0 += kCs) {
        const int rows = min(kCs, Nh - t0);
        for (int idx = tid; idx < kCs * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            float a = 0.f, b = 0.f;
            if (i < rows) {
                a = phi_accurate(to_f32(qh[(long long)(t0 + i) * D + d]));
                b = phi_accurate(to_f32(kh[(long long)(t0 + i) * D + d]));
            }
            fq[i * ldq + d] = a;
            fk[i * ldq + d] = b;
        }
        for (int idx = tid; idx < kCs * M; idx += kThreads) {
            const int i = idx / M, m = idx - i * M;
            vv[idx] = i < rows ? to_f32(vh[(long long)(t0 + i) * M + m]) : 0.f;
        }
        __syncthreads();
        if (oh) {
            for (int idx = tid; idx < kCs * kCs; idx += kThreads) {
                const int i = idx / kCs, j = idx - i * kCs;
                float s = 0.f;
                if (j <= i && i < rows)
                    for (int d = 0; d < D; ++d) s += fq[i * ldq + d] * fk[j * ldq + d];
                A[i * lda + j] = s;
            }
            __syncthreads();
            for (int i = tid; i < rows; i += kThreads) {
                float s = 0.f, t = 0.f;
                for (int j = 0; j <= i; ++j) s += A[i * lda + j];
                for (int d = 0; d < D; ++d) t += fq[i * ldq + d] * z[d];
                den[i] = s + t;
            }
            __syncthreads();
            for (int idx = tid; idx < rows * M; idx += kThreads) {
                const int i = idx / M, m = idx - i * M;
                float intra = 0.f, inter = 0.f;
                for (int j = 0; j <= i; ++j) intra += A[i * lda + j] * vv[j * M + m];
                for (int d = 0; d < D; ++d) inter += fq[i * ldq + d] * S[d * M + m];
                oh[(long long)(t0 + i) * M + m] = from_f32<T>((intra + inter) / den[i]);
            }
            __syncthreads();
        }
        for (int idx = tid; idx < D * M; idx += kThreads) {
            const int d = idx / M, m = idx - d * M;
            float s = 0.f;
            for (int j = 0; j < rows; ++j) s += fk[j * ldq + d] * vv[j * M + m];
            S[idx] += s;
        }
        for (int d = tid; d < D; d += kThreads) {
            float s = 0.f;
            for (int j = 0; j < rows; ++j) s += fk[j * ldq + d];
            z[d] += s;
        }
        __syncthreads();
    }
    if (S_io)
        for (int i = tid; i < D * M; i += kThreads) S_io[h * D * M + i] = S[i];
    if (z_io)
        for (int i = tid; i < D; i += kThreads) z_io[h * D + i] = z[i];
}

// Non-causal form, sec. 3.2 eq. (5), phase 1: each CTA reduces
// sum phi(K_j) V_j^T and sum phi(K_j) over its slice of keys into fp32
// partials (workspace [BH][nsplit][D*M + D]).
template <typename T>
__global__ void __launch_bounds__(kThreads)
nc_reduce_simt_kernel(const T *__restrict__ k, const T *__restrict__ v, float *__restrict__ ws,
                      int N, int D, int M, int nsplit, int L, long long ws_floats, int *err, int inject_oob)
{
    extern __shared__ float sm[];
    const int ldq = D + 1;
    float *acc = sm;                  // [D*M + D]
    float *fk = acc + D * M + D;      // [kCs][ldq]
    float *vv = fk + kCs * ldq;       // [kCs][M]
    const long long h = blockIdx.x;
    const int sp = blockIdx.y, tid = threadIdx.x;
    const int t_begin = sp * L, t_end = min(N, t_begin + L);
    const T *kh = k + h * N * D, *vh = v + h * N * M;
    for (int i = tid; i < D * M + D; i += kThreads) acc[i] = 0.f;
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
            float s = 0.f;
            for (int j = 0; j < rows; ++j) s += fk[j * ldq + d] * vv[j * M + m];
            acc[idx] += s;
        }
        for (int d = tid; d < D; d += kThreads) {
            float s = 0.f;
            for (int j = 0; j < rows; ++j) s += fk[j * ldq + d];
            acc[D * M + d] += s;
        }
    }
    __syncthreads();
    long long base = (h * nsplit + sp) * (long long)(D * M + D);
#ifdef LA_CHECKED
    if (inject_oob) base += ws_floats;   // test hook: one workspace length past, caught below
#endif
    if (!LA_IN_BOUNDS(base + D * M + D <= ws_floats, tid == 0 ? err : nullptr)) return;
    float *dst = ws + base;
    for (int i = tid; i < D * M + D; i += kThreads) dst[i] = acc[i];
}

// Phase 2: sum the partials of one head, then V'_i = phi(Q_i)^T KV / phi(Q_i)^T ksum
// for the CTA's block of R query rows.
template <typename T>
__global__ void __launch_bounds__(kThreads)
nc_readout_simt_kernel(const T *__restrict__ q, const float *__restrict__ ws, T *__restrict__ out,
                       int N, int D, int M, int nsplit, int R, long long ws_floats, int *err)
{
    extern __shared__ float sm[];
    const int ldq = D + 1;
    float *kv = sm;                  // [D*M + D]
    float *fq = kv + D * M + D;      // [kCs][ldq]
    float *den = fq + kCs * ldq;     // [kCs]
    const long long h = blockIdx.x;
    const int tid = threadIdx.x;
    const int r0 = blockIdx.y * R, r1 = min(N, r0 + R);
    if (!LA_IN_BOUNDS((h + 1) * nsplit * (long long)(D * M + D) <= ws_floats, tid == 0 ? err : nullptr)) return;
    const float *src = ws + h * nsplit * (long long)(D * M + D);
    for (int i = tid; i < D * M + D; i += kThreads) {
        float s = 0.f;
        for (int sp = 0; sp < nsplit; ++sp) s += src[sp * (long long)(D * M + D) + i];
        kv[i] = s;
    }
    const T *qh = q + h * N * D;
    T *oh = out + h * N * M;
    for (int t0 = r0; t0 < r1; t0 += kCs) {
        const int rows = min(kCs, r1 - t0);
        __syncthreads();
        for (int idx = tid; idx < kCs * D; idx += kThreads) {
            const int i = idx / D, d = idx - i * D;
            fq[i * ldq + d] = i < rows ? phi_accurate(to_f32(qh[(long long)(t0 + i) * D + d])) : 0.f;
        }
        __syncthreads();
        for (int i = tid; i < rows; i += kThreads) {
            float t = 0.f;
            for (int d = 0; d < D; ++d) t += fq[i * ldq + d] * kv[D * M + d];
            den[i] = t;
        }
        __syncthreads();
        for (int idx = tid; idx < rows * M; idx += kThreads) {
            const int i = idx / M, m = idx - i * M;
            float num = 0.f;
            for (int d = 0; d < D; ++d) num += fq[i * ldq + d] * kv[d * M + m];
            oh[(long long)(t0 + i) * M + m] = from_f32<T>(num / den[i]);
        }
    }
}

// Recurrent step, sec. 3.4 eqs. (18)-(20), one CTA per head.  Thread t owns
// the float4 column group t % (M/4) of rows t / (M/4) + r * (256 / (M/4)):
// a warp covers whole 128-bit-aligned rows, so every load and store of the
// state is a coalesced 16-byte access; the state is read once and written once.
template <typename T, int D, int M>
__global__ void __launch_bounds__(kThreads)
decode_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
              T *__restrict__ y, float *__restrict__ S, float *__restrict__ z)
{
    constexpr int C4 = M / 4;                 // float4 per state row
    constexpr int RP = kThreads / C4;         // rows per pass
    constexpr int NR = (D + RP - 1) / RP;     // passes
    __shared__ float fq[D], fk[D], vs[M], dz[D];
    __shared__ float4 red[RP][C4];
    __shared__ float den_s;
    const long long h = blockIdx.x;
    const int tid = threadIdx.x;
    const int c4 = tid % C4, r = tid / C4;
    pdl_wait_cta();

    float4 s[NR];
    float4 *Sh = reinterpret_cast<float4 *>(S + h * D * M);
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int d = r + i * RP;
        if (d < D) s[i] = Sh[d * C4 + c4];
    }
    if (tid < D) {
        fq[tid] = phi_accurate(to_f32(q[h * D + tid]));
        fk[tid] = phi_accurate(to_f32(k[h * D + tid]));
    }
    if (tid < M) vs[tid] = to_f32(v[h * M + tid]);
    __syncthreads();
    const float4 v4 = make_float4(vs[4 * c4], vs[4 * c4 + 1], vs[4 * c4 + 2], vs[4 * c4 + 3]);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int d = r + i * RP;
        if (d < D) {
            const float a = fk[d], b = fq[d];
            float4 t = s[i];
            t.x = fmaf(a, v4.x, t.x);      // eq. (18): s_i = s_{i-1} + phi(k) v^T
            t.y = fmaf(a, v4.y, t.y);
            t.z = fmaf(a, v4.z, t.z);
            t.w = fmaf(a, v4.w, t.w);
            Sh[d * C4 + c4] = t;
            acc.x = fmaf(b, t.x, acc.x);   // eq. (20) numerator uses the updated s_i
            acc.y = fmaf(b, t.y, acc.y);
            acc.z = fmaf(b, t.z, acc.z);
            acc.w = fmaf(b, t.w, acc.w);
        }
    }
    if (r < RP) red[r][c4] = acc;
    if (tid < D) {
        const float zn = z[h * D + tid] + fk[tid];   // eq. (19)
        z[h * D + tid] = zn;
        dz[tid] = fq[tid] * zn;
    }
    __syncthreads();
    if (tid < 32) {
        float a = 0.f;
        for (int d = tid; d < D; d += 32) a += dz[d];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
        if (tid == 0) den_s = a;
    }
    __syncthreads();
    if (tid < M) {
        const float *redf = reinterpret_cast<const float *>(red);
        float num = 0.f;
#pragma unroll 4
        for (int rr = 0; rr < RP && rr < D; ++rr) num += redf[rr * M + tid];
        y[h * M + tid] = from_f32<T>(num / den_s);
    }
}

template <typename T, int D, int M>
cudaError_t launch_decode(const Problem &p) {
    const cudaError_t e = launch_pdl(decode_kernel<T, D, M>, dim3((unsigned)p.BH), dim3(kThreads), 0, p.stream, 0u,
                                     (const T *)p.q, (const T *)p.k, (const T *)p.v, (T *)p.out, p.S, p.z);
    count_launches(1);
    return e;
}

template <typename T, int D>
cudaError_t decode_m(const Problem &p) {
    switch (p.M) {
        case 16: return launch_decode<T, D, 16>(p);
        case 32: return launch_decode<T, D, 32>(p);
        case 64: return launch_decode<T, D, 64>(p);
        case 128: return launch_decode<T, D, 128>(p);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t decode_dm(const Problem &p) {
    switch (p.D) {
        case 16: return decode_m<T, 16>(p);
        case 32: return decode_m<T, 32>(p);
        case 64: return decode_m<T, 64>(p);
        case 128: return decode_m<T, 128>(p);
    }
    return cudaErrorInvalidValue;
}

int nc_nsplit(long long BH, int N, int sm_count) {
    long long want = (2LL * std::max(sm_count, 1) + BH - 1) / BH;
    long long most = (N + kCs - 1) / kCs;
    return (int)std::max(1LL, std::min(want, std::min(most, 16LL)));
}

template <typename T>
cudaError_t simt_noncausal_t(const Problem &p, const DeviceInfo &dev) {
    const int nsplit = nc_nsplit(p.BH, p.N, dev.sm_count);
    const int L = (p.N + nsplit - 1) / nsplit;
    const int ldq = p.D + 1;
    size_t sm1 = sizeof(float) * ((size_t)p.D * p.M + p.D + kCs * ldq + (size_t)kCs * p.M);
    size_t sm2 = sizeof(float) * ((size_t)p.D * p.M + p.D + kCs * ldq + kCs);
    cudaError_t e = cudaFuncSetAttribute(nc_reduce_simt_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(nc_readout_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm2);
    if (e != cudaSuccess) return e;
    nc_reduce_simt_kernel<T><<<dim3((unsigned)p.BH, nsplit), kThreads, sm1, p.stream>>>(
        (const T *)p.k, (const T *)p.v, (float *)p.ws, p.N, p.D, p.M, nsplit, L,
        (long long)(p.ws_bytes / sizeof(float)), dev.err_word, g_inject_bounds);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int R = 256;
    const int nrb = (p.N + R - 1) / R;
    nc_readout_simt_kernel<T><<<dim3((unsigned)p.BH, nrb), kThreads, sm2, p.stream>>>(
        (const T *)p.q, (const float *)p.ws, (T *)p.out, p.N, p.D, p.M, nsplit, R,
        (long long)(p.ws_bytes / sizeof(float)), dev.err_word);
    count_launches(1);
    return cudaGetLastError();
}

template <typename T>
cudaError_t simt_causal_t(const Problem &p) {
    const size_t smem = causal_smem_bytes(p.D, p.M);
    cudaError_t e = cudaFuncSetAttribute(causal_simt_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    causal_simt_kernel<T><<<(unsigned)p.BH, kThreads, smem, p.stream>>>(
        (const T *)p.q, (const T *)p.k, (const T *)p.v, (T *)p.out, p.S, p.z, p.N, p.D, p.M, p.lens,
        p.H > 0 ? p.H : 1);
    count_launches(1);
    return cudaGetLastError();
}

// T recurrent steps of sec. 3.4 eqs. (18)-(20) in one launch, one CTA per
// head: the head's state is read into registers once (same thread layout as
// decode_kernel), updated and read out T times, and written back once, so the
// steps cost only their q, k, v, y traffic.  Inputs are step-major:
// q, k [T][BH][D], v, y [T][BH][M].  Batch entry b runs steps[b] steps (all
// T if steps is null); its later outputs are left untouched.
template <typename T, int D, int M>
__global__ void __launch_bounds__(kThreads)
decode_steps_kernel(const T *__restrict__ q, const T *__restrict__ k, const T *__restrict__ v,
                    T *__restrict__ y, float *__restrict__ S, float *__restrict__ z,
                    const int *__restrict__ steps, int Tn, long long BH, int H)
{
    constexpr int C4 = M / 4;
    constexpr int RP = kThreads / C4;
    constexpr int NR = (D + RP - 1) / RP;
    __shared__ float fq[D], fk[D], vs[M], dz[D];
    __shared__ float4 red[RP][C4];
    __shared__ float den_s;
    const long long h = blockIdx.x;
    const int tid = threadIdx.x;
    const int c4 = tid % C4, r = tid / C4;
    pdl_wait_cta();
    const int nsteps = steps ? max(0, min(Tn, steps[h / H])) : Tn;

    float4 s[NR];
    float4 *Sh = reinterpret_cast<float4 *>(S + h * D * M);
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int d = r + i * RP;
        if (d < D) s[i] = Sh[d * C4 + c4];
    }
    float zr = tid < D ? z[h * D + tid] : 0.f;
    // the inputs of the next kPre steps are in flight while a step runs: each
    // thread prefetches its own element of q, k (tid < D) and v (tid < M)
    constexpr int kPre = 8;
    float pq[kPre], pk[kPre], pv[kPre];
    auto fetch = [&](int t, float &a, float &b, float &c) {
        if (t < nsteps) {
            const long long row = (long long)t * BH + h;
            a = tid < D ? to_f32(q[row * D + tid]) : 0.f;
            b = tid < D ? to_f32(k[row * D + tid]) : 0.f;
            c = tid < M ? to_f32(v[row * M + tid]) : 0.f;
        }
    };
#pragma unroll
    for (int u = 0; u < kPre; ++u) fetch(u, pq[u], pk[u], pv[u]);
    for (int t0 = 0; t0 < nsteps; t0 += kPre) {
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
            const int t = t0 + u;
            if (t >= nsteps) break;   // CTA-uniform
            const long long row = (long long)t * BH + h;
            if (tid < D) {
                fq[tid] = phi_accurate(pq[u]);
                fk[tid] = phi_accurate(pk[u]);
            }
            if (tid < M) vs[tid] = pv[u];
            fetch(t + kPre, pq[u], pk[u], pv[u]);
            __syncthreads();
            const float4 v4 = make_float4(vs[4 * c4], vs[4 * c4 + 1], vs[4 * c4 + 2], vs[4 * c4 + 3]);
            float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int i = 0; i < NR; ++i) {
                const int d = r + i * RP;
                if (d < D) {
                    const float a = fk[d], b = fq[d];
                    float4 w4 = s[i];
                    w4.x = fmaf(a, v4.x, w4.x);      // eq. (18)
                    w4.y = fmaf(a, v4.y, w4.y);
                    w4.z = fmaf(a, v4.z, w4.z);
                    w4.w = fmaf(a, v4.w, w4.w);
                    s[i] = w4;
                    acc.x = fmaf(b, w4.x, acc.x);    // eq. (20) numerator, updated state
                    acc.y = fmaf(b, w4.y, acc.y);
                    acc.z = fmaf(b, w4.z, acc.z);
                    acc.w = fmaf(b, w4.w, acc.w);
                }
            }
            if (r < RP) red[r][c4] = acc;
            if (tid < D) {
                zr += fk[tid];                       // eq. (19)
                dz[tid] = fq[tid] * zr;
            }
            __syncthreads();
            if (tid < 32) {
                float a = 0.f;
                for (int d = tid; d < D; d += 32) a += dz[d];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                if (tid == 0) den_s = a;
            }
            __syncthreads();
            if (tid < M) {
                const float *redf = reinterpret_cast<const float *>(red);
                float num = 0.f;
#pragma unroll 4
                for (int rr = 0; rr < RP && rr < D; ++rr) num += redf[rr * M + tid];
                y[row * M + tid] = from_f32<T>(num / den_s);
            }
        }
    }
#pragma unroll
    for (int i = 0; i < NR; ++i) {
        const int d = r + i * RP;
        if (d < D) Sh[d * C4 + c4] = s[i];
    }
    if (tid < D) z[h * D + tid] = zr;
}

template <typename T, int D, int M>
cudaError_t launch_decode_steps(const Problem &p, const int *steps, int Tn) {
    const cudaError_t e = launch_pdl(decode_steps_kernel<T, D, M>, dim3((unsigned)p.BH), dim3(kThreads), 0, p.stream,
                                     0u, (const T *)p.q, (const T *)p.k, (const T *)p.v, (T *)p.out, p.S, p.z, steps,
                                     Tn, p.BH, (int)(p.H > 0 ? p.H : 1));
    count_launches(1);
    return e;
}

template <typename T, int D>
cudaError_t decode_steps_m(const Problem &p, const int *steps, int Tn) {
    switch (p.M) {
        case 16: return launch_decode_steps<T, D, 16>(p, steps, Tn);
        case 32: return launch_decode_steps<T, D, 32>(p, steps, Tn);
        case 64: return launch_decode_steps<T, D, 64>(p, steps, Tn);
        case 128: return launch_decode_steps<T, D, 128>(p, steps, Tn);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t decode_steps_dm(const Problem &p, const int *steps, int Tn) {
    switch (p.D) {
        case 16: return decode_steps_m<T, 16>(p, steps, Tn);
        case 32: return decode_steps_m<T, 32>(p, steps, Tn);
        case 64: return decode_steps_m<T, 64>(p, steps, Tn);
        case 128: return decode_steps_m<T, 128>(p, steps, Tn);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t simt_noncausal_capped_t(const Problem &p, const DeviceInfo &dev, int max_splits) {
    const int nsplit = std::max(1, std::min(nc_nsplit(p.BH, p.N, dev.sm_count), max_splits));
    const int L = (p.N + nsplit - 1) / nsplit;
    const int ldq = p.D + 1;
    size_t sm1 = sizeof(float) * ((size_t)p.D * p.M + p.D + kCs * ldq + (size_t)kCs * p.M);
    size_t sm2 = sizeof(float) * ((size_t)p.D * p.M + p.D + kCs * ldq + kCs);
    cudaError_t e = cudaFuncSetAttribute(nc_reduce_simt_kernel<T>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm1);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(nc_readout_simt_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)sm2);
    if (e != cudaSuccess) return e;
    nc_reduce_simt_kernel<T><<<dim3((unsigned)p.BH, nsplit), kThreads, sm1, p.stream>>>(
        (const T *)p.k, (const T *)p.v, (float *)p.ws, p.N, p.D, p.M, nsplit, L,
        (long long)(p.ws_bytes / sizeof(float)), dev.err_word, g_inject_bounds);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    const int R = 256;
    const int nrb = (p.N + R - 1) / R;
    nc_readout_simt_kernel<T><<<dim3((unsigned)p.BH, nrb), kThreads, sm2, p.stream>>>(
        (const T *)p.q, (const float *)p.ws, (T *)p.out, p.N, p.D, p.M, nsplit, R,
        (long long)(p.ws_bytes / sizeof(float)), dev.err_word);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

cudaError_t simt_noncausal_capped(const Problem &p, const DeviceInfo &dev, int max_splits) {
    return p.dtype == LA_DTYPE_F32 ? simt_noncausal_capped_t<float>(p, dev, max_splits)
                                   : simt_noncausal_capped_t<__nv_bfloat16>(p, dev, max_splits);
}

size_t simt_noncausal_ws_bytes(const la_shape &s) {
    // Sized for the largest split count any device could pick (16 splits max).
    const long long BH = (long long)s.B * s.H;
    const int nsplit = std::min(16, std::max(1, (s.N + kCs - 1) / kCs));
    return sizeof(float) * (size_t)BH * nsplit * ((size_t)s.D * s.M + s.D);
}

cudaError_t simt_noncausal(const Problem &p, const DeviceInfo &dev) {
    return p.dtype == LA_DTYPE_F32 ? simt_noncausal_t<float>(p, dev)
                                   : simt_noncausal_t<__nv_bfloat16>(p, dev);
}

cudaError_t simt_causal(const Problem &p, const DeviceInfo &) {
    return p.dtype == LA_DTYPE_F32 ? simt_causal_t<float>(p) : simt_causal_t<__nv_bfloat16>(p);
}

cudaError_t decode_step(const Problem &p, const DeviceInfo &) {
    return p.dtype == LA_DTYPE_F32 ? decode_dm<float>(p) : decode_dm<__nv_bfloat16>(p);
}

cudaError_t decode_steps(const Problem &p, const int *steps, int Tn) {
    return p.dtype == LA_DTYPE_F32 ? decode_steps_dm<float>(p, steps, Tn) : decode_steps_dm<__nv_bfloat16>(p, steps, Tn);
}

}  // namespace la

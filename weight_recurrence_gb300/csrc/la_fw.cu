// la_fw.cu - CUDA-core kernels for the variants of kernelised linear attention:
// other feature maps, sum-normalised features and the delta update rule.
//
// Sources:
//  [TaR] "Transformers are RNNs" (Katharopoulos et al.): eq. (7) elu + 1,
//        sec. 3.2.1 (degree-2 polynomial kernel, exact feature map x x^T),
//        eqs. (10)-(12) and (18)-(20) (update, then read out).
//  [FWP] "Linear Transformers Are Secretly Fast Weight Programmers" (Schlag,
//        Irie, Schmidhuber): DPFP-nu, sum normalisation of phi(q) and phi(k),
//        and the update that replaces the value paired with a key by
//        beta v + (1 - beta) vbar:  S += phi(k) (beta (v - S^T phi(k)))^T.
//
// Per head the state S is F x M (F = feature width).  Every update rule here
// is separable along M: column m of S evolves from phi(k), v_m and beta alone
// (retrieval S^T phi(k) and read-out S^T phi(q) are per column too).  So:
//
// fw_causal_kernel - one CTA of 256 threads per (head, 16 state columns).
//   Per chunk of 32 tokens all threads stage the raw q, k rows, evaluate the
//   feature map into shared memory (sum-normalising the rows if asked), and,
//   with the TaR denominator, form den_t = phi(q_t) . z_t from a running
//   per-feature prefix of phi(k).  Then each warp walks the chunk's tokens on
//   its own: a warp owns two state columns, 16 lanes per column, each lane
//   holding E = F/16 entries of the column in registers.  A token costs a few
//   FMAs per lane and one (sum rule) or two (delta rule) 16-lane shuffle
//   reductions - no block-wide barrier inside a chunk.
//
// fw_nc_reduce_kernel / fw_nc_readout_kernel - the non-causal form ([TaR]
//   eq. (5) with the variant's phi and read-out): per (head, key split, 16
//   columns) partial sums of phi(K)^T V (and phi(K)^T 1) into the workspace,
//   then per (head, row block, 16 columns) the read-out.
//
// All arithmetic is fp32; phi of elu uses expf.  The feature index order is
// the one the state layout [B, H, F, M] exposes (see la.h).
#include <algorithm>

#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr int kFwThreads = 256;
constexpr int kFwL = 32;                       // tokens per chunk
constexpr int kFwG = 16;                       // lanes per state column
constexpr int kFwCols = kFwThreads / kFwG;     // state columns per CTA (16)
constexpr int kFwWarps = kFwThreads / 32;

// Feature f < F of the raw row x (fp32, length D); 0 for padding f >= F.
__device__ __forceinline__ float feature_at(const float *x, int f, int fm, int D, int nu, int F) {
    if (f >= F) return 0.f;
    if (fm == LA_FM_ELU1) return phi_accurate(x[f]);
    if (fm == LA_FM_DPFP) {
        // r = [relu(x), relu(-x)]; feature (s-1)*2D + i is r_i * r_{(i+s) mod 2D}
        const int twoD = 2 * D;
        const int s = f / twoD + 1, i = f - (s - 1) * twoD;
        int j = i + s;
        if (j >= twoD) j -= twoD;                // s <= nu < 2D
        const float a = i < D ? fmaxf(x[i], 0.f) : fmaxf(-x[i - D], 0.f);
        const float b = j < D ? fmaxf(x[j], 0.f) : fmaxf(-x[j - D], 0.f);
        return a * b;
    }
    const int a = f / D, b = f - a * D;          // degree-2 polynomial: x_a x_b
    return x[a] * x[b];
}

// feature_at on a raw row of dtype T (values converted as read).
template <typename T>
__device__ __forceinline__ float feature_raw(const T *x, int f, int fm, int D, int nu, int F) {
    if (f >= F) return 0.f;
    if (fm == LA_FM_ELU1) return phi_accurate(to_f32(x[f]));
    if (fm == LA_FM_DPFP) {
        const int twoD = 2 * D;
        const int s = f / twoD + 1, i = f - (s - 1) * twoD;
        int j = i + s;
        if (j >= twoD) j -= twoD;                // s <= nu < 2D
        const float a = i < D ? fmaxf(to_f32(x[i]), 0.f) : fmaxf(-to_f32(x[i - D]), 0.f);
        const float b = j < D ? fmaxf(to_f32(x[j]), 0.f) : fmaxf(-to_f32(x[j - D]), 0.f);
        return a * b;
    }
    const int a = f / D, b = f - a * D;          // degree-2 polynomial: x_a x_b
    return to_f32(x[a]) * to_f32(x[b]);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

struct FwArgs {
    const void *q, *k, *v, *beta;
    void *out;               // may be null (state only)
    float *S, *z;            // [BH, F, M], [BH, F] or null
    int N, D, M, F, Fp;      // Fp: padded feature width of the kernel's layout
    int fm, nu, norm;
    int cpc;                 // causal kernel: state columns per CTA
};

// Loads `rows` raw rows of q and k (and of v's 16-column slice) for the chunk
// starting at token t0, and evaluates the feature map into fq, fk [L][Fp];
// sum-normalises the rows for LA_NORM_SUM.  Rows past `rows` are zero.
template <typename T>
__device__ void chunk_features(const FwArgs &a, long long h, int t0, int rows, float *xq, float *xk,
                               float *fq, float *fk, bool want_q) {
    const int tid = threadIdx.x;
    const T *qh = (const T *)a.q + h * a.N * a.D, *kh = (const T *)a.k + h * a.N * a.D;
    for (int idx = tid; idx < kFwL * a.D; idx += kFwThreads) {
        const int t = idx / a.D;
        const bool ok = t < rows;
        xk[idx] = ok ? to_f32(kh[(long long)t0 * a.D + idx]) : 0.f;
        if (want_q) xq[idx] = ok ? to_f32(qh[(long long)t0 * a.D + idx]) : 0.f;
    }
    __syncthreads();
    for (int idx = tid; idx < kFwL * a.Fp; idx += kFwThreads) {
        const int t = idx / a.Fp, f = idx - t * a.Fp;
        const bool ok = t < rows;
        fk[idx] = ok ? feature_at(xk + t * a.D, f, a.fm, a.D, a.nu, a.F) : 0.f;
        if (want_q) fq[idx] = ok ? feature_at(xq + t * a.D, f, a.fm, a.D, a.nu, a.F) : 0.f;
    }
    __syncthreads();
    if (a.norm == LA_NORM_SUM) {
        const int warp = tid >> 5, lane = tid & 31;
        for (int r = warp; r < 2 * kFwL; r += kFwWarps) {
            if (r >= kFwL && !want_q) continue;
            float *row = (r < kFwL ? fk : fq) + (r % kFwL) * a.Fp;
            float s = 0.f;
            for (int f = lane; f < a.Fp; f += 32) s += row[f];
            s = warp_sum(s);
            if (s > 0.f)
                for (int f = lane; f < a.Fp; f += 32) row[f] = row[f] / s;
        }
        __syncthreads();
    }
}

// 16-byte asynchronous copy global -> shared; src_bytes < 16 zero-fills the
// rest (0: nothing is read, the source address is then only a placeholder).
__device__ __forceinline__ void cp_async16(void *dst, const void *src, int src_bytes) {
    const uint32_t d = (uint32_t)__cvta_generic_to_shared(dst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(d), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Raw inputs of one chunk as they are in memory (dtype T): q, k rows [L][D],
// the CTA's 16 value columns [L][16], beta [L].
template <typename T>
struct RawChunk {
    T *q, *k, *v;
    float *b;
};

// Causal form of every variant.  A warp owns CW = 32 / G state columns, G
// lanes per column; lane = cl * G + g owns column warp * CW + cl of the CTA's
// block and the column entries f = 4 (e4 G + g) + j (e4 < E / 4, j < 4), so a
// lane's features come in float4 loads and the G lanes of a column read one
// contiguous span (no bank conflicts; the other columns of the warp read the
// same addresses).  A CTA holds a.cpc columns (one warp per CW of them) and
// evaluates its head's features once per chunk.
// Per chunk: the raw rows of the next chunk are copied asynchronously into the
// other raw buffer while this chunk's tokens run.
template <typename T, int G, int E, bool DELTA, bool DEN>
__global__ void __launch_bounds__(kFwThreads)
fw_causal_kernel(FwArgs a)
{
    static_assert(E % 4 == 0 && 32 % G == 0, "lane layout");
    constexpr int CW = 32 / G;
    extern __shared__ __align__(16) float sm[];
    const int nthr = blockDim.x, nwarps = nthr >> 5;
    const int cpc = a.cpc;                                     // columns of this CTA
    const int rawqk = kFwL * a.D * (int)sizeof(T);            // bytes of one raw q or k chunk
    const int rawv = kFwL * cpc * (int)sizeof(T);
    const int rawb = kFwL * 4;
    const int rawsz = 2 * rawqk + rawv + rawb;                 // multiple of 16
    uint8_t *rawbase = reinterpret_cast<uint8_t *>(sm);
    auto raw = [&](int buf) {
        uint8_t *p = rawbase + buf * rawsz;
        return RawChunk<T>{reinterpret_cast<T *>(p), reinterpret_cast<T *>(p + rawqk),
                           reinterpret_cast<T *>(p + 2 * rawqk), reinterpret_cast<float *>(p + 2 * rawqk + rawv)};
    };
    float *fq = reinterpret_cast<float *>(rawbase + 2 * rawsz);   // [L][Fp] features
    float *fk = fq + kFwL * a.Fp;             // [L][Fp]
    float *ys = fk + kFwL * a.Fp;             // [L][cpc] outputs of the chunk
    float *den = ys + kFwL * cpc;             // [L]
    float *dpart = den + kFwL;                // [8 warps][L]
    float *zs = dpart + kFwWarps * kFwL;      // [Fp] running z (DEN)

    const long long h = blockIdx.x;
    const int m0 = blockIdx.y * cpc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cl = lane / G, g = lane % G;
    const int mc = warp * CW + cl;            // column within the CTA's block

    const T *qh = (const T *)a.q + h * a.N * a.D, *kh = (const T *)a.k + h * a.N * a.D;
    const T *vh = (const T *)a.v + h * a.N * a.M;
    const T *bh = DELTA ? (const T *)a.beta + h * a.N : nullptr;
    T *oh = a.out ? (T *)a.out + h * a.N * a.M : nullptr;
    const bool want_q = oh != nullptr;

    // copies of chunk t0's raw rows into buffer `buf` (one commit group);
    // beta (whose rows need not be 16-byte aligned) is loaded into a register
    // by the first 32 threads and stored after the current chunk's tokens
    auto issue = [&](int buf, int t0, float &bnext) {
        const int rows = min(kFwL, a.N - t0);
        RawChunk<T> r = raw(buf);
        const int rowb = a.D * (int)sizeof(T);                 // multiple of 32 bytes
        for (int vi = tid; vi < rawqk / 16; vi += nthr) {
            const int row = vi * 16 / rowb;
            const bool ok = row < rows;
            const size_t off = (size_t)t0 * rowb + (size_t)vi * 16;
            cp_async16(reinterpret_cast<uint8_t *>(r.k) + vi * 16,
                       ok ? reinterpret_cast<const uint8_t *>(kh) + off : reinterpret_cast<const uint8_t *>(kh),
                       ok ? 16 : 0);
            if (want_q)
                cp_async16(reinterpret_cast<uint8_t *>(r.q) + vi * 16,
                           ok ? reinterpret_cast<const uint8_t *>(qh) + off : reinterpret_cast<const uint8_t *>(qh),
                           ok ? 16 : 0);
        }
        const int vpr = cpc * (int)sizeof(T) / 16;             // 16-byte pieces per value row
        for (int vi = tid; vi < kFwL * vpr; vi += nthr) {
            const int row = vi / vpr, part = vi - row * vpr;
            const bool ok = row < rows;
            const T *src = ok ? vh + (size_t)(t0 + row) * a.M + m0 : vh;
            cp_async16(reinterpret_cast<uint8_t *>(r.v) + vi * 16,
                       reinterpret_cast<const uint8_t *>(src) + (ok ? part * 16 : 0), ok ? 16 : 0);
        }
        cp_async_commit();
        if (DELTA && tid < kFwL) bnext = tid < rows ? to_f32(bh[t0 + tid]) : 0.f;
    };

    // carried-in state, staged through shared memory (the fq, fk buffers) for coalesced loads
    float s[E];
    auto ent = [&](int e) { return 4 * ((e >> 2) * G + g) + (e & 3); };   // feature index of entry e
    {
        float *stage = fq;                    // [Fp][cpc], fits in 2 [L][Fp] (cpc <= 64)
        for (int idx = tid; idx < a.Fp * cpc; idx += nthr) {
            const int f = idx / cpc, cc = idx - f * cpc;
            stage[idx] = (a.S && f < a.F) ? a.S[(h * a.F + f) * a.M + m0 + cc] : 0.f;
        }
        if (DEN)
            for (int f = tid; f < a.Fp; f += nthr) zs[f] = (a.z && f < a.F) ? a.z[h * a.F + f] : 0.f;
        __syncthreads();
#pragma unroll
        for (int e = 0; e < E; ++e) s[e] = stage[ent(e) * cpc + mc];
    }

    float bnext = 0.f;
    if (a.N > 0) issue(0, 0, bnext);
    if (DELTA && tid < kFwL) raw(0).b[tid] = bnext;
    int buf = 0;
    for (int t0 = 0; t0 < a.N; t0 += kFwL, buf ^= 1) {
        const int rows = min(kFwL, a.N - t0);
        const RawChunk<T> r = raw(buf);
        cp_async_wait_all();
        __syncthreads();                      // chunk t0's raw rows (and beta) are in shared memory
        // features of the chunk (rows past `rows` are zero)
        for (int idx = tid; idx < kFwL * a.Fp; idx += nthr) {
            const int t = idx / a.Fp, f = idx - t * a.Fp;
            float vk = 0.f, vq = 0.f;
            if (t < rows) {
                vk = feature_raw<T>(r.k + t * a.D, f, a.fm, a.D, a.nu, a.F);
                if (want_q) vq = feature_raw<T>(r.q + t * a.D, f, a.fm, a.D, a.nu, a.F);
            }
            fk[idx] = vk;
            if (want_q) fq[idx] = vq;
        }
        __syncthreads();
        if (a.norm == LA_NORM_SUM) {
            for (int rr = warp; rr < 2 * kFwL; rr += nwarps) {
                if (rr >= kFwL && !want_q) continue;
                float *row = (rr < kFwL ? fk : fq) + (rr % kFwL) * a.Fp;
                float sum = 0.f;
                for (int f = lane; f < a.Fp; f += 32) sum += row[f];
                sum = warp_sum(sum);
                if (sum > 0.f)
                    for (int f = lane; f < a.Fp; f += 32) row[f] = row[f] / sum;
            }
            __syncthreads();
        }
        // the next chunk's raw rows stream in while this chunk's tokens run (its
        // buffer was last read by the previous chunk's tokens, before the barriers above)
        if (t0 + kFwL < a.N) issue(buf ^ 1, t0 + kFwL, bnext);

        if (DEN && want_q) {
            // den_t = phi(q_t) . (z_prev + sum_{s <= t} phi(k_s)): warp w owns the
            // features w*32 + lane + 32 nwarps p and keeps their running z
            if (lane == 0)
                for (int t = 0; t < kFwL; ++t) dpart[warp * kFwL + t] = 0.f;
            __syncwarp();
            for (int f0 = warp * 32; f0 < a.Fp; f0 += nthr) {   // warp-uniform
                const int f = f0 + lane;
                const bool ok = f < a.Fp;
                float zf = ok ? zs[f] : 0.f;
                for (int t = 0; t < rows; ++t) {
                    zf += ok ? fk[t * a.Fp + f] : 0.f;
                    const float p = warp_sum(ok ? fq[t * a.Fp + f] * zf : 0.f);
                    if (lane == 0) dpart[warp * kFwL + t] += p;
                }
                if (ok) zs[f] = zf;
            }
            __syncthreads();
            if (tid < kFwL) {
                float d = 0.f;
                for (int w = 0; w < nwarps; ++w) d += dpart[w * kFwL + tid];
                den[tid] = d;
            }
            __syncthreads();
        } else if (DEN) {
            for (int f = tid; f < a.Fp; f += nthr) {
                float zf = zs[f];
                for (int t = 0; t < rows; ++t) zf += fk[t * a.Fp + f];
                zs[f] = zf;
            }
        }

        // the recurrence over the chunk's tokens, each warp on its own columns
        auto dot = [&](const float *row, float &acc0, float &acc1) {   // row points at [f = 0]
#pragma unroll
            for (int e4 = 0; e4 < E / 4; ++e4) {
                const float4 x = *reinterpret_cast<const float4 *>(row + 4 * (e4 * G + g));
                acc0 = fmaf(x.x, s[4 * e4], acc0);
                acc1 = fmaf(x.y, s[4 * e4 + 1], acc1);
                acc0 = fmaf(x.z, s[4 * e4 + 2], acc0);
                acc1 = fmaf(x.w, s[4 * e4 + 3], acc1);
            }
        };
        if (DELTA) {
            // the read-out of token t-1 and the retrieval of token t both read the
            // state after token t-1, so their reductions run together
            for (int t = 0; t <= rows; ++t) {
                const bool has_k = t < rows, has_y = want_q && t > 0;   // warp-uniform
                float kr[E];
                float r0 = 0.f, r1 = 0.f, y0 = 0.f, y1 = 0.f;
                if (has_k) {
                    const float *fkt = fk + t * a.Fp;
#pragma unroll
                    for (int e4 = 0; e4 < E / 4; ++e4) {
                        const float4 x = *reinterpret_cast<const float4 *>(fkt + 4 * (e4 * G + g));
                        kr[4 * e4] = x.x;
                        kr[4 * e4 + 1] = x.y;
                        kr[4 * e4 + 2] = x.z;
                        kr[4 * e4 + 3] = x.w;
                    }
#pragma unroll
                    for (int e = 0; e < E; e += 2) {
                        r0 = fmaf(kr[e], s[e], r0);
                        r1 = fmaf(kr[e + 1], s[e + 1], r1);
                    }
                }
                if (has_y) dot(fq + (t - 1) * a.Fp, y0, y1);
                float rr = r0 + r1, y = y0 + y1;
#pragma unroll
                for (int o = G / 2; o > 0; o >>= 1) {
                    rr += __shfl_xor_sync(0xffffffffu, rr, o);
                    y += __shfl_xor_sync(0xffffffffu, y, o);
                }
                if (has_y && g == 0) ys[(t - 1) * cpc + mc] = y;
                if (has_k) {
                    const float u = r.b[t] * (to_f32(r.v[t * cpc + mc]) - rr);
#pragma unroll
                    for (int e = 0; e < E; ++e) s[e] = fmaf(kr[e], u, s[e]);
                }
            }
        } else {
#pragma unroll 2
            for (int t = 0; t < rows; ++t) {
                const float *fkt = fk + t * a.Fp;
                const float vt = to_f32(r.v[t * cpc + mc]);
#pragma unroll
                for (int e4 = 0; e4 < E / 4; ++e4) {
                    const float4 x = *reinterpret_cast<const float4 *>(fkt + 4 * (e4 * G + g));
                    s[4 * e4] = fmaf(x.x, vt, s[4 * e4]);
                    s[4 * e4 + 1] = fmaf(x.y, vt, s[4 * e4 + 1]);
                    s[4 * e4 + 2] = fmaf(x.z, vt, s[4 * e4 + 2]);
                    s[4 * e4 + 3] = fmaf(x.w, vt, s[4 * e4 + 3]);
                }
                if (want_q) {
                    float y0 = 0.f, y1 = 0.f;            // read-out S^T phi(q), after the update
                    dot(fq + t * a.Fp, y0, y1);
                    float y = y0 + y1;
#pragma unroll
                    for (int o = G / 2; o > 0; o >>= 1) y += __shfl_xor_sync(0xffffffffu, y, o);
                    if (g == 0) ys[t * cpc + mc] = DEN ? y / den[t] : y;
                }
            }
        }
        __syncthreads();
        if (want_q)
            for (int idx = tid; idx < rows * cpc; idx += nthr) {
                const int t = idx / cpc, cc = idx - t * cpc;
                oh[(long long)(t0 + t) * a.M + m0 + cc] = from_f32<T>(ys[idx]);
            }
        if (DELTA && tid < kFwL && t0 + kFwL < a.N) raw(buf ^ 1).b[tid] = bnext;
        // the next iteration's first barrier orders these stores before any reuse
    }

    if (a.S) {
        __syncthreads();
        float *stage = fq;
#pragma unroll
        for (int e = 0; e < E; ++e) stage[ent(e) * cpc + mc] = s[e];
        __syncthreads();
        for (int idx = tid; idx < a.F * cpc; idx += nthr) {
            const int f = idx / cpc, cc = idx - f * cpc;
            a.S[(h * a.F + f) * a.M + m0 + cc] = stage[idx];
        }
    }
    if (DEN && a.z && blockIdx.y == 0) {
        __syncthreads();
        for (int f = tid; f < a.F; f += nthr) a.z[h * a.F + f] = zs[f];
    }
}

// Non-causal, phase 1: partial sums over keys [sp*L, ...) of one head for the
// CTA's 16 columns: acc[f][c] = sum_j phi(K_j)_f V_{j, m0+c} and, for the CTA
// of the first column block, ksum[f] = sum_j phi(K_j)_f.
// Workspace layout: ws[(h * nsplit + sp) * (F*M + F)]: F x M row-major, then F.
template <typename T, int E>
__global__ void __launch_bounds__(kFwThreads)
fw_nc_reduce_kernel(FwArgs a, float *__restrict__ ws, int nsplit, int L)
{
    extern __shared__ float sm[];
    float *xk = sm;                           // [Lc][D]
    float *fk = xk + kFwL * a.D;              // [Lc][Fp]
    float *vs = fk + kFwL * a.Fp;             // [Lc][16]
    const long long h = blockIdx.x;
    const int sp = blockIdx.y, m0 = blockIdx.z * kFwCols;
    const int tid = threadIdx.x, c = tid & 15, fg = tid >> 4;
    const int t_begin = sp * L, t_end = min(a.N, t_begin + L);
    const T *vh = (const T *)a.v + h * a.N * a.M;
    float acc[E], ks[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = ks[e] = 0.f;
    for (int t0 = t_begin; t0 < t_end; t0 += kFwL) {
        const int rows = min(kFwL, t_end - t0);
        __syncthreads();
        for (int idx = tid; idx < kFwL * kFwCols; idx += kFwThreads) {
            const int t = idx / kFwCols, cc = idx - t * kFwCols;
            vs[idx] = t < rows ? to_f32(vh[(long long)(t0 + t) * a.M + m0 + cc]) : 0.f;
        }
        chunk_features<T>(a, h, t0, rows, nullptr, xk, nullptr, fk, false);
        for (int t = 0; t < rows; ++t) {
            const float vt = vs[t * kFwCols + c];
#pragma unroll
            for (int e = 0; e < E; ++e) {
                const float f = fk[t * a.Fp + fg + kFwG * e];
                acc[e] = fmaf(f, vt, acc[e]);
                ks[e] += f;
            }
        }
    }
    float *dst = ws + (h * nsplit + sp) * (long long)(a.F * a.M + a.F);
#pragma unroll
    for (int e = 0; e < E; ++e) {
        const int f = fg + kFwG * e;
        if (f < a.F) {
            dst[f * a.M + m0 + c] = acc[e];
            if (blockIdx.z == 0 && c == 0) dst[a.F * a.M + f] = ks[e];
        }
    }
}

// Non-causal, phase 2: sum the head's partials for the CTA's 16 columns, then
// y_i = phi(Q_i)^T KV (/ phi(Q_i)^T ksum) for the rows [r0, r0 + R).
template <typename T>
__global__ void __launch_bounds__(kFwThreads)
fw_nc_readout_kernel(FwArgs a, const float *__restrict__ ws, int nsplit, int R)
{
    extern __shared__ float sm[];
    float *xq = sm;                           // [L][D]
    float *fq = xq + kFwL * a.D;              // [L][Fp]
    float *kv = fq + kFwL * a.Fp;             // [Fp][16]
    float *ks = kv + a.Fp * kFwCols;          // [Fp]
    float *den = ks + a.Fp;                   // [L]
    const long long h = blockIdx.x;
    const int m0 = blockIdx.z * kFwCols;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int r0 = blockIdx.y * R, r1 = min(a.N, r0 + R);
    const float *src = ws + h * nsplit * (long long)(a.F * a.M + a.F);
    for (int idx = tid; idx < a.Fp * kFwCols; idx += kFwThreads) {
        const int f = idx / kFwCols, cc = idx - f * kFwCols;
        float s = 0.f;
        if (f < a.F)
            for (int sp = 0; sp < nsplit; ++sp) s += src[sp * (long long)(a.F * a.M + a.F) + f * a.M + m0 + cc];
        kv[idx] = s;
    }
    for (int f = tid; f < a.Fp; f += kFwThreads) {
        float s = 0.f;
        if (f < a.F)
            for (int sp = 0; sp < nsplit; ++sp) s += src[sp * (long long)(a.F * a.M + a.F) + a.F * a.M + f];
        ks[f] = s;
    }
    T *oh = (T *)a.out + h * a.N * a.M;
    const bool use_den = a.norm == LA_NORM_DEN;
    FwArgs aq = a;
    aq.k = a.q;                               // the query rows go through the key staging path
    for (int t0 = r0; t0 < r1; t0 += kFwL) {
        const int rows = min(kFwL, r1 - t0);
        __syncthreads();
        chunk_features<T>(aq, h, t0, rows, nullptr, xq, nullptr, fq, false);
        if (use_den) {
            for (int t = warp; t < rows; t += kFwWarps) {
                float d = 0.f;
                for (int f = lane; f < a.Fp; f += 32) d = fmaf(fq[t * a.Fp + f], ks[f], d);
                d = warp_sum(d);
                if (lane == 0) den[t] = d;
            }
            __syncthreads();
        }
        for (int idx = tid; idx < rows * kFwCols; idx += kFwThreads) {
            const int t = idx / kFwCols, cc = idx - t * kFwCols;
            float y = 0.f;
            for (int f = 0; f < a.Fp; ++f) y = fmaf(fq[t * a.Fp + f], kv[f * kFwCols + cc], y);
            if (use_den) y = y / den[t];
            oh[(long long)(t0 + t) * a.M + m0 + cc] = from_f32<T>(y);
        }
    }
}

// E = entries per lane for a feature width F (F <= 16 * 32), padded to an
// instantiated value; Fp = 16 * E.
int entries_for(int F) {
    const int e = (F + kFwG - 1) / kFwG;
    for (int cand : {1, 2, 4, 8, 16, 24, 32})
        if (e <= cand) return cand;
    return 0;
}

template <typename T>
size_t causal_smem(int D, int Fp, int cpc) {
    const size_t raw = (size_t)2 * kFwL * D * sizeof(T) + (size_t)kFwL * cpc * sizeof(T) + kFwL * 4;
    return 2 * raw + sizeof(float) * ((size_t)2 * kFwL * Fp + (size_t)kFwL * cpc + kFwL + kFwWarps * kFwL + Fp);
}

// Lane layout of the causal kernel for feature width F: G lanes per column and
// E entries per lane, Fp = G * E >= F; the instantiated (G, E) pairs.
struct CausalLayout {
    int G, E;
};
CausalLayout causal_layout(int F) {
    static const CausalLayout kLayouts[] = {{4, 4}, {4, 8}, {4, 16}, {4, 24}, {4, 32},
                                            {8, 24}, {8, 32}, {16, 24}, {16, 32}};
    for (const CausalLayout &l : kLayouts)
        if (l.G * l.E >= F) return l;
    return {0, 0};
}

template <typename T, int G, int E, bool DELTA, bool DEN>
cudaError_t launch_causal_ge(FwArgs a, long long BH, cudaStream_t st) {
    constexpr int CW = 32 / G;
    a.Fp = G * E;
    a.cpc = std::min(a.M, kFwWarps * CW);            // columns per CTA, one warp per CW columns
    const size_t smem = causal_smem<T>(a.D, a.Fp, a.cpc);
    cudaError_t e = cudaFuncSetAttribute(fw_causal_kernel<T, G, E, DELTA, DEN>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fw_causal_kernel<T, G, E, DELTA, DEN><<<dim3((unsigned)BH, a.M / a.cpc), 32 * (a.cpc / CW), smem, st>>>(a);
    count_launches(1);
    return cudaGetLastError();
}

template <typename T, bool DELTA, bool DEN>
cudaError_t launch_causal_upd(const FwArgs &a, long long BH, cudaStream_t st) {
    const CausalLayout l = causal_layout(a.F);
    switch (l.G * 100 + l.E) {
        case 404: return launch_causal_ge<T, 4, 4, DELTA, DEN>(a, BH, st);
        case 408: return launch_causal_ge<T, 4, 8, DELTA, DEN>(a, BH, st);
        case 416: return launch_causal_ge<T, 4, 16, DELTA, DEN>(a, BH, st);
        case 424: return launch_causal_ge<T, 4, 24, DELTA, DEN>(a, BH, st);
        case 432: return launch_causal_ge<T, 4, 32, DELTA, DEN>(a, BH, st);
        case 824: return launch_causal_ge<T, 8, 24, DELTA, DEN>(a, BH, st);
        case 832: return launch_causal_ge<T, 8, 32, DELTA, DEN>(a, BH, st);
        case 1624: return launch_causal_ge<T, 16, 24, DELTA, DEN>(a, BH, st);
        case 1632: return launch_causal_ge<T, 16, 32, DELTA, DEN>(a, BH, st);
    }
    return cudaErrorInvalidValue;
}

template <typename T>
cudaError_t fw_causal_t(const FwArgs &a, long long BH, int update, cudaStream_t st) {
    if (update == LA_UPDATE_DELTA) return launch_causal_upd<T, true, false>(a, BH, st);
    if (a.norm == LA_NORM_DEN) return launch_causal_upd<T, false, true>(a, BH, st);
    return launch_causal_upd<T, false, false>(a, BH, st);
}

int fw_nsplit(long long BH, int N, int M, int sm_count) {
    const long long ctas = BH * (M / kFwCols);
    long long want = (2LL * std::max(sm_count, 1) + ctas - 1) / ctas;
    long long most = (N + kFwL - 1) / kFwL;
    return (int)std::max(1LL, std::min(want, std::min(most, 16LL)));
}

template <typename T, int E>
cudaError_t launch_nc_reduce_e(const FwArgs &a, long long BH, float *ws, int nsplit, int L, cudaStream_t st) {
    const size_t smem = sizeof(float) * ((size_t)kFwL * a.D + (size_t)kFwL * a.Fp + kFwL * kFwCols);
    cudaError_t e = cudaFuncSetAttribute(fw_nc_reduce_kernel<T, E>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    fw_nc_reduce_kernel<T, E><<<dim3((unsigned)BH, nsplit, a.M / kFwCols), kFwThreads, smem, st>>>(a, ws, nsplit, L);
    count_launches(1);
    return cudaGetLastError();
}

template <typename T>
cudaError_t fw_noncausal_t(const FwArgs &a, long long BH, void *ws, const DeviceInfo &dev, cudaStream_t st) {
    const int nsplit = fw_nsplit(BH, a.N, a.M, dev.sm_count);
    const int L = (a.N + nsplit - 1) / nsplit;
    float *w = (float *)ws;
    cudaError_t e = cudaErrorInvalidValue;
    switch (a.Fp / kFwG) {
        case 1: e = launch_nc_reduce_e<T, 1>(a, BH, w, nsplit, L, st); break;
        case 2: e = launch_nc_reduce_e<T, 2>(a, BH, w, nsplit, L, st); break;
        case 4: e = launch_nc_reduce_e<T, 4>(a, BH, w, nsplit, L, st); break;
        case 8: e = launch_nc_reduce_e<T, 8>(a, BH, w, nsplit, L, st); break;
        case 16: e = launch_nc_reduce_e<T, 16>(a, BH, w, nsplit, L, st); break;
        case 24: e = launch_nc_reduce_e<T, 24>(a, BH, w, nsplit, L, st); break;
        case 32: e = launch_nc_reduce_e<T, 32>(a, BH, w, nsplit, L, st); break;
    }
    if (e != cudaSuccess) return e;
    const int R = 128;
    const int nrb = (a.N + R - 1) / R;
    const size_t smem = sizeof(float) * ((size_t)kFwL * a.D + (size_t)kFwL * a.Fp + (size_t)a.Fp * kFwCols +
                                         a.Fp + kFwL);
    e = cudaFuncSetAttribute(fw_nc_readout_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    fw_nc_readout_kernel<T><<<dim3((unsigned)BH, nrb, a.M / kFwCols), kFwThreads, smem, st>>>(a, w, nsplit, R);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

int fw_feature_dim(const la_variant &v, int D) {
    if (D <= 0) return 0;
    switch (v.feature_map) {
        case LA_FM_ELU1: return D;
        case LA_FM_DPFP: return (v.nu >= 1 && v.nu < 2 * D) ? 2 * D * v.nu : 0;
        case LA_FM_POLY2: return D * D;
    }
    return 0;
}

la_status fw_check_variant(const la_variant &v, int D) {
    if (v.feature_map != LA_FM_ELU1 && v.feature_map != LA_FM_DPFP && v.feature_map != LA_FM_POLY2)
        return LA_ERR_INVALID_ARG;
    if (v.norm != LA_NORM_DEN && v.norm != LA_NORM_SUM && v.norm != LA_NORM_NONE) return LA_ERR_INVALID_ARG;
    if (v.update != LA_UPDATE_SUM && v.update != LA_UPDATE_DELTA) return LA_ERR_INVALID_ARG;
    if (v.feature_map == LA_FM_DPFP && (v.nu < 1 || v.nu >= 2 * D)) return LA_ERR_INVALID_ARG;
    const int F = fw_feature_dim(v, D);
    if (F <= 0 || F > kFwMaxFeatures) return LA_ERR_UNSUPPORTED;
    // DPFP features of a query can miss every key seen so far, making the
    // denominator zero; polynomial features can be negative, so their sum is
    // no normaliser; the delta rule needs |phi(k)|^2 <= 1 to stay bounded.
    if (v.feature_map == LA_FM_DPFP && v.norm == LA_NORM_DEN) return LA_ERR_UNSUPPORTED;
    if (v.feature_map == LA_FM_POLY2 && v.norm == LA_NORM_SUM) return LA_ERR_UNSUPPORTED;
    if (v.update == LA_UPDATE_DELTA && v.norm != LA_NORM_SUM) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

size_t fw_noncausal_ws_bytes(const la_shape &s, const la_variant &v) {
    const int F = fw_feature_dim(v, s.D);
    const long long BH = (long long)s.B * s.H;
    const int nsplit = std::min(16, std::max(1, (s.N + kFwL - 1) / kFwL));
    return sizeof(float) * (size_t)BH * nsplit * ((size_t)F * s.M + F);
}

static FwArgs make_args(const Problem &p, const void *beta, const la_variant &v) {
    const int F = fw_feature_dim(v, p.D);
    const int E = entries_for(F);
    return FwArgs{p.q, p.k, p.v, beta, p.out, p.S, p.z, p.N, p.D, p.M, F, E * kFwG, v.feature_map, v.nu, v.norm, 0};
}

cudaError_t fw_causal(const Problem &p, const void *beta, const la_variant &v) {
    const FwArgs a = make_args(p, beta, v);
    if (a.Fp == 0) return cudaErrorInvalidValue;
    return p.dtype == LA_DTYPE_F32 ? fw_causal_t<float>(a, p.BH, v.update, p.stream)
                                   : fw_causal_t<__nv_bfloat16>(a, p.BH, v.update, p.stream);
}

cudaError_t fw_noncausal(const Problem &p, const la_variant &v, const DeviceInfo &dev) {
    const FwArgs a = make_args(p, nullptr, v);
    if (a.Fp == 0) return cudaErrorInvalidValue;
    return p.dtype == LA_DTYPE_F32 ? fw_noncausal_t<float>(a, p.BH, p.ws, dev, p.stream)
                                   : fw_noncausal_t<__nv_bfloat16>(a, p.BH, p.ws, dev, p.stream);
}

}  // namespace la

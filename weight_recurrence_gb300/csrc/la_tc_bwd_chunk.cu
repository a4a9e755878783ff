// la_tc_bwd_chunk.cu - tensor-core (tcgen05 + TMA) backward of the causal
// form, "Transformers are RNNs" sec. 3.3 eqs. (10)-(12) (the gradient the
// page describes as cumulative sums, sec. 3.3.1, through the chain rule), for
// bf16 tensors with D, M in {64, 128}, every chunk of C = 128 rows at once.
//
// With S_c, z_c the state entering chunk c (the sums over the chunks before
// it, plus a carried-in state) and R_c, r_c the reverse sums after it
// (R = sum phi(Q_i) g_i^T, r = sum phi(Q_i) e_i over the later chunks, plus
// the gradient reaching the final state), every chunk's gradients depend on
// its own rows and these four sums only:
//   P = phi(Q) phi(K)^T masked to j <= i;  num = P V + phi(Q) S_c;
//   den = P 1 + phi(Q) . z_c;  g = dO / den;  e_i = -(g_i . num_i) / den_i;
//   A = (g V^T + e 1^T) masked to j <= i;
//   dphi(Q) = A phi(K) + g S_c^T + e z_c^T;   dR_c = phi(Q)^T [g | e];
//   dphi(K) = A^T phi(Q) + V R_c^T + 1 r_c^T;  dV = P^T g + phi(K) R_c;
//   dQ = dphi(Q) min(phi(Q), 1),  dK = dphi(K) min(phi(K), 1).
// Five launches: the per-chunk sums [dS_c | dz_c] = phi(K_c)^T [V_c | 1] (the
// causal forward's segment-sum pre-pass, one chunk per split); an exclusive
// scan over the chunks turning them into [S_c | z_c]; the query pass, one
// CTA per chunk (dQ, g as bf16 and e kept for the key pass, dR_c); the
// reverse exclusive scan turning [dR_c | dr_c] into [R_c | r_c] (started from
// the final state's gradient; its total is the carried-in state's gradient);
// the key pass, one CTA per chunk (dK, dV).  The sums enter the products as
// bf16 hi + lo pairs in the tile form of tc_bwd_common.cuh, and e is formed
// from the bf16 g the products use, as in the non-causal backward, so that
// terms which cancel in exact arithmetic cancel to fp32 rounding.  One CTA of
// 128 threads per chunk: thread r owns row r (TMEM lane r); the phases run
// one after another.  Every wait is bounded; a CTA that gives up records
// LA_ERR_TIMEOUT and skips the rest of its work.
#include <algorithm>

#include "la_common.cuh"
#include "la_internal.h"
#include "tc_bwd_common.cuh"
#include "tc_host.h"
#include "tc_kernels.cuh"
#include "tc_ptx.cuh"

// Optional per-phase timestamps of the first 1024 CTAs of the query (0) and
// key (1) kernels for performance work: compiled only with -DLA_TRACE (never
// in the library build).  Slot 15 holds %globaltimer at the CTA's start.
#ifdef LA_TRACE
__device__ unsigned long long g_la_trace_chunk[2][1024][16];
extern "C" int la_trace_read_chunk(unsigned long long *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_la_trace_chunk, sizeof(g_la_trace_chunk));
}
#define CH_TRACE(pass, ev)                                                                    \
    do {                                                                                      \
        if (blockIdx.x < 1024 && threadIdx.x == 0) {                                          \
            g_la_trace_chunk[pass][blockIdx.x][ev] = clock64();                               \
            if ((ev) == 0) g_la_trace_chunk[pass][blockIdx.x][15] = globaltimer_ns();         \
        }                                                                                     \
    } while (0)
#else
#define CH_TRACE(pass, ev) ((void)0)
#endif

namespace la {
namespace {

using namespace tc;

// ------------------------------------------------------------------ scans
// Exclusive scan of per-chunk vectors of W = D*M + D floats, in place, over
// the chunks of each head (reverse: from the last chunk down).  The running
// sum starts from `init` ([BH][D*M] then [BH][D], the vector's two parts;
// null: zero) and its final value goes to `total` (same layout; may be null).
// Thread (head, e4) owns elements 4 e4 .. 4 e4 + 3; the loads of sixteen
// chunks are issued before their sums.
__global__ void __launch_bounds__(256)
chunk_scan_kernel(float *ws, int nch, int DM, int D, const float *init_s, const float *init_z, float *tot_s,
                  float *tot_z, int reverse)
{
    const long long W4 = ((long long)DM + D) / 4;   // float4 per vector (DM and D are multiples of 4)
    const int e4 = blockIdx.y * 256 + threadIdx.x;
    const long long bh = blockIdx.x;
    pdl_wait_cta();
    if (e4 >= W4) return;
    const int e = 4 * e4;   // elements e..e+3: all of S or all of z
    float4 run = make_float4(0.f, 0.f, 0.f, 0.f);
    if (e < DM) {
        if (init_s) run = *reinterpret_cast<const float4 *>(init_s + bh * DM + e);
    } else if (init_z) {
        run = *reinterpret_cast<const float4 *>(init_z + bh * D + (e - DM));
    }
    float4 *base = reinterpret_cast<float4 *>(ws) + bh * nch * W4 + e4;
    constexpr int U = 16;
    for (int c0 = 0; c0 < nch; c0 += U) {
        float4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = reverse ? nch - 1 - (c0 + u) : c0 + u;
            x[u] = (c0 + u < nch) ? __ldcg(base + (long long)c * W4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (c0 + u >= nch) break;
            const int c = reverse ? nch - 1 - (c0 + u) : c0 + u;
            base[(long long)c * W4] = run;
            run.x += x[u].x;
            run.y += x[u].y;
            run.z += x[u].z;
            run.w += x[u].w;
        }
    }
    if (e < DM) {
        if (tot_s) *reinterpret_cast<float4 *>(tot_s + bh * DM + e) = run;
    } else if (tot_z) {
        *reinterpret_cast<float4 *>(tot_z + bh * D + (e - DM)) = run;
    }
}

struct ChunkBwdArgs {
    const float *ws_s;       // [BH, nch, D*M + D]: [S_c | z_c]
    float *ws_r;             // [BH, nch, D*M + D]: [dR_c | dr_c] (query pass) then [R_c | r_c]
    __nv_bfloat16 *ws_g;     // [BH, N, M]: g (query pass writes it)
    float *ws_e;             // [BH, N]: e
    __nv_bfloat16 *g0, *g1;  // query pass: dQ; key pass: dK, dV
    int N, nch;
    int total;               // BH * nch chunks, walked by the grid's CTAs in strides of gridDim.x
    int *err;
};

// TMEM columns of the two passes (all 512: one CTA per SM).
//   query pass: P (fp32, 128) -> A as bf16 hi (at Q_AH) and lo parts (at
//   Q_AL, in P's place); [num | den] (M + 16), then dphi(Q) (D) in its place;
//   A2 = g V^T (fp32, 128, in P's place) -> A2' (bf16, 64, in A_hi's place);
//   [dR | dr] (M + 16).
//   key pass: P^T and A^T (fp32, 128 each) -> bf16 in place; dV (M) and
//   dphi(K) (D).
template <int D, int M>
struct ChunkCols {
    static constexpr uint32_t Q_P = 0, Q_AL = 0, Q_AH = 128, Q_NUM = 192, Q_DQ = 192;
    static constexpr uint32_t Q_A2 = 0, Q_A2B = 128;
    static constexpr uint32_t Q_R = 192 + (M + 16 > D ? M + 16 : D);
    static constexpr uint32_t K_PT = 0, K_AT = 128, K_DV = 256, K_DK = 256 + M;
    static constexpr uint32_t COLS = 512;
    static_assert(Q_R + M + 16 <= COLS && K_DK + D <= COLS, "TMEM budget");
};

// Row r of the fp32 TMEM columns [c_begin, c_end) of a 128-column block at
// `src`: x_j = value + add(j) where keep(j), else 0, as bf16 into the packed
// columns at dst + j / 2.  Returns the fp32 sum of the x_j's bf16 roundings:
// the row sum of what the products will see.  dst may be src: each
// 32-column piece is read before the 16 packed columns it yields are
// written, at or below it, as long as no other thread writes this range.
template <typename Keep, typename Add>
__device__ __forceinline__ float tmem_mask_to_bf16(uint32_t src, uint32_t dst, int c_begin, int c_end, Keep keep,
                                                   Add add) {
    float sum = 0.f;
#pragma unroll 1
    for (int c0 = c_begin; c0 < c_end; c0 += 32) {
        float x[32];
        tmem_ld32f(src + c0, x);
        uint32_t w[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int c = c0 + 2 * j;
            const float a = keep(c) ? x[2 * j] + add(c) : 0.f;
            const float b = keep(c + 1) ? x[2 * j + 1] + add(c + 1) : 0.f;
            w[j] = pack_bf16x2(a, b);
            sum += bf16lo(w[j]) + bf16hi(w[j]);
        }
        tmem_st16(dst + c0 / 2, w);
        tmem_wait_st();
    }
    return sum;
}

// Both passes run two warpgroups: thread t handles row r = t mod 128 (TMEM
// lane r) and half h = t / 128 of the columns of every CUDA-core phase (or,
// where two operands are formed at once, one of them).
constexpr int kCT = 256;

// ------------------------------------------------------------- query pass
template <int D, int M>
struct CQCfg {
    static constexpr int TQ = kC * D * 2, TV = kC * M * 2;
    static constexpr int OFF_K = TQ, OFF_V = 2 * TQ, OFF_G = 2 * TQ + TV;
    static constexpr int OFF_SNAP = 2 * TQ + 2 * TV;                 // [S_hi | z | S_lo]
    static constexpr int OFF_E = OFF_SNAP + XwTile<D, M>::BYTES;     // (e_hi, e_hi, e_lo, e_lo) atom
    static constexpr int OFF_X = OFF_E + kC * 128;                   // fp32 [2][2][128] row-sum halves
    static constexpr int OFF_BAR = OFF_X + 2 * 2 * kC * 4;
    static constexpr int SMEM = OFF_BAR + 64;
    static_assert(SMEM <= (int)kSmemMax, "shared memory budget");
};

template <int D, int M>
__global__ void __launch_bounds__(kCT, 1)
chunk_bwd_query_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                       const ChunkBwdArgs args)
{
    using C = CQCfg<D, M>;
    using T = ChunkCols<D, M>;
    constexpr int MH = M / 2, DH = D / 2;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int t = threadIdx.x, r = t & (kC - 1), h = t >> 7;
    uint8_t *tq = smem, *tk = smem + C::OFF_K, *tv = smem + C::OFF_V, *tg = smem + C::OFF_G;
    uint8_t *snap = smem + C::OFF_SNAP, *eat = smem + C::OFF_E;
    float *xa = reinterpret_cast<float *>(smem + C::OFF_X), *xb = xa + 2 * kC;   // [half][row] each
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR), *mbar = full + 1;
    uint32_t *slot = reinterpret_cast<uint32_t *>(mbar + 1);

    CH_TRACE(0, 0);
    bool ok = (smem_u32(smem) & 1023u) == 0;
    if (t == 0) {
        mbar_init(full, 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    if (t < 32) {
        tmem_alloc(slot, T::COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + ((uint32_t)(32 * (r >> 5)) << 16);
    CH_TRACE(0, 1);
    pdl_wait_cta();   // the scanned sums of the previous launch are complete

    uint32_t phase = 0, fphase = 0;
    bool pending = false;   // MMAs committed but not complete (error path)
    bool loading = false;   // tiles requested but not landed (error path)
    constexpr uint32_t ID_P = idesc_bf16(128, 128, 0, 0);      // K-major A and B
    constexpr uint32_t ID_NV = idesc_bf16(128, M, 0, 1);       // A (TMEM) x V MN-major
    constexpr uint32_t ID_NS = idesc_bf16(128, M + 16, 0, 1);  // phi(Q) x [S_hi | z] MN-major
    constexpr uint32_t ID_DQ = idesc_bf16(128, D, 0, 0);       // [g | e | g] x [S_hi | z | S_lo]^T, K-major
    constexpr uint32_t ID_DQ2 = idesc_bf16(128, D, 0, 1);      // A2' (TMEM) x psi(K) MN-major
    constexpr uint32_t ID_R = idesc_bf16(128, M, 1, 1);        // phi(Q)^T x g, MN-major
    constexpr uint32_t ID_RZ = idesc_bf16(128, 16, 1, 1);
    auto mma_wait_all = [&]() {
        if (t == 0) mma_commit(mbar);
        const bool got = mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
        if (got) phase ^= 1u;
        tc_fence_after();
        return __syncthreads_and(got ? 1 : 0) != 0;
    };
    // Chunks u = blockIdx.x, + gridDim.x, ...: once one's tiles have landed,
    // the next one's tiles and sums are prefetched into L2 while it computes,
    // so that HBM is not idle between the CTAs' load phases
    for (int u = blockIdx.x; ok && u < args.total; u += gridDim.x) {
    const int bh = u / args.nch, c = u % args.nch;
    const int t0 = c * kC, valid = min(kC, args.N - t0);
    CH_TRACE(0, 2);
    if (t == 0) {
        mbar_arrive_expect_tx(full, 2 * C::TQ + 2 * C::TV);
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
            tma_load_3d(tq + j * kC * 128, &tm_q, full, j * 64, t0, bh);
            tma_load_3d(tk + j * kC * 128, &tm_k, full, j * 64, t0, bh);
        }
#pragma unroll
        for (int j = 0; j < M / 64; ++j) {
            tma_load_3d(tv + j * kC * 128, &tm_v, full, j * 64, t0, bh);
            tma_load_3d(tg + j * kC * 128, &tm_g, full, j * 64, t0, bh);
        }
    }
    loading = true;
    // [S_c hi | z_c | S_c lo]
    load_sum_tile<D, M, kCT>(args.ws_s + (size_t)u * (D * M + D), snap, t);
    CH_TRACE(0, 3);
    {
        const bool landed = mbar_wait_bounded(full, fphase, now_ns() + kWaitNs, nullptr);
        if (landed) {
            fphase ^= 1u;
            loading = false;
        }
        ok = __syncthreads_and(landed) != 0;
    }
    // the next chunk into L2 while this one computes
    if (t == 0 && ok) {
        const int un = u + gridDim.x;
        if (un < args.total) {
            const int bn = un / args.nch, tn = (un % args.nch) * kC;
#pragma unroll
            for (int j = 0; j < D / 64; ++j) {
                tma_prefetch_3d(&tm_q, j * 64, tn, bn);
                tma_prefetch_3d(&tm_k, j * 64, tn, bn);
            }
#pragma unroll
            for (int j = 0; j < M / 64; ++j) {
                tma_prefetch_3d(&tm_v, j * 64, tn, bn);
                tma_prefetch_3d(&tm_g, j * 64, tn, bn);
            }
            bulk_prefetch_l2(args.ws_s + (size_t)un * (D * M + D), (D * M + D) * 4);
        }
    }
    CH_TRACE(0, 4);
    // phi(Q) (half 0) and psi(K) = phi(K) - 1 (half 1; the 1 enters as the
    // row sums of phi(Q)); rows past the end become zeros
    float sq = 0.f;
    if (ok) {
        if (h == 0) phi_tile<D>(tq, r, valid);
        else psi_tile<D>(tk, r, valid);
        ok = operands_ready(true);
        sq = row_sum<D>(tq, r);
    }
    CH_TRACE(0, 5);
    // ---- phi(Q) psi(K)^T
    if (ok) {
        if (t == 0)
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::Q_P, kmajor_base(smem_u32(tq)) + kmajor_step(ks),
                           kmajor_base(smem_u32(tk)) + kmajor_step(ks), ID_P, ks > 0);
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(0, 6);
    // ---- A = P = phi(Q) psi(K)^T + sq masked to j <= r, as bf16 hi and lo
    // parts (num feeds e, which enters every entry of A2'); its row sum.  Each
    // half reads its 64 columns of P before either writes (A_lo replaces P's
    // first 64 columns)
    if (ok) {
        float x[64];
        tmem_ld32f(trow + T::Q_P + 64 * h, *reinterpret_cast<float(*)[32]>(x));
        tmem_ld32f(trow + T::Q_P + 64 * h + 32, *reinterpret_cast<float(*)[32]>(x + 32));
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        float rsp = 0.f;
#pragma unroll
        for (int p = 0; p < 2; ++p) {
            uint32_t w[16], l[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const int cc = 64 * h + 32 * p + 2 * j;
                const float a = cc <= r ? x[32 * p + 2 * j] + sq : 0.f;
                const float b = cc + 1 <= r ? x[32 * p + 2 * j + 1] + sq : 0.f;
                w[j] = pack_bf16x2(a, b);
                l[j] = pack_bf16x2(a - bf16lo(w[j]), b - bf16hi(w[j]));
                rsp += a + b;
            }
            tmem_st16(trow + T::Q_AH + 32 * h + 16 * p, w);
            tmem_st16(trow + T::Q_AL + 32 * h + 16 * p, l);
        }
        xa[h * kC + r] = rsp;
        ok = operands_ready(true);
    }
    CH_TRACE(0, 7);
    // ---- [num | den] = phi(Q) [S_hi | z] + A_hi V + A_lo V + phi(Q) [S_lo | -]
    // (the first product covers all M + 16 columns, so it starts the sum)
    if (ok) {
        if (t == 0) {
            const uint64_t dq = kmajor_base(smem_u32(tq));
            const uint64_t db = smem_desc(smem_u32(snap), D * 128, 1024);
            const uint64_t dl = smem_desc(smem_u32(snap + XwTile<D, M>::LO), D * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::Q_NUM, dq + kmajor_step(ks), db + mnmajor_step(ks), ID_NS, ks > 0);
            const uint64_t dv = smem_desc(smem_u32(tv), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + T::Q_NUM, tmem + T::Q_AH + ks * 8, dv + mnmajor_step(ks), ID_NV, 1);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + T::Q_NUM, tmem + T::Q_AL + ks * 8, dv + mnmajor_step(ks), ID_NV, 1);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::Q_NUM, dq + kmajor_step(ks), dl + mnmajor_step(ks), ID_NV, 1);
        }
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(0, 8);
    // ---- g = dO / den as bf16 (over dO; columns of half h), e = -(g . num) / den;
    // g and e kept for the key pass
    float e = 0.f;
    if (ok) {
        float dz[32];
        tmem_ld32f(trow + T::Q_NUM + M, dz);   // phi(Q) . z: the z_hi and z_lo columns
        const float den = xa[r] + xa[kC + r] + dz[0] + dz[1];
        const float inv = r < valid ? 1.f / den : 0.f;
        float dot = 0.f, gh[MH];
#pragma unroll
        for (int c0 = 0; c0 < MH; c0 += 32) {
            float x[32], gv[32];
            tmem_ld32f(trow + T::Q_NUM + MH * h + c0, x);
            load_row32(tg, r, MH * h + c0, gv);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                gv[j] = __bfloat162float(__float2bfloat16_rn(gv[j] * inv));
                dot = fmaf(gv[j], x[j], dot);
                gh[c0 + j] = gv[j];
            }
            store_snap32<kC>(tg, r, MH * h + c0, gv);
        }
        if (r < valid) store_row_bf16<MH>(args.ws_g + ((size_t)bh * args.N + t0 + r) * M + MH * h, gh);
        xb[h * kC + r] = dot;
        __syncthreads();
        e = -(xb[r] + xb[kC + r]) * inv;
        if (h == 0) {
            const float eh = __bfloat162float(__float2bfloat16_rn(e));
            const uint32_t hh = pack_bf16x2(eh, eh), ll = pack_bf16x2(e - eh, e - eh);
#pragma unroll
            for (int cc = 0; cc < 64; cc += 8)
                *reinterpret_cast<uint4 *>(eat + sw128_offset(r, cc)) =
                    make_uint4(cc == 0 ? hh : 0u, cc == 0 ? ll : 0u, 0u, 0u);
            if (r < valid) args.ws_e[(size_t)bh * args.N + t0 + r] = e;
        }
        ok = operands_ready(true);
    }
    CH_TRACE(0, 9);
    // ---- A2 = g V^T;  dphi(Q) = [g | e | g] [S_hi | z | S_lo]^T;  [dR | dr] = phi(Q)^T [g | e]
    if (ok) {
        if (t == 0) {
            const uint64_t dg = kmajor_base(smem_u32(tg)), de = kmajor_base(smem_u32(eat));
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::Q_A2, dg + kmajor_step(ks), kmajor_base(smem_u32(tv)) + kmajor_step(ks), ID_P, ks > 0);
            const uint64_t db = kmajor_base(smem_u32(snap)), dl = kmajor_base(smem_u32(snap + XwTile<D, M>::LO));
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::Q_DQ, dg + kmajor_step(ks), db + kmajor_step(ks, D), ID_DQ, ks > 0);
            mma_f16_ss(tmem + T::Q_DQ, de, db + kmajor_step(M / 16, D), ID_DQ, 1);   // the z atom
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::Q_DQ, dg + kmajor_step(ks), dl + kmajor_step(ks, D), ID_DQ, 1);
            // A read MN-major; at D = 64 with M-atom stride 0 (lanes 64-127
            // repeat lanes 0-63 and are not read)
            const uint64_t da = smem_desc(smem_u32(tq), D == 64 ? 0 : kC * 128, 1024);
            const uint64_t dgb = smem_desc(smem_u32(tg), kC * 128, 1024), deb = smem_desc(smem_u32(eat), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks) {
                mma_f16_ss(tmem + T::Q_R, da + mnmajor_step(ks), dgb + mnmajor_step(ks), ID_R, ks > 0);
                mma_f16_ss(tmem + T::Q_R + M, da + mnmajor_step(ks), deb + mnmajor_step(ks), ID_RZ, ks > 0);
            }
        }
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(0, 10);
    // ---- A2' = (A2 + e_r) masked to j <= r, as bf16 (columns of half h); its
    // row sum (the product with the 1 of phi(K) = psi(K) + 1).  [dR_c | dr_c]
    // is final: its rows are staged in the operand tile of the sums (last read
    // by the products just completed) and leave with coalesced stores while
    // the last product runs
    float *dst_r = args.ws_r + (size_t)u * (D * M + D);
    float *stage = reinterpret_cast<float *>(snap);
    static_assert(D * M * 4 <= XwTile<D, M>::BYTES, "staging area");
    if (ok) {
        xa[h * kC + r] = tmem_mask_to_bf16(trow + T::Q_A2, trow + T::Q_A2B, 64 * h, 64 * h + 64,
                                           [&](int j) { return j <= r; }, [&](int) { return e; });
        if (r < D) {
            float y[32];
#pragma unroll 1
            for (int c0 = MH * h; c0 < MH * h + MH; c0 += 32) {
                tmem_ld32f(trow + T::Q_R + c0, y);
                stage_row32_f32<M>(stage, r, c0, y);
            }
            if (h == 0) {
                tmem_ld32f(trow + T::Q_R + M, y);
                dst_r[D * M + r] = y[0] + y[2];   // the e_hi and e_lo columns
            }
        }
        ok = operands_ready(true);
    }
    CH_TRACE(0, 11);
    // ---- dphi(Q) += A2' psi(K)
    if (ok) {
        if (t == 0) {
            const uint64_t dk = smem_desc(smem_u32(tk), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + T::Q_DQ, tmem + T::Q_A2B + ks * 8, dk + mnmajor_step(ks), ID_DQ2, 1);
        }
        store_staged_f32<D, M>(dst_r, stage, t, kCT);
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(0, 12);
    // ---- dQ = (dphi(Q) + asum) min(phi(Q), 1), columns of half h
    if (ok) {
        const float asum = xa[r] + xa[kC + r];
        float x[DH];
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 32) {
            float d32[32], f[32];
            tmem_ld32f(trow + T::Q_DQ + DH * h + c0, d32);
            load_row32(tq, r, DH * h + c0, f);
#pragma unroll
            for (int j = 0; j < 32; ++j) x[c0 + j] = (d32[j] + asum) * fminf(f[j], 1.f);
        }
        if (r < valid) store_row_bf16<DH>(args.g0 + ((size_t)bh * args.N + t0 + r) * D + DH * h, x);
    }
    // the chunk's tiles, tile of sums, row-sum halves and TMEM are free for
    // the next one
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    }
    CH_TRACE(0, 13);
    if (!ok && t == 0) {
        record_error(args.err, kErrTimeout);
        if (loading) mbar_wait_bounded(full, fphase, now_ns() + kWaitNs, nullptr);
        if (pending) mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (t < 32) tmem_dealloc(tmem, T::COLS);
    CH_TRACE(0, 14);
}

// --------------------------------------------------------------- key pass
template <int D, int M>
struct CKCfg {
    static constexpr int TQ = kC * D * 2, TV = kC * M * 2;
    static constexpr int OFF_K = TQ, OFF_V = 2 * TQ, OFF_G = 2 * TQ + TV;
    static constexpr int OFF_SNAP = 2 * TQ + 2 * TV;                 // [R_hi | r | R_lo]
    static constexpr int OFF_ONES = OFF_SNAP + XwTile<D, M>::BYTES;  // [1 1 0 ..] atom
    static constexpr int OFF_E = OFF_ONES + kC * 128;                // e of the chunk's queries, fp32
    static constexpr int OFF_BAR = OFF_E + kC * 4;
    static constexpr int SMEM = OFF_BAR + 64;
    static_assert(SMEM <= (int)kSmemMax, "shared memory budget");
};

template <int D, int M>
__global__ void __launch_bounds__(kCT, 1)
chunk_bwd_key_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_gw,
                     const ChunkBwdArgs args)
{
    using C = CKCfg<D, M>;
    using T = ChunkCols<D, M>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int t = threadIdx.x, r = t & (kC - 1), h = t >> 7;
    uint8_t *tq = smem, *tk = smem + C::OFF_K, *tv = smem + C::OFF_V, *tg = smem + C::OFF_G;
    uint8_t *snap = smem + C::OFF_SNAP, *ones = smem + C::OFF_ONES;
    float *es = reinterpret_cast<float *>(smem + C::OFF_E);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR), *mbar = full + 1;
    uint32_t *slot = reinterpret_cast<uint32_t *>(mbar + 1);

    CH_TRACE(1, 0);
    bool ok = (smem_u32(smem) & 1023u) == 0;
    if (t == 0) {
        mbar_init(full, 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    if (t < 32) {
        tmem_alloc(slot, T::COLS);
        tmem_relinquish();
    }
    if (h == 0)
#pragma unroll
        for (int cc = 0; cc < 64; cc += 8)
            *reinterpret_cast<uint4 *>(ones + sw128_offset(r, cc)) = make_uint4(cc == 0 ? 0x3F803F80u : 0u, 0u, 0u, 0u);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + ((uint32_t)(32 * (r >> 5)) << 16);
    CH_TRACE(1, 1);
    pdl_wait_cta();   // the query pass and the reverse scan are complete

    uint32_t phase = 0, fphase = 0;
    bool pending = false, loading = false;
    constexpr uint32_t ID_P = idesc_bf16(128, 128, 0, 0);      // K-major A and B
    constexpr uint32_t ID_DV = idesc_bf16(128, M, 0, 1);       // P^T (TMEM) or phi(K) x MN-major
    constexpr uint32_t ID_DK = idesc_bf16(128, D, 0, 0);       // [V | 1 | V] x [R_hi | r | R_lo]^T, K-major
    constexpr uint32_t ID_DK2 = idesc_bf16(128, D, 0, 1);      // A^T (TMEM) x psi(Q) MN-major
    auto mma_wait_all = [&]() {
        if (t == 0) mma_commit(mbar);
        const bool got = mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
        if (got) phase ^= 1u;
        tc_fence_after();
        return __syncthreads_and(got ? 1 : 0) != 0;
    };
    // chunks in strides of gridDim.x, the next one prefetched into L2 (as in
    // the query pass)
    for (int u = blockIdx.x; ok && u < args.total; u += gridDim.x) {
    const int bh = u / args.nch, c = u % args.nch;
    const int t0 = c * kC, valid = min(kC, args.N - t0);
    CH_TRACE(1, 2);
    if (t == 0) {
        mbar_arrive_expect_tx(full, 2 * C::TQ + 2 * C::TV);
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
            tma_load_3d(tq + j * kC * 128, &tm_q, full, j * 64, t0, bh);
            tma_load_3d(tk + j * kC * 128, &tm_k, full, j * 64, t0, bh);
        }
#pragma unroll
        for (int j = 0; j < M / 64; ++j) {
            tma_load_3d(tv + j * kC * 128, &tm_v, full, j * 64, t0, bh);
            tma_load_3d(tg + j * kC * 128, &tm_gw, full, j * 64, t0, bh);
        }
    }
    loading = true;
    if (h == 0) es[r] = r < valid ? __ldcg(args.ws_e + (size_t)bh * args.N + t0 + r) : 0.f;
    // [R_c hi | r_c | R_c lo]
    load_sum_tile<D, M, kCT>(args.ws_r + (size_t)u * (D * M + D), snap, t);
    CH_TRACE(1, 3);
    {
        const bool landed = mbar_wait_bounded(full, fphase, now_ns() + kWaitNs, nullptr);
        if (landed) {
            fphase ^= 1u;
            loading = false;
        }
        ok = __syncthreads_and(landed) != 0;
    }
    // the next chunk into L2 while this one computes
    if (t == 0 && ok) {
        const int un = u + gridDim.x;
        if (un < args.total) {
            const int bn = un / args.nch, tn = (un % args.nch) * kC;
#pragma unroll
            for (int j = 0; j < D / 64; ++j) {
                tma_prefetch_3d(&tm_q, j * 64, tn, bn);
                tma_prefetch_3d(&tm_k, j * 64, tn, bn);
            }
#pragma unroll
            for (int j = 0; j < M / 64; ++j) {
                tma_prefetch_3d(&tm_v, j * 64, tn, bn);
                tma_prefetch_3d(&tm_gw, j * 64, tn, bn);
            }
            bulk_prefetch_l2(args.ws_r + (size_t)un * (D * M + D), (D * M + D) * 4);
        }
    }
    CH_TRACE(1, 4);
    // psi(Q) = phi(Q) - 1 (half 0; the 1 enters as the row sums of phi(K))
    // and phi(K) (half 1); rows past the end become zeros
    float sk = 0.f;
    if (ok) {
        if (h == 0) psi_tile<D>(tq, r, valid);
        else phi_tile<D>(tk, r, valid);
        ok = operands_ready(true);
        if (h == 0) sk = row_sum<D>(tk, r);
    }
    CH_TRACE(1, 5);
    // ---- phi(K) psi(Q)^T;  A^T (raw) = V g^T
    if (ok) {
        if (t == 0) {
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::K_PT, kmajor_base(smem_u32(tk)) + kmajor_step(ks),
                           kmajor_base(smem_u32(tq)) + kmajor_step(ks), ID_P, ks > 0);
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::K_AT, kmajor_base(smem_u32(tv)) + kmajor_step(ks),
                           kmajor_base(smem_u32(tg)) + kmajor_step(ks), ID_P, ks > 0);
        }
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(1, 6);
    // ---- P^T = phi(K) psi(Q)^T + sk (half 0) and A^T + e_i (half 1), masked
    // to r <= i < valid (key r, query i), as bf16 in place; the row sum of A^T
    // (its product with the 1 of phi(Q) = psi(Q) + 1)
    float asum = 0.f;
    if (ok) {
        auto keep = [&](int i) { return i >= r && i < valid; };
        if (h == 0) tmem_mask_to_bf16(trow + T::K_PT, trow + T::K_PT, 0, 128, keep, [&](int) { return sk; });
        else asum = tmem_mask_to_bf16(trow + T::K_AT, trow + T::K_AT, 0, 128, keep, [&](int i) { return es[i]; });
        ok = operands_ready(true);
    }
    CH_TRACE(1, 7);
    // ---- dV = P^T g + phi(K) (R_hi + R_lo);  dphi(K) = A^T psi(Q) + [V | 1 | V] [R_hi | r | R_lo]^T
    if (ok) {
        if (t == 0) {
            const uint64_t dgb = smem_desc(smem_u32(tg), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + T::K_DV, tmem + T::K_PT + ks * 8, dgb + mnmajor_step(ks), ID_DV, ks > 0);
            const uint64_t dk = kmajor_base(smem_u32(tk));
            const uint64_t ds = smem_desc(smem_u32(snap), D * 128, 1024);
            const uint64_t dsl = smem_desc(smem_u32(snap + XwTile<D, M>::LO), D * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::K_DV, dk + kmajor_step(ks), ds + mnmajor_step(ks), ID_DV, 1);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::K_DV, dk + kmajor_step(ks), dsl + mnmajor_step(ks), ID_DV, 1);
            const uint64_t dqb = smem_desc(smem_u32(tq), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + T::K_DK, tmem + T::K_AT + ks * 8, dqb + mnmajor_step(ks), ID_DK2, ks > 0);
            const uint64_t dv = kmajor_base(smem_u32(tv)), d1 = kmajor_base(smem_u32(ones));
            const uint64_t db = kmajor_base(smem_u32(snap)), dl = kmajor_base(smem_u32(snap + XwTile<D, M>::LO));
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::K_DK, dv + kmajor_step(ks), db + kmajor_step(ks, D), ID_DK, 1);
            mma_f16_ss(tmem + T::K_DK, d1, db + kmajor_step(M / 16, D), ID_DK, 1);   // the r atom
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::K_DK, dv + kmajor_step(ks), dl + kmajor_step(ks, D), ID_DK, 1);
        }
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(1, 8);
    // ---- dK = (dphi(K) + asum) min(phi(K), 1) (half 1, which holds asum); dV (half 0)
    if (ok) {
        if (h == 1) {
            float x[D];
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float d32[32], f[32];
                tmem_ld32f(trow + T::K_DK + c0, d32);
                load_row32(tk, r, c0, f);
#pragma unroll
                for (int j = 0; j < 32; ++j) x[c0 + j] = (d32[j] + asum) * fminf(f[j], 1.f);
            }
            if (r < valid) store_row_bf16<D>(args.g0 + ((size_t)bh * args.N + t0 + r) * D, x);
        } else {
            float x[M];
#pragma unroll
            for (int c0 = 0; c0 < M; c0 += 32) tmem_ld32f(trow + T::K_DV + c0, *reinterpret_cast<float(*)[32]>(x + c0));
            if (r < valid) store_row_bf16<M>(args.g1 + ((size_t)bh * args.N + t0 + r) * M, x);
        }
    }
    // the chunk's tiles, tile of sums, e values and TMEM are free for the next one
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    }
    CH_TRACE(1, 9);
    if (!ok && t == 0) {
        record_error(args.err, kErrTimeout);
        if (loading) mbar_wait_bounded(full, fphase, now_ns() + kWaitNs, nullptr);
        if (pending) mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (t < 32) tmem_dealloc(tmem, T::COLS);
    CH_TRACE(1, 10);
}

struct ChunkWs {
    size_t s_floats, g_elems, e_floats;
};

ChunkWs chunk_ws(long long BH, int N, int D, int M) {
    const long long nch = (N + kC - 1) / kC;
    return ChunkWs{(size_t)BH * nch * ((size_t)D * M + D), (size_t)BH * N * M, (size_t)BH * N};
}

// [S | z] and [R | r] per chunk, then g (bf16), then e; each part starts on
// a 256-byte boundary
size_t round256(size_t b) { return (b + 255) / 256 * 256; }
size_t chunk_ws_bytes(const ChunkWs &w) {
    return 2 * round256(w.s_floats * sizeof(float)) + round256(w.g_elems * 2) + w.e_floats * sizeof(float);
}

template <int D, int M>
cudaError_t launch_chunk_bwd(const BwdProblem &p, const DeviceInfo &dev) {
    const int nch = (p.N + kC - 1) / kC;
    const ChunkWs w = chunk_ws(p.BH, p.N, D, M);
    if (p.ws_bytes < chunk_ws_bytes(w)) return cudaErrorInvalidValue;
    uint8_t *base = (uint8_t *)p.ws;
    const size_t sb = round256(w.s_floats * sizeof(float));
    float *ws_s = (float *)base, *ws_r = (float *)(base + sb);
    __nv_bfloat16 *ws_g = (__nv_bfloat16 *)(base + 2 * sb);
    float *ws_e = (float *)(base + 2 * sb + round256(w.g_elems * 2));
    CUtensorMap tq, tk, tv, tg, tgw;
    if (!cached_tmap_bf16_3d(&tq, p.q, D, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tk, p.k, D, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tv, p.v, M, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tg, p.dout, M, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tgw, ws_g, M, p.N, p.BH, 64, kC))
        return cudaErrorInvalidValue;
    // per-chunk key sums
    cudaError_t e = tc_key_sums(p.k, p.v, p.BH, p.N, D, M, nch, 1, ws_s, w.s_floats * sizeof(float), p.stream, dev);
    if (e != cudaSuccess) return e;
    const int W = D * M + D;
    const dim3 sgrid((unsigned)p.BH, (unsigned)((W / 4 + 255) / 256));
    e = launch_pdl(chunk_scan_kernel, sgrid, dim3(256), 0, p.stream, 0u, ws_s, nch, D * M, D, p.S0, p.z0,
                   (float *)nullptr, (float *)nullptr, 0);
    count_launches(1);
    if (e != cudaSuccess) return e;
    // one CTA per SM (the shared memory and the 512 TMEM columns each CTA
    // holds allow no more), each walking chunks in strides of the grid
    const long long total = p.BH * nch;
    if (total > INT32_MAX) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)std::min<long long>(total, std::max(1, dev.sm_count))), block(kCT);
    ChunkBwdArgs a{ws_s, ws_r, ws_g, ws_e, (__nv_bfloat16 *)p.dq, nullptr, p.N, nch, (int)total, dev.err_word};
    if ((e = set_smem(chunk_bwd_query_kernel<D, M>, CQCfg<D, M>::SMEM)) != cudaSuccess) return e;
    e = launch_pdl(chunk_bwd_query_kernel<D, M>, grid, block, CQCfg<D, M>::SMEM, p.stream, 0u, tq, tk, tv, tg, a);
    count_launches(1);
    if (e != cudaSuccess) return e;
    e = launch_pdl(chunk_scan_kernel, sgrid, dim3(256), 0, p.stream, 0u, ws_r, nch, D * M, D, p.dSN, p.dzN, p.dS0,
                   p.dz0, 1);
    count_launches(1);
    if (e != cudaSuccess) return e;
    a.g0 = (__nv_bfloat16 *)p.dk;
    a.g1 = (__nv_bfloat16 *)p.dv;
    if ((e = set_smem(chunk_bwd_key_kernel<D, M>, CKCfg<D, M>::SMEM)) != cudaSuccess) return e;
    e = launch_pdl(chunk_bwd_key_kernel<D, M>, grid, block, CKCfg<D, M>::SMEM, p.stream, 0u, tq, tk, tv, tgw, a);
    count_launches(1);
    return e;
}

}  // namespace

bool tc_chunk_backward_supported(const la_shape &s) {
    return s.dtype == LA_DTYPE_BF16 && (s.D == 64 || s.D == 128) && (s.M == 64 || s.M == 128) &&
           !(s.D == 64 && s.M == 64);
}

size_t tc_chunk_backward_ws_bytes(const la_shape &s) {
    const long long BH = (long long)s.B * s.H;
    if (BH <= 0 || s.N <= 0) return 0;
    return chunk_ws_bytes(chunk_ws(BH, s.N, s.D, s.M));
}

cudaError_t tc_chunk_causal_backward(const BwdProblem &p, const DeviceInfo &dev) {
    if (p.D == 64 && p.M == 128) return launch_chunk_bwd<64, 128>(p, dev);
    if (p.D == 128 && p.M == 64) return launch_chunk_bwd<128, 64>(p, dev);
    if (p.D == 128 && p.M == 128) return launch_chunk_bwd<128, 128>(p, dev);
    return cudaErrorInvalidValue;
}

}  // namespace la

// la_tc_bwd.cu - tensor-core (tcgen05 + TMA) backward of the causal form for
// bf16 tensors with D = M = 64.
//
// The chain rule through "Transformers are RNNs" sec. 3.3 eqs. (10)-(12)
// (the page describes the gradient as cumulative sums in constant memory,
// sec. 3.3.1, without printing eqs. (13)-(15)), regrouped by chunks of C = 128
// rows.  For the chunk's rows i (queries) and j (keys), with S, Z the state
// before the chunk and R, r the reverse sums after it:
//   pass 1 (chunks in order):
//     P = phi(Q) phi(K)^T masked to j <= i;  num = P V + phi(Q) S;
//     den_i = sum_j P_ij + phi(Q_i) . Z;  g_i = dO_i / den_i;
//     e_i = -(g_i . num_i) / den_i;  A = (g V^T + e 1^T) masked to j <= i;
//     dphi(Q) = A phi(K) + g S^T + e Z^T;  dQ = dphi(Q) * min(phi(Q), 1);
//     S += phi(K)^T V,  Z += sum_j phi(K_j);  g (bf16) and e (fp32) kept.
//   pass 2 (chunks in reverse):
//     P^T = phi(K) phi(Q)^T masked to i >= j;  A^T = (V g^T + 1 e^T) masked;
//     dV = P^T g + phi(K) R;  dphi(K) = A^T phi(Q) + V R^T + 1 r^T;
//     dK = dphi(K) * min(phi(K), 1);  R += phi(Q)^T g,  r += sum_i e_i phi(Q_i).
// Every product is a tcgen05 MMA (bf16 operands, fp32 accumulators in TMEM);
// the masks, divisions and the rank-one terms run on CUDA cores between the
// MMAs.  One CTA of 128 threads per head; thread t owns row t of every
// 128-row accumulator (TMEM lane t).  The phases of a chunk run one after
// the other, the next chunk's tiles loading by TMA meanwhile (two stages).
// Every wait is bounded; a CTA that gives up records LA_ERR_TIMEOUT and
// skips the rest of its work.
#include "la_common.cuh"
#include "la_internal.h"
#include "tc_host.h"
#include "tc_kernels.cuh"
#include "tc_ptx.cuh"

// Optional per-phase timeline of CTA 0 of the forward sweep for performance
// work: compiled only with -DLA_TRACE (never in the library build).
#ifdef LA_TRACE
__device__ unsigned long long g_la_trace_bwd[32][12];
extern "C" int la_trace_read_bwd(unsigned long long *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_la_trace_bwd, sizeof(g_la_trace_bwd));
}
#define BWD_TRACE(it, ev)                                                                            \
    do {                                                                                             \
        if (blockIdx.x == 0 && threadIdx.x == 0 && (it) < 32) g_la_trace_bwd[it][ev] = clock64();    \
    } while (0)
#else
#define BWD_TRACE(it, ev) ((void)0)
#endif

namespace la {
namespace {

constexpr int kBD = 64;                     // D = M
constexpr int kBT = 128;                    // threads
constexpr int kTile = kC * kBD * 2;         // one 128 x 64 bf16 tile, 16 KB
constexpr int kStage = 4 * kTile;           // Q, K, V, dO (pass 1) or Q, K, V, g (pass 2)
constexpr int kOffGT = 2 * kStage;          // pass 1: g of the chunk as an MMA operand
constexpr int kOffSnap = kOffGT + kTile;    // state S or R as bf16 hi then lo parts, [64 rows][64] each
constexpr int kSnap = kBD * kBD * 2;        // 8 KB
constexpr int kOffZ = kOffSnap + 2 * kSnap; // fp32 Z or r [64]
constexpr int kOffE = kOffZ + kBD * 4;      // fp32 e of the chunk [128]
constexpr int kOffPart = kOffE + kC * 4;    // fp32 [2][64] column-sum halves
constexpr int kOffPsi = ((kOffPart + 2 * kBD * 4 + 1023) / 1024) * 1024;   // psi(K) (pass 1) or psi(Q) (pass 2)
constexpr int kOffBar = kOffPsi + kTile;
constexpr int kOffSlot = kOffBar + 8 * 4;
constexpr int kBwdSmem = kOffSlot + 16;
constexpr uint32_t kBwdTmemCols = 512;
static_assert(kBwdSmem <= (int)kSmemMax, "shared memory budget");

// TMEM columns.  Pass 1: P, then A, in [0, 128) (A as bf16 in [0, 64)); num
// in [128, 192); dphi(Q) in [192, 256); S in [256, 320).  Pass 2: P^T in
// [0, 128) (bf16 in [0, 64)), A^T in [128, 256) (bf16 in [128, 192)); dV in
// [256, 320); dphi(K) in [320, 384); R in [384, 448).
constexpr uint32_t kColP = 0, kColA2 = 128, kColNum = 128, kColDQ = 192, kColS = 256;
constexpr uint32_t kColDV = 256, kColDK = 320, kColR = 384;

struct BwdArgs {
    __nv_bfloat16 *dq, *dk, *dv;
    __nv_bfloat16 *g_ws;     // [BH, N, 64] bf16
    float *e_ws;             // [BH, N]
    const float *S0, *z0, *dSN, *dzN;
    float *dS0, *dz0;
    int N;
    int *err;
};

// Synchronous MMA step: thread 0 commits everything it issued to `bar`;
// every thread waits for that phase.  Returns false (CTA-uniform) if the wait
// gave up.
__device__ __forceinline__ bool mma_sync_all(uint64_t *bar, uint32_t &phase, bool ok, int *err) {
    if (threadIdx.x == 0 && ok) mma_commit(bar);
    bool mine = ok && mbar_wait_bounded(bar, phase, now_ns() + kWaitNs, nullptr);
    if (ok && !mine && threadIdx.x == 0) record_error(err, kErrTimeout);
    const bool all = __syncthreads_and(mine ? 1 : 0) != 0;
    if (ok) phase ^= 1u;
    tc_fence_after();
    return all;
}

// All threads finished their TMEM stores and generic shared-memory writes:
// make them visible to the MMAs thread 0 issues next.
__device__ __forceinline__ void operands_ready() {
    tmem_wait_st();
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Loads the chunk's four tiles (64-column boxes) into stage `st`.
__device__ __forceinline__ void load_chunk(uint8_t *st, uint64_t *full, const CUtensorMap *t0m,
                                           const CUtensorMap *t1m, const CUtensorMap *t2m,
                                           const CUtensorMap *t3m, int t0, int bh) {
    mbar_arrive_expect_tx(full, kStage);
    tma_load_3d(st, t0m, full, 0, t0, bh);
    tma_load_3d(st + kTile, t1m, full, 0, t0, bh);
    tma_load_3d(st + 2 * kTile, t2m, full, 0, t0, bh);
    tma_load_3d(st + 3 * kTile, t3m, full, 0, t0, bh);
}

// Reads this thread's row of a 128-column fp32 accumulator, applies the
// causal mask (pass 1 keeps columns j <= r, pass 2 keeps i >= r) and adds
// `colv[c]` (if given) or `rowv` to the kept entries, writes the row back as
// bf16 in the first 64 columns of the block, and returns the fp32 sum of
// the kept entries (after the addition, before rounding).
__device__ __forceinline__ float mask_to_bf16(uint32_t tbase, int r, bool lower, float rowv, const float *colv,
                                              bool hilo = false) {
    float sum = 0.f;
    uint32_t packed[4][16], packed_lo[4][16];
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        const int c0 = 32 * b;
        float x[32];
        tmem_ld32f(tbase + c0, x);
#pragma unroll
        for (int j = 0; j < 32; j += 2) {
            const int c = c0 + j;
            const bool k0 = lower ? (c <= r) : (c >= r);
            const bool k1 = lower ? (c + 1 <= r) : (c + 1 >= r);
            const float add0 = colv ? colv[c] : rowv, add1 = colv ? colv[c + 1] : rowv;
            const float a0 = k0 ? x[j] + add0 : 0.f, a1 = k1 ? x[j + 1] + add1 : 0.f;
            sum += a0 + a1;
            const uint32_t hp = pack_bf16x2(a0, a1);
            packed[b][j / 2] = hp;
            packed_lo[b][j / 2] = pack_bf16x2(a0 - bf16lo(hp), a1 - bf16hi(hp));
        }
    }
#pragma unroll
    for (int b = 0; b < 4; ++b) tmem_st16(tbase + 16 * b, packed[b]);
    if (hilo)   // the rounding error of each entry as a second bf16 operand
#pragma unroll
        for (int b = 0; b < 4; ++b) tmem_st16(tbase + 64 + 16 * b, packed_lo[b]);
    return sum;
}

// Column sums over the chunk's 128 rows of a phi-applied bf16 tile, each row
// weighted by w[row] (or 1): thread t sums column t % 64 over rows of half
// t / 64; the halves meet in `part`; threads 0..63 add the total to acc[t].
__device__ __forceinline__ void colsum_add(const uint8_t *tile, const float *w, float *part, float *acc) {
    const int t = threadIdx.x, d = t & 63, half = t >> 6;
    float s = 0.f;
#pragma unroll 8
    for (int i = 64 * half; i < 64 * half + 64; ++i) {
        const float x = __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + sw128_offset(i, d)));
        s = fmaf(w ? w[i] : 1.f, x, s);
    }
    part[half * 64 + d] = s;
    __syncthreads();
    if (t < 64) acc[t] += part[t] + part[64 + t];
}

// Stores this thread's 64-column fp32 row `v` (scaled elementwise by `scale`
// when given) as bf16 to `dst` (128 bytes).
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16 *dst, const float *v) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int c8 = 0; c8 < 8; ++c8) {
        uint4 w;
        w.x = pack_bf16x2(v[8 * c8], v[8 * c8 + 1]);
        w.y = pack_bf16x2(v[8 * c8 + 2], v[8 * c8 + 3]);
        w.z = pack_bf16x2(v[8 * c8 + 4], v[8 * c8 + 5]);
        w.w = pack_bf16x2(v[8 * c8 + 6], v[8 * c8 + 7]);
        d4[c8] = w;
    }
}

// Row r, columns c0..c0+31 of a fp32 state as two bf16 parts (hi, then lo =
// the rounding error of hi), so that MMAs against the state keep about 16
// bits: the gradient terms S g and e Z (and V R^T and r) cancel in large part.
__device__ __forceinline__ void store_state32(uint8_t *snap, int r, int c0, const float *v) {
    float hi[32], lo[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        hi[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
        lo[j] = v[j] - hi[j];
    }
    store_snap32<kBD>(snap, r, c0, hi);
    store_snap32<kBD>(snap + kSnap, r, c0, lo);
}

// psi(x) = phi(x) - 1 (x for x > 0, e^x - 1 otherwise) of a raw bf16 tile into
// `dst` (same layout), rows >= zero_from as zeros.  Where the inputs are
// small, phi(x) is close to 1 and its bf16 rounding swamps x; the gradient
// products use psi and add the row sums of the other factor separately.
// Same chunk-to-thread assignment as phi_tile, so a thread may apply phi_tile
// to `raw` right after this without a barrier.
__device__ __forceinline__ void psi_tile(const uint8_t *raw, uint8_t *dst, int t, int zero_from) {
    constexpr int CHUNKS = kC * kBD * 2 / 16;
#pragma unroll 1
    for (int u0 = t; u0 < CHUNKS; u0 += 4 * kGrp) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t off = (uint32_t)(u0 + i * kGrp) * 16u;
            const int row = (int)((off % (kC * 128u)) >> 7);
            const uint4 w = *reinterpret_cast<const uint4 *>(raw + off);
            const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
            uint32_t o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float a = bf16lo(ww[u]), b = bf16hi(ww[u]);
                float ea, eb;
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ea) : "f"(a * 1.4426950408889634f));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(eb) : "f"(b * 1.4426950408889634f));
                o[u] = pack_bf16x2(a > 0.f ? a : ea - 1.f, b > 0.f ? b : eb - 1.f);
            }
            *reinterpret_cast<uint4 *>(dst + off) =
                row >= zero_from ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(o[0], o[1], o[2], o[3]);
        }
    }
}

// phi'(x) from the stored bf16 phi(x): 1 where phi > 1 (x > 0), else phi.
__device__ __forceinline__ float dphi_at(const uint8_t *tile, int r, int c) {
    return fminf(__bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + sw128_offset(r, c))), 1.f);
}

// ------------------------------------------------------------------ pass 1
__global__ void __launch_bounds__(kBT, 1)
bwd_tc_pass1_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const BwdArgs args)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int r = threadIdx.x, q4 = r >> 5;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int bh = blockIdx.x, N = args.N;
    const int nch = (N + kC - 1) / kC;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar), *mbar = full + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + kOffSlot);
    uint8_t *gt = smem + kOffGT, *snap = smem + kOffSnap;
    float *zs = reinterpret_cast<float *>(smem + kOffZ), *part = reinterpret_cast<float *>(smem + kOffPart);

    bool ok = (smem_u32(smem) & 1023u) == 0;
    if (r == 0) {
        if (!ok) record_error(args.err, kErrTimeout);
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    if (q4 == 0) {
        tmem_alloc(slot, kBwdTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + lane_off;

    // the starting state: S (TMEM, fp32; lanes 64-127 unused) and its bf16
    // snapshot, Z (shared memory, fp32)
    {
        float v[32];
        for (int c0 = 0; c0 < kBD; c0 += 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = (r < kBD && args.S0) ? args.S0[((size_t)bh * kBD + r) * kBD + c0 + j] : 0.f;
            tmem_st32f(trow + kColS + c0, v);
            if (r < kBD) store_state32(snap, r, c0, v);
        }
        if (r < kBD) zs[r] = args.z0 ? args.z0[(size_t)bh * kBD + r] : 0.f;
    }
    if (r == 0 && ok && nch > 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
        load_chunk(smem, &full[0], &tm_q, &tm_k, &tm_v, &tm_do, 0, bh);
    }
    operands_ready();

    uint32_t phase = 0;
    constexpr uint32_t ID_P = idesc_bf16(128, 128, 0, 0);     // K-major A and B
    constexpr uint32_t ID_MN = idesc_bf16(128, kBD, 0, 1);    // K-major A, MN-major B
    constexpr uint32_t ID_KK = idesc_bf16(128, kBD, 0, 0);    // K-major A and B
    constexpr uint32_t ID_S = idesc_bf16(128, kBD, 1, 1);     // MN-major A and B
    for (int it = 0; it < nch && ok; ++it) {
        BWD_TRACE(it, 0);
        const int s = it & 1, t0 = it * kC;
        uint8_t *st = smem + s * kStage;
        uint8_t *tq = st, *tk = st + kTile, *tv = st + 2 * kTile, *tdo = st + 3 * kTile;
        // next chunk's tiles into the other stage (freed at the end of the previous chunk)
        if (r == 0 && it + 1 < nch)
            load_chunk(smem + (s ^ 1) * kStage, &full[s ^ 1], &tm_q, &tm_k, &tm_v, &tm_do, t0 + kC, bh);
        const bool landed = mbar_wait_bounded(&full[s], (it >> 1) & 1, now_ns() + kWaitNs, nullptr);
        if (!landed && r == 0) record_error(args.err, kErrTimeout);
        if (!(ok = __syncthreads_and(landed) != 0)) break;
        // feature map in place (rows past the sequence end become zero), and
        // psi(K) = phi(K) - 1 for the dQ product
        phi_tile<kBD>(tq, r, min(kC, N - t0));
        psi_tile(tk, smem + kOffPsi, r, min(kC, N - t0));
        phi_tile<kBD>(tk, r, min(kC, N - t0));
        operands_ready();
        BWD_TRACE(it, 1);
        const uint32_t aq = smem_u32(tq), ak = smem_u32(tk), av = smem_u32(tv), ag = smem_u32(gt), as = smem_u32(snap);
        // P = phi(Q) phi(K)^T
        if (r == 0)
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColP, kmajor_base(aq) + kmajor_step(ks), kmajor_base(ak) + kmajor_step(ks), ID_P, ks > 0);
        if (!(ok = mma_sync_all(mbar, phase, ok, args.err))) break;
        BWD_TRACE(it, 2);
        // mask (j <= i), row sums, A as bf16 hi and lo parts (num feeds e, where
        // the output's error would enter every entry of A)
        const float rowsum = mask_to_bf16(trow + kColP, r, true, 0.f, nullptr, true);
        const float den = rowsum + q_dot_z<kBD>(tq, r, zs);
        operands_ready();
        BWD_TRACE(it, 3);
        // num = A V + phi(Q) S
        if (r == 0) {
            const uint64_t dv = smem_desc(av, kC * 128, 1024), ds = smem_desc(as, kBD * 128, 1024);
#pragma unroll
            for (int part2 = 0; part2 < 2; ++part2)
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_f16_ts(tmem + kColNum, tmem + kColP + 64 * part2 + ks * 8, dv + mnmajor_step(ks), ID_MN,
                               part2 > 0 || ks > 0);
#pragma unroll
            for (int part2 = 0; part2 < 2; ++part2)
#pragma unroll
                for (int ks = 0; ks < kBD / 16; ++ks)
                    mma_f16_ss(tmem + kColNum, kmajor_base(aq) + kmajor_step(ks),
                               ds + (uint64_t)(part2 * kSnap / 16) + mnmajor_step(ks), ID_MN, 1);
        }
        if (!(ok = mma_sync_all(mbar, phase, ok, args.err))) break;
        BWD_TRACE(it, 4);
        // g_i = dO_i / den_i, e_i = -(g_i . num_i) / den_i; g as bf16 into the
        // operand tile and the workspace, e into the workspace
        const bool valid = t0 + r < N;
        float e = 0.f;
        {
            float num[64], g[64];
            tmem_ld32f(trow + kColNum, *reinterpret_cast<float(*)[32]>(num));
            tmem_ld32f(trow + kColNum + 32, *reinterpret_cast<float(*)[32]>(num + 32));
            const float inv = valid ? 1.f / den : 0.f;
            float gn = 0.f;
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const uint4 w = *reinterpret_cast<const uint4 *>(tdo + sw128_offset(r, 8 * c8));
                const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    g[8 * c8 + 2 * u] = bf16lo(ww[u]) * inv;
                    g[8 * c8 + 2 * u + 1] = bf16hi(ww[u]) * inv;
                }
            }
            // the MMAs (and pass 2) use g rounded to bf16; e is formed from that same
            // g, so that the terms A phi(K), g S^T and e Z stay consistent
#pragma unroll
            for (int c = 0; c < 64; ++c) g[c] = __bfloat162float(__float2bfloat16_rn(g[c]));
#pragma unroll
            for (int c0 = 0; c0 < 64; c0 += 32) store_snap32<kC>(gt, r, c0, g + c0);
#pragma unroll
            for (int c = 0; c < 64; ++c) gn = fmaf(g[c], num[c], gn);
            e = valid ? -gn * inv : 0.f;
            if (valid) {
                store_row_bf16(args.g_ws + ((size_t)bh * N + t0 + r) * kBD, g);
                args.e_ws[(size_t)bh * N + t0 + r] = e;
            }
        }
        operands_ready();
        BWD_TRACE(it, 5);
        // A2 = g V^T
        if (r == 0)
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColP, kmajor_base(ag) + kmajor_step(ks), kmajor_base(av) + kmajor_step(ks), ID_P, ks > 0);
        if (!(ok = mma_sync_all(mbar, phase, ok, args.err))) break;
        BWD_TRACE(it, 6);
        // A = (A2 + e_i) masked to j <= i, as bf16; asum its fp32 row sum
        const float asum = mask_to_bf16(trow + kColP, r, true, e, nullptr);
        operands_ready();
        BWD_TRACE(it, 7);
        // dphi(Q) = A psi(K) + g S^T  (+ asum: the product with the 1 of phi = psi + 1)
        if (r == 0) {
            const uint64_t dk = smem_desc(smem_u32(smem + kOffPsi), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + kColDQ, tmem + kColP + ks * 8, dk + mnmajor_step(ks), ID_MN, ks > 0);
#pragma unroll
            for (int part2 = 0; part2 < 2; ++part2)
#pragma unroll
                for (int ks = 0; ks < kBD / 16; ++ks)
                    mma_f16_ss(tmem + kColDQ, kmajor_base(ag) + kmajor_step(ks),
                               kmajor_base(as + part2 * kSnap) + kmajor_step(ks, kBD), ID_KK, 1);
        }
        if (!(ok = mma_sync_all(mbar, phase, ok, args.err))) break;
        BWD_TRACE(it, 8);
        // dQ = (dphi(Q) + e_i Z) * phi'(Q)
        {
            float dq[64];
            tmem_ld32f(trow + kColDQ, *reinterpret_cast<float(*)[32]>(dq));
            tmem_ld32f(trow + kColDQ + 32, *reinterpret_cast<float(*)[32]>(dq + 32));
#pragma unroll
            for (int c = 0; c < 64; ++c) dq[c] = (fmaf(e, zs[c], dq[c]) + asum) * dphi_at(tq, r, c);
            if (valid) store_row_bf16(args.dq + ((size_t)bh * N + t0 + r) * kBD, dq);
        }
        __syncthreads();   // every thread has read Z before it changes
        // S += phi(K)^T V (A read MN-major with M-atom stride 0: lanes 64-127
        // repeat lanes 0-63), Z += column sums of phi(K)
        if (r == 0) {
            const uint64_t da = smem_desc(ak, 0, 1024), db = smem_desc(av, kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ss(tmem + kColS, da + mnmajor_step(ks), db + mnmajor_step(ks), ID_S, 1);
        }
        colsum_add(tk, nullptr, part, zs);
        if (!(ok = mma_sync_all(mbar, phase, ok, args.err))) break;
        BWD_TRACE(it, 9);
        // the new state's bf16 snapshot for the next chunk
        if (r < kBD) {
            float v[32];
            for (int c0 = 0; c0 < kBD; c0 += 32) {
                tmem_ld32f(trow + kColS + c0, v);
                store_state32(snap, r, c0, v);
            }
        }
        operands_ready();   // also: every thread is done with this stage
        BWD_TRACE(it, 10);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (q4 == 0) tmem_dealloc(tmem, kBwdTmemCols);
}

// ------------------------------------------------------------------ pass 2
__global__ void __launch_bounds__(kBT, 1)
bwd_tc_pass2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                    const BwdArgs args)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int r = threadIdx.x, q4 = r >> 5;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int bh = blockIdx.x, N = args.N;
    const int nch = (N + kC - 1) / kC;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar), *mbar = full + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + kOffSlot);
    uint8_t *snap = smem + kOffSnap;
    float *rs = reinterpret_cast<float *>(smem + kOffZ), *es = reinterpret_cast<float *>(smem + kOffE);
    float *part = reinterpret_cast<float *>(smem + kOffPart);

    bool ok = (smem_u32(smem) & 1023u) == 0;
    if (r == 0) {
        if (!ok) record_error(args.err, kErrTimeout);
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    if (q4 == 0) {
        tmem_alloc(slot, kBwdTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + lane_off;

    // R, r start from the gradient reaching the final state (or zero)
    {
        float v[32];
        for (int c0 = 0; c0 < kBD; c0 += 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = (r < kBD && args.dSN) ? args.dSN[((size_t)bh * kBD + r) * kBD + c0 + j] : 0.f;
            tmem_st32f(trow + kColR + c0, v);
            if (r < kBD) store_state32(snap, r, c0, v);
        }
        if (r < kBD) rs[r] = args.dzN ? args.dzN[(size_t)bh * kBD + r] : 0.f;
    }
    if (r == 0 && ok && nch > 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_g);
        load_chunk(smem, &full[0], &tm_q, &tm_k, &tm_v, &tm_g, (nch - 1) * kC, bh);
    }
    operands_ready();

    uint32_t phase = 0;
    constexpr uint32_t ID_P = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t ID_MN = idesc_bf16(128, kBD, 0, 1);
    constexpr uint32_t ID_KK = idesc_bf16(128, kBD, 0, 0);
    constexpr uint32_t ID_S = idesc_bf16(128, kBD, 1, 1);
    for (int it = 0; it < nch && ok; ++it) {
        const int c = nch - 1 - it, s = it & 1, t0 = c * kC;
        uint8_t *st = smem + s * kStage;
        uint8_t *tq = st, *tk = st + kTile, *tv = st + 2 * kTile, *tg = st + 3 * kTile;
        if (r == 0 && it + 1 < nch)
            load_chunk(smem + (s ^ 1) * kStage, &full[s ^ 1], &tm_q, &tm_k, &tm_v, &tm_g, t0 - kC, bh);
        es[r] = t0 + r < N ? args.e_ws[(size_t)bh * N + t0 + r] : 0.f;
        const bool landed = mbar_wait_bounded(&full[s], (it >> 1) & 1, now_ns() + kWaitNs, nullptr);
        if (!landed && r == 0) record_error(args.err, kErrTimeout);
        if (!(ok = __syncthreads_and(landed) != 0)) break;
        psi_tile(tq, smem + kOffPsi, r, min(kC, N - t0));
        phi_tile<kBD>(tq, r, min(kC, N - t0));
        phi_tile<kBD>(tk, r, min(kC, N - t0));
        operands_ready();
        const uint32_t aq = smem_u32(tq), ak = smem_u32(tk), av = smem_u32(tv), ag = smem_u32(tg), as = smem_u32(snap);
        // P^T = phi(K) phi(Q)^T and A^T = V g^T (rows j, columns i)
        if (r == 0) {
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColP, kmajor_base(ak) + kmajor_step(ks), kmajor_base(aq) + kmajor_step(ks), ID_P, ks > 0);
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColA2, kmajor_base(av) + kmajor_step(ks), kmajor_base(ag) + kmajor_step(ks), ID_P, ks > 0);
        }
        if (!(ok = mma_sync_all(mbar, phase, ok, args.err))) break;
        // masks (i >= j), e_i added to the kept entries of A^T; both as bf16
        mask_to_bf16(trow + kColP, r, false, 0.f, nullptr);
        const float asum = mask_to_bf16(trow + kColA2, r, false, 0.f, es);
        operands_ready();
        // dV = P^T g + phi(K) R;  dphi(K) = A^T psi(Q) + V R^T (+ asum)
        if (r == 0) {
            const uint64_t dg = smem_desc(ag, kC * 128, 1024), dqm = smem_desc(smem_u32(smem + kOffPsi), kC * 128, 1024);
            const uint64_t ds = smem_desc(as, kBD * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + kColDV, tmem + kColP + ks * 8, dg + mnmajor_step(ks), ID_MN, ks > 0);
#pragma unroll
            for (int part2 = 0; part2 < 2; ++part2)
#pragma unroll
                for (int ks = 0; ks < kBD / 16; ++ks)
                    mma_f16_ss(tmem + kColDV, kmajor_base(ak) + kmajor_step(ks),
                               ds + (uint64_t)(part2 * kSnap / 16) + mnmajor_step(ks), ID_MN, 1);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + kColDK, tmem + kColA2 + ks * 8, dqm + mnmajor_step(ks), ID_MN, ks > 0);
#pragma unroll
            for (int part2 = 0; part2 < 2; ++part2)
#pragma unroll
                for (int ks = 0; ks < kBD / 16; ++ks)
                    mma_f16_ss(tmem + kColDK, kmajor_base(av) + kmajor_step(ks),
                               kmajor_base(as + part2 * kSnap) + kmajor_step(ks, kBD), ID_KK, 1);
        }
        if (!(ok = mma_sync_all(mbar, phase, ok, args.err))) break;
        {
            const bool valid = t0 + r < N;
            float x[64];
            tmem_ld32f(trow + kColDV, *reinterpret_cast<float(*)[32]>(x));
            tmem_ld32f(trow + kColDV + 32, *reinterpret_cast<float(*)[32]>(x + 32));
            if (valid) store_row_bf16(args.dv + ((size_t)bh * N + t0 + r) * kBD, x);
            tmem_ld32f(trow + kColDK, *reinterpret_cast<float(*)[32]>(x));
            tmem_ld32f(trow + kColDK + 32, *reinterpret_cast<float(*)[32]>(x + 32));
#pragma unroll
            for (int cc = 0; cc < 64; ++cc) x[cc] = (x[cc] + rs[cc] + asum) * dphi_at(tk, r, cc);
            if (valid) store_row_bf16(args.dk + ((size_t)bh * N + t0 + r) * kBD, x);
        }
        __syncthreads();   // every thread has read r before it changes
        // R += phi(Q)^T g (A read MN-major, M-atom stride 0), r += sum_i e_i phi(Q_i)
        if (r == 0) {
            const uint64_t da = smem_desc(aq, 0, 1024), db = smem_desc(ag, kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ss(tmem + kColR, da + mnmajor_step(ks), db + mnmajor_step(ks), ID_S, 1);
        }
        colsum_add(tq, es, part, rs);
        if (!(ok = mma_sync_all(mbar, phase, ok, args.err))) break;
        if (r < kBD) {
            float v[32];
            for (int c0 = 0; c0 < kBD; c0 += 32) {
                tmem_ld32f(trow + kColR + c0, v);
                store_state32(snap, r, c0, v);
            }
        }
        operands_ready();
    }
    // dL/dS_0 = R, dL/dZ_0 = r after the first chunk
    if (ok && args.dS0 && r < kBD) {
        float v[32];
        for (int c0 = 0; c0 < kBD; c0 += 32) {
            tmem_ld32f(trow + kColR + c0, v);
#pragma unroll
            for (int j = 0; j < 32; ++j) args.dS0[((size_t)bh * kBD + r) * kBD + c0 + j] = v[j];
        }
        args.dz0[(size_t)bh * kBD + r] = rs[r];
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (q4 == 0) tmem_dealloc(tmem, kBwdTmemCols);
}

}  // namespace

bool tc_backward_supported(const la_shape &s) { return s.dtype == LA_DTYPE_BF16 && s.D == kBD && s.M == kBD; }

// Workspace: g as bf16 [BH, N, 64] then e as fp32 [BH, N].
cudaError_t tc_causal_backward(const BwdProblem &p, const DeviceInfo &dev) {
    if (p.D != kBD || p.M != kBD) return cudaErrorInvalidValue;
    const size_t g_bytes = (size_t)p.BH * p.N * kBD * 2;
    if (p.ws_bytes < g_bytes + (size_t)p.BH * p.N * 4) return cudaErrorInvalidValue;
    __nv_bfloat16 *g_ws = (__nv_bfloat16 *)p.ws;
    float *e_ws = (float *)((uint8_t *)p.ws + g_bytes);
    CUtensorMap tq, tk, tv, tdo, tg;
    if (!cached_tmap_bf16_3d(&tq, p.q, kBD, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tk, p.k, kBD, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tv, p.v, kBD, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tdo, p.dout, kBD, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tg, g_ws, kBD, p.N, p.BH, 64, kC))
        return cudaErrorInvalidValue;
    BwdArgs a;
    a.dq = (__nv_bfloat16 *)p.dq;
    a.dk = (__nv_bfloat16 *)p.dk;
    a.dv = (__nv_bfloat16 *)p.dv;
    a.g_ws = g_ws;
    a.e_ws = e_ws;
    a.S0 = p.S0;
    a.z0 = p.z0;
    a.dSN = p.dSN;
    a.dzN = p.dzN;
    a.dS0 = p.dS0;
    a.dz0 = p.dz0;
    a.N = p.N;
    a.err = dev.err_word;
    cudaError_t e;
    if ((e = set_smem(bwd_tc_pass1_kernel, kBwdSmem)) != cudaSuccess) return e;
    if ((e = set_smem(bwd_tc_pass2_kernel, kBwdSmem)) != cudaSuccess) return e;
    bwd_tc_pass1_kernel<<<(unsigned)p.BH, kBT, kBwdSmem, p.stream>>>(tq, tk, tv, tdo, a);
    count_launches(1);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    bwd_tc_pass2_kernel<<<(unsigned)p.BH, kBT, kBwdSmem, p.stream>>>(tq, tk, tv, tg, a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace la

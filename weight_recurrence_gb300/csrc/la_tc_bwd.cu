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
// MMAs.  One CTA of two warpgroups (256 threads) per head: thread t owns row
// t % 128 of every 128-row accumulator (TMEM lane t % 128), and the two
// warpgroups split each CUDA-core phase by columns (or by operand), meeting
// in shared memory where a row reduction spans both halves.  The phases of a
// chunk run one after the other; around them:
//   - the state products (S += phi(K)^T V in pass 1, R += phi(Q)^T g in
//     pass 2) and the column sums of Z and r are issued with the chunk's
//     first product, since the chunk's own gradient terms read the bf16
//     snapshot of the state taken before it;
//   - the next chunk's tiles are requested by TMA after the chunk's first
//     products (two stages), and its feature maps (and, in pass 2, its e)
//     are computed while the chunk's largest products run;
//   - the products against the state's bf16 hi and lo parts that share an
//     A operand run as one N = 128 MMA ([hi | lo] are adjacent atoms);
//   - g, dQ, dK and dV leave through TMA stores from swizzled tiles (dQ, dK
//     and dV from stage tiles whose last reader has finished).
// Every wait is bounded; a CTA that gives up records LA_ERR_TIMEOUT and skips
// the rest of its work.
#include "la_common.cuh"
#include "la_internal.h"
#include "tc_host.h"
#include "tc_kernels.cuh"
#include "tc_ptx.cuh"

// Optional per-phase timeline of CTA 0 of the forward sweep for performance
// work: compiled only with -DLA_TRACE (never in the library build).
#ifdef LA_TRACE
__device__ unsigned long long g_la_trace_bwd[2][32][12];
extern "C" int la_trace_read_bwd(unsigned long long *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_la_trace_bwd, sizeof(g_la_trace_bwd));
}
#define BWD_TRACE(pass, it, ev)                                                                      \
    do {                                                                                             \
        if (blockIdx.x == 0 && threadIdx.x == 0 && (it) < 32) g_la_trace_bwd[pass][it][ev] = clock64(); \
    } while (0)
#else
#define BWD_TRACE(pass, it, ev) ((void)0)
#endif

namespace la {
namespace {

constexpr int kBD = 64;                     // D = M
constexpr int kBT = 256;                    // threads: two warpgroups
constexpr int kTile = kC * kBD * 2;         // one 128 x 64 bf16 tile, 16 KB
constexpr int kStage = 4 * kTile;           // Q, K, V, dO (pass 1) or Q, K, V, g (pass 2)
constexpr int kOffGT = 2 * kStage;          // pass 1: g of the chunk (MMA operand, store source)
constexpr int kOffPsi = kOffGT + kTile;     // [2] psi(K) (pass 1) or psi(Q) (pass 2), an MMA operand, per chunk parity
constexpr int kOffSnap = kOffPsi + 2 * kTile;   // state S or R as bf16 hi then lo parts, [64 rows][64] each
constexpr int kSnap = kBD * kBD * 2;        // 8 KB
constexpr int kOffZ = kOffSnap + 2 * kSnap; // fp32 Z or r, [2][64]: before and after the chunk
constexpr int kOffE = kOffZ + 2 * kBD * 4;  // pass 2: fp32 e of the chunk, [2][128] by chunk parity
constexpr int kOffPart = kOffE + 2 * kC * 4;    // fp32 [8][64] column-sum parts
constexpr int kOffX = kOffPart + 8 * kBD * 4;   // fp32 [3][2][128] row-reduction halves
constexpr int kOffBar = kOffX + 3 * 2 * kC * 4;
constexpr int kOffSlot = kOffBar + 8 * 8;
constexpr int kBwdSmem = kOffSlot + 16;
constexpr uint32_t kBwdTmemCols = 512;
static_assert(kBwdSmem <= (int)kSmemMax, "shared memory budget");
static_assert(kOffGT % 1024 == 0 && kOffPsi % 1024 == 0 && kOffSnap % 1024 == 0, "swizzled tiles on 1 KB");

// TMEM columns.  Pass 1: P, then A, in [0, 128); num in [128, 256) as two
// halves to be added (P V + phi(Q) S_hi, then phi(Q) S_lo: one N = 128
// product against [S_hi | S_lo]); S in [256, 320); P as bf16 hi parts in
// [320, 384) (later A as bf16) and lo parts in [384, 448); dphi(Q) in
// [448, 512).  Pass 2: P^T in [0, 128) (bf16 in [0, 64)), A^T in [128, 256)
// (bf16 in [128, 192)); dV in [256, 384) as two halves (P^T g + phi(K) R_hi,
// then phi(K) R_lo); R in [384, 448); dphi(K) in [448, 512).
constexpr uint32_t kColP = 0, kColNum = 128, kColS = 256, kColPH = 320, kColPL = 384, kColDQ = 448;
constexpr uint32_t kColA2 = 128, kColDV = 256, kColR = 384, kColDK = 448;

struct BwdArgs {
    float *e_ws;             // [BH, N]
    const float *S0, *z0, *dSN, *dzN;
    float *dS0, *dz0;
    int N;
    int *err;
};

// This thread waits (bounded) for the next phase of an MMA-completion
// barrier, which thread 0 arrives on with tcgen05.commit; TMEM reads may
// follow.  Returns false if the wait gave up (the caller makes it CTA-uniform
// at its next barrier_and).
__device__ __forceinline__ bool mma_wait(uint64_t *bar, uint32_t &phase) {
    const bool got = mbar_wait_bounded(bar, phase, now_ns() + kWaitNs, nullptr);
    phase ^= 1u;
    tc_fence_after();
    return got;
}

// All threads finished their TMEM stores and generic shared-memory writes:
// make them visible to the MMAs and TMA stores thread 0 issues next.  Returns
// true iff every thread passed `mine`; records a timeout otherwise.
__device__ __forceinline__ bool barrier_and(bool mine, int *err) {
    tmem_wait_st();
    fence_proxy_async();
    tc_fence_before();
    const bool all = __syncthreads_and(mine ? 1 : 0) != 0;
    tc_fence_after();
    if (!all && threadIdx.x == 0) record_error(err, kErrTimeout);
    return all;
}

__device__ __forceinline__ void operands_ready() { barrier_and(true, nullptr); }

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

// Columns [c0, c0 + 64) of this thread's row r of a 128-column fp32
// accumulator at `src`: keeps columns j <= r (lower) or j >= r, adds colv[j]
// (if given) or rowv to the kept entries, writes them as 32 packed bf16
// pairs at `dst` and, if HILO, the rounding error of each as a second bf16
// operand at `dst_lo`.  Returns the fp32 sum of the kept entries (after the
// addition, before rounding).  All four loads are in flight before the wait.
template <bool HILO>
__device__ __forceinline__ float mask64(uint32_t src, int c0, int r, bool lower, float rowv, const float *colv,
                                        uint32_t dst, uint32_t dst_lo) {
    uint32_t x[4][16];
#pragma unroll
    for (int b = 0; b < 4; ++b) tmem_ld16(src + c0 + 16 * b, x[b]);
    tmem_wait_ld();
    float sum = 0.f;
    uint32_t hp[2][16], lp[2][16];
#pragma unroll
    for (int j = 0; j < 64; j += 2) {
        const int c = c0 + j;
        const bool k0 = lower ? (c <= r) : (c >= r);
        const bool k1 = lower ? (c + 1 <= r) : (c + 1 >= r);
        const float2 cv = colv ? *reinterpret_cast<const float2 *>(colv + c) : make_float2(rowv, rowv);
        const float add0 = cv.x, add1 = cv.y;
        const float a0 = k0 ? __uint_as_float(x[j / 16][j % 16]) + add0 : 0.f;
        const float a1 = k1 ? __uint_as_float(x[j / 16][j % 16 + 1]) + add1 : 0.f;
        sum += a0 + a1;
        const uint32_t h = pack_bf16x2(a0, a1);
        hp[j / 32][(j % 32) / 2] = h;
        if (HILO) lp[j / 32][(j % 32) / 2] = pack_bf16x2(a0 - bf16lo(h), a1 - bf16hi(h));
    }
    tmem_st16(dst, hp[0]);
    tmem_st16(dst + 16, hp[1]);
    if (HILO) {
        tmem_st16(dst_lo, lp[0]);
        tmem_st16(dst_lo + 16, lp[1]);
    }
    return sum;
}

// Column sums of a 128 x 64 bf16 tile (swizzled), each row weighted by w[row]
// (or 1), in eight parts: thread t sums the column pair 2(t % 32), 2(t % 32)+1
// over rows 16(t / 32) .. +16 into part[t / 32][.].  A warp reads one
// 128-byte row per step.
__device__ __forceinline__ void colsum_part(const uint8_t *tile, const float *w, float *part) {
    const int t = threadIdx.x, cp = t & 31, rg = t >> 5;
    float s0 = 0.f, s1 = 0.f;
#pragma unroll
    for (int i = 16 * rg; i < 16 * rg + 16; ++i) {
        const uint32_t x = *reinterpret_cast<const uint32_t *>(tile + sw128_offset(i, 2 * cp));
        const float wi = w ? w[i] : 1.f;
        s0 = fmaf(wi, bf16lo(x), s0);
        s1 = fmaf(wi, bf16hi(x), s1);
    }
    part[rg * kBD + 2 * cp] = s0;
    part[rg * kBD + 2 * cp + 1] = s1;
}

// The eight parts of column c summed.
__device__ __forceinline__ float colsum_total(const float *part, int c) {
    float s = 0.f;
#pragma unroll
    for (int g = 0; g < 8; ++g) s += part[g * kBD + c];
    return s;
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

// sum_c a[c] z[c] over 32 columns, z 16-byte aligned in shared memory.
__device__ __forceinline__ float dot32(const float *a, const float *z) {
    float acc = 0.f;
#pragma unroll
    for (int c4 = 0; c4 < 8; ++c4) {
        const float4 w = reinterpret_cast<const float4 *>(z)[c4];
        acc = fmaf(a[4 * c4], w.x, acc);
        acc = fmaf(a[4 * c4 + 1], w.y, acc);
        acc = fmaf(a[4 * c4 + 2], w.z, acc);
        acc = fmaf(a[4 * c4 + 3], w.w, acc);
    }
    return acc;
}

// Columns [c0, c0 + 32) of row r of a swizzled 128 x 64 bf16 tile as fp32.
__device__ __forceinline__ void tile_row32(const uint8_t *tile, int r, int c0, float *v) {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        const uint4 w = *reinterpret_cast<const uint4 *>(tile + sw128_offset(r, c0 + 8 * c8));
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            v[8 * c8 + 2 * u] = bf16lo(ww[u]);
            v[8 * c8 + 2 * u + 1] = bf16hi(ww[u]);
        }
    }
}

// phi in place on a 128 x 64 bf16 tile by all 256 threads, four 16-byte
// chunks per thread (rows >= zero_from become zeros).
__device__ __forceinline__ void phi_tile_all(uint8_t *tile, int t, int zero_from) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4 *>(tile + (t + i * kBT) * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[i].x = phi_bf16x2(v[i].x);
        v[i].y = phi_bf16x2(v[i].y);
        v[i].z = phi_bf16x2(v[i].z);
        v[i].w = phi_bf16x2(v[i].w);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t off = (uint32_t)(t + i * kBT) * 16u;
        *reinterpret_cast<uint4 *>(tile + off) = (int)(off >> 7) >= zero_from ? make_uint4(0u, 0u, 0u, 0u) : v[i];
    }
}

// psi(x) = phi(x) - 1 (x for x > 0, e^x - 1 otherwise) of a raw bf16 tile into
// `psi` (same layout) and phi(x) = psi(x) + 1 in place, from one fp32
// exponential per element; rows >= zero_from as zeros in both.  Where the
// inputs are small, phi(x) is close to 1 and its bf16 rounding swamps x; the
// gradient products use psi and add the row sums of the other factor
// separately.
__device__ __forceinline__ void psi_phi_tile(uint8_t *tile, uint8_t *psi, int t, int zero_from) {
    uint4 v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4 *>(tile + (t + i * kBT) * 16);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t off = (uint32_t)(t + i * kBT) * 16u;
        const uint32_t ww[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint32_t ps[4], ph[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float a = bf16lo(ww[u]), b = bf16hi(ww[u]);
            float ea, eb;
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ea) : "f"(a * 1.4426950408889634f));
            asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(eb) : "f"(b * 1.4426950408889634f));
            ps[u] = pack_bf16x2(a > 0.f ? a : ea - 1.f, b > 0.f ? b : eb - 1.f);
            ph[u] = pack_bf16x2(a > 0.f ? a + 1.f : ea, b > 0.f ? b + 1.f : eb);
        }
        const bool zero = (int)(off >> 7) >= zero_from;
        *reinterpret_cast<uint4 *>(psi + off) = zero ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(ps[0], ps[1], ps[2], ps[3]);
        *reinterpret_cast<uint4 *>(tile + off) = zero ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(ph[0], ph[1], ph[2], ph[3]);
    }
}

// ------------------------------------------------------------------ pass 1
__global__ void __launch_bounds__(kBT, 1)
bwd_tc_pass1_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                    const __grid_constant__ CUtensorMap tm_g, const __grid_constant__ CUtensorMap tm_dq,
                    const BwdArgs args)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, r = tid & (kC - 1), wg = tid >> 7, q4 = (tid >> 5) & 3;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int bh = blockIdx.x, N = args.N;
    const int nch = (N + kC - 1) / kC;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar), *mbar = full + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + kOffSlot);
    uint8_t *gt = smem + kOffGT, *psi = smem + kOffPsi, *snap = smem + kOffSnap;
    float *zs = reinterpret_cast<float *>(smem + kOffZ), *part = reinterpret_cast<float *>(smem + kOffPart);
    float *xr = reinterpret_cast<float *>(smem + kOffX), *xg = xr + 2 * kC, *xa = xg + 2 * kC;

    bool ok = (smem_u32(smem) & 1023u) == 0;
    if (tid == 0) {
        if (!ok) record_error(args.err, kErrTimeout);
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        mbar_init(&mbar[2], 1);
        fence_mbar_init();
    }
    if (tid < 32) {
        tmem_alloc(slot, kBwdTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + lane_off;
    pdl_wait_cta();   // set-up above touched no global memory

    // the starting state: S (TMEM, fp32; lanes 64-127 unused) and its bf16
    // snapshot, Z (shared memory, fp32); warpgroup h takes columns 32h..32h+31
    {
        float v[32];
        const int c0 = 32 * wg;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (r < kBD && args.S0) ? args.S0[((size_t)bh * kBD + r) * kBD + c0 + j] : 0.f;
        tmem_st32f(trow + kColS + c0, v);
        if (r < kBD) store_state32(snap, r, c0, v);
        if (tid < kBD) zs[tid] = args.z0 ? args.z0[(size_t)bh * kBD + tid] : 0.f;
    }
    if (tid == 0 && ok && nch > 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_do);
        prefetch_tmap(&tm_g);
        prefetch_tmap(&tm_dq);
        load_chunk(smem, &full[0], &tm_q, &tm_k, &tm_v, &tm_do, 0, bh);
    }
    operands_ready();

    uint32_t ph0 = 0, ph1 = 0, ph2 = 0;
    constexpr uint32_t ID_P = idesc_bf16(128, 128, 0, 0);     // K-major A and B
    constexpr uint32_t ID_MN = idesc_bf16(128, kBD, 0, 1);    // K-major A, MN-major B
    constexpr uint32_t ID_MN2 = idesc_bf16(128, 2 * kBD, 0, 1);   // ... N = 128: [hi | lo] of the state
    constexpr uint32_t ID_KK = idesc_bf16(128, kBD, 0, 0);    // K-major A and B
    constexpr uint32_t ID_S = idesc_bf16(128, kBD, 1, 1);     // MN-major A and B
    for (int it = 0; it < nch && ok; ++it) {
        BWD_TRACE(0, it, 0);
        const int s = it & 1, t0 = it * kC, rows = min(kC, N - t0);
        uint8_t *st = smem + s * kStage;
        uint8_t *tq = st, *tk = st + kTile, *tv = st + 2 * kTile, *tdo = st + 3 * kTile;
        const float *zc = zs + kBD * s;   // Z before this chunk
        float *zn = zs + kBD * (s ^ 1);   // Z after it
        uint8_t *psi_c = psi + s * kTile;
        // feature maps in place (rows past the sequence end become zero), and
        // psi(K) = phi(K) - 1 for the dQ product: the first chunk's here, every
        // later chunk's while the previous chunk's num product runs (made
        // visible by that chunk's last barrier)
        if (it == 0) {
            const bool landed = mbar_wait_bounded(&full[0], 0, now_ns() + kWaitNs, nullptr);
            if (!(ok = barrier_and(landed, args.err))) break;
            phi_tile_all(tq, tid, rows);
            psi_phi_tile(tk, psi_c, tid, rows);
            operands_ready();
        }
        BWD_TRACE(0, it, 1);
        const uint32_t aq = smem_u32(tq), ak = smem_u32(tk), av = smem_u32(tv), ag = smem_u32(gt), as = smem_u32(snap);
        // P = phi(Q) phi(K)^T;  S += phi(K)^T V (A read MN-major with M-atom
        // stride 0: lanes 64-127 repeat lanes 0-63).  Then the next chunk's
        // tiles into the other stage, once the TMA stores out of it (dQ) and
        // of the g tile have read their sources.
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColP, kmajor_base(aq) + kmajor_step(ks), kmajor_base(ak) + kmajor_step(ks), ID_P, ks > 0);
            const uint64_t da = smem_desc(ak, 0, 1024), db = smem_desc(av, kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ss(tmem + kColS, da + mnmajor_step(ks), db + mnmajor_step(ks), ID_S, 1);
            mma_commit(&mbar[0]);
            tma_store_wait_read0();
            if (it + 1 < nch) load_chunk(smem + (s ^ 1) * kStage, &full[s ^ 1], &tm_q, &tm_k, &tm_v, &tm_do, t0 + kC, bh);
        }
        // meanwhile: the column sums of phi(K), this half of phi(Q_i) . Z
        colsum_part(tk, nullptr, part);
        float qz;
        {
            float pq[32];
            tile_row32(tq, r, 32 * wg, pq);
            qz = dot32(pq, zc + 32 * wg);
        }
        bool mine = mma_wait(&mbar[0], ph0);
        BWD_TRACE(0, it, 2);
        // mask (j <= i) as bf16 hi and lo parts (num feeds e, where the output's
        // error would enter every entry of A); the halves of the row sums
        xr[wg * kC + r] = qz + mask64<true>(trow + kColP, 64 * wg, r, true, 0.f, nullptr, trow + kColPH + 32 * wg,
                                            trow + kColPL + 32 * wg);
        if (!(ok = barrier_and(mine, args.err))) break;
        BWD_TRACE(0, it, 3);
        if (tid < kBD) zn[tid] = zc[tid] + colsum_total(part, tid);
        const bool valid = t0 + r < N;
        const float inv = valid ? 1.f / (xr[r] + xr[kC + r]) : 0.f;
        // num = phi(Q) [S_hi | S_lo] (one N = 128 product: the snapshot's lo part
        // is its second 64-column atom), then + P V into the first half
        if (tid == 0) {
            const uint64_t dv = smem_desc(av, kC * 128, 1024), ds = smem_desc(as, kSnap, 1024);
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColNum, kmajor_base(aq) + kmajor_step(ks), ds + mnmajor_step(ks), ID_MN2, ks > 0);
#pragma unroll
            for (int part2 = 0; part2 < 2; ++part2)
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_f16_ts(tmem + kColNum, tmem + (part2 ? kColPL : kColPH) + ks * 8, dv + mnmajor_step(ks), ID_MN, 1);
            mma_commit(&mbar[1]);
        }
        // meanwhile g_i = dO_i / den_i (columns 32h..32h+31 by warpgroup h),
        // rounded to bf16 as the MMAs (and pass 2) use it, into the operand tile
        float g[32];
        tile_row32(tdo, r, 32 * wg, g);
#pragma unroll
        for (int c = 0; c < 32; ++c) g[c] = __bfloat162float(__float2bfloat16_rn(g[c] * inv));
        store_snap32<kC>(gt, r, 32 * wg, g);
        operands_ready();
        // g to the workspace (rows past the end are not written); A2 = g V^T
        // and the g S^T part of dphi(Q)
        if (tid == 0) {
            tma_store_3d(&tm_g, gt, 0, t0, bh);
            tma_store_commit();
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColP, kmajor_base(ag) + kmajor_step(ks), kmajor_base(av) + kmajor_step(ks), ID_P, ks > 0);
            mma_commit(&mbar[2]);
#pragma unroll
            for (int part2 = 0; part2 < 2; ++part2)
#pragma unroll
                for (int ks = 0; ks < kBD / 16; ++ks)
                    mma_f16_ss(tmem + kColDQ, kmajor_base(ag) + kmajor_step(ks),
                               kmajor_base(as + part2 * kSnap) + kmajor_step(ks, kBD), ID_KK, part2 > 0 || ks > 0);
        }
        // meanwhile the next chunk's feature maps (its tiles were issued after
        // this chunk's first products)
        bool nxt = true;
        if (it + 1 < nch) {
            nxt = mbar_wait_bounded(&full[s ^ 1], ((it + 1) >> 1) & 1, now_ns() + kWaitNs, nullptr);
            if (nxt) {
                uint8_t *st1 = smem + (s ^ 1) * kStage;
                const int rows1 = min(kC, N - t0 - kC);
                phi_tile_all(st1, tid, rows1);
                psi_phi_tile(st1 + kTile, psi + (s ^ 1) * kTile, tid, rows1);
            }
        }
        // e_i = -(g_i . num_i) / den_i, from the same bf16 g, so that the terms
        // A phi(K), g S^T and e Z stay consistent
        mine = mma_wait(&mbar[1], ph1) && nxt;
        BWD_TRACE(0, it, 4);
        {
            float num[32], lo[32];
            tmem_ld32f(trow + kColNum + 32 * wg, num);
            tmem_ld32f(trow + kColNum + kBD + 32 * wg, lo);
            float gn = 0.f;
#pragma unroll
            for (int c = 0; c < 32; ++c) gn = fmaf(g[c], num[c] + lo[c], gn);
            xg[wg * kC + r] = gn;
        }
        if (!(ok = barrier_and(mine, args.err))) break;
        const float e = valid ? -(xg[r] + xg[kC + r]) * inv : 0.f;
        if (wg == 0 && valid) args.e_ws[(size_t)bh * N + t0 + r] = e;
        mine = mma_wait(&mbar[2], ph2);
        BWD_TRACE(0, it, 5);
        // A = (A2 + e_i) masked to j <= i, as bf16; the halves of its row sum
        xa[wg * kC + r] = mask64<false>(trow + kColP, 64 * wg, r, true, e, nullptr, trow + kColPH + 32 * wg, 0u);
        if (!(ok = barrier_and(mine, args.err))) break;
        BWD_TRACE(0, it, 6);
        const float asum = xa[r] + xa[kC + r];
        // dphi(Q) += A psi(K)  (+ asum: the product with the 1 of phi = psi + 1)
        if (tid == 0) {
            const uint64_t dk = smem_desc(smem_u32(psi_c), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + kColDQ, tmem + kColPH + ks * 8, dk + mnmajor_step(ks), ID_MN, 1);
            mma_commit(&mbar[0]);
        }
        mine = mma_wait(&mbar[0], ph0);
        BWD_TRACE(0, it, 7);
        // dQ = (dphi(Q) + e_i Z) * phi'(Q), phi' = min(phi, 1), into the dO tile
        // (its last reader has finished) for the TMA store; the new state's
        // bf16 snapshot for the next chunk
        {
            float dq[32], pq[32];
            tmem_ld32f(trow + kColDQ + 32 * wg, dq);
            tile_row32(tq, r, 32 * wg, pq);
            const float4 *z4 = reinterpret_cast<const float4 *>(zc + 32 * wg);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 z = z4[c4];
                dq[4 * c4] = (fmaf(e, z.x, dq[4 * c4]) + asum) * fminf(pq[4 * c4], 1.f);
                dq[4 * c4 + 1] = (fmaf(e, z.y, dq[4 * c4 + 1]) + asum) * fminf(pq[4 * c4 + 1], 1.f);
                dq[4 * c4 + 2] = (fmaf(e, z.z, dq[4 * c4 + 2]) + asum) * fminf(pq[4 * c4 + 2], 1.f);
                dq[4 * c4 + 3] = (fmaf(e, z.w, dq[4 * c4 + 3]) + asum) * fminf(pq[4 * c4 + 3], 1.f);
            }
            store_snap32<kC>(tdo, r, 32 * wg, dq);
            if (q4 < 2) {
                float v[32];
                tmem_ld32f(trow + kColS + 32 * wg, v);
                store_state32(snap, r, 32 * wg, v);
            }
        }
        if (!(ok = barrier_and(mine, args.err))) break;   // also: every thread is done with this stage
        if (tid == 0) {
            tma_store_3d(&tm_dq, tdo, 0, t0, bh);
            tma_store_commit();
        }
        BWD_TRACE(0, it, 8);
    }
    if (tid == 0) tma_store_wait_all0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid < 32) tmem_dealloc(tmem, kBwdTmemCols);
}

// ------------------------------------------------------------------ pass 2
__global__ void __launch_bounds__(kBT, 1)
bwd_tc_pass2_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                    const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                    const BwdArgs args)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, r = tid & (kC - 1), wg = tid >> 7, q4 = (tid >> 5) & 3;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int bh = blockIdx.x, N = args.N;
    const int nch = (N + kC - 1) / kC;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kOffBar), *mbar = full + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + kOffSlot);
    uint8_t *psi = smem + kOffPsi, *snap = smem + kOffSnap;
    float *rs = reinterpret_cast<float *>(smem + kOffZ), *es = reinterpret_cast<float *>(smem + kOffE);
    float *part = reinterpret_cast<float *>(smem + kOffPart), *xa = reinterpret_cast<float *>(smem + kOffX);

    bool ok = (smem_u32(smem) & 1023u) == 0;
    if (tid == 0) {
        if (!ok) record_error(args.err, kErrTimeout);
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(&mbar[0], 1);
        mbar_init(&mbar[1], 1);
        mbar_init(&mbar[2], 1);
        fence_mbar_init();
    }
    if (tid < 32) {
        tmem_alloc(slot, kBwdTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + lane_off;
    pdl_wait_cta();   // set-up above touched no global memory

    // R, r start from the gradient reaching the final state (or zero)
    {
        float v[32];
        const int c0 = 32 * wg;
#pragma unroll
        for (int j = 0; j < 32; ++j) v[j] = (r < kBD && args.dSN) ? args.dSN[((size_t)bh * kBD + r) * kBD + c0 + j] : 0.f;
        tmem_st32f(trow + kColR + c0, v);
        if (r < kBD) store_state32(snap, r, c0, v);
        if (tid < kBD) rs[tid] = args.dzN ? args.dzN[(size_t)bh * kBD + tid] : 0.f;
    }
    if (tid == 0 && ok && nch > 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_g);
        prefetch_tmap(&tm_dk);
        prefetch_tmap(&tm_dv);
        load_chunk(smem, &full[0], &tm_q, &tm_k, &tm_v, &tm_g, (nch - 1) * kC, bh);
    }
    operands_ready();

    uint32_t ph0 = 0, ph1 = 0, ph2 = 0;
    constexpr uint32_t ID_P = idesc_bf16(128, 128, 0, 0);
    constexpr uint32_t ID_MN = idesc_bf16(128, kBD, 0, 1);
    constexpr uint32_t ID_MN2 = idesc_bf16(128, 2 * kBD, 0, 1);
    constexpr uint32_t ID_KK = idesc_bf16(128, kBD, 0, 0);
    constexpr uint32_t ID_S = idesc_bf16(128, kBD, 1, 1);
    for (int it = 0; it < nch && ok; ++it) {
        BWD_TRACE(1, it, 0);
        const int c = nch - 1 - it, s = it & 1, t0 = c * kC, rows = min(kC, N - t0);
        uint8_t *st = smem + s * kStage;
        uint8_t *tq = st, *tk = st + kTile, *tv = st + 2 * kTile, *tg = st + 3 * kTile;
        const float *rc = rs + kBD * s;   // r after this chunk (the reverse sum of the later ones)
        float *rn = rs + kBD * (s ^ 1);   // r including this chunk
        uint8_t *psi_c = psi + s * kTile;
        float *es_c = es + kC * s;
        // the first chunk's feature maps and e here, every later chunk's while
        // the previous chunk's dV and dphi(K) products run (made visible by
        // that chunk's last barrier)
        if (it == 0) {
            if (wg == 0) es_c[r] = t0 + r < N ? args.e_ws[(size_t)bh * N + t0 + r] : 0.f;
            const bool landed = mbar_wait_bounded(&full[0], 0, now_ns() + kWaitNs, nullptr);
            if (!(ok = barrier_and(landed, args.err))) break;
            psi_phi_tile(tq, psi_c, tid, rows);
            phi_tile_all(tk, tid, rows);
            operands_ready();
        }
        // the next chunk's e, loaded now and stored below, so that the load's
        // latency passes under this chunk's work
        const float e_next = (wg == 0 && it + 1 < nch) ? args.e_ws[(size_t)bh * N + t0 - kC + r] : 0.f;
        BWD_TRACE(1, it, 1);
        const uint32_t aq = smem_u32(tq), ak = smem_u32(tk), av = smem_u32(tv), ag = smem_u32(tg), as = smem_u32(snap);
        // P^T = phi(K) phi(Q)^T, then A^T = V g^T (rows j, columns i) and
        // R += phi(Q)^T g (A read MN-major, M-atom stride 0); then the next
        // chunk's tiles into the other stage, once the TMA stores out of it
        // (dV, dK) have read their sources
        if (tid == 0) {
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColP, kmajor_base(ak) + kmajor_step(ks), kmajor_base(aq) + kmajor_step(ks), ID_P, ks > 0);
            mma_commit(&mbar[0]);
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColA2, kmajor_base(av) + kmajor_step(ks), kmajor_base(ag) + kmajor_step(ks), ID_P, ks > 0);
            const uint64_t da = smem_desc(aq, 0, 1024), db = smem_desc(ag, kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ss(tmem + kColR, da + mnmajor_step(ks), db + mnmajor_step(ks), ID_S, 1);
            mma_commit(&mbar[1]);
            tma_store_wait_read0();
            if (it + 1 < nch) load_chunk(smem + (s ^ 1) * kStage, &full[s ^ 1], &tm_q, &tm_k, &tm_v, &tm_g, t0 - kC, bh);
        }
        // meanwhile the column sums sum_i e_i phi(Q_i)
        colsum_part(tq, es_c, part);
        // masks (i >= j) as bf16: warpgroup 0 P^T, warpgroup 1 A^T with e_i
        // added to the kept entries (and its row sums)
        bool mine = mma_wait(&mbar[0], ph0);
        if (wg == 0) {
            mask64<false>(trow + kColP, 0, r, false, 0.f, nullptr, trow + kColP, 0u);
            mask64<false>(trow + kColP, 64, r, false, 0.f, nullptr, trow + kColP + 32, 0u);
        }
        mine = mma_wait(&mbar[1], ph1) && mine;
        BWD_TRACE(1, it, 2);
        if (wg == 1) {
            float a = mask64<false>(trow + kColA2, 0, r, false, 0.f, es_c, trow + kColA2, 0u);
            a += mask64<false>(trow + kColA2, 64, r, false, 0.f, es_c, trow + kColA2 + 32, 0u);
            xa[r] = a;
        }
        if (!(ok = barrier_and(mine, args.err))) break;
        BWD_TRACE(1, it, 3);
        if (tid < kBD) rn[tid] = rc[tid] + colsum_total(part, tid);
        const float asum = xa[r];
        // dV = phi(K) [R_hi | R_lo] (one N = 128 product) + P^T g into its first
        // half;  dphi(K) = A^T psi(Q) + V R^T (+ asum)
        if (tid == 0) {
            const uint64_t dg = smem_desc(ag, kC * 128, 1024), dqm = smem_desc(smem_u32(psi_c), kC * 128, 1024);
            const uint64_t ds = smem_desc(as, kSnap, 1024);
#pragma unroll
            for (int ks = 0; ks < kBD / 16; ++ks)
                mma_f16_ss(tmem + kColDV, kmajor_base(ak) + kmajor_step(ks), ds + mnmajor_step(ks), ID_MN2, ks > 0);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + kColDV, tmem + kColP + ks * 8, dg + mnmajor_step(ks), ID_MN, 1);
            mma_commit(&mbar[2]);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + kColDK, tmem + kColA2 + ks * 8, dqm + mnmajor_step(ks), ID_MN, ks > 0);
#pragma unroll
            for (int part2 = 0; part2 < 2; ++part2)
#pragma unroll
                for (int ks = 0; ks < kBD / 16; ++ks)
                    mma_f16_ss(tmem + kColDK, kmajor_base(av) + kmajor_step(ks),
                               kmajor_base(as + part2 * kSnap) + kmajor_step(ks, kBD), ID_KK, 1);
            mma_commit(&mbar[0]);
        }
        // dV into the V tile (its last reader, the dphi(K) product, runs after
        // dV's: wait for both before writing), dK = (dphi(K) + r + asum) * phi'(K)
        // into the g tile (columns 32h..32h+31 by warpgroup h); the new R's
        // bf16 snapshot
        // meanwhile the next (earlier) chunk's e and feature maps
        if (it + 1 < nch) {
            if (wg == 0) es[kC * (s ^ 1) + r] = e_next;
            const bool nxt = mbar_wait_bounded(&full[s ^ 1], ((it + 1) >> 1) & 1, now_ns() + kWaitNs, nullptr);
            if (nxt) {
                uint8_t *st1 = smem + (s ^ 1) * kStage;
                const int rows1 = min(kC, N - (t0 - kC));
                psi_phi_tile(st1, psi + (s ^ 1) * kTile, tid, rows1);
                phi_tile_all(st1 + kTile, tid, rows1);
            }
            mine = mine && nxt;
        }
        float x[32];
        mine = mma_wait(&mbar[2], ph2) && mine;
        BWD_TRACE(1, it, 4);
        {
            float lo[32];
            tmem_ld32f(trow + kColDV + 32 * wg, x);
            tmem_ld32f(trow + kColDV + kBD + 32 * wg, lo);
#pragma unroll
            for (int c = 0; c < 32; ++c) x[c] += lo[c];
        }
        mine = mma_wait(&mbar[0], ph0) && mine;
        BWD_TRACE(1, it, 5);
        store_snap32<kC>(tv, r, 32 * wg, x);
        {
            float pk[32];
            tmem_ld32f(trow + kColDK + 32 * wg, x);
            tile_row32(tk, r, 32 * wg, pk);
            const float4 *r4 = reinterpret_cast<const float4 *>(rc + 32 * wg);
#pragma unroll
            for (int c4 = 0; c4 < 8; ++c4) {
                const float4 rv = r4[c4];
                x[4 * c4] = (x[4 * c4] + rv.x + asum) * fminf(pk[4 * c4], 1.f);
                x[4 * c4 + 1] = (x[4 * c4 + 1] + rv.y + asum) * fminf(pk[4 * c4 + 1], 1.f);
                x[4 * c4 + 2] = (x[4 * c4 + 2] + rv.z + asum) * fminf(pk[4 * c4 + 2], 1.f);
                x[4 * c4 + 3] = (x[4 * c4 + 3] + rv.w + asum) * fminf(pk[4 * c4 + 3], 1.f);
            }
            store_snap32<kC>(tg, r, 32 * wg, x);
            if (q4 < 2) {
                float v[32];
                tmem_ld32f(trow + kColR + 32 * wg, v);
                store_state32(snap, r, 32 * wg, v);
            }
        }
        if (!(ok = barrier_and(mine, args.err))) break;   // also: every thread is done with this stage
        if (tid == 0) {
            tma_store_3d(&tm_dv, tv, 0, t0, bh);
            tma_store_3d(&tm_dk, tg, 0, t0, bh);
            tma_store_commit();
        }
        BWD_TRACE(1, it, 6);
    }
    // dL/dS_0 = R, dL/dZ_0 = r after the first chunk
    if (ok && args.dS0 && r < kBD) {
        float v[32];
        tmem_ld32f(trow + kColR + 32 * wg, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) args.dS0[((size_t)bh * kBD + r) * kBD + 32 * wg + j] = v[j];
        if (wg == 0) args.dz0[(size_t)bh * kBD + r] = rs[kBD * (nch & 1) + r];
    }
    if (tid == 0) tma_store_wait_all0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid < 32) tmem_dealloc(tmem, kBwdTmemCols);
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
    CUtensorMap tq, tk, tv, tdo, tg, tdq, tdk, tdv;
    if (!cached_tmap_bf16_3d(&tq, p.q, kBD, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tk, p.k, kBD, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tv, p.v, kBD, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tdo, p.dout, kBD, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tg, g_ws, kBD, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tdq, p.dq, kBD, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tdk, p.dk, kBD, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tdv, p.dv, kBD, p.N, p.BH, 64, kC))
        return cudaErrorInvalidValue;
    BwdArgs a;
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
    e = launch_pdl(bwd_tc_pass1_kernel, dim3((unsigned)p.BH), dim3(kBT), kBwdSmem, p.stream, 0u, tq, tk, tv, tdo, tg,
                   tdq, a);
    count_launches(1);
    if (e != cudaSuccess) return e;
    // the reverse sweep's pdl_wait_cta() holds it until the forward sweep's g and e are written
    e = launch_pdl(bwd_tc_pass2_kernel, dim3((unsigned)p.BH), dim3(kBT), kBwdSmem, p.stream, 0u, tq, tk, tv, tg, tdk,
                   tdv, a);
    count_launches(1);
    return e;
}

}  // namespace la

// la_tc_delta.cu - the delta update rule of "Linear Transformers Are Secretly
// Fast Weight Programmers" (Schlag, Irie, Schmidhuber) with sum-normalised
// features, chunked onto tensor cores, for bf16 with feature width F = 64 and
// M = 64.
//
// Per token t (state S: F x M, retrieval S^T k):
//   vbar_t = S_{t-1}^T k_t,  S_t = S_{t-1} + k_t (beta_t (v_t - vbar_t))^T,
//   y_t = S_t^T q_t          (k, q the sum-normalised features).
// Regrouped by chunks of C = 128 tokens (exact in real arithmetic): with the
// pseudo-values u_t = beta_t (v_t - vbar_t) the state inside a chunk is
// S_t = S_0 + sum_{s<=t} k_s u_s^T, so the u_t solve the unit lower triangular
// system
//   u_t + beta_t sum_{s<t} (k_t . k_s) u_s = beta_t (v_t - S_0^T k_t),
// i.e. (I + diag(beta) tril(K K^T, -1)) U = diag(beta) (V - K S_0), and then
//   Y = Q S_0 + tril(Q K^T) U   (the diagonal kept: read-out after the update)
//   S_C = S_0 + K^T U.
// The products run on tcgen05 (bf16 operands, fp32 accumulators in TMEM; the
// state and U enter as bf16 hi + lo pairs); the triangular solve runs on CUDA
// cores in fp32, by blocks of 16 rows: rows of block b first take the product
// with the finished rows before it, then the block's own 16 x 16 unit lower
// triangular inverse.  It is done in two 64-row halves: between them the
// bottom rows take off L[64:128, 0:64] U[0:64] in one tcgen05 product (L as
// bf16, U as bf16 hi + lo).  One CTA of 256 threads per head; thread r < 128
// owns row r of every 128-row accumulator (TMEM lane r), threads 128..255
// share the CUDA-core phases.  The next chunk's tiles load by TMA meanwhile
// (two stages), and its beta and feature maps are computed while this chunk's
// last products run.  Every wait is bounded; a CTA that gives up records
// LA_ERR_TIMEOUT and skips the rest of its work.
#include "la_common.cuh"
#include "la_internal.h"
#include "tc_host.h"
#include "tc_kernels.cuh"
#include "tc_ptx.cuh"

// Optional per-phase timeline of CTA 0 for performance work: compiled only with
// -DLA_TRACE (never in the library build); read with la_trace_read_delta().
#ifdef LA_TRACE
__device__ unsigned long long g_la_trace_delta[64][8];
__device__ unsigned long long g_la_trace_solve[8][3];
extern "C" int la_trace_read_solve(unsigned long long *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_la_trace_solve, sizeof(g_la_trace_solve));
}
#define SOLVE_TRACE(it, b, ev)                                                                            \
    do {                                                                                                  \
        if (blockIdx.x == 0 && threadIdx.x == 0 && (it) == 2) g_la_trace_solve[b][ev] = clock64();        \
    } while (0)
extern "C" int la_trace_read_delta(unsigned long long *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_la_trace_delta, sizeof(g_la_trace_delta));
}
#define DELTA_TRACE(it, ev)                                                                       \
    do {                                                                                          \
        if (blockIdx.x == 0 && threadIdx.x == 0 && (it) < 64) g_la_trace_delta[it][ev] = clock64(); \
    } while (0)
#else
#define DELTA_TRACE(it, ev) ((void)0)
#define SOLVE_TRACE(it, b, ev) ((void)0)
#endif

namespace la {
namespace {

constexpr int kDF = 64;                       // feature width F (= M)
constexpr int kDT = 256;                      // threads
constexpr int kDTile = kC * 64 * 2;           // one 128 x 64 bf16 tile, 16 KB
constexpr int kDStage = 3 * kDTile;           // Q, K, V
constexpr int kDSnap = kDF * kDF * 2;         // state as bf16, [64 rows][64], 8 KB per part
constexpr int kDOffSnap = 2 * kDStage;        // S hi, S lo
constexpr int kDOffL = kDOffSnap + 2 * kDSnap;                 // L by 16-column blocks, fp32; later U hi, U lo tiles
constexpr int kDLBytes = 16 * (128 * 8 - 8 * 8 * 7) * 4;       // column blocks b = 0..7: rows 16 b .. 127 x 16
constexpr int kDUS = 68;                                       // row stride of the U work rows (floats)
constexpr int kDOffU = kDOffL + kDLBytes;                      // U work rows [128][kDUS] fp32
constexpr int kDOffA = kDOffU + kC * kDUS * 4;                   // a block's right-hand sides and solution, 2 x [16][64] fp32
constexpr int kDOffT = kDOffA + 2 * 16 * 64 * 4;               // diagonal block inverses [8][16][16] fp32
constexpr int kDOffB = kDOffT + 8 * 16 * 16 * 4;               // beta [2][128] fp32, by chunk parity
constexpr int kDOffBar = kDOffB + 2 * kC * 4;
constexpr int kDOffSlot = kDOffBar + 8 * 4;
constexpr int kDeltaSmem = kDOffSlot + 16;
static_assert(kDOffL % 1024 == 0 && kDOffSnap % 1024 == 0, "swizzled operand tiles need 1024-byte alignment");
static_assert(kDLBytes >= 2 * kDTile && kDLBytes % 1024 == 0, "L region also holds the U tiles");
static_assert(kDeltaSmem <= (int)kSmemMax, "shared memory budget");

// TMEM columns: G = K K^T at [0, 128) (then O at [0, 64)); P = Q K^T at
// [128, 256) (its masked bf16 form in [128, 192)); W = K S at [256, 320);
// the fp32 state S at [320, 384) (lanes 0-63); the solve's off-diagonal
// product L[64:128, 0:64] U[0:64] at [384, 448) (lanes 64-127).
constexpr uint32_t kTColG = 0, kTColO = 0, kTColP = 128, kTColW = 256, kTColS = 320, kTColC = 384;
// Bytes of L's column blocks 0-3 (the left 64 columns), free once the
// off-diagonal operand has been built from them: the top half of U goes
// there as bf16 hi and lo operand tiles ([64 rows][64], 8 KB each).
constexpr int kDLLeft = 16 * (128 * 4 - 8 * 4 * 3) * 4;
static_assert(kDLLeft >= 2 * 64 * 128 && kDLLeft % 1024 == 0, "left column blocks hold the U top tiles");
constexpr uint32_t kDeltaTmemCols = 512;

struct DeltaArgs {
    __nv_bfloat16 *out;            // [BH, N, 64] or null
    const __nv_bfloat16 *beta;     // [BH, N]
    float *S;                      // [BH, 64, 64] in/out or null
    int N;
    int feat, dr, nu;              // feature map of the rows (kFeatElu1Sum or kFeatDpfp, sum-normalised)
    int *err;
};

// L = diag(beta) tril(K K^T, -1) is kept by 16-column blocks: block b holds
// rows 16 b .. 127 of columns 16 b .. 16 b + 15, 16 floats per row (64-byte
// aligned rows), the four float4 slots of row i permuted by (i >> 1) & 3 so
// that 32 rows written at once by 32 lanes spread over all banks.  Offset of
// L[i][16 b + j] for i >= 16 b:
__device__ __forceinline__ int lblk(int b) { return 16 * (128 * b - 8 * b * (b - 1)); }
__device__ __forceinline__ int lrow16(int i, int b) { return lblk(b) + (i - 16 * b) * 16; }
__device__ __forceinline__ int lslot(int i, int j4) { return 4 * (j4 ^ ((i >> 1) & 3)); }

// Thread 0 commits the MMAs it issued to `bar`; every thread waits for that
// phase.  CTA-uniform result: false if any wait gave up (the phase is then
// left as it was, so that the exit path can wait for those MMAs once more).
__device__ __forceinline__ bool delta_mma_sync(uint64_t *bar, uint32_t &phase, bool ok, int *err) {
    if (threadIdx.x == 0 && ok) mma_commit(bar);
    const bool mine = ok && mbar_wait_bounded(bar, phase, now_ns() + kWaitNs, nullptr);
    if (ok && !mine && threadIdx.x == 0) record_error(err, kErrTimeout);
    const bool all = __syncthreads_and(mine ? 1 : 0) != 0;
    if (all) phase ^= 1u;
    tc_fence_after();
    return all;
}

// TMEM stores and generic shared-memory writes of all threads visible to the
// MMAs thread 0 issues next.
__device__ __forceinline__ void delta_operands_ready() {
    tmem_wait_st();
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Columns c0..c0+31 of row r of a fp32 64-column matrix as a bf16 hi part
// and the bf16 rounding error of hi (lo) into two MN-major tiles of `rows` rows.
template <int ROWS>
__device__ __forceinline__ void store_hilo32(uint8_t *hi_tile, uint8_t *lo_tile, int r, int c0, const float *v) {
    float hi[32], lo[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        hi[j] = __bfloat162float(__float2bfloat16_rn(v[j]));
        lo[j] = v[j] - hi[j];
    }
    store_snap32<ROWS>(hi_tile, r, c0, hi);
    store_snap32<ROWS>(lo_tile, r, c0, lo);
}

__global__ void __launch_bounds__(kDT, 1)
delta_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const DeltaArgs args)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, wg = tid >> 7, r = tid & 127, q4 = (tid >> 5) & 3;
    const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
    const int bh = blockIdx.x, N = args.N;
    const int nch = (N + kC - 1) / kC;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kDOffBar), *mbar = full + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(smem + kDOffSlot);
    uint8_t *snap = smem + kDOffSnap;
    float *Lp = reinterpret_cast<float *>(smem + kDOffL);
    uint8_t *uhi = smem + kDOffL, *ulo = smem + kDOffL + kDTile;   // U operand tiles (after the solve)
    float *Us = reinterpret_cast<float *>(smem + kDOffU);
    float *Ab = reinterpret_cast<float *>(smem + kDOffA);
    float *Tb = reinterpret_cast<float *>(smem + kDOffT);
    float *bs = reinterpret_cast<float *>(smem + kDOffB);

    bool ok = (smem_u32(smem) & 1023u) == 0;
    if (tid == 0) {
        if (!ok) record_error(args.err, kErrTimeout);
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    if (tid < 32) {
        tmem_alloc(slot, kDeltaTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + lane_off;
    pdl_wait_cta();   // set-up above touched no global memory

    // the starting state: S in TMEM (fp32, lanes 0-63) and its bf16 hi/lo snapshot
    if (wg == 0) {
        float v[32];
        for (int c0 = 0; c0 < kDF; c0 += 32) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = (r < kDF && args.S) ? args.S[((size_t)bh * kDF + r) * kDF + c0 + j] : 0.f;
            tmem_st32f(trow + kTColS + c0, v);
            if (r < kDF) store_hilo32<kDF>(snap, snap + kDSnap, r, c0, v);
        }
    }
    int issued = 0, consumed = 0;   // chunks whose tiles were requested / have landed
    bool mma_pending = false;       // an MMA wait gave up
    auto load_chunk = [&](int s, int t0) {
        ++issued;
        uint8_t *st = smem + s * kDStage;
        mbar_arrive_expect_tx(&full[s], kDStage);
        tma_load_3d(st, &tm_q, &full[s], 0, t0, bh);
        tma_load_3d(st + kDTile, &tm_k, &full[s], 0, t0, bh);
        tma_load_3d(st + 2 * kDTile, &tm_v, &full[s], 0, t0, bh);
    };
    if (tid == 0 && ok && nch > 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        load_chunk(0, 0);
    }
    delta_operands_ready();

    uint32_t phase = 0;
    constexpr uint32_t ID_P = idesc_bf16(128, 128, 0, 0);     // K-major A and B
    constexpr uint32_t ID_MN = idesc_bf16(128, kDF, 0, 1);    // K-major A, MN-major B
    constexpr uint32_t ID_S = idesc_bf16(128, kDF, 1, 1);     // MN-major A and B
    for (int it = 0; it < nch && ok; ++it) {
        const int s = it & 1, t0 = it * kC;
        const int valid = min(kC, N - t0);
        uint8_t *st = smem + s * kDStage;
        uint8_t *tq = st, *tk = st + kDTile, *tv = st + 2 * kDTile;
        float *bs_c = bs + kC * s;
        DELTA_TRACE(it, 0);
        if (tid == 0 && it + 1 < nch) load_chunk(s ^ 1, t0 + kC);
        // the next chunk's beta, loaded now and stored under this chunk's last
        // products, so that the load's latency passes under this chunk's work
        const int valid1 = it + 1 < nch ? min(kC, N - t0 - kC) : 0;
        const float b_next = (wg == 1 && r < valid1) ? __bfloat162float(args.beta[(size_t)bh * N + t0 + kC + r]) : 0.f;
        // ---- features in place: K rows (rows past the end zeroed) by the first
        // warpgroup, Q rows by the second; the first chunk's here, every later
        // chunk's (and its beta) under the previous chunk's last products
        if (it == 0) {
            if (wg == 1) bs_c[r] = r < valid ? __bfloat162float(args.beta[(size_t)bh * N + t0 + r]) : 0.f;
            const bool landed = mbar_wait_bounded(&full[s], 0, now_ns() + kWaitNs, nullptr);
            if (!landed && tid == 0) record_error(args.err, kErrTimeout);
            if (!(ok = __syncthreads_and(landed) != 0)) break;
            ++consumed;
            feature_row<kDF>(wg == 0 ? tk : tq, r, wg == 0 ? valid : kC, args.feat, args.dr, args.nu, true);
            delta_operands_ready();
        }
        DELTA_TRACE(it, 1);
        DELTA_TRACE(it, 2);
        const uint32_t aq = smem_u32(tq), ak = smem_u32(tk), as = smem_u32(snap);
        // ---- G = K K^T, P = Q K^T, W = K S_0 (S as hi + lo)
        if (tid == 0) {
            const uint64_t ds = smem_desc(as, kDF * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kDF / 16; ++ks) {
                mma_f16_ss(tmem + kTColG, kmajor_base(ak) + kmajor_step(ks), kmajor_base(ak) + kmajor_step(ks), ID_P, ks > 0);
                mma_f16_ss(tmem + kTColP, kmajor_base(aq) + kmajor_step(ks), kmajor_base(ak) + kmajor_step(ks), ID_P, ks > 0);
            }
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < kDF / 16; ++ks)
                    mma_f16_ss(tmem + kTColW, kmajor_base(ak) + kmajor_step(ks),
                               ds + (uint64_t)(part * kDSnap / 16) + mnmajor_step(ks), ID_MN, part > 0 || ks > 0);
        }
        if (!(ok = delta_mma_sync(mbar, phase, ok, args.err))) {
            mma_pending = true;
            break;
        }
        DELTA_TRACE(it, 3);
        if (wg == 0) {
            // row r of L = diag(beta) tril(G, -1) into the column blocks that hold
            // row r (zeros on and above the diagonal); P masked to j <= r as bf16 in place
            const float br = bs_c[r];
#pragma unroll 1
            for (int c0 = 0; c0 < kC; c0 += 32) {
                if (c0 > 32 * q4 + 31) break;        // warp-uniform: past every row of this warp
                float x[32];
                tmem_ld32f(trow + kTColG + c0, x);
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const int c = c0 + 4 * j4, b = c >> 4;
                    if (16 * b <= r) {
                        float4 o;
                        o.x = c < r ? br * x[4 * j4] : 0.f;
                        o.y = c + 1 < r ? br * x[4 * j4 + 1] : 0.f;
                        o.z = c + 2 < r ? br * x[4 * j4 + 2] : 0.f;
                        o.w = c + 3 < r ? br * x[4 * j4 + 3] : 0.f;
                        *reinterpret_cast<float4 *>(Lp + lrow16(r, b) + lslot(r, (c & 15) >> 2)) = o;
                    }
                }
            }
            uint32_t packed[4][16];
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                float x[32];
                tmem_ld32f(trow + kTColP + 32 * b, x);
#pragma unroll
                for (int j = 0; j < 32; j += 2) {
                    const int c = 32 * b + j;
                    packed[b][j / 2] = pack_bf16x2(c <= r ? x[j] : 0.f, c + 1 <= r ? x[j + 1] : 0.f);
                }
            }
#pragma unroll
            for (int b = 0; b < 4; ++b) tmem_st16(trow + kTColP + 16 * b, packed[b]);
        } else {
            // row r of the right-hand side diag(beta) (V - K S_0), fp32
            const float br = bs_c[r];
            float w[64];
            tmem_ld32f(trow + kTColW, *reinterpret_cast<float(*)[32]>(w));
            tmem_ld32f(trow + kTColW + 32, *reinterpret_cast<float(*)[32]>(w + 32));
#pragma unroll
            for (int c8 = 0; c8 < 8; ++c8) {
                const uint4 vv = *reinterpret_cast<const uint4 *>(tv + sw128_offset(r, 8 * c8));
                const uint32_t ww[4] = {vv.x, vv.y, vv.z, vv.w};
                float4 o0, o1;
                o0.x = br * (bf16lo(ww[0]) - w[8 * c8]);
                o0.y = br * (bf16hi(ww[0]) - w[8 * c8 + 1]);
                o0.z = br * (bf16lo(ww[1]) - w[8 * c8 + 2]);
                o0.w = br * (bf16hi(ww[1]) - w[8 * c8 + 3]);
                o1.x = br * (bf16lo(ww[2]) - w[8 * c8 + 4]);
                o1.y = br * (bf16hi(ww[2]) - w[8 * c8 + 5]);
                o1.z = br * (bf16lo(ww[3]) - w[8 * c8 + 6]);
                o1.w = br * (bf16hi(ww[3]) - w[8 * c8 + 7]);
                *reinterpret_cast<float4 *>(Us + r * kDUS + 8 * c8) = o0;
                *reinterpret_cast<float4 *>(Us + r * kDUS + 8 * c8 + 4) = o1;
            }
        }
        tmem_wait_st();
        __syncthreads();
        DELTA_TRACE(it, 4);
        // ---- inverses of the eight 16 x 16 diagonal blocks of I + L: thread
        // (block b, column c) solves column c by forward substitution
        if (tid < 128) {
            const int b = tid >> 4, c = tid & 15, base = 16 * b;
            float x[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                float a = i == c ? 1.f : 0.f;
                if (i > 0) {
                    // row i of the diagonal block: its (i + 3) / 4 first float4 slots
                    float lv[16];
#pragma unroll
                    for (int j4 = 0; j4 < (i + 3) / 4; ++j4) {
                        const float4 t = *reinterpret_cast<const float4 *>(Lp + lrow16(base + i, b) + lslot(base + i, j4));
                        lv[4 * j4] = t.x; lv[4 * j4 + 1] = t.y; lv[4 * j4 + 2] = t.z; lv[4 * j4 + 3] = t.w;
                    }
#pragma unroll
                    for (int j = 0; j < i; ++j) a = fmaf(-lv[j], x[j], a);
                }
                x[i] = i < c ? 0.f : a;
            }
#pragma unroll
            for (int i = 0; i < 16; ++i) Tb[(b * 16 + i) * 16 + c] = x[i];
        }
        __syncthreads();
        DELTA_TRACE(it, 5);
        // ---- forward substitution by blocks of 16 rows, right-looking, with the
        // right-hand sides in registers: warp g owns rows i = g (mod 8), lane l
        // columns l and l + 32.  For block b the two owned rows of the block go
        // to Ab, are solved with the block's 16 x 16 inverse into Ab2, and every
        // later owned row of the same half takes off L[i][block b] U_b.  The
        // two 64-row halves are solved apart: between them the bottom rows
        // take off L[64:128, 0:64] U[0:64] in one tensor-core product (L in
        // bf16, U as bf16 hi + lo), which is 4/7 of the solve's FMAs.
        {
            const int g = tid >> 5, l = tid & 31;
            float acc[16][2];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                acc[k][0] = Us[(g + 8 * k) * kDUS + l];
                acc[k][1] = Us[(g + 8 * k) * kDUS + l + 32];
            }
            float *Ab2 = Ab + 16 * 64;
            auto solve_block = [&](const int b, const int kend) {
                SOLVE_TRACE(it, b, 0);
                // the block's rows owned here: local rows g and g + 8 (k = 2b, 2b + 1)
                Ab[g * 64 + l] = acc[2 * b][0];
                Ab[g * 64 + l + 32] = acc[2 * b][1];
                Ab[(g + 8) * 64 + l] = acc[2 * b + 1][0];
                Ab[(g + 8) * 64 + l + 32] = acc[2 * b + 1][1];
                __syncthreads();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int lr = g + 8 * h;                       // local row, warp-uniform
                    const float *Ti = Tb + (b * 16 + lr) * 16;
                    float x0 = 0.f, x1 = 0.f;
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        if (j > lr) break;
                        const float t = Ti[j];
                        x0 = fmaf(t, Ab[j * 64 + l], x0);
                        x1 = fmaf(t, Ab[j * 64 + l + 32], x1);
                    }
                    acc[2 * b + h][0] = x0;
                    acc[2 * b + h][1] = x1;
                    Ab2[lr * 64 + l] = x0;
                    Ab2[lr * 64 + l + 32] = x1;
                }
                __syncthreads();
                SOLVE_TRACE(it, b, 1);
                float ub[16][2];
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    ub[j][0] = Ab2[j * 64 + l];
                    ub[j][1] = Ab2[j * 64 + l + 32];
                }
#pragma unroll
                for (int k = 2 * b + 2; k < kend; ++k) {
                    const int row = g + 8 * k;
                    const float *Lr = Lp + lrow16(row, b);
                    float a0 = acc[k][0], a1 = acc[k][1], c0 = 0.f, c1 = 0.f;
#pragma unroll
                    for (int j4 = 0; j4 < 4; ++j4) {
                        const float4 lv = *reinterpret_cast<const float4 *>(Lr + lslot(row, j4));
                        a0 = fmaf(-lv.x, ub[4 * j4][0], a0);
                        a1 = fmaf(-lv.x, ub[4 * j4][1], a1);
                        c0 = fmaf(-lv.y, ub[4 * j4 + 1][0], c0);
                        c1 = fmaf(-lv.y, ub[4 * j4 + 1][1], c1);
                        a0 = fmaf(-lv.z, ub[4 * j4 + 2][0], a0);
                        a1 = fmaf(-lv.z, ub[4 * j4 + 2][1], a1);
                        c0 = fmaf(-lv.w, ub[4 * j4 + 3][0], c0);
                        c1 = fmaf(-lv.w, ub[4 * j4 + 3][1], c1);
                    }
                    acc[k][0] = a0 + c0;
                    acc[k][1] = a1 + c1;
                }
                SOLVE_TRACE(it, b, 2);
            };
#pragma unroll
            for (int b = 0; b < 4; ++b) solve_block(b, 8);
            // U[0:64] to the work rows
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                Us[(g + 8 * k) * kDUS + l] = acc[k][0];
                Us[(g + 8 * k) * kDUS + l + 32] = acc[k][1];
            }
            __syncthreads();
            // operands of the off-diagonal product: A = L[:, 0:64] as bf16 (rows
            // 0-63 zero) into the V tile, dead since the right-hand sides were
            // formed; then U[0:64] as bf16 hi + lo into L's left column blocks
            {
                const int row = tid & (kC - 1), c0 = 32 * (tid >> 7);
                float a[32];
#pragma unroll
                for (int j4 = 0; j4 < 8; ++j4) {
                    const int c = c0 + 4 * j4, b = c >> 4;
                    float4 lv = make_float4(0.f, 0.f, 0.f, 0.f);
                    if (row >= kDF) lv = *reinterpret_cast<const float4 *>(Lp + lrow16(row, b) + lslot(row, (c & 15) >> 2));
                    a[4 * j4] = lv.x; a[4 * j4 + 1] = lv.y; a[4 * j4 + 2] = lv.z; a[4 * j4 + 3] = lv.w;
                }
                store_snap32<kC>(tv, row, c0, a);
            }
            __syncthreads();
            uint8_t *uth = smem + kDOffL, *utl = uth + kDF * 128;
            if (tid < 2 * kDF) {
                const int row = tid & (kDF - 1), c0 = 32 * (tid >> 6);
                float u[32];
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(Us + row * kDUS + c0 + j);
                    u[j] = x.x; u[j + 1] = x.y; u[j + 2] = x.z; u[j + 3] = x.w;
                }
                store_hilo32<kDF>(uth, utl, row, c0, u);
            }
            delta_operands_ready();
            if (tid == 0) {
#pragma unroll
                for (int part = 0; part < 2; ++part) {
                    const uint64_t du = smem_desc(smem_u32(part ? utl : uth), kDF * 128, 1024);
#pragma unroll
                    for (int ks = 0; ks < kDF / 16; ++ks)
                        mma_f16_ss(tmem + kTColC, kmajor_base(smem_u32(tv)) + kmajor_step(ks), du + mnmajor_step(ks), ID_MN,
                                   part > 0 || ks > 0);
                }
            }
            if (!(ok = delta_mma_sync(mbar, phase, ok, args.err))) {
                mma_pending = true;
                break;
            }
            // the bottom rows' corrections through the work rows (TMEM lanes
            // 64-127: warps 2, 3 and 6, 7, 32 columns each)
            if (q4 >= 2) {
                float cv[32];
                tmem_ld32f(trow + kTColC + 32 * wg, cv);
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(Us + r * kDUS + 32 * wg + j) = make_float4(cv[j], cv[j + 1], cv[j + 2], cv[j + 3]);
            }
            __syncthreads();
#pragma unroll
            for (int k = 8; k < 16; ++k) {
                acc[k][0] -= Us[(g + 8 * k) * kDUS + l];
                acc[k][1] -= Us[(g + 8 * k) * kDUS + l + 32];
            }
            __syncthreads();   // the corrections are read before the rows are overwritten below
#pragma unroll
            for (int b = 4; b < 8; ++b) solve_block(b, 16);
            // U (all rows) back to the work rows for the tile conversion below
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                Us[(g + 8 * k) * kDUS + l] = acc[k][0];
                Us[(g + 8 * k) * kDUS + l + 32] = acc[k][1];
            }
            __syncthreads();
        }
        DELTA_TRACE(it, 6);
        // ---- U as bf16 hi + lo operand tiles (over the dead L): row r, half wg
        {
            float u[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {
                const float4 x = *reinterpret_cast<const float4 *>(Us + r * kDUS + 32 * wg + j);
                u[j] = x.x; u[j + 1] = x.y; u[j + 2] = x.z; u[j + 3] = x.w;
            }
            store_hilo32<kC>(uhi, ulo, r, 32 * wg, u);
        }
        delta_operands_ready();
        DELTA_TRACE(it, 7);
        // ---- O = Q S_0 + tril(P) U;  S += K^T U
        if (tid == 0) {
            const uint64_t ds = smem_desc(as, kDF * 128, 1024);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int ks = 0; ks < kDF / 16; ++ks)
                    mma_f16_ss(tmem + kTColO, kmajor_base(aq) + kmajor_step(ks),
                               ds + (uint64_t)(part * kDSnap / 16) + mnmajor_step(ks), ID_MN, part > 0 || ks > 0);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const uint64_t du = smem_desc(smem_u32(part ? ulo : uhi), kC * 128, 1024);
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_f16_ts(tmem + kTColO, tmem + kTColP + ks * 8, du + mnmajor_step(ks), ID_MN, 1);
            }
            // K^T read MN-major with M-atom stride 0 (lanes 64-127 repeat 0-63)
            const uint64_t da = smem_desc(ak, 0, 1024);
#pragma unroll
            for (int part = 0; part < 2; ++part) {
                const uint64_t du = smem_desc(smem_u32(part ? ulo : uhi), kC * 128, 1024);
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks)
                    mma_f16_ss(tmem + kTColS, da + mnmajor_step(ks), du + mnmajor_step(ks), ID_S, 1);
            }
        }
        // meanwhile the next chunk's beta and feature maps (its tiles were
        // requested at the top of this chunk)
        bool nxt = true;
        if (it + 1 < nch) {
            if (wg == 1) bs[kC * (s ^ 1) + r] = b_next;
            nxt = mbar_wait_bounded(&full[s ^ 1], ((it + 1) >> 1) & 1, now_ns() + kWaitNs, nullptr);
            if (nxt) {
                uint8_t *st1 = smem + (s ^ 1) * kDStage;
                feature_row<kDF>(wg == 0 ? st1 + kDTile : st1, r, wg == 0 ? valid1 : kC, args.feat, args.dr, args.nu,
                                 true);
            }
        }
        if (!(ok = delta_mma_sync(mbar, phase, ok, args.err))) {
            mma_pending = true;
            break;
        }
        if (!(ok = __syncthreads_and(nxt) != 0)) {
            if (tid == 0) record_error(args.err, kErrTimeout);
            break;
        }
        if (it + 1 < nch) ++consumed;
        // ---- output rows; the new state's bf16 snapshot for the next chunk
        if (wg == 0) {
            if (args.out) {                          // warp-uniform: the TMEM loads are warp-collective
                float o[64];
                tmem_ld32f(trow + kTColO, *reinterpret_cast<float(*)[32]>(o));
                tmem_ld32f(trow + kTColO + 32, *reinterpret_cast<float(*)[32]>(o + 32));
                if (r < valid) {
                    uint4 *dst = reinterpret_cast<uint4 *>(args.out + ((size_t)bh * N + t0 + r) * kDF);
                    uint4 w[8];
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8)
                        w[c8] = make_uint4(pack_bf16x2(o[8 * c8], o[8 * c8 + 1]), pack_bf16x2(o[8 * c8 + 2], o[8 * c8 + 3]),
                                           pack_bf16x2(o[8 * c8 + 4], o[8 * c8 + 5]), pack_bf16x2(o[8 * c8 + 6], o[8 * c8 + 7]));
                    if ((reinterpret_cast<uintptr_t>(args.out) & 31u) == 0) {   // 256-bit stores
#pragma unroll
                        for (int c16 = 0; c16 < 4; ++c16) st_global_v8(dst + 2 * c16, w[2 * c16], w[2 * c16 + 1]);
                    } else {
#pragma unroll
                        for (int c8 = 0; c8 < 8; ++c8) dst[c8] = w[c8];
                    }
                }
            }
        } else if (r < kDF) {
            float v[32];
            for (int c0 = 0; c0 < kDF; c0 += 32) {
                tmem_ld32f(trow + kTColS + c0, v);
                store_hilo32<kDF>(snap, snap + kDSnap, r, c0, v);
            }
        }
        delta_operands_ready();   // also: every thread is done with this stage
    }
    // the final state
    if (ok && args.S && wg == 1 && r < kDF && nch > 0) {
        float v[32];
        for (int c0 = 0; c0 < kDF; c0 += 32) {
            tmem_ld32f(trow + kTColS + c0, v);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(args.S + ((size_t)bh * kDF + r) * kDF + c0 + j) =
                    make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
        }
    }
    // on the error path: no copy may still be writing shared memory and no MMA
    // may still be running when the CTA frees its TMEM and exits (bounded waits)
    if (!ok && tid == 0) {
        for (int c = consumed; c < issued; ++c)
            mbar_wait_bounded(&full[c & 1], (c >> 1) & 1, now_ns() + kWaitNs, nullptr);
        if (mma_pending) mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid < 32) tmem_dealloc(tmem, kDeltaTmemCols);
}

}  // namespace

bool tc_delta_supported(const la_shape &s, const la_variant &v) {
    if (s.dtype != LA_DTYPE_BF16 || v.update != LA_UPDATE_DELTA || v.norm != LA_NORM_SUM || s.M != kDF) return false;
    if (v.feature_map == LA_FM_ELU1) return s.D == kDF;
    if (v.feature_map == LA_FM_DPFP) return (s.D == 32 && v.nu == 1) || (s.D == 16 && v.nu == 2);
    return false;
}

cudaError_t tc_delta(const Problem &p, const void *beta, const la_variant &v, const DeviceInfo &dev) {
    CUtensorMap tq, tk, tv;
    if (!tc::cached_tmap_bf16_3d(&tq, p.q, p.D, p.N, p.BH, 64, kC) ||
        !tc::cached_tmap_bf16_3d(&tk, p.k, p.D, p.N, p.BH, 64, kC) ||
        !tc::cached_tmap_bf16_3d(&tv, p.v, kDF, p.N, p.BH, 64, kC))
        return cudaErrorInvalidValue;
    DeltaArgs a;
    a.out = reinterpret_cast<__nv_bfloat16 *>(p.out);
    a.beta = reinterpret_cast<const __nv_bfloat16 *>(beta);
    a.S = p.S;
    a.N = p.N;
    a.feat = v.feature_map == LA_FM_ELU1 ? kFeatElu1Sum : kFeatDpfp;
    a.dr = p.D;
    a.nu = v.nu;
    a.err = dev.err_word;
    cudaError_t e = set_smem(delta_tc_kernel, kDeltaSmem);
    if (e != cudaSuccess) return e;
    e = launch_pdl(delta_tc_kernel, dim3((unsigned)p.BH), dim3(kDT), kDeltaSmem, p.stream, 0u, tq, tk, tv, a);
    count_launches(1);
    return e;
}

}  // namespace la

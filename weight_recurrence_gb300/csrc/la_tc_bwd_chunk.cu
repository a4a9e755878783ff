// la_tc_bwd_chunk.cu - tensor-core (tcgen05 + TMA) backward of the causal
// form, "Transformers are RNNs" sec. 3.3 eqs. (10)-(12) (the gradient the
// page describes as cumulative sums, sec. 3.3.1, through the chain rule), for
// bf16 tensors with D, M in {64, 128}: each head's 128-row chunks are cut into
// segments of consecutive chunks, one CTA per segment and pass.
//
// With S_c, z_c the state entering chunk c (the sums over the chunks before
// it, plus a carried-in state) and R_c, r_c the reverse sums after it
// (R = sum phi(Q_i) g_i^T, r = sum e_i phi(Q_i) over the later chunks, plus
// the gradient reaching the final state), every chunk's gradients depend on
// its own rows and these four sums only:
//   P = phi(Q) phi(K)^T masked to j <= i;  num = P V + phi(Q) S_c;
//   den = P 1 + phi(Q) . z_c;  g = dO / den;  e_i = -(g_i . num_i) / den_i;
//   A = (g V^T + e 1^T) masked to j <= i;
//   dphi(Q) = A phi(K) + g S_c^T + e z_c^T;
//   dphi(K) = A^T phi(Q) + V R_c^T + 1 r_c^T;  dV = P^T g + phi(K) R_c;
//   dQ = dphi(Q) min(phi(Q), 1),  dK = dphi(K) min(phi(K), 1).
// Five launches: the key sums [S | z] of every segment (the causal forward's
// segment-sum pre-pass; skipped with one segment per head); an exclusive scan
// over each head's segments into the state entering each segment; the query
// pass, one CTA per segment walking its chunks in order with S in TMEM
// (S += phi(K_c)^T V_c after each chunk) and z on CUDA cores: dQ, g (bf16) and
// e kept for the key pass, and the segment's [dR | dr] = sum phi(Q)^T [g | e];
// the reverse scan of those into the sums after each segment (started from the
// final state's gradient; its total is the carried-in state's gradient); the
// key pass, one CTA per segment walking its chunks backwards with R in TMEM:
// dK, dV.  The sums enter the products as bf16 hi + lo pairs, the masked P
// that forms num as hi + lo, e is formed from the bf16 g the products use, and
// the products whose terms cancel along the 1 of phi take psi = phi - 1 as
// the operand with the 1 added in fp32 (row sums, and column sums for the
// state updates), so that terms which cancel in exact arithmetic cancel to
// fp32 rounding.  Two warpgroups per CTA: thread t owns row t mod 128 (TMEM
// lane) and one half of the columns (or one of two operands) of every
// CUDA-core phase.  Every wait is bounded; a CTA that gives up records
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
// Exclusive scan of per-segment vectors of W = D*M + D floats, in place, over
// the segments of each head (reverse: from the last segment down).  The
// running sum starts from `init` ([BH][D*M] then [BH][D], the vector's two
// parts; null: zero) and its final value goes to `total` (same layout; may be
// null).  has_x = 0: the slots hold no input (taken as zero), so each slot
// receives the initial value.  Thread (head, e4) owns elements 4 e4 .. 4 e4 + 3;
// the loads of sixteen slots are issued before their sums.
__global__ void __launch_bounds__(256)
seg_scan_kernel(float *ws, int nseg, int DM, int D, const float *init_s, const float *init_z, float *tot_s,
                float *tot_z, int reverse, int has_x)
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
    float4 *base = reinterpret_cast<float4 *>(ws) + bh * nseg * W4 + e4;
    constexpr int U = 16;
    for (int c0 = 0; c0 < nseg; c0 += U) {
        float4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int c = reverse ? nseg - 1 - (c0 + u) : c0 + u;
            x[u] = (has_x && c0 + u < nseg) ? __ldcg(base + (long long)c * W4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            if (c0 + u >= nseg) break;
            const int c = reverse ? nseg - 1 - (c0 + u) : c0 + u;
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

struct SegBwdArgs {
    const float *ws_s;       // [BH, nseg, D*M + D]: [S | z] entering each segment
    float *ws_r;             // [BH, nseg, D*M + D]: query pass: each segment's [dR | dr];
                             // after the reverse scan: [R | r] after each segment
    __nv_bfloat16 *ws_g;     // [BH, N, M]: g (query pass writes it)
    float *ws_e;             // [BH, N]: e
    __nv_bfloat16 *g0, *g1;  // query pass: dQ; key pass: dK, dV
    int N, nch, nseg, L;     // rows and chunks per head, segments per head, chunks per segment (the last may be shorter)
    int *err;
};

// Both passes run two warpgroups: thread t handles row r = t mod 128 (TMEM
// lane r) and half h = t / 128 of the columns of every CUDA-core phase (or,
// where two operands are formed at once, one of them).
constexpr int kCT = 256;

// TMEM columns (512: one CTA per SM).
//   query pass: P (fp32, 128), then A as bf16 hi (0..63) and lo (64..127);
//   then A2 = g V^T (fp32, 128) and A2' (bf16, 0..63); num (M), then dphi(Q)
//   (D) in its place; the state S (M columns on lanes 0..D-1, without the
//   column sums of V, which are added in fp32 when it is read); dR summed over
//   the segment (M).
//   key pass: P^T (fp32, 0..127) and A^T (fp32, 128..255), then as bf16 at
//   0..63 (in place) and 192..255 (A^T's pieces converted last to first, so
//   each is read before the packed columns of an earlier one land on it);
//   dV (M) in between; dphi(K) (D); R (M columns on lanes 0..D-1, without the
//   column sums of g).
template <int D, int M>
struct SegCols {
    static constexpr uint32_t Q_P = 0, Q_AH = 0, Q_AL = 64, Q_A2 = 0, Q_NUM = 128, Q_DQ = 128;
    static constexpr uint32_t Q_S = 128 + (M > D ? M : D), Q_R = Q_S + M;
    static constexpr uint32_t K_PT = 0, K_AT = 128, K_PTB = 0, K_ATB = 192, K_DV = 64, K_DK = 256, K_R = 256 + D;
    static constexpr uint32_t COLS = 512;
    static_assert(Q_R + M <= COLS && K_R + M <= COLS && K_DV + M <= K_ATB, "TMEM budget");
};

// Operand tile of a D x M fp32 sum as bf16 [X_hi | X_lo], each part M/64
// swizzled atoms of D rows; read MN-major (as the B operand of phi X) and
// K-major (as the B operand of g X^T).  Also the fp32 staging area of a
// D x M block.
template <int D, int M>
struct SnapTile {
    static constexpr int ATOM = D * 128;
    static constexpr int LO = (M / 64) * ATOM;
    static constexpr int BYTES = 2 * LO;
    static_assert(D * M * 4 <= BYTES, "staging area");
};

// Columns [c0, c0 + 32) of row r of the fp32 state in TMEM at
// `col`, plus the column sums `cs` not held there, into the bf16 hi and lo
// parts of the operand tile.
template <int D, int M>
__device__ __forceinline__ void snap_from_tmem(uint32_t trow, uint32_t col, int r, int c0, const float *cs,
                                               uint8_t *snap) {
    float x[32], lo[32];
    tmem_ld32f(trow + col + c0, x);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
        const float v = x[j] + cs[c0 + j];
        const float hi = __bfloat162float(__float2bfloat16_rn(v));
        x[j] = hi;
        lo[j] = v - hi;
    }
    store_snap32<D>(snap, r, c0, x);
    store_snap32<D>(snap + SnapTile<D, M>::LO, r, c0, lo);
}

// The fp32 slot [X (D x M) | w (D)] into TMEM columns col.. (row d of X on
// lane d) and w into vec: coalesced 16-byte loads staged in `stage`, then each
// row's two threads store their halves of the row.  Ends with the stores
// complete and visible (block barrier).
template <int D, int M>
__device__ __forceinline__ void slot_to_tmem(const float *slot, float *stage, float *vec, uint32_t trow, uint32_t col,
                                             int t, int r, int h) {
    constexpr int R4 = M / 4;
    const float4 *src = reinterpret_cast<const float4 *>(slot);
    float4 *s4 = reinterpret_cast<float4 *>(stage);
    for (int f = t; f < D * R4; f += kCT) {
        const int row = f / R4, c4 = f % R4;
        s4[row * R4 + (c4 ^ (row % R4))] = __ldcg(src + f);
    }
    if (t < D) vec[t] = __ldcg(slot + D * M + t);
    __syncthreads();
    if (r < D) {
#pragma unroll 1
        for (int c0 = h * (M / 2); c0 < (h + 1) * (M / 2); c0 += 32) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 a = s4[r * R4 + ((c0 / 4 + j) ^ (r % R4))];
                v[4 * j] = a.x; v[4 * j + 1] = a.y; v[4 * j + 2] = a.z; v[4 * j + 3] = a.w;
            }
            tmem_st32f(trow + col + c0, v);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
}

// Partial column sums of a swizzled bf16 [kC x NC] tile (NC = 64 or 128),
// each row weighted by w[i] if W, and with ONEP of 1 + x (x a psi row: the
// column sums of phi): lane l of warp w sums the 8 columns of group l mod
// NC/8 over its rows with 16-byte loads, the warp's row shares are added by
// shuffles, and the warp's partial goes to part[w][column].
constexpr int kCW = kCT / 32;   // warps
template <int NC, bool W, bool ONEP>
__device__ __forceinline__ void colsum_part(const uint8_t *tile, const float *w, float *part, int t) {
    constexpr int CG = NC / 8, SPW = 32 / CG, RPT = kC / (kCW * SPW);
    const int lane = t & 31, wp = t >> 5, g = lane % CG, sh = lane / CG;
    const int row0 = (wp * SPW + sh) * RPT;
    const uint8_t *base = tile + (g / 8) * kC * 128;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.f;
#pragma unroll
    for (int i = row0; i < row0 + RPT; ++i) {
        const uint4 v = *reinterpret_cast<const uint4 *>(base + sw128_offset(i, (g % 8) * 8));
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
        const float wi = W ? w[i] : 1.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const float a = bf16lo(u[q]) + (ONEP ? 1.f : 0.f), b = bf16hi(u[q]) + (ONEP ? 1.f : 0.f);
            acc[2 * q] = fmaf(wi, a, acc[2 * q]);
            acc[2 * q + 1] = fmaf(wi, b, acc[2 * q + 1]);
        }
    }
#pragma unroll
    for (int off = CG; off < 32; off <<= 1)
#pragma unroll
        for (int k = 0; k < 8; ++k) acc[k] += __shfl_xor_sync(0xffffffffu, acc[k], off);
    if (lane < CG) {
        float4 *dst = reinterpret_cast<float4 *>(part + wp * kC + g * 8);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
}
template <int NC>
__device__ __forceinline__ float colsum_total(const float *part, int c) {
    float s = 0.f;
#pragma unroll
    for (int wp = 0; wp < kCW; ++wp) s += part[wp * kC + c];
    return s;
}

// Row r's 64 fp32 TMEM columns of half h at `src` (+ add(j) where keep(j),
// else 0) into bf16 at dst_hi (and the rounding remainders at dst_lo if LO):
// every thread first reads its columns, then (block barrier) writes, so the
// destinations may overlap any source column.  Returns the sum of the kept
// values (LO) or of their bf16 roundings.
template <bool LO, typename Keep, typename Add>
__device__ __forceinline__ float tmem_half_to_bf16(uint32_t src, uint32_t dst_hi, uint32_t dst_lo, int h, Keep keep,
                                                   Add add) {
    float x[64];
    tmem_ld32f(src + 64 * h, *reinterpret_cast<float(*)[32]>(x));
    tmem_ld32f(src + 64 * h + 32, *reinterpret_cast<float(*)[32]>(x + 32));
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    float sum = 0.f;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
        uint32_t w[16], l[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            const int c = 64 * h + 32 * p + 2 * j;
            const float a = keep(c) ? x[32 * p + 2 * j] + add(c) : 0.f;
            const float b = keep(c + 1) ? x[32 * p + 2 * j + 1] + add(c + 1) : 0.f;
            w[j] = pack_bf16x2(a, b);
            if (LO) {
                l[j] = pack_bf16x2(a - bf16lo(w[j]), b - bf16hi(w[j]));
                sum += a + b;
            } else {
                sum += bf16lo(w[j]) + bf16hi(w[j]);
            }
        }
        tmem_st16(dst_hi + 32 * h + 16 * p, w);
        if (LO) tmem_st16(dst_lo + 32 * h + 16 * p, l);
    }
    return sum;
}

// Row r's 128 fp32 TMEM columns at `src` (+ add(j) where keep(j), else 0) as
// bf16 into the 64 packed columns at dst, 32 columns at a time: in order when
// dst = src, last piece first when dst = src + 64, so that each piece is read
// before packed columns land on it.  Returns the sum of the bf16 roundings.
template <bool REV, typename Keep, typename Add>
__device__ __forceinline__ float tmem_row_to_bf16(uint32_t src, uint32_t dst, Keep keep, Add add) {
    float sum = 0.f;
#pragma unroll 1
    for (int p = 0; p < 4; ++p) {
        const int c0 = 32 * (REV ? 3 - p : p);
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

// Small fp32 arrays of both passes, after the tiles.
struct SegSmall {
    static constexpr int VEC = 0;               // z (query) or r (key), [128]
    static constexpr int CS = VEC + 128;        // column sums of V (query) or g (key) not in TMEM, [128]
    static constexpr int DR = CS + 128;         // query: dr summed over the segment, [128]
    static constexpr int ES = DR + 128;         // e of the chunk's rows, [128]
    static constexpr int XA = ES + 128;         // row-sum halves, [2][128]
    static constexpr int XB = XA + 256;         // [2][128]
    static constexpr int PA = XB + 256;         // column-sum partials, [warps][128] each
    static constexpr int PB = PA + kCW * 128;
    static constexpr int PC = PB + kCW * 128;
    static constexpr int FLOATS = PC + kCW * 128;
};

// ------------------------------------------------------------- query pass
template <int D, int M>
struct SQCfg {
    static constexpr int TQ = kC * D * 2, TV = kC * M * 2;
    static constexpr int OFF_K = TQ, OFF_V = 2 * TQ, OFF_G = 2 * TQ + TV;
    static constexpr int OFF_SNAP = 2 * TQ + 2 * TV;                    // [S_hi | S_lo]; fp32 staging
    static constexpr int OFF_SM = OFF_SNAP + SnapTile<D, M>::BYTES;     // SegSmall
    static constexpr int OFF_BAR = OFF_SM + SegSmall::FLOATS * 4;
    static constexpr int SMEM = OFF_BAR + 64;
    static_assert(SMEM <= (int)kSmemMax, "shared memory budget");
};

template <int D, int M>
__global__ void __launch_bounds__(kCT, 1)
seg_bwd_query_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_g,
                     const __grid_constant__ CUtensorMap tm_gw, const __grid_constant__ CUtensorMap tm_dq,
                     const SegBwdArgs args)
{
    using C = SQCfg<D, M>;
    using T = SegCols<D, M>;
    using SS = SegSmall;
    constexpr int MH = M / 2, DH = D / 2;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int t = threadIdx.x, r = t & (kC - 1), h = t >> 7;
    uint8_t *tq = smem, *tk = smem + C::OFF_K, *tv = smem + C::OFF_V, *tg = smem + C::OFF_G;
    uint8_t *snap = smem + C::OFF_SNAP;
    float *sm = reinterpret_cast<float *>(smem + C::OFF_SM);
    float *zs = sm + SS::VEC, *cv = sm + SS::CS, *drs = sm + SS::DR, *es = sm + SS::ES;
    float *xa = sm + SS::XA, *xb = sm + SS::XB, *pa = sm + SS::PA, *pb = sm + SS::PB, *pc = sm + SS::PC;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR), *mbar = full + 1;
    uint32_t *slot = reinterpret_cast<uint32_t *>(mbar + 1);
    const int bh = blockIdx.x / args.nseg, sg = blockIdx.x % args.nseg;
    const int c_begin = sg * args.L, c_end = min(args.nch, c_begin + args.L);

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
    if (t < 128) {
        cv[t] = 0.f;
        drs[t] = 0.f;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + ((uint32_t)(32 * (r >> 5)) << 16);
    CH_TRACE(0, 1);
    pdl_wait_cta();   // the scanned segment sums of the previous launch are complete
    // the state entering the segment: S into TMEM, z into zs
    slot_to_tmem<D, M>(args.ws_s + ((size_t)bh * args.nseg + sg) * (D * M + D), reinterpret_cast<float *>(snap), zs,
                       trow, T::Q_S, t, r, h);

    uint32_t phase = 0, fphase = 0;
    bool pending = false;   // MMAs committed but not complete (error path)
    bool loading = false;   // tiles requested but not landed (error path)
    constexpr uint32_t ID_P = idesc_bf16(128, 128, 0, 0);   // K-major A and B
    constexpr uint32_t ID_NV = idesc_bf16(128, M, 0, 1);    // A x (V or S) MN-major
    constexpr uint32_t ID_DQ = idesc_bf16(128, D, 0, 0);    // [g | g] x [S_hi | S_lo]^T, K-major
    constexpr uint32_t ID_DQ2 = idesc_bf16(128, D, 0, 1);   // A2' (TMEM) x psi(K) MN-major
    constexpr uint32_t ID_T = idesc_bf16(128, M, 1, 1);     // X^T x Y, both MN-major (dR, S updates)
    auto mma_wait_all = [&]() {
        if (t == 0) mma_commit(mbar);
        const bool got = mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
        if (got) phase ^= 1u;
        tc_fence_after();
        return __syncthreads_and(got ? 1 : 0) != 0;
    };
    for (int c = c_begin; ok && c < c_end; ++c) {
    const int t0 = c * kC, valid = min(kC, args.N - t0);
    CH_TRACE(0, 2);
    if (t == 0) {
        tma_store_wait_read0();   // the previous chunk's g and dQ stores have read their tiles
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
    // [S_c hi | S_c lo] from the TMEM state plus the column sums of V
    if (r < D)
#pragma unroll 1
        for (int c0 = MH * h; c0 < MH * h + MH; c0 += 32) snap_from_tmem<D, M>(trow, T::Q_S, r, c0, cv, snap);
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
    if (t == 0 && ok && c + 1 < c_end) {
        const int tn = t0 + kC;
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
            tma_prefetch_3d(&tm_q, j * 64, tn, bh);
            tma_prefetch_3d(&tm_k, j * 64, tn, bh);
        }
#pragma unroll
        for (int j = 0; j < M / 64; ++j) {
            tma_prefetch_3d(&tm_v, j * 64, tn, bh);
            tma_prefetch_3d(&tm_g, j * 64, tn, bh);
        }
    }
    CH_TRACE(0, 4);
    // phi(Q) (half 0) and psi(K) = phi(K) - 1 (half 1; the 1 enters as the row
    // sums of phi(Q)); rows past the end become zeros.  Then the row sums of
    // phi(Q) and phi(Q) . z
    float sq = 0.f, qz = 0.f;
    if (ok) {
        if (h == 0) phi_tile<D>(tq, r, valid);
        else psi_tile<D>(tk, r, valid);
        ok = operands_ready(true);
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            float f[32];
            load_row32(tq, r, c0, f);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                sq += f[j];
                qz = fmaf(f[j], zs[c0 + j], qz);
            }
        }
    }
    CH_TRACE(0, 5);
    // ---- phi(Q) psi(K)^T; meanwhile the column sums of V and psi(K) (the
    // state update's 1 terms)
    if (ok) {
        if (t == 0)
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::Q_P, kmajor_base(smem_u32(tq)) + kmajor_step(ks),
                           kmajor_base(smem_u32(tk)) + kmajor_step(ks), ID_P, ks > 0);
        colsum_part<M, false, false>(tv, nullptr, pa, t);
        colsum_part<D, false, false>(tk, nullptr, pb, t);
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(0, 6);
    // ---- A = P = phi(Q) psi(K)^T + sq masked to j <= r, as bf16 hi and lo
    // parts (num feeds e, which enters every entry of A2'); its row sum
    if (ok) {
        xa[h * kC + r] = tmem_half_to_bf16<true>(trow + T::Q_P, trow + T::Q_AH, trow + T::Q_AL, h,
                                                 [&](int j) { return j <= r; }, [&](int) { return sq; });
        ok = operands_ready(true);
    }
    CH_TRACE(0, 7);
    // ---- num = phi(Q) S_hi + A_hi V + A_lo V + phi(Q) S_lo
    if (ok) {
        if (t == 0) {
            const uint64_t dq = kmajor_base(smem_u32(tq));
            const uint64_t db = smem_desc(smem_u32(snap), D * 128, 1024);
            const uint64_t dl = smem_desc(smem_u32(snap + SnapTile<D, M>::LO), D * 128, 1024);
            const uint64_t dv = smem_desc(smem_u32(tv), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::Q_NUM, dq + kmajor_step(ks), db + mnmajor_step(ks), ID_NV, ks > 0);
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
        const float den = xa[r] + xa[kC + r] + qz;
        const float inv = r < valid ? 1.f / den : 0.f;
        float dot = 0.f;
#pragma unroll
        for (int c0 = 0; c0 < MH; c0 += 32) {
            float x[32], gv[32];
            tmem_ld32f(trow + T::Q_NUM + MH * h + c0, x);
            load_row32(tg, r, MH * h + c0, gv);
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                gv[j] = __bfloat162float(__float2bfloat16_rn(gv[j] * inv));
                dot = fmaf(gv[j], x[j], dot);
            }
            store_snap32<kC>(tg, r, MH * h + c0, gv);
        }
        xb[h * kC + r] = dot;
        __syncthreads();
        e = -(xb[r] + xb[kC + r]) * inv;
        if (h == 0) {
            es[r] = e;
            if (r < valid) args.ws_e[(size_t)bh * args.N + t0 + r] = e;
        }
        ok = operands_ready(true);
    }
    CH_TRACE(0, 9);
    // ---- g to the workspace (TMA store; rows past the end are not written);
    // A2 = g V^T;  dphi(Q) = [g | g] [S_hi | S_lo]^T;  dR += phi(Q)^T g;
    // meanwhile dr's partial sums of e_i phi(Q_i)
    if (ok) {
        if (t == 0) {
#pragma unroll
            for (int j = 0; j < M / 64; ++j) tma_store_3d(&tm_gw, tg + j * kC * 128, j * 64, t0, bh);
            tma_store_commit();
            const uint64_t dg = kmajor_base(smem_u32(tg));
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::Q_A2, dg + kmajor_step(ks), kmajor_base(smem_u32(tv)) + kmajor_step(ks), ID_P, ks > 0);
            const uint64_t db = kmajor_base(smem_u32(snap)), dl = kmajor_base(smem_u32(snap + SnapTile<D, M>::LO));
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::Q_DQ, dg + kmajor_step(ks), db + kmajor_step(ks, D), ID_DQ, ks > 0);
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::Q_DQ, dg + kmajor_step(ks), dl + kmajor_step(ks, D), ID_DQ, 1);
            // A read MN-major; at D = 64 with M-atom stride 0 (lanes 64-127
            // repeat lanes 0-63 and are never read)
            const uint64_t da = smem_desc(smem_u32(tq), D == 64 ? 0 : kC * 128, 1024);
            const uint64_t dgb = smem_desc(smem_u32(tg), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ss(tmem + T::Q_R, da + mnmajor_step(ks), dgb + mnmajor_step(ks), ID_T, c > c_begin || ks > 0);
        }
        colsum_part<D, true, false>(tq, es, pc, t);
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(0, 10);
    // ---- A2' = (A2 + e_r) masked to j <= r, as bf16 (columns of half h); its
    // row sum (the product with the 1 of phi(K) = psi(K) + 1)
    if (ok) {
        xa[h * kC + r] = tmem_half_to_bf16<false>(trow + T::Q_A2, trow + T::Q_A2, 0u, h, [&](int j) { return j <= r; },
                                                  [&](int) { return e; });
        ok = operands_ready(true);
    }
    CH_TRACE(0, 11);
    // ---- dphi(Q) += A2' psi(K);  S += psi(K)^T V (the chunk's state update;
    // its 1 terms are the column sums taken above)
    if (ok) {
        if (t == 0) {
            const uint64_t dk = smem_desc(smem_u32(tk), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + T::Q_DQ, tmem + T::Q_A2 + ks * 8, dk + mnmajor_step(ks), ID_DQ2, 1);
            const uint64_t dka = smem_desc(smem_u32(tk), D == 64 ? 0 : kC * 128, 1024);
            const uint64_t dvb = smem_desc(smem_u32(tv), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ss(tmem + T::Q_S, dka + mnmajor_step(ks), dvb + mnmajor_step(ks), ID_T, 1);
        }
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(0, 12);
    // ---- dQ = (dphi(Q) + asum + e z) min(phi(Q), 1), columns of half h, over
    // phi(Q) in its tile (each thread reads its row's values before writing
    // them), then stored by TMA (rows past the end are not written)
    if (ok) {
        const float asum = xa[r] + xa[kC + r];
#pragma unroll
        for (int c0 = 0; c0 < DH; c0 += 32) {
            float d32[32], f[32];
            tmem_ld32f(trow + T::Q_DQ + DH * h + c0, d32);
            load_row32(tq, r, DH * h + c0, f);
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = (d32[j] + asum + e * zs[DH * h + c0 + j]) * fminf(f[j], 1.f);
            store_snap32<kC>(tq, r, DH * h + c0, f);
        }
    }
    // the chunk's tiles and TMEM are free for the next one (once the dQ store
    // has read its tile); then the column sums move z, the V sums and dr on to
    // the next chunk
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (ok) {
        if (t == 0) {
#pragma unroll
            for (int j = 0; j < D / 64; ++j) tma_store_3d(&tm_dq, tq + j * kC * 128, j * 64, t0, bh);
            tma_store_commit();
        }
        if (t < M) cv[t] += colsum_total<M>(pa, t);
        if (t < D) {
            zs[t] += (float)valid + colsum_total<D>(pb, t);
            drs[t] += colsum_total<D>(pc, t);
        }
    }
    __syncthreads();
    }
    CH_TRACE(0, 13);
    // the segment's [dR | dr]: rows staged in the operand tile, coalesced stores
    if (ok) {
        float *dst = args.ws_r + ((size_t)bh * args.nseg + sg) * (D * M + D);
        float *stage = reinterpret_cast<float *>(snap);
        if (r < D) {
            float y[32];
#pragma unroll 1
            for (int c0 = MH * h; c0 < MH * h + MH; c0 += 32) {
                tmem_ld32f(trow + T::Q_R + c0, y);
                stage_row32_f32<M>(stage, r, c0, y);
            }
        }
        if (t < D) dst[D * M + t] = drs[t];
        __syncthreads();
        store_staged_f32<D, M>(dst, stage, t, kCT);
    }
    if (!ok && t == 0) {
        record_error(args.err, kErrTimeout);
        if (loading) mbar_wait_bounded(full, fphase, now_ns() + kWaitNs, nullptr);
        if (pending) mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
    }
    if (t == 0) tma_store_wait_all0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (t < 32) tmem_dealloc(tmem, T::COLS);
    CH_TRACE(0, 14);
}

// --------------------------------------------------------------- key pass
template <int D, int M>
struct SKCfg {
    static constexpr int TQ = kC * D * 2, TV = kC * M * 2;
    static constexpr int OFF_K = TQ, OFF_V = 2 * TQ, OFF_G = 2 * TQ + TV;
    static constexpr int OFF_SNAP = 2 * TQ + 2 * TV;                    // [R_hi | R_lo]; fp32 staging
    static constexpr int OFF_SM = OFF_SNAP + SnapTile<D, M>::BYTES;     // SegSmall
    static constexpr int OFF_BAR = OFF_SM + SegSmall::FLOATS * 4;
    static constexpr int SMEM = OFF_BAR + 64;
    static_assert(SMEM <= (int)kSmemMax, "shared memory budget");
};

template <int D, int M>
__global__ void __launch_bounds__(kCT, 1)
seg_bwd_key_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_gw,
                   const __grid_constant__ CUtensorMap tm_dk, const __grid_constant__ CUtensorMap tm_dv,
                   const SegBwdArgs args)
{
    using C = SKCfg<D, M>;
    using T = SegCols<D, M>;
    using SS = SegSmall;
    constexpr int MH = M / 2;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int t = threadIdx.x, r = t & (kC - 1), h = t >> 7;
    uint8_t *tq = smem, *tk = smem + C::OFF_K, *tv = smem + C::OFF_V, *tg = smem + C::OFF_G;
    uint8_t *snap = smem + C::OFF_SNAP;
    float *sm = reinterpret_cast<float *>(smem + C::OFF_SM);
    float *rsv = sm + SS::VEC, *cg = sm + SS::CS, *es = sm + SS::ES, *pa = sm + SS::PA, *pb = sm + SS::PB;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR), *mbar = full + 1;
    uint32_t *slot = reinterpret_cast<uint32_t *>(mbar + 1);
    const int bh = blockIdx.x / args.nseg, sg = blockIdx.x % args.nseg;
    const int c_begin = sg * args.L, c_end = min(args.nch, c_begin + args.L);

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
    if (t < 128) cg[t] = 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + ((uint32_t)(32 * (r >> 5)) << 16);
    CH_TRACE(1, 1);
    pdl_wait_cta();   // the query pass and the reverse scan are complete
    // the sums after the segment: R into TMEM, r into rsv
    slot_to_tmem<D, M>(args.ws_r + ((size_t)bh * args.nseg + sg) * (D * M + D), reinterpret_cast<float *>(snap), rsv,
                       trow, T::K_R, t, r, h);

    uint32_t phase = 0, fphase = 0;
    bool pending = false, loading = false;
    constexpr uint32_t ID_P = idesc_bf16(128, 128, 0, 0);    // K-major A and B
    constexpr uint32_t ID_DV = idesc_bf16(128, M, 0, 1);     // P^T (TMEM) or phi(K) x MN-major
    constexpr uint32_t ID_DK = idesc_bf16(128, D, 0, 0);     // [V | V] x [R_hi | R_lo]^T, K-major
    constexpr uint32_t ID_DK2 = idesc_bf16(128, D, 0, 1);    // A^T (TMEM) x psi(Q) MN-major
    constexpr uint32_t ID_T = idesc_bf16(128, M, 1, 1);      // psi(Q)^T x g, both MN-major
    auto mma_wait_all = [&]() {
        if (t == 0) mma_commit(mbar);
        const bool got = mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
        if (got) phase ^= 1u;
        tc_fence_after();
        return __syncthreads_and(got ? 1 : 0) != 0;
    };
    for (int c = c_end - 1; ok && c >= c_begin; --c) {
    const int t0 = c * kC, valid = min(kC, args.N - t0);
    CH_TRACE(1, 2);
    if (t == 0) {
        tma_store_wait_read0();   // the previous chunk's dK and dV stores have read their tiles
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
    // e of the chunk's rows (the load is in flight during the operand tile)
    const float ev = (h == 0 && r < valid) ? __ldcg(args.ws_e + (size_t)bh * args.N + t0 + r) : 0.f;
    // [R_c hi | R_c lo] from the TMEM sums plus the column sums of g
    if (r < D)
#pragma unroll 1
        for (int c0 = MH * h; c0 < MH * h + MH; c0 += 32) snap_from_tmem<D, M>(trow, T::K_R, r, c0, cg, snap);
    if (h == 0) es[r] = ev;
    CH_TRACE(1, 3);
    {
        const bool landed = mbar_wait_bounded(full, fphase, now_ns() + kWaitNs, nullptr);
        if (landed) {
            fphase ^= 1u;
            loading = false;
        }
        ok = __syncthreads_and(landed) != 0;
    }
    // the next (earlier) chunk into L2 while this one computes
    if (t == 0 && ok && c > c_begin) {
        const int tn = t0 - kC;
#pragma unroll
        for (int j = 0; j < D / 64; ++j) {
            tma_prefetch_3d(&tm_q, j * 64, tn, bh);
            tma_prefetch_3d(&tm_k, j * 64, tn, bh);
        }
#pragma unroll
        for (int j = 0; j < M / 64; ++j) {
            tma_prefetch_3d(&tm_v, j * 64, tn, bh);
            tma_prefetch_3d(&tm_gw, j * 64, tn, bh);
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
    // ---- phi(K) psi(Q)^T;  A^T (raw) = V g^T;  meanwhile the column sums of g
    // and of e_i (1 + psi(Q_i)) (the 1 terms of the R and r updates)
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
        colsum_part<M, false, false>(tg, nullptr, pa, t);
        colsum_part<D, true, true>(tq, es, pb, t);
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(1, 6);
    // ---- P^T = phi(K) psi(Q)^T + sk (half 0) and A^T + e_i (half 1), masked
    // to r <= i < valid (key r, query i), as bf16 at K_PTB / K_ATB; the row
    // sum of A^T (its product with the 1 of phi(Q) = psi(Q) + 1)
    float asum = 0.f;
    if (ok) {
        auto keep = [&](int i) { return i >= r && i < valid; };
        if (h == 0) tmem_row_to_bf16<false>(trow + T::K_PT, trow + T::K_PTB, keep, [&](int) { return sk; });
        else asum = tmem_row_to_bf16<true>(trow + T::K_AT, trow + T::K_ATB, keep, [&](int i) { return es[i]; });
        ok = operands_ready(true);
    }
    CH_TRACE(1, 7);
    // ---- dV = P^T g + phi(K) (R_hi + R_lo);  dphi(K) = A^T psi(Q) + [V | V] [R_hi | R_lo]^T;
    // R += psi(Q)^T g (the chunk's update; its 1 terms are the column sums above)
    if (ok) {
        if (t == 0) {
            const uint64_t dgb = smem_desc(smem_u32(tg), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + T::K_DV, tmem + T::K_PTB + ks * 8, dgb + mnmajor_step(ks), ID_DV, ks > 0);
            const uint64_t dk = kmajor_base(smem_u32(tk));
            const uint64_t ds = smem_desc(smem_u32(snap), D * 128, 1024);
            const uint64_t dsl = smem_desc(smem_u32(snap + SnapTile<D, M>::LO), D * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::K_DV, dk + kmajor_step(ks), ds + mnmajor_step(ks), ID_DV, 1);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + T::K_DV, dk + kmajor_step(ks), dsl + mnmajor_step(ks), ID_DV, 1);
            const uint64_t dqb = smem_desc(smem_u32(tq), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ts(tmem + T::K_DK, tmem + T::K_ATB + ks * 8, dqb + mnmajor_step(ks), ID_DK2, ks > 0);
            const uint64_t dv = kmajor_base(smem_u32(tv));
            const uint64_t db = kmajor_base(smem_u32(snap)), dl = kmajor_base(smem_u32(snap + SnapTile<D, M>::LO));
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::K_DK, dv + kmajor_step(ks), db + kmajor_step(ks, D), ID_DK, 1);
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + T::K_DK, dv + kmajor_step(ks), dl + kmajor_step(ks, D), ID_DK, 1);
            // A read MN-major; at D = 64 with M-atom stride 0 (lanes 64-127
            // repeat lanes 0-63 and are never read)
            const uint64_t dqa = smem_desc(smem_u32(tq), D == 64 ? 0 : kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks)
                mma_f16_ss(tmem + T::K_R, dqa + mnmajor_step(ks), dgb + mnmajor_step(ks), ID_T, 1);
        }
        pending = true;
        ok = mma_wait_all();
        pending = !ok;
    }
    CH_TRACE(1, 8);
    // ---- dK = (dphi(K) + asum + r) min(phi(K), 1) (half 1, which holds asum)
    // over phi(K) in its tile, dV (half 0) over V in its tile (both last read
    // by the products just completed); then stored by TMA
    if (ok) {
        if (h == 1) {
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float d32[32], f[32];
                tmem_ld32f(trow + T::K_DK + c0, d32);
                load_row32(tk, r, c0, f);
#pragma unroll
                for (int j = 0; j < 32; ++j) f[j] = (d32[j] + asum + rsv[c0 + j]) * fminf(f[j], 1.f);
                store_snap32<kC>(tk, r, c0, f);
            }
        } else {
#pragma unroll
            for (int c0 = 0; c0 < M; c0 += 32) {
                float x[32];
                tmem_ld32f(trow + T::K_DV + c0, x);
                store_snap32<kC>(tv, r, c0, x);
            }
        }
    }
    // the chunk's tiles, e values and TMEM are free for the next one (once the
    // dK, dV stores have read their tiles); then the column sums move r and
    // the g sums on to the earlier chunk
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (ok) {
        if (t == 0) {
#pragma unroll
            for (int j = 0; j < D / 64; ++j) tma_store_3d(&tm_dk, tk + j * kC * 128, j * 64, t0, bh);
#pragma unroll
            for (int j = 0; j < M / 64; ++j) tma_store_3d(&tm_dv, tv + j * kC * 128, j * 64, t0, bh);
            tma_store_commit();
        }
        if (t < M) cg[t] += colsum_total<M>(pa, t);
        if (t < D) rsv[t] += colsum_total<D>(pb, t);
    }
    __syncthreads();
    }
    CH_TRACE(1, 9);
    if (!ok && t == 0) {
        record_error(args.err, kErrTimeout);
        if (loading) mbar_wait_bounded(full, fphase, now_ns() + kWaitNs, nullptr);
        if (pending) mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
    }
    if (t == 0) tma_store_wait_all0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (t < 32) tmem_dealloc(tmem, T::COLS);
    CH_TRACE(1, 10);
}

// Segments per head: as many as give every SM one CTA (at least one per
// head, at most one per chunk), on a device of `sms` SMs; then the chunks per
// segment, and the segment count without empty segments.
void seg_grid(long long BH, int nch, int sms, int &nseg, int &L) {
    nseg = (int)std::max(1LL, std::min<long long>(nch, sms / std::max(1LL, BH)));
    L = (nch + nseg - 1) / nseg;
    nseg = (nch + L - 1) / L;
}

struct SegWs {
    size_t s_floats, g_elems, e_floats;
};

SegWs seg_ws(long long BH, int nseg, int N, int D, int M) {
    return SegWs{(size_t)BH * nseg * ((size_t)D * M + D), (size_t)BH * N * M, (size_t)BH * N};
}

// [S | z] and [R | r] per segment, then g (bf16), then e; each part starts on
// a 256-byte boundary
size_t round256(size_t b) { return (b + 255) / 256 * 256; }
size_t seg_ws_bytes(const SegWs &w) {
    return 2 * round256(w.s_floats * sizeof(float)) + round256(w.g_elems * 2) + w.e_floats * sizeof(float);
}

template <int D, int M>
cudaError_t launch_seg_bwd(const BwdProblem &p, const DeviceInfo &dev) {
    const int nch = (p.N + kC - 1) / kC;
    int nseg, L;
    seg_grid(p.BH, nch, std::min(192, std::max(1, dev.sm_count)), nseg, L);
    const SegWs w = seg_ws(p.BH, nseg, p.N, D, M);
    if (p.ws_bytes < seg_ws_bytes(w)) return cudaErrorInvalidValue;
    if (p.BH * nseg > INT32_MAX) return cudaErrorInvalidValue;
    uint8_t *base = (uint8_t *)p.ws;
    const size_t sb = round256(w.s_floats * sizeof(float));
    float *ws_s = (float *)base, *ws_r = (float *)(base + sb);
    __nv_bfloat16 *ws_g = (__nv_bfloat16 *)(base + 2 * sb);
    float *ws_e = (float *)(base + 2 * sb + round256(w.g_elems * 2));
    CUtensorMap tq, tk, tv, tg, tgw, tdq, tdk, tdv;
    if (!cached_tmap_bf16_3d(&tq, p.q, D, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tk, p.k, D, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tv, p.v, M, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tg, p.dout, M, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tgw, ws_g, M, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tdq, p.dq, D, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tdk, p.dk, D, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tdv, p.dv, M, p.N, p.BH, 64, kC))
        return cudaErrorInvalidValue;
    cudaError_t e = cudaSuccess;
    // key sums of every segment (with one segment the carried-in state alone enters it)
    if (nseg > 1) {
        e = tc_key_sums(p.k, p.v, p.BH, p.N, D, M, nseg, L, ws_s, w.s_floats * sizeof(float), p.stream, dev);
        if (e != cudaSuccess) return e;
    }
    const int W = D * M + D;
    const dim3 sgrid((unsigned)p.BH, (unsigned)((W / 4 + 255) / 256));
    e = launch_pdl(seg_scan_kernel, sgrid, dim3(256), 0, p.stream, 0u, ws_s, nseg, D * M, D, p.S0, p.z0,
                   (float *)nullptr, (float *)nullptr, 0, nseg > 1 ? 1 : 0);
    count_launches(1);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(p.BH * nseg)), block(kCT);
    SegBwdArgs a{ws_s, ws_r, ws_g, ws_e, (__nv_bfloat16 *)p.dq, nullptr, p.N, nch, nseg, L, dev.err_word};
    if ((e = set_smem(seg_bwd_query_kernel<D, M>, SQCfg<D, M>::SMEM)) != cudaSuccess) return e;
    e = launch_pdl(seg_bwd_query_kernel<D, M>, grid, block, SQCfg<D, M>::SMEM, p.stream, 0u, tq, tk, tv, tg, tgw, tdq,
                   a);
    count_launches(1);
    if (e != cudaSuccess) return e;
    e = launch_pdl(seg_scan_kernel, sgrid, dim3(256), 0, p.stream, 0u, ws_r, nseg, D * M, D, p.dSN, p.dzN, p.dS0,
                   p.dz0, 1, 1);
    count_launches(1);
    if (e != cudaSuccess) return e;
    a.g0 = (__nv_bfloat16 *)p.dk;
    a.g1 = (__nv_bfloat16 *)p.dv;
    if ((e = set_smem(seg_bwd_key_kernel<D, M>, SKCfg<D, M>::SMEM)) != cudaSuccess) return e;
    e = launch_pdl(seg_bwd_key_kernel<D, M>, grid, block, SKCfg<D, M>::SMEM, p.stream, 0u, tq, tk, tv, tgw, tdk, tdv,
                   a);
    count_launches(1);
    return e;
}

}  // namespace

bool tc_chunk_backward_supported(const la_shape &s) {
    return s.dtype == LA_DTYPE_BF16 && (s.D == 64 || s.D == 128) && (s.M == 64 || s.M == 128) &&
           !(s.D == 64 && s.M == 64);
}

size_t tc_chunk_backward_ws_bytes(const la_shape &s) {
    // sized for the most segments any device picks (up to 192 SMs)
    const long long BH = (long long)s.B * s.H;
    if (BH <= 0 || s.N <= 0) return 0;
    int nseg, L;
    seg_grid(BH, (s.N + kC - 1) / kC, 192, nseg, L);
    return seg_ws_bytes(seg_ws(BH, nseg, s.N, s.D, s.M));
}

cudaError_t tc_chunk_causal_backward(const BwdProblem &p, const DeviceInfo &dev) {
    if (p.D == 64 && p.M == 128) return launch_seg_bwd<64, 128>(p, dev);
    if (p.D == 128 && p.M == 64) return launch_seg_bwd<128, 64>(p, dev);
    if (p.D == 128 && p.M == 128) return launch_seg_bwd<128, 128>(p, dev);
    return cudaErrorInvalidValue;
}

}  // namespace la

// la_tc_bwd_nc.cu - tensor-core (tcgen05 + TMA) backward of the non-causal
// form, "Transformers are RNNs" sec. 3.2 eq. (5), for bf16 tensors with D, M
// in {64, 128}.
//
// With S = sum_j phi(K_j) V_j^T and z = sum_j phi(K_j) over all N keys, the
// forward is V'_i = phi(Q_i)^T S / phi(Q_i)^T z.  Given dO = dL/dV' the chain
// rule gives, per query row i and key row j,
//   den_i = phi(Q_i) . z,  g_i = dO_i / den_i,  e_i = -(dO_i . V'_i) / den_i,
//   dphi(Q_i) = S g_i + e_i z,    dS = sum_i phi(Q_i) g_i^T,  dz = sum_i e_i phi(Q_i),
//   dphi(K_j) = dS V_j + dz,      dV_j = dS^T phi(K_j),
// and dQ = dphi(Q) phi'(Q), dK = dphi(K) phi'(K) with phi'(x) = 1 for x > 0,
// e^x otherwise, i.e. min(phi(x), 1).  Three launches, each over BH x nsplit
// CTAs (a head's rows in nsplit ranges of cps chunks of C = 128 rows):
//   1. key sums: [S | z] partials of each key range (the segment-sum pre-pass
//      of the causal forward, la_tc.cu);
//   2. query kernel: sums the head's [S | z] partials into the bf16 operand
//      below; per query chunk: [num | den] = phi(Q) [S | z] (MMAs), g and e
//      on CUDA cores (V' recomputed, not read), dphi(Q) = S g + z e (MMAs),
//      dQ; and the partials dS += phi(Q)^T g, dz += phi(Q)^T e (MMAs
//      accumulating over the range);
//   3. key kernel: sums the [dS | dz] partials into the same form; per key
//      chunk: dphi(K) = dS V + dz and dV = dS^T phi(K) (MMAs), dK.
// The sums enter the products as bf16 hi + lo pairs, in one row-major tile
// [X_hi | w | X_lo] of 64-column swizzled atoms whose w atom holds
// (w_hi, w_lo, w_hi, w_lo) in its first four columns; the tile is read both
// as an MN-major B operand ([K = D] x [N]: phi(Q) [S | z]) and as a K-major
// one ([N = D] x [K]: [g | e | g] [S_hi | z | S_lo]^T), so one copy serves
// both products.  e also enters as (e_hi, e_hi, e_lo, e_lo), so that the
// four columns meet as (e_hi + e_lo)(z_hi + z_lo), and e is formed from the
// bf16 g the products use: where the terms S g and e z cancel (one key: the
// output is V whatever Q is) they cancel to fp32 rounding.  One CTA of 128 threads: thread r owns row r of each chunk (TMEM
// lane r); the phases of a chunk run in order, the next chunk's tiles load
// by TMA meanwhile (two stages).  Every wait is bounded; a CTA that gives up
// records LA_ERR_TIMEOUT and skips the rest of its work.
#include <algorithm>

#include "la_common.cuh"
#include "la_internal.h"
#include "tc_host.h"
#include "tc_bwd_common.cuh"
#include "tc_kernels.cuh"
#include "tc_ptx.cuh"

// Optional per-phase timeline of CTA 0 of the query kernel for performance
// work: compiled only with -DLA_TRACE (never in the library build).
#ifdef LA_TRACE
__device__ unsigned long long g_la_trace_ncbwd[32][8];
extern "C" int la_trace_read_ncbwd(unsigned long long *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_la_trace_ncbwd, sizeof(g_la_trace_ncbwd));
}
#define NCB_TRACE(it, ev)                                                                          \
    do {                                                                                           \
        if (blockIdx.x == 0 && threadIdx.x == 0 && (it) < 32) g_la_trace_ncbwd[it][ev] = clock64(); \
    } while (0)
#else
#define NCB_TRACE(it, ev) ((void)0)
#endif

namespace la {
namespace {

using namespace tc;

struct NcBwdArgs {
    const float *ws_in;      // [BH, nsplit, D*M + D]: the partials this kernel sums
    float *ws_out;           // [BH, nsplit, D*M + D]: the partials this kernel writes (query kernel)
    __nv_bfloat16 *g0, *g1;  // query kernel: dQ; key kernel: dK, dV
    int N, nsplit, cps;
    int *err;
    long long ws_floats;     // floats in each of ws_in, ws_out (checked build)
};

// ------------------------------------------------------------ query kernel
template <int D, int M>
struct QCfg {
    static constexpr int TQ = kC * D * 2, TG = kC * M * 2;
    static constexpr int STAGE = TQ + TG;
    static constexpr int OFF_SNAP = 2 * STAGE;                       // [S_hi | z | S_lo]
    static constexpr int OFF_E = OFF_SNAP + XwTile<D, M>::BYTES;     // (e_hi, e_hi, e_lo, e_lo) atom, 128 rows
    static constexpr int OFF_BAR = OFF_E + kC * 128;
    static constexpr int SMEM = OFF_BAR + 64;
    // TMEM: [num | den parts] (M + 16), then dphi(Q) (D) over it once read;
    // [dS | dz parts] (M + 16)
    static constexpr uint32_t COL_O = 0, COL_DQ = 0, COL_DS = (M + 16 > D ? M + 16 : D);
    static constexpr uint32_t TMEM_COLS = COL_DS + M + 16 <= 256 ? 256 : 512;
    static_assert(SMEM <= (int)kSmemMax, "shared memory budget");
};

template <int D, int M>
__global__ void __launch_bounds__(kNT, 1)
nc_bwd_query_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_g,
                    const __grid_constant__ CUtensorMap tm_dq, const NcBwdArgs args)
{
    using C = QCfg<D, M>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int r = threadIdx.x;
    const int bh = blockIdx.x / args.nsplit, sp = blockIdx.x % args.nsplit;
    const int nch = (args.N + kC - 1) / kC;
    const int c_begin = sp * args.cps;
    const int n = max(0, min(nch, c_begin + args.cps) - c_begin);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR), *mbar = full + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(mbar + 1);
    uint8_t *snap = smem + C::OFF_SNAP, *eat = smem + C::OFF_E;

    bool ok = (smem_u32(smem) & 1023u) == 0;
    if (r == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    if (r < 32) {
        tmem_alloc(slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + ((uint32_t)(32 * (r >> 5)) << 16);
    pdl_wait_cta();   // the key sums of the previous launch are complete

    int issued = 0, consumed = 0;
    auto load_chunk = [&](int it) {
        ++issued;
        uint8_t *st = smem + (it & 1) * C::STAGE;
        const int t0 = (c_begin + it) * kC;
        mbar_arrive_expect_tx(&full[it & 1], C::STAGE);
#pragma unroll
        for (int j = 0; j < D / 64; ++j) tma_load_3d(st + j * kC * 128, &tm_q, &full[it & 1], j * 64, t0, bh);
#pragma unroll
        for (int j = 0; j < M / 64; ++j) tma_load_3d(st + C::TQ + j * kC * 128, &tm_g, &full[it & 1], j * 64, t0, bh);
    };
    if (r == 0 && ok && n > 0) {
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_g);
        load_chunk(0);
    }
    // [S | z_hi z_lo] of the head from the key-sum partials
    // the head's slots lie inside the workspace (checked build)
    const bool ws_ok = LA_IN_BOUNDS(((long long)bh + 1) * args.nsplit * (D * M + D) <= args.ws_floats, args.err);
    if (ws_ok)
        sum_partials_to_tile<D, M>(args.ws_in + (size_t)bh * args.nsplit * (D * M + D), args.nsplit, snap, r);
    ok = operands_ready(ok);
    if (!ok && r == 0) record_error(args.err, kErrTimeout);

    constexpr uint32_t ID_O = idesc_bf16(128, M + 16, 0, 1);   // phi(Q) K-major, [S | z] MN-major
    constexpr uint32_t ID_OL = idesc_bf16(128, M, 0, 1);
    constexpr uint32_t ID_DQ = idesc_bf16(128, D, 0, 0);       // [g | e] K-major, [S | z] K-major
    constexpr uint32_t ID_DS = idesc_bf16(128, M, 1, 1);       // phi(Q)^T MN-major, g MN-major
    constexpr uint32_t ID_DZ = idesc_bf16(128, 16, 1, 1);
    uint32_t phase = 0;
    bool mma_pending = false;
    for (int it = 0; it < n && ok; ++it) {
        const int s = it & 1, t0 = (c_begin + it) * kC;
        const int valid = min(kC, args.N - t0);
        uint8_t *tq = smem + s * C::STAGE, *tg = tq + C::TQ;
        NCB_TRACE(it, 0);
        if (r == 0 && it + 1 < n) {
            tma_store_wait_read0();   // chunk it - 1's dQ store has read the stage
            load_chunk(it + 1);       // into the stage released at the end of it - 1
        }
        const bool landed = mbar_wait_bounded(&full[s], (it >> 1) & 1, now_ns() + kWaitNs, nullptr);
        if (!(ok = __syncthreads_and(landed) != 0)) {
            if (r == 0) record_error(args.err, kErrTimeout);
            break;
        }
        ++consumed;
        NCB_TRACE(it, 1);
        phi_tile<D>(tq, r, valid);   // rows past the end become zeros
        ok = operands_ready(true);
        NCB_TRACE(it, 2);
        // ---- [num | den] = phi(Q) [S_hi | z] + phi(Q) [S_lo | -]
        if (r == 0) {
            const uint64_t dq = kmajor_base(smem_u32(tq));
            const uint64_t db = smem_desc(smem_u32(snap), D * 128, 1024);
            const uint64_t dl = smem_desc(smem_u32(snap + XwTile<D, M>::LO), D * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + C::COL_O, dq + kmajor_step(ks), db + mnmajor_step(ks), ID_O, ks > 0);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + C::COL_O, dq + kmajor_step(ks), dl + mnmajor_step(ks), ID_OL, 1);
        }
        if (!(ok = mma_done(mbar, phase))) {
            mma_pending = true;
            break;
        }
        NCB_TRACE(it, 3);
        // ---- g = dO / den as bf16 (over dO in place), e = -(g . V'), V' = num / den
        {
            float dz[32];
            tmem_ld32f(trow + C::COL_O + M, dz);   // den parts (z_hi, z_lo columns), then unused columns
            const float den = dz[0] + dz[1];
            const float inv = r < valid ? 1.f / den : 0.f;
            float dot = 0.f;
#pragma unroll 1
            for (int c0 = 0; c0 < M; c0 += 32) {
                float x[32], gv[32];
                tmem_ld32f(trow + C::COL_O + c0, x);
                load_row32(tg, r, c0, gv);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    gv[j] = __bfloat162float(__float2bfloat16_rn(gv[j] * inv));
                    dot = fmaf(gv[j], x[j] * inv, dot);
                }
                store_snap32<kC>(tg, r, c0, gv);
            }
            const float e = -dot;
            const float eh = __bfloat162float(__float2bfloat16_rn(e));
            const uint32_t hh = pack_bf16x2(eh, eh), ll = pack_bf16x2(e - eh, e - eh);
#pragma unroll
            for (int c = 0; c < 64; c += 8)
                *reinterpret_cast<uint4 *>(eat + sw128_offset(r, c)) =
                    make_uint4(c == 0 ? hh : 0u, c == 0 ? ll : 0u, 0u, 0u);
        }
        ok = operands_ready(ok);
        NCB_TRACE(it, 4);
        // ---- dphi(Q) = [g | e | g] [S_hi | z | S_lo]^T;  [dS | dz] += phi(Q)^T [g | e]
        if (r == 0) {
            const uint64_t dg = kmajor_base(smem_u32(tg)), de = kmajor_base(smem_u32(eat));
            const uint64_t db = kmajor_base(smem_u32(snap)), dl = kmajor_base(smem_u32(snap + XwTile<D, M>::LO));
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + C::COL_DQ, dg + kmajor_step(ks), db + kmajor_step(ks, D), ID_DQ, ks > 0);
            mma_f16_ss(tmem + C::COL_DQ, de, db + kmajor_step(M / 16, D), ID_DQ, 1);   // the z atom
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + C::COL_DQ, dg + kmajor_step(ks), dl + kmajor_step(ks, D), ID_DQ, 1);
            // phi(Q)^T read MN-major; at D = 64 its 64 rows are read twice
            // (M-atom stride 0) and accumulator lanes 64-127 are not used
            const uint64_t da = smem_desc(smem_u32(tq), D == 64 ? 0 : kC * 128, 1024);
            const uint64_t dgb = smem_desc(smem_u32(tg), kC * 128, 1024), deb = smem_desc(smem_u32(eat), kC * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < kC / 16; ++ks) {
                mma_f16_ss(tmem + C::COL_DS, da + mnmajor_step(ks), dgb + mnmajor_step(ks), ID_DS, it > 0 || ks > 0);
                mma_f16_ss(tmem + C::COL_DS + M, da + mnmajor_step(ks), deb + mnmajor_step(ks), ID_DZ, it > 0 || ks > 0);
            }
        }
        if (!(ok = mma_done(mbar, phase))) {
            mma_pending = true;
            break;
        }
        NCB_TRACE(it, 5);
        // ---- dQ = dphi(Q) min(phi(Q), 1), over phi(Q) in its tile (each thread
        // reads its row's values before writing them), then stored by TMA (rows
        // past the end are not written)
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            float d32[32], f[32];
            tmem_ld32f(trow + C::COL_DQ + c0, d32);
            load_row32(tq, r, c0, f);
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = d32[j] * fminf(f[j], 1.f);
            store_snap32<kC>(tq, r, c0, f);
        }
        NCB_TRACE(it, 6);
        fence_proxy_async();
        __syncthreads();   // the stage is free for the load two chunks on, once the store has read it
        if (r == 0) {
#pragma unroll
            for (int j = 0; j < D / 64; ++j) tma_store_3d(&tm_dq, tq + j * kC * 128, j * 64, t0, bh);
            tma_store_commit();
        }
    }
    // [dS | dz] partial of this query range (zero for an empty range)
    if (ok && r < D && ws_ok) {
        float *dst = args.ws_out + ((size_t)bh * args.nsplit + sp) * (D * M + D);
        float x[32];
        for (int c0 = 0; c0 < M; c0 += 32) {
            if (n > 0) {
                tmem_ld32f(trow + C::COL_DS + c0, x);
            } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) x[j] = 0.f;
            }
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(dst + r * M + c0 + j) = make_float4(x[j], x[j + 1], x[j + 2], x[j + 3]);
        }
        if (n > 0) tmem_ld32f(trow + C::COL_DS + M, x);
        dst[D * M + r] = n > 0 ? x[0] + x[2] : 0.f;   // the e_hi and e_lo columns
    }
    if (!ok && r == 0) {
        record_error(args.err, kErrTimeout);
        for (int c = consumed; c < issued; ++c)
            mbar_wait_bounded(&full[c & 1], (c >> 1) & 1, now_ns() + kWaitNs, nullptr);
        if (mma_pending) mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
    }
    if (r == 0) tma_store_wait_all0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (r < 32) tmem_dealloc(tmem, C::TMEM_COLS);
}

// -------------------------------------------------------------- key kernel
template <int D, int M>
struct KCfg {
    static constexpr int TK = kC * D * 2, TV = kC * M * 2;
    static constexpr int STAGE = TK + TV;
    static constexpr int OFF_SNAP = 2 * STAGE;                       // [dS_hi | dz | dS_lo]
    static constexpr int OFF_ONES = OFF_SNAP + XwTile<D, M>::BYTES;  // [1 1 0 ..] atom, 128 rows
    static constexpr int OFF_BAR = OFF_ONES + kC * 128;
    static constexpr int SMEM = OFF_BAR + 64;
    static constexpr uint32_t COL_DK = 0, COL_DV = D;
    static constexpr uint32_t TMEM_COLS = D + M <= 256 ? 256 : 512;
    static_assert(SMEM <= (int)kSmemMax, "shared memory budget");
};

template <int D, int M>
__global__ void __launch_bounds__(kNT, 1)
nc_bwd_key_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const __grid_constant__ CUtensorMap tm_dk,
                  const __grid_constant__ CUtensorMap tm_dv, const NcBwdArgs args)
{
    using C = KCfg<D, M>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int r = threadIdx.x;
    const int bh = blockIdx.x / args.nsplit, sp = blockIdx.x % args.nsplit;
    const int nch = (args.N + kC - 1) / kC;
    const int c_begin = sp * args.cps;
    const int n = max(0, min(nch, c_begin + args.cps) - c_begin);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR), *mbar = full + 2;
    uint32_t *slot = reinterpret_cast<uint32_t *>(mbar + 1);
    uint8_t *snap = smem + C::OFF_SNAP, *ones = smem + C::OFF_ONES;

    bool ok = (smem_u32(smem) & 1023u) == 0;
    if (r == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_init(mbar, 1);
        fence_mbar_init();
    }
    if (r < 32) {
        tmem_alloc(slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    // the ones atom: columns 0 and 1 of every row are 1 (they meet dz_hi, dz_lo)
#pragma unroll
    for (int c = 0; c < 64; c += 8)
        *reinterpret_cast<uint4 *>(ones + sw128_offset(r, c)) = make_uint4(c == 0 ? 0x3F803F80u : 0u, 0u, 0u, 0u);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *slot;
    const uint32_t trow = tmem + ((uint32_t)(32 * (r >> 5)) << 16);
    pdl_wait_cta();   // the query kernel's partials are complete

    int issued = 0, consumed = 0;
    auto load_chunk = [&](int it) {
        ++issued;
        uint8_t *st = smem + (it & 1) * C::STAGE;
        const int t0 = (c_begin + it) * kC;
        mbar_arrive_expect_tx(&full[it & 1], C::STAGE);
#pragma unroll
        for (int j = 0; j < D / 64; ++j) tma_load_3d(st + j * kC * 128, &tm_k, &full[it & 1], j * 64, t0, bh);
#pragma unroll
        for (int j = 0; j < M / 64; ++j) tma_load_3d(st + C::TK + j * kC * 128, &tm_v, &full[it & 1], j * 64, t0, bh);
    };
    if (r == 0 && ok && n > 0) {
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        load_chunk(0);
    }
    // the head's slots lie inside the workspace (checked build)
    const bool ws_ok = LA_IN_BOUNDS(((long long)bh + 1) * args.nsplit * (D * M + D) <= args.ws_floats, args.err);
    if (ws_ok)
        sum_partials_to_tile<D, M>(args.ws_in + (size_t)bh * args.nsplit * (D * M + D), args.nsplit, snap, r);
    ok = operands_ready(ok);
    if (!ok && r == 0) record_error(args.err, kErrTimeout);

    constexpr uint32_t ID_DK = idesc_bf16(128, D, 0, 0);   // [V | 1 1] K-major, [dS | dz] K-major
    constexpr uint32_t ID_DV = idesc_bf16(128, M, 0, 1);   // phi(K) K-major, dS MN-major
    uint32_t phase = 0;
    bool mma_pending = false;
    for (int it = 0; it < n && ok; ++it) {
        const int s = it & 1, t0 = (c_begin + it) * kC;
        const int valid = min(kC, args.N - t0);
        uint8_t *tk = smem + s * C::STAGE, *tv = tk + C::TK;
        if (r == 0 && it + 1 < n) {
            tma_store_wait_read0();   // chunk it - 1's dK, dV stores have read the stage
            load_chunk(it + 1);
        }
        const bool landed = mbar_wait_bounded(&full[s], (it >> 1) & 1, now_ns() + kWaitNs, nullptr);
        if (!(ok = __syncthreads_and(landed) != 0)) {
            if (r == 0) record_error(args.err, kErrTimeout);
            break;
        }
        ++consumed;
        phi_tile<D>(tk, r, valid);
        ok = operands_ready(true);
        // ---- dphi(K) = [V | 1 | V] [dS_hi | dz | dS_lo]^T,  dV = phi(K) (dS_hi + dS_lo)
        if (r == 0) {
            const uint64_t dv = kmajor_base(smem_u32(tv)), d1 = kmajor_base(smem_u32(ones));
            const uint64_t db = kmajor_base(smem_u32(snap)), dl = kmajor_base(smem_u32(snap + XwTile<D, M>::LO));
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + C::COL_DK, dv + kmajor_step(ks), db + kmajor_step(ks, D), ID_DK, ks > 0);
            mma_f16_ss(tmem + C::COL_DK, d1, db + kmajor_step(M / 16, D), ID_DK, 1);   // the dz atom
#pragma unroll
            for (int ks = 0; ks < M / 16; ++ks)
                mma_f16_ss(tmem + C::COL_DK, dv + kmajor_step(ks), dl + kmajor_step(ks, D), ID_DK, 1);
            const uint64_t dk = kmajor_base(smem_u32(tk));
            const uint64_t ds = smem_desc(smem_u32(snap), D * 128, 1024);
            const uint64_t dsl = smem_desc(smem_u32(snap + XwTile<D, M>::LO), D * 128, 1024);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + C::COL_DV, dk + kmajor_step(ks), ds + mnmajor_step(ks), ID_DV, ks > 0);
#pragma unroll
            for (int ks = 0; ks < D / 16; ++ks)
                mma_f16_ss(tmem + C::COL_DV, dk + kmajor_step(ks), dsl + mnmajor_step(ks), ID_DV, 1);
        }
        if (!(ok = mma_done(mbar, phase))) {
            mma_pending = true;
            break;
        }
        // ---- dK = dphi(K) min(phi(K), 1) over phi(K) in its tile, dV over V in
        // its tile (last read by the products just completed); then stored by
        // TMA (rows past the end are not written)
#pragma unroll
        for (int c0 = 0; c0 < D; c0 += 32) {
            float d32[32], f[32];
            tmem_ld32f(trow + C::COL_DK + c0, d32);
            load_row32(tk, r, c0, f);
#pragma unroll
            for (int j = 0; j < 32; ++j) f[j] = d32[j] * fminf(f[j], 1.f);
            store_snap32<kC>(tk, r, c0, f);
        }
#pragma unroll
        for (int c0 = 0; c0 < M; c0 += 32) {
            float x[32];
            tmem_ld32f(trow + C::COL_DV + c0, x);
            store_snap32<kC>(tv, r, c0, x);
        }
        fence_proxy_async();
        __syncthreads();   // the stage is free for the load two chunks on, once the stores have read it
        if (r == 0) {
#pragma unroll
            for (int j = 0; j < D / 64; ++j) tma_store_3d(&tm_dk, tk + j * kC * 128, j * 64, t0, bh);
#pragma unroll
            for (int j = 0; j < M / 64; ++j) tma_store_3d(&tm_dv, tv + j * kC * 128, j * 64, t0, bh);
            tma_store_commit();
        }
    }
    if (!ok && r == 0) {
        record_error(args.err, kErrTimeout);
        for (int c = consumed; c < issued; ++c)
            mbar_wait_bounded(&full[c & 1], (c >> 1) & 1, now_ns() + kWaitNs, nullptr);
        if (mma_pending) mbar_wait_bounded(mbar, phase, now_ns() + kWaitNs, nullptr);
    }
    if (r == 0) tma_store_wait_all0();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (r < 32) tmem_dealloc(tmem, C::TMEM_COLS);
}

// Key/query ranges per head: as many CTAs as fit on the device at once (two
// per SM at D = M = 64, where both kernels fit twice), so that all run in one
// wave (measured on 128 heads x 3072 rows: 3 ranges a head, 1.26 waves,
// 185 us for the three launches; 2 ranges, one wave, 137 us), at most 16,
// whole chunks each.
void nc_tc_grid(long long BH, int N, int sm_count, bool two_per_sm, int &nsplit, int &cps) {
    const long long nch = (N + kC - 1) / kC;
    const long long slots = (long long)std::max(sm_count, 1) * (two_per_sm ? 2 : 1);
    long long want = slots / BH;
    want = std::max(1LL, std::min(std::min(want, nch), 16LL));
    cps = (int)((nch + want - 1) / want);
    nsplit = (int)((nch + cps - 1) / cps);
}

template <int D, int M>
cudaError_t launch_nc_bwd(const BwdProblem &p, const DeviceInfo &dev) {
    int nsplit, cps;
    nc_tc_grid(p.BH, p.N, dev.sm_count, D == 64 && M == 64, nsplit, cps);
    const size_t part = (size_t)p.BH * nsplit * (D * M + D) * sizeof(float);
    if (p.ws_bytes < 2 * part) return cudaErrorInvalidValue;
    float *ws_s = (float *)p.ws, *ws_r = ws_s + part / sizeof(float);
    CUtensorMap tq, tg, tk, tv, tdq, tdk, tdv;
    if (!cached_tmap_bf16_3d(&tq, p.q, D, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tg, p.dout, M, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tk, p.k, D, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tv, p.v, M, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tdq, p.dq, D, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&tdk, p.dk, D, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tdv, p.dv, M, p.N, p.BH, 64, kC))
        return cudaErrorInvalidValue;
    cudaError_t e = tc_key_sums(p.k, p.v, p.BH, p.N, D, M, nsplit, cps, ws_s, part, p.stream, dev);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)(p.BH * nsplit)), block(kNT);
    const long long part_floats = (long long)(part / sizeof(float));
    NcBwdArgs qa{ws_s, ws_r, (__nv_bfloat16 *)p.dq, nullptr, p.N, nsplit, cps, dev.err_word, part_floats};
    if ((e = set_smem(nc_bwd_query_kernel<D, M>, QCfg<D, M>::SMEM)) != cudaSuccess) return e;
    e = launch_pdl(nc_bwd_query_kernel<D, M>, grid, block, QCfg<D, M>::SMEM, p.stream, 0u, tq, tg, tdq, qa);
    count_launches(1);
    if (e != cudaSuccess) return e;
    NcBwdArgs ka{ws_r, nullptr, (__nv_bfloat16 *)p.dk, (__nv_bfloat16 *)p.dv, p.N, nsplit, cps, dev.err_word,
                 part_floats};
    if ((e = set_smem(nc_bwd_key_kernel<D, M>, KCfg<D, M>::SMEM)) != cudaSuccess) return e;
    e = launch_pdl(nc_bwd_key_kernel<D, M>, grid, block, KCfg<D, M>::SMEM, p.stream, 0u, tk, tv, tdk, tdv, ka);
    count_launches(1);
    return e;
}

}  // namespace

size_t tc_nc_backward_ws_bytes(const la_shape &s) {
    // the most ranges nc_tc_grid picks on any device (up to 192 SMs, two CTAs each)
    const long long BH = (long long)s.B * s.H;
    if (BH <= 0 || s.N <= 0) return 0;
    int nsplit, cps;
    nc_tc_grid(BH, s.N, 192, true, nsplit, cps);
    return (size_t)2 * BH * nsplit * ((size_t)s.D * s.M + s.D) * sizeof(float);
}

bool tc_nc_backward_supported(const la_shape &s) {
    return s.dtype == LA_DTYPE_BF16 && (s.D == 64 || s.D == 128) && (s.M == 64 || s.M == 128);
}

cudaError_t tc_noncausal_backward(const BwdProblem &p, const DeviceInfo &dev) {
    if (p.D == 64 && p.M == 64) return launch_nc_bwd<64, 64>(p, dev);
    if (p.D == 64 && p.M == 128) return launch_nc_bwd<64, 128>(p, dev);
    if (p.D == 128 && p.M == 64) return launch_nc_bwd<128, 64>(p, dev);
    if (p.D == 128 && p.M == 128) return launch_nc_bwd<128, 128>(p, dev);
    return cudaErrorInvalidValue;
}

}  // namespace la

// la_tc.cu - tensor-core (tcgen05 + TMA) kernels of liblinattn.so for bf16
// inputs with D, M in {64, 128}.
//
// Method ("Transformers are RNNs", Chinese translation "線性變換器"):
// causal attention, sec. 3.3 eqs. (9)-(12), regrouped into chunks of C = 128
// rows.  For chunk c with rows t0..t0+C-1 of one head:
//   P      = phi(Q_c) phi(K_c)^T                       (C x C, fp32 in TMEM)
//   A      = P with A_ij = 0 for j > i (diagonal kept, eq. (8)), rounded to bf16
//   num    = A V_c + phi(Q_c) S_prev                    (C x M, fp32 in TMEM)
//   den_i  = sum_j A_ij + phi(Q_c)_i . z_prev            (fp32)
//   out_i  = num_i / den_i                               (eq. (12))
//   S_prev += phi(K_c)^T V_c,  z_prev += phi(K_c)^T 1   (eqs. (10), (11))
// Exact in real arithmetic: the j <= i sum of eq. (9) is split at the chunk
// start into the in-chunk part and the carried prefix state.
//
// Roles per CTA (one CTA = one head segment, 192 threads):
//   warp 0     TMA producer: Q, K, V chunk tiles into a ring of NS stages,
//              128-byte swizzled (the tcgen05 canonical K-major layout);
//   warp 1     MMA issuer (one thread): all tcgen05.mma, completion through
//              tcgen05.commit on mbarriers;
//   warps 2-5  "working group", one thread per TMEM lane / chunk row: applies
//              phi in place in shared memory, masks P and writes it back to
//              TMEM as bf16 (the A operand of A V), snapshots the fp32 state to
//              a bf16 shared-memory copy (the B operand of phi(Q) S_prev),
//              divides and stores the output rows.
// The state S (D x M) and z (D) stay in TMEM in fp32 for the whole segment.
// Long sequences are cut into segments; the state entering segment g is the
// carried-in state plus the fp32 sums of segments < g, which
// state_reduce_kernel computes beforehand (two passes, no inter-CTA waits).
// Every mbarrier wait is bounded; a CTA that gives up records LA_ERR_TIMEOUT,
// lets its copies and MMAs drain, frees its TMEM and returns.
#include <algorithm>

#include "la_common.cuh"
#include "la_internal.h"
#include "tc_host.h"
#include "tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;                          // chunk rows (MMA M)
constexpr int kWg = 128;                         // working-group threads
constexpr int kThreads = 64 + kWg;
constexpr uint64_t kWaitNs = 2000000000ull;      // 2 s per wait
constexpr uint32_t kSmemMax = 232448;            // 227 KB opt-in per CTA
constexpr int kOnesBytes = 2048;                 // 16 K-rows x 64 bf16 ones

template <int D, int M>
struct Cfg {
    static constexpr int TILE_QK = kC * D * 2;
    static constexpr int TILE_V = kC * M * 2;
    static constexpr int STAGE = 2 * TILE_QK + TILE_V;
    static constexpr int SNAP = D * M * 2;
    static constexpr int NPB = (M == 64) ? 2 : 1;      // P buffers in TMEM
    static constexpr bool O_IN_P = (M == 64);          // O shares the P buffer's upper 64 columns
    static constexpr int NBARS_FIXED = 4 + 4 * 2;      // snap, s_full, never, drain, 4 per-buffer x2
    static constexpr int FIXED = SNAP + kOnesBytes + D * 4 + 8 * (NBARS_FIXED + 3 * 8) + 16;
    static constexpr int NS_FIT = (int)((kSmemMax - FIXED) / STAGE);
    static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
    static_assert(NS >= 2, "pipeline needs two stages");
    // shared-memory map (from a 1024-byte aligned base)
    static constexpr int OFF_SNAP = NS * STAGE;
    static constexpr int OFF_ONES = OFF_SNAP + SNAP;
    static constexpr int OFF_Z = OFF_ONES + kOnesBytes;
    static constexpr int OFF_BAR = OFF_Z + D * 4;
    static constexpr int NBARS = 3 * NS + 4 * NPB + 4;
    static constexpr int OFF_TSLOT = OFF_BAR + 8 * NBARS;
    static constexpr int SMEM = OFF_TSLOT + 16;
    static_assert(SMEM <= (int)kSmemMax, "shared memory budget");
    // TMEM columns
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = 256;
    static constexpr uint32_t COL_Z = 256 + M;
    static __device__ __forceinline__ uint32_t col_p(int b) { return O_IN_P ? 128u * b : 0u; }
    static __device__ __forceinline__ uint32_t col_o(int b) { return O_IN_P ? 128u * b + 64u : 128u; }
};

struct CausalArgs {
    void *out;               // [BH, N, M] bf16 or null
    float *S;                // [BH, D, M] in/out or null
    float *z;                // [BH, D] in/out or null
    const float *seg_ws;     // [BH, nseg, D*M + D] segment sums (segments < nseg-1) or null
    int N;
    int nseg;                // segments per head
    int cps;                 // chunks per segment
    int *err;
    uint64_t inject_ns;      // test hook: wait this long on a flag nobody sets
};

struct Bars {
    uint64_t *full, *empty, *phi;          // [NS]
    uint64_t *p_full, *a_ready, *o_full, *o_free;  // [NPB]
    uint64_t *snap, *s_full, *never, *drain;
};

template <typename C>
__device__ __forceinline__ Bars carve_bars(uint8_t *sm) {
    uint64_t *b = reinterpret_cast<uint64_t *>(sm + C::OFF_BAR);
    Bars r;
    r.full = b;
    r.empty = b + C::NS;
    r.phi = b + 2 * C::NS;
    r.p_full = b + 3 * C::NS;
    r.a_ready = r.p_full + C::NPB;
    r.o_full = r.a_ready + C::NPB;
    r.o_free = r.o_full + C::NPB;
    r.snap = r.o_free + C::NPB;
    r.s_full = r.snap + 1;
    r.never = r.s_full + 1;
    r.drain = r.never + 1;
    return r;
}

__device__ __forceinline__ uint64_t now_ns() { return globaltimer_ns(); }

// Bounded wait that also gives up as soon as another role has aborted.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (*abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    return mbar_wait_bounded(bar, parity, now_ns() + kWaitNs, abort);
}

__device__ __forceinline__ void set_abort(volatile int *abort, int *err) {
    *abort = 1;
    record_error(err, kErrTimeout);
}

// phi in place on one 16-byte chunk (8 bf16) of a swizzled tile; zero = write zeros.
__device__ __forceinline__ void phi_chunk(uint8_t *p, bool zero) {
    uint4 v = *reinterpret_cast<uint4 *>(p);
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float lo = phi_fast(bf16lo(w[i])), hi = phi_fast(bf16hi(w[i]));
        w[i] = zero ? 0u : pack_bf16x2(lo, hi);
    }
    *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Applies phi to the C x DD tile at `tile` (sub-tiles of 64 columns, each
// C rows x 128 bytes).  Rows >= zero_from are written as zeros.
template <int DD>
__device__ __forceinline__ void phi_tile(uint8_t *tile, int t, int zero_from) {
    constexpr int CHUNKS = kC * DD * 2 / 16;
#pragma unroll 4
    for (int u = t; u < CHUNKS; u += kWg) {
        const uint32_t off = (uint32_t)u * 16u;
        const int row = (int)((off % (kC * 128u)) >> 7);
        phi_chunk(tile + off, row >= zero_from);
    }
}

// Writes row r of a D x M fp32 state (values in v, M entries) as bf16 into the
// MN-major swizzled snapshot [D rows x M cols] (sub-tiles of 64 columns).
template <int D, int M>
__device__ __forceinline__ void store_snap_row(uint8_t *snap, int r, const float *v) {
#pragma unroll
    for (int c8 = 0; c8 < M / 8; ++c8) {
        const int c = c8 * 8;
        uint8_t *dst = snap + (c / 64) * D * 128 + sw128_offset(r, c % 64);
        uint4 w;
        w.x = pack_bf16x2(v[c + 0], v[c + 1]);
        w.y = pack_bf16x2(v[c + 2], v[c + 3]);
        w.z = pack_bf16x2(v[c + 4], v[c + 5]);
        w.w = pack_bf16x2(v[c + 6], v[c + 7]);
        *reinterpret_cast<uint4 *>(dst) = w;
    }
}

// phi(Q)_r . z with phi(Q) read back (bf16) from the swizzled tile.
template <int D>
__device__ __forceinline__ float q_dot_z(const uint8_t *qt, int r, const float *zs) {
    float acc = 0.f;
#pragma unroll
    for (int c8 = 0; c8 < D / 8; ++c8) {
        const int c = c8 * 8;
        const uint4 w = *reinterpret_cast<const uint4 *>(qt + (c / 64) * kC * 128 + sw128_offset(r, c % 64));
        const float4 z0 = *reinterpret_cast<const float4 *>(zs + c);
        const float4 z1 = *reinterpret_cast<const float4 *>(zs + c + 4);
        acc = fmaf(bf16lo(w.x), z0.x, acc);
        acc = fmaf(bf16hi(w.x), z0.y, acc);
        acc = fmaf(bf16lo(w.y), z0.z, acc);
        acc = fmaf(bf16hi(w.y), z0.w, acc);
        acc = fmaf(bf16lo(w.z), z1.x, acc);
        acc = fmaf(bf16hi(w.z), z1.y, acc);
        acc = fmaf(bf16lo(w.w), z1.z, acc);
        acc = fmaf(bf16hi(w.w), z1.w, acc);
    }
    return acc;
}

__device__ __forceinline__ void wg_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// ----------------------------------------------------------------------------
// Causal chunked kernel.
template <int D, int M>
__global__ void __launch_bounds__(kThreads, 1)
causal_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const CausalArgs args)
{
    using C = Cfg<D, M>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_TSLOT + 4);

    const int item = blockIdx.x;
    const int bh = item / args.nseg, seg = item % args.nseg;
    const int nch_total = (args.N + kC - 1) / kC;
    const int c_begin = seg * args.cps;
    const int c_end = min(nch_total, c_begin + args.cps);
    const int n = max(0, c_end - c_begin);

    Bars bars = carve_bars<C>(smem);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::OFF_TSLOT);
    uint8_t *snap = smem + C::OFF_SNAP;
    uint8_t *ones = smem + C::OFF_ONES;
    float *zs = reinterpret_cast<float *>(smem + C::OFF_Z);

    if (tid == 0) {
        *abort = (smem_u32(smem) & 1023u) ? 1 : 0;   // layout needs a 1024-byte aligned base
        if (*abort) record_error(args.err, kErrTimeout);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(&bars.full[s], 1);
            mbar_init(&bars.empty[s], 1);
            mbar_init(&bars.phi[s], kWg);
        }
        for (int b = 0; b < C::NPB; ++b) {
            mbar_init(&bars.p_full[b], 1);
            mbar_init(&bars.a_ready[b], kWg);
            mbar_init(&bars.o_full[b], 1);
            mbar_init(&bars.o_free[b], kWg);
        }
        mbar_init(bars.snap, kWg);
        mbar_init(bars.s_full, 1);
        mbar_init(bars.never, 1);
        mbar_init(bars.drain, 1);
        fence_mbar_init();
    }
    for (int i = tid; i < kOnesBytes / 4; i += kThreads) reinterpret_cast<uint32_t *>(ones)[i] = 0x3F803F80u;
    if (warp == 0) {
        tmem_alloc(tslot, C::TMEM_COLS);
        tmem_relinquish();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;

    // Test hook: wait on a barrier that nothing arrives on, then give up.
    if (args.inject_ns && tid == 0) {
        if (!mbar_wait_bounded(bars.never, 0, now_ns() + args.inject_ns, nullptr)) set_abort(abort, args.err);
    }
    __syncthreads();

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0 && !*abort) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued = 0;
            for (int it = 0; it < n; ++it) {
                const int s = it % C::NS, k = it / C::NS;
                if (it >= C::NS && !wait_bar(&bars.empty[s], (k - 1) & 1, abort)) break;
                uint8_t *st = smem + s * C::STAGE;
                const int t0 = (c_begin + it) * kC;
                mbar_arrive_expect_tx(&bars.full[s], C::STAGE);
#pragma unroll
                for (int j = 0; j < D / 64; ++j) tma_load_3d(st + j * kC * 128, &tm_q, &bars.full[s], j * 64, t0, bh);
#pragma unroll
                for (int j = 0; j < D / 64; ++j)
                    tma_load_3d(st + C::TILE_QK + j * kC * 128, &tm_k, &bars.full[s], j * 64, t0, bh);
#pragma unroll
                for (int j = 0; j < M / 64; ++j)
                    tma_load_3d(st + 2 * C::TILE_QK + j * kC * 128, &tm_v, &bars.full[s], j * 64, t0, bh);
                ++issued;
            }
            if (*abort) {
                // let the copies in flight land before the CTA exits
                const int first = max(0, issued - C::NS);
                for (int it = first; it < issued; ++it)
                    mbar_wait_bounded(&bars.full[it % C::NS], (it / C::NS) & 1, now_ns() + kWaitNs, nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && !*abort) {
            constexpr uint32_t ID_P = idesc_bf16(128, kC, 0, 0);
            constexpr uint32_t ID_O = idesc_bf16(128, M, 0, 1);
            constexpr uint32_t ID_S = idesc_bf16(128, M, 1, 1);
            constexpr uint32_t ID_Z = idesc_bf16(128, 16, 1, 1);
            const uint32_t ones_a = smem_u32(ones);
            for (int it = 0; it < n; ++it) {
                const int s = it % C::NS, k = it / C::NS;
                const int pb = it % C::NPB, kb = it / C::NPB;
                const uint32_t st = smem_u32(smem + s * C::STAGE);
                const uint32_t qa = st, ka = st + C::TILE_QK, va = st + 2 * C::TILE_QK;
                if (!wait_bar(&bars.phi[s], k & 1, abort)) break;
                if (kb > 0) {
                    // P buffer pb is free once the chunk that used it last has been read out
                    if (C::O_IN_P) {
                        if (!wait_bar(&bars.o_free[pb], (kb - 1) & 1, abort)) break;
                    } else {
                        if (!wait_bar(&bars.o_full[pb], (kb - 1) & 1, abort)) break;
                    }
                }
                tc_fence_after();
                // P = phi(Q) phi(K)^T  (K-major A and B, K = D)
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (ks / 4) * kC * 128 + (ks % 4) * 32;
                    mma_f16_ss(tmem + C::col_p(pb), smem_desc(qa + off, 16, 1024), smem_desc(ka + off, 16, 1024),
                               ID_P, ks > 0);
                }
                mma_commit(&bars.p_full[pb]);
                // snapshot of the state before this chunk is in shared memory
                if (!wait_bar(bars.snap, it & 1, abort)) break;
                if (C::O_IN_P) {
                    if (!wait_bar(&bars.a_ready[pb], kb & 1, abort)) break;
                } else if (it > 0) {
                    if (!wait_bar(&bars.o_free[0], (it - 1) & 1, abort)) break;
                }
                tc_fence_after();
                // O = phi(Q) S_prev   (A = phi(Q) K-major, B = S snapshot MN-major, K = D)
                const uint32_t sa = smem_u32(snap);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t aoff = (ks / 4) * kC * 128 + (ks % 4) * 32;
                    mma_f16_ss(tmem + C::col_o(pb), smem_desc(qa + aoff, 16, 1024),
                               smem_desc(sa + ks * 2048, D * 128, 1024), ID_O, ks > 0);
                }
                // S += phi(K)^T V and z += phi(K)^T 1  (A = phi(K) read MN-major; M = 128 rows,
                // rows >= D of the accumulator are never read)
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks) {
                    const uint64_t adesc = smem_desc(ka + ks * 2048, kC * 128, 1024);
                    mma_f16_ss(tmem + C::COL_S, adesc, smem_desc(va + ks * 2048, kC * 128, 1024), ID_S, 1);
                    mma_f16_ss(tmem + C::COL_Z, adesc, smem_desc(ones_a, 1024, 1024), ID_Z, 1);
                }
                mma_commit(bars.s_full);
                if (!C::O_IN_P && !wait_bar(&bars.a_ready[pb], kb & 1, abort)) break;
                tc_fence_after();
                // O += A V  (A = masked P as bf16 in TMEM, B = V MN-major, K = C)
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks) {
                    const uint64_t bdesc = smem_desc(va + ks * 2048, kC * 128, 1024);
                    const uint32_t a_t = tmem + C::col_p(pb) + ks * 8;
                    asm volatile(
                        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem + C::col_o(pb)),
                        "r"(a_t), "l"(bdesc), "r"(ID_O), "r"(1)
                        : "memory");
                }
                mma_commit(&bars.o_full[pb]);
                mma_commit(&bars.empty[s]);
            }
            // no MMA may still be running when the CTA frees its TMEM
            mma_commit(bars.drain);
            mbar_wait_bounded(bars.drain, 0, now_ns() + kWaitNs, nullptr);
        }
    } else {
        // ------------------------------------------------------ working group
        const int t = tid - 64;
        const int q4 = warp & 3;                 // TMEM lane quarter this warp may access
        const int r = 32 * q4 + lane;            // chunk row / state row owned by this thread
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const bool srow = r < D;                 // owns a state row
        const bool swarp = 32 * q4 < D;          // warp-uniform
        const float *ws_h = args.seg_ws ? args.seg_ws + (size_t)bh * args.nseg * (D * M + D) : nullptr;
        float *S_h = args.S ? args.S + (size_t)bh * D * M : nullptr;
        float *z_h = args.z ? args.z + (size_t)bh * D : nullptr;
        __nv_bfloat16 *out_h = args.out ? reinterpret_cast<__nv_bfloat16 *>(args.out) + (size_t)bh * args.N * M
                                        : nullptr;

        // initial state: carried-in state plus the sums of earlier segments
        if (swarp) {
            float v[M];
            float zr = 0.f;
#pragma unroll
            for (int c = 0; c < M; ++c) v[c] = 0.f;
            if (srow) {
                if (S_h) {
#pragma unroll
                    for (int c = 0; c < M; c += 4) {
                        const float4 x = *reinterpret_cast<const float4 *>(S_h + r * M + c);
                        v[c] = x.x; v[c + 1] = x.y; v[c + 2] = x.z; v[c + 3] = x.w;
                    }
                    zr = z_h[r];
                }
                for (int g = 0; g < seg; ++g) {
                    const float *src = ws_h + (size_t)g * (D * M + D);
#pragma unroll
                    for (int c = 0; c < M; c += 4) {
                        const float4 x = *reinterpret_cast<const float4 *>(src + r * M + c);
                        v[c] += x.x; v[c + 1] += x.y; v[c + 2] += x.z; v[c + 3] += x.w;
                    }
                    zr += src[D * M + r];
                }
                store_snap_row<D, M>(snap, r, v);
                zs[r] = zr;
            }
#pragma unroll
            for (int c0 = 0; c0 < M; c0 += 16) {
                uint32_t w[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) w[j] = __float_as_uint(v[c0 + j]);
                tmem_st16(tmem + lane_off + C::COL_S + c0, w);
            }
            uint32_t w[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) w[j] = 0u;
            w[0] = __float_as_uint(zr);
            tmem_st16(tmem + lane_off + C::COL_Z, w);
            tmem_wait_st();
        }
        tc_fence_before();
        fence_proxy_async();
        mbar_arrive(bars.snap);

        float den = 0.f;
        // phi of the first chunk
        if (n > 0) {
            if (wait_bar(&bars.full[0], 0, abort)) {
                uint8_t *st = smem;
                const int valid = min(kC, args.N - c_begin * kC);
                phi_tile<D>(st, t, kC);
                phi_tile<D>(st + C::TILE_QK, t, valid);
            }
            fence_proxy_async();
            mbar_arrive(&bars.phi[0]);
        }
        for (int it = 0; it < n; ++it) {
            const int s = it % C::NS;
            const int pb = it % C::NPB, kb = it / C::NPB;
            const int t0 = (c_begin + it) * kC;
            const int valid = min(kC, args.N - t0);
            uint8_t *st = smem + s * C::STAGE;
            // ---- P: mask j > r, row sums of the bf16-rounded values, back to TMEM as bf16
            bool ok = wait_bar(&bars.p_full[pb], kb & 1, abort);
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                float rs = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t pv[64];
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        tmem_ld16(tmem + lane_off + C::col_p(pb) + h * 64 + j * 16,
                                  *reinterpret_cast<uint32_t(*)[16]>(&pv[j * 16]));
                    tmem_wait_ld();
                    uint32_t a[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int c = h * 64 + 2 * j;
                        const float x0 = (c <= r) ? __uint_as_float(pv[2 * j]) : 0.f;
                        const float x1 = (c + 1 <= r) ? __uint_as_float(pv[2 * j + 1]) : 0.f;
                        a[j] = pack_bf16x2(x0, x1);
                        rs += bf16lo(a[j]) + bf16hi(a[j]);
                    }
                    tmem_st16(tmem + lane_off + C::col_p(pb) + h * 32, *reinterpret_cast<uint32_t(*)[16]>(&a[0]));
                    tmem_st16(tmem + lane_off + C::col_p(pb) + h * 32 + 16,
                              *reinterpret_cast<uint32_t(*)[16]>(&a[16]));
                }
                tmem_wait_st();
                den = rs + q_dot_z<D>(st, r, zs);
            }
            tc_fence_before();
            mbar_arrive(&bars.a_ready[pb]);
            if (it + 1 < n) {
                // ---- phi of the next chunk (lets the next P = phi(Q) phi(K)^T start early)
                const int s1 = (it + 1) % C::NS, k1 = (it + 1) / C::NS;
                if (wait_bar(&bars.full[s1], k1 & 1, abort)) {
                    uint8_t *st1 = smem + s1 * C::STAGE;
                    const int valid1 = min(kC, args.N - t0 - kC);
                    phi_tile<D>(st1, t, kC);
                    phi_tile<D>(st1 + C::TILE_QK, t, valid1);
                }
                fence_proxy_async();
                mbar_arrive(&bars.phi[s1]);
            }
            wg_sync();   // every thread is done reading z_prev before it is replaced
            if (it + 1 < n) {
                // ---- snapshot of the state after this chunk, for the next chunk
                bool ok2 = wait_bar(bars.s_full, it & 1, abort);
                ok2 = __all_sync(0xffffffffu, ok2);
                if (ok2 && swarp) {
                    tc_fence_after();
                    uint32_t sv[M];
#pragma unroll
                    for (int c0 = 0; c0 < M; c0 += 16)
                        tmem_ld16(tmem + lane_off + C::COL_S + c0, *reinterpret_cast<uint32_t(*)[16]>(&sv[c0]));
                    uint32_t zv[16];
                    tmem_ld16(tmem + lane_off + C::COL_Z, zv);
                    tmem_wait_ld();
                    if (srow) {
                        store_snap_row<D, M>(snap, r, reinterpret_cast<const float *>(sv));
                        zs[r] = __uint_as_float(zv[0]);
                    }
                }
                tc_fence_before();
                fence_proxy_async();
                mbar_arrive(bars.snap);
            }
            // ---- output rows
            bool ok3 = wait_bar(&bars.o_full[pb], kb & 1, abort);
            ok3 = __all_sync(0xffffffffu, ok3);
            if (ok3) {
                tc_fence_after();
                uint32_t ov[M];
#pragma unroll
                for (int c0 = 0; c0 < M; c0 += 16)
                    tmem_ld16(tmem + lane_off + C::col_o(pb) + c0, *reinterpret_cast<uint32_t(*)[16]>(&ov[c0]));
                tmem_wait_ld();
                tc_fence_before();
                mbar_arrive(&bars.o_free[pb]);
                if (out_h && r < valid) {
                    const float inv = 1.f / den;
                    uint4 *dst = reinterpret_cast<uint4 *>(out_h + (size_t)(t0 + r) * M);
#pragma unroll
                    for (int c = 0; c < M; c += 8) {
                        uint4 w;
                        w.x = pack_bf16x2(__uint_as_float(ov[c]) * inv, __uint_as_float(ov[c + 1]) * inv);
                        w.y = pack_bf16x2(__uint_as_float(ov[c + 2]) * inv, __uint_as_float(ov[c + 3]) * inv);
                        w.z = pack_bf16x2(__uint_as_float(ov[c + 4]) * inv, __uint_as_float(ov[c + 5]) * inv);
                        w.w = pack_bf16x2(__uint_as_float(ov[c + 6]) * inv, __uint_as_float(ov[c + 7]) * inv);
                        dst[c / 8] = w;
                    }
                }
            } else {
                tc_fence_before();
                mbar_arrive(&bars.o_free[pb]);
            }
        }
        // ---- final state of the sequence (last segment only)
        if (S_h && seg == args.nseg - 1 && n > 0) {
            bool ok4 = wait_bar(bars.s_full, (n - 1) & 1, abort);
            ok4 = __all_sync(0xffffffffu, ok4);
            if (ok4 && swarp) {
                tc_fence_after();
                uint32_t sv[M];
#pragma unroll
                for (int c0 = 0; c0 < M; c0 += 16)
                    tmem_ld16(tmem + lane_off + C::COL_S + c0, *reinterpret_cast<uint32_t(*)[16]>(&sv[c0]));
                uint32_t zv[16];
                tmem_ld16(tmem + lane_off + C::COL_Z, zv);
                tmem_wait_ld();
                if (srow) {
#pragma unroll
                    for (int c = 0; c < M; c += 4)
                        *reinterpret_cast<float4 *>(S_h + r * M + c) =
                            make_float4(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1]),
                                        __uint_as_float(sv[c + 2]), __uint_as_float(sv[c + 3]));
                    z_h[r] = __uint_as_float(zv[0]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int D, int M>
cudaError_t launch_causal(const Problem &p, const DeviceInfo &dev) {
    using C = Cfg<D, M>;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bf16_3d(&tq, p.q, D, p.N, p.BH, 64, kC) || !make_tmap_bf16_3d(&tk, p.k, D, p.N, p.BH, 64, kC) ||
        !make_tmap_bf16_3d(&tv, p.v, M, p.N, p.BH, 64, kC))
        return cudaErrorInvalidValue;
    CausalArgs a;
    a.out = p.out;
    a.S = p.S;
    a.z = p.z;
    a.seg_ws = nullptr;
    a.N = p.N;
    a.nseg = 1;
    a.cps = (p.N + kC - 1) / kC;
    a.err = dev.err_word;
    a.inject_ns = g_inject_timeout ? (uint64_t)g_inject_limit_us * 1000ull : 0ull;
    cudaError_t e = cudaFuncSetAttribute(causal_tc_kernel<D, M>, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
    if (e != cudaSuccess) return e;
    causal_tc_kernel<D, M><<<(unsigned)(p.BH * a.nseg), kThreads, C::SMEM, p.stream>>>(tq, tk, tv, a);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

bool tc_causal_supported(const la_shape &s, int chunk) {
    return s.dtype == LA_DTYPE_BF16 && (s.D == 64 || s.D == 128) && (s.M == 64 || s.M == 128) &&
           (chunk == 0 || chunk == 128);
}

size_t tc_causal_ws_bytes(const la_shape &, int) { return 0; }

cudaError_t tc_causal(const Problem &p, const DeviceInfo &dev) {
    if (p.D == 64 && p.M == 64) return launch_causal<64, 64>(p, dev);
    if (p.D == 64 && p.M == 128) return launch_causal<64, 128>(p, dev);
    if (p.D == 128 && p.M == 64) return launch_causal<128, 64>(p, dev);
    if (p.D == 128 && p.M == 128) return launch_causal<128, 128>(p, dev);
    return cudaErrorInvalidValue;
}

bool tc_noncausal_supported(const la_shape &) { return false; }
size_t tc_noncausal_ws_bytes(const la_shape &) { return 0; }
cudaError_t tc_noncausal(const Problem &, const DeviceInfo &) { return cudaErrorNotSupported; }

}  // namespace la

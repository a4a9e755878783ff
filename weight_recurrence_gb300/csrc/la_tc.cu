// la_tc.cu - tensor-core (tcgen05 + TMA) kernels of liblinattn.so for bf16
// inputs with D, M in {64, 128}.
//
// Method ("Transformers are RNNs", read in its Chinese translation):
// causal attention, sec. 3.3 eqs. (9)-(12), regrouped into chunks of C = 128
// rows.  For chunk c with rows t0..t0+C-1 of one head:
//   P      = phi(Q_c) phi(K_c)^T                       (C x C, fp32 in TMEM)
//   A      = P with A_ij = 0 for j > i (diagonal kept, eq. (8)), rounded to bf16
//   num    = A V_c + phi(Q_c) S_prev                    (C x M, fp32 in TMEM)
//   den_i  = sum_j A_ij + phi(Q_c)_i . z_prev            (fp32)
//   out_i  = num_i / den_i                               (eq. (12))
//   S_prev += phi(K_c)^T V_c,  z_prev += phi(K_c)^T 1   (eqs. (10), (11))
// Exact in real arithmetic: the j <= i sum of eq. (9) is split at the chunk
// start into the in-chunk part and the carried prefix state.  The non-causal
// form (sec. 3.2 eq. (5)) is the same two summaries taken over all keys
// followed by the read-out phi(Q) S / phi(Q) z (noncausal_tc_kernel, one
// launch, the CTAs of a head exchanging partial sums within a cluster).
//
// Roles of the causal CTA (480 threads; 608 with two feature-map groups):
//   warp 0      TMA producer: chunk tiles into a ring of NS stages, 128-byte
//               swizzled (the tcgen05 canonical K-major layout);
//   warp 1      P issuer (one thread): P = phi(Q) phi(K)^T as soon as the
//               feature map is applied; at D = M = 64 also the chunk's state
//               increment phi(K)^T [V | 1] into a fresh TMEM buffer;
//   warp 2      output issuer (one thread): at other sizes first the state
//               update S += phi(K)^T V (accumulated in TMEM), then A V and
//               phi(Q) S_prev; completion through tcgen05.commit on mbarriers;
//   warps 3-6   P group, one thread per TMEM lane: masks P and writes it back to
//               TMEM as bf16 (the A operand of A V), and forms phi(Q_i).z_prev;
//   warps 7-10  O group: keeps the state (in registers at D = M = 64, adding
//               each increment; else in TMEM), writes the bf16 shared-memory
//               snapshot that is the B operand of phi(Q) S_prev, divides the
//               output rows and writes them out (at D = M = 64 staged in the
//               stage's dead Q and K tiles for one TMA store per chunk; else
//               straight from registers);
//   warps 11-14 feature-map group: applies phi in place to the Q and K tiles as
//               they land, running ahead of the MMAs by up to NS chunks.
// The segment-sum and non-causal kernels use warps 0-9 the same way with one
// epilogue group (320 threads).
// The state S (D x M) and z (D) stay on chip in fp32 for the whole segment.
// Launches are programmatic (launch_pdl): a CTA's set-up overlaps the previous
// launch's tail, it may prefetch its first tiles into L2 meanwhile, and one
// thread waits for the previous grid before any global-memory read.
// Long sequences with few heads are cut into segments; the state entering
// segment g is the carried-in state plus the fp32 sums of segments < g,
// computed beforehand by state_reduce_kernel (two passes, no inter-CTA waits).
// Every mbarrier wait is bounded; a CTA that gives up records LA_ERR_TIMEOUT,
// lets its copies and MMAs drain, frees its TMEM and returns.
#include <algorithm>
#include <mutex>
#include <utility>
#include <vector>

#include "la_common.cuh"
#include "la_internal.h"
#include "tc_host.h"
#include "tc_ptx.cuh"
#include "tc_kernels.cuh"

// Optional timeline of CTA 0 for performance work: compiled only with
// -DLA_TRACE (never in the library build); read with la_trace_read().
#ifdef LA_TRACE
__device__ unsigned long long g_la_trace[5][64][8];
extern "C" int la_trace_read(unsigned long long *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_la_trace, sizeof(g_la_trace));
}
#define LA_TRACE_AT(role, it, ev)                                                     \
    do {                                                                              \
        if (blockIdx.x == 0 && (it) < 64) g_la_trace[role][it][ev] = (unsigned long long)clock64(); \
    } while (0)
// per-CTA global-timer events of the last eight launches (slot = launch % 8);
// event 11 holds the SM id
__device__ unsigned long long g_la_cta[8][512][12];
__device__ unsigned int g_la_cta_ctr;
extern "C" int la_trace_read_cta(unsigned long long *dst) {
    return (int)cudaMemcpyFromSymbol(dst, g_la_cta, sizeof(g_la_cta));
}
extern "C" int la_trace_reset_cta() {
    const unsigned int z = 0;
    return (int)cudaMemcpyToSymbol(g_la_cta_ctr, &z, sizeof(z));
}
// (the slot of each CTA lives in global memory: no static shared memory,
// which would change the CTAs' shared-memory footprint and so the occupancy)
__device__ unsigned int g_la_cta_slot[512];
#define LA_CTA_BEGIN()                                                                \
    if (threadIdx.x == 0 && blockIdx.x < 512) {                                       \
        const unsigned int sl_ = atomicAdd(&g_la_cta_ctr, 1u) / gridDim.x;            \
        g_la_cta_slot[blockIdx.x] = sl_;                                              \
        unsigned int sm_;                                                             \
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm_));                              \
        g_la_cta[sl_ & 7][blockIdx.x][11] = sm_;                                      \
    }
#define LA_CTA_AT(ev)                                                                 \
    do {                                                                              \
        if (blockIdx.x < 512) {                                                       \
            unsigned long long t_;                                                    \
            asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t_));                    \
            g_la_cta[*(volatile unsigned int *)&g_la_cta_slot[blockIdx.x] & 7][blockIdx.x][ev] = t_; \
        }                                                                             \
    } while (0)
#else
#define LA_TRACE_AT(role, it, ev) ((void)0)
#define LA_CTA_BEGIN()
#define LA_CTA_AT(ev) ((void)0)
#endif

namespace la {
namespace {

using namespace tc;

// ------------------------------------------------------------ causal kernel

// Warps of the causal CTA: 0 producer, 1 P issuer, 2 output issuer, 3-6 P
// group, 7-10 O group, 11-14 feature-map group (phi(Q) and phi(K)), or 11-14
// phi(Q) and 15-18 phi(K) with two feature-map groups.
constexpr int kWarpP = 3, kWarpO = 7, kWarpPhi = 11;

template <int D, int M>
struct Cfg {
    static constexpr int TILE_QK = kC * D * 2;
    static constexpr int TILE_V = kC * M * 2;
    static constexpr int STAGE = 2 * TILE_QK + TILE_V;
    static constexpr int SNAP = D * M * 2;
    // M = 64: O shares its P buffer; V is read as [V | ones] (N = 80) so that
    // the state update also yields z and A V also yields the row sums; and the
    // snapshot is read as [S | z] (N = 80) so that phi(Q) S_prev also yields
    // phi(Q).z_prev.  The ones operand is a [C x 64] MN-major tile with ones in
    // column 0; z of snapshot b is stored as two bf16 parts (hi, lo) in its
    // columns 16(b+1)+1 and 16(b+1)+2, read as an N-atom that starts 32(b+1)
    // bytes into the tile (the 128-byte swizzle acts on address bits, so a
    // 16-column window of a swizzled tile is itself a valid atom).
    static constexpr bool O_IN_P = (M == 64);
    static constexpr bool ZMMA = O_IN_P;
    // D = M = 64: each chunk's state increment dS = phi(K)^T [V | 1] goes to a
    // fresh TMEM buffer (two of them) and the O group adds it to an fp32 copy
    // of the state held in its registers, so the state MMAs never wait for a
    // snapshot.  The increment's A operand repeats its 64 rows (M-atom stride
    // 0), so accumulator lanes 64-127 hold a second copy and all four warps of
    // the O group can each take one row and half of its columns.
    static constexpr bool DS = (D == 64 && M == 64);
    static constexpr int NPB = DS ? 2 : (O_IN_P ? 3 : 1);   // P buffers in TMEM
    // D = M = 64: output rows are staged (swizzled) in the stage's dead Q and K
    // tiles and stored by TMA, the stage being released once the store has
    // read them; one feature-map group.  Other sizes: each O-group thread
    // stores its own output row, and two feature-map groups share the tiles
    // (measured choices: at D = M = 128 the feature map, not the stage ring,
    // limits the pipeline).
    static constexpr bool OUT_TMA = DS;
    // D = M = 64: a stage is two parts with barriers of their own, the Q and K
    // tiles and the V tile, and the output rows are staged in the V tile.  The
    // Q and K tiles are handed back as soon as the chunk's MMAs have read them,
    // so the next loads into the stage (and their feature map, on the critical
    // path) start before the output store has read the staged rows.
    static constexpr bool SPLITV = DS;
    static constexpr int NPHI = DS ? 1 : 2;
    static constexpr int THREADS = 32 * (kWarpPhi + 4 * NPHI);
    static constexpr int NDZ = ZMMA ? 1 : 2;           // phi(Q).z_prev hand-over slots (TMEM)
    static constexpr int ONES = O_IN_P ? kC * 128 : kOnesBytes;
    static constexpr int ZS_BYTES = ZMMA ? 0 : 2 * D * 4;
    static constexpr int NBARS_MAX = 3 * 4 + 4 * 3 + 2 + 5 + 4 + 2 * 4;
    static constexpr int FIXED1 = SNAP + ONES + ZS_BYTES + 8 * NBARS_MAX + 16;
    // two state snapshots when two stages still fit beside them
    static constexpr bool DB = (kSmemMax - FIXED1 - SNAP) / STAGE >= 2;
    static constexpr int NSB = DB ? 2 : 1;
    static constexpr int FIXED = FIXED1 + (NSB - 1) * SNAP;
    static constexpr int NS_FIT = (int)((kSmemMax - FIXED) / STAGE);
    static constexpr int NS = NS_FIT > 4 ? 4 : NS_FIT;
    static_assert(NS >= 2, "pipeline needs two stages");
    static constexpr int NBARS = 3 * NS + 4 * NPB + NDZ + 5 + 4 + 2 * NS;
    static constexpr int OFF_SNAP = NS * STAGE;
    static constexpr int OFF_ONES = OFF_SNAP + NSB * SNAP;
    static constexpr int OFF_Z = OFF_ONES + ONES;           // z snapshots [2][D] fp32 (without ZMMA)
    static constexpr int OFF_BAR = OFF_Z + ZS_BYTES;
    static constexpr int OFF_TSLOT = OFF_BAR + 8 * NBARS;
    static constexpr int SMEM = OFF_TSLOT + 16;
    static_assert(SMEM <= (int)kSmemMax, "shared memory budget");
    // TMEM columns.  D = M = 64: two 144-column P/O buffers (as below) and two
    // 80-column increment buffers at 288 and 368.  M = 64: three 144-column buffers, each holding P
    // (128 fp32 columns), then A (bf16, columns 0-63) and O (columns 64-143:
    // 64 numerator columns, then row sum, phi(Q).z_hi, phi(Q).z_lo); S and z
    // in 432-511.  M = 128: P, a separate A, O, S, z, a 16-column row-sum
    // block and two 16-column slots handing phi(Q).z_prev from the P group to
    // the O group.
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t COL_S = O_IN_P ? 432 : 320;
    static constexpr uint32_t COL_Z = COL_S + M;
    static __device__ __forceinline__ uint32_t col_p(int b) { return O_IN_P ? 144u * b : 0u; }
    static __device__ __forceinline__ uint32_t col_a(int b) { return O_IN_P ? 144u * b : 128u; }
    static __device__ __forceinline__ uint32_t col_o(int b) { return O_IN_P ? 144u * b + 64u : 192u; }
    static __device__ __forceinline__ uint32_t col_den(int b) { return O_IN_P ? 144u * b + 128u : 464u; }
    static __device__ __forceinline__ uint32_t col_dz(int j) { return 480u + 16u * (j & 1); }
    static __device__ __forceinline__ uint32_t col_ds(int j) { return 288u + 80u * (j & 1); }
    static_assert(O_IN_P ? (COL_Z + 16 <= TMEM_COLS) : (COL_Z + 16 <= 464), "TMEM budget");
};

struct CausalArgs {
    __nv_bfloat16 *out;      // [BH, N, M] or null (state only)
    float *S;                // [BH, D, M] in/out or null
    float *z;                // [BH, D] in/out or null
    const float *seg_ws;     // nseg > 1: [BH, nseg, D*M + D]; slots < nseg-1 hold segment sums,
                             // slot nseg-1 the state carried in
    int N;
    int nseg;                // segments per head
    int cps;                 // chunks per segment
    int *err;
    uint64_t inject_ns;      // test hook: wait this long on a flag nobody sets
    const int *lens;         // per-batch sequence lengths (device) or null: rows past them are ignored
    int H;                   // heads per batch entry
    long long o_rs, o_hs;    // output row and head strides (elements) for the direct stores
    int feat;                // kFeatPhi (elu + 1 in place) or a row feature map of a variant
    int dr, nu;              // raw width of Q, K rows and DPFP shifts (feat != kFeatPhi)
    int sum_norm;            // DPFP: divide each feature row by its sum
    int no_den;              // read-out without the denominator: out = num
    // extents the checked build tests direct accesses against (elements)
    long long nheads, state_elems, ws_floats, out_elems;
    int inject_oob;          // checked build test hook: state loads offset past the state
};

// Named barrier of the O group's 128 threads.
__device__ __forceinline__ void o_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// VAR: a variant's feature map and read-out (CausalArgs feat, no_den); the
// plain instantiation compiles without that code.
template <int D, int M, bool VAR>
__global__ void __launch_bounds__(Cfg<D, M>::THREADS, 1)
causal_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                 const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                 const CausalArgs args)
{
    using C = Cfg<D, M>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    if (tid == 0) LA_TRACE_AT(0, 63, 0);
    LA_CTA_BEGIN();
    if (tid == 0) LA_CTA_AT(0);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_TSLOT + 4);

    const int bh = blockIdx.x / args.nseg, seg = blockIdx.x % args.nseg;
    const int c_begin = seg * args.cps;
    // the next launch on the stream may start its own set-up now (it reads
    // nothing of ours before its griddepcontrol.wait).  Measured: this early
    // trigger helps the plain kernel; with a variant's feature map the next
    // grid's early CTAs slowed the running one (91 -> 105 us for DPFP-1), so
    // that instantiation triggers implicitly, at exit.
    if (!VAR) pdl_launch_dependents();

    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full = bar, *empty = bar + C::NS, *phi_done = bar + 2 * C::NS;
    uint64_t *p_full = bar + 3 * C::NS, *a_ready = p_full + C::NPB, *o_full = a_ready + C::NPB,
             *o_free = o_full + C::NPB, *dz_ready = o_free + C::NPB;
    // snapshot of the state entering chunk j: barrier j & 1, phase j >> 1 (two
    // barriers, so that no waiter can fall two phases behind one barrier)
    uint64_t *snap_bar = dz_ready + C::NDZ, *s_full = snap_bar + 2, *never = s_full + 1, *drain = never + 1;
    uint64_t *ds_full = drain + 1, *ds_free = ds_full + 2;   // increment buffers (DS)
    uint64_t *full_v = ds_free + 2, *empty_v = full_v + C::NS;  // the V part of each stage (SPLITV)
    auto snap_wait = [&](int j) { return wait_bar(&snap_bar[j & 1], (j >> 1) & 1, abort); };
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::OFF_TSLOT);
    uint8_t *snap0 = smem + C::OFF_SNAP;
    uint8_t *ones = smem + C::OFF_ONES;
    float *zs0 = reinterpret_cast<float *>(smem + C::OFF_Z);
    auto snap_buf = [&](int j) { return snap0 + (C::DB ? (j & 1) : 0) * C::SNAP; };
    // column of the ones tile holding z_hi of snapshot j (z_lo in the next one)
    auto zcol = [&](int j) { return 16 * (1 + (C::DB ? (j & 1) : 0)) + 1; };
    auto zs_buf = [&](int j) { return zs0 + (j & 1) * D; };

    if (tid == 0) {
        *abort = (smem_u32(smem) & 1023u) ? 1 : 0;   // the swizzled layouts need a 1024-byte aligned base
        if (*abort) record_error(args.err, kErrTimeout);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(&full[s], 1);
            // released by the output issuer's commit, with DS also by the P
            // issuer's (state increment), and without ZMMA by the P group once it
            // has read phi(Q) for phi(Q).z_prev
            mbar_init(&empty[s], (C::DS ? 2 : 1) + (C::ZMMA ? 0 : kGrp) + (C::OUT_TMA && !C::SPLITV ? 1 : 0));
            mbar_init(&phi_done[s], C::NPHI * kGrp);
            // V part: the state increment's and the output MMAs' commits, and the
            // output store having read the staged rows
            mbar_init(&full_v[s], 1);
            mbar_init(&empty_v[s], 3);
        }
        for (int b = 0; b < C::NPB; ++b) {
            mbar_init(&p_full[b], 1);
            mbar_init(&a_ready[b], kGrp);
            mbar_init(&o_full[b], 1);
            mbar_init(&o_free[b], kGrp);
        }
        for (int b = 0; b < C::NDZ; ++b) mbar_init(&dz_ready[b], kGrp);
        mbar_init(&snap_bar[0], kGrp);
        mbar_init(&snap_bar[1], kGrp);
        mbar_init(s_full, 1);
        mbar_init(never, 1);
        mbar_init(drain, 2);
        for (int b = 0; b < 2; ++b) {
            mbar_init(&ds_full[b], 1);
            mbar_init(&ds_free[b], kGrp);
        }
        fence_mbar_init();
    }
    // ones operand, MN-major, ones in column 0 and zeros elsewhere: [C K-rows x 64]
    // when it is read as the second N-atom of [V | ones], else one 8-row atom
    for (int i = tid; i < C::ONES / 4; i += C::THREADS) reinterpret_cast<uint32_t *>(ones)[i] = 0u;
    __syncthreads();
    for (int k = tid; k < C::ONES / 128; k += C::THREADS)
        *reinterpret_cast<uint16_t *>(ones + sw128_offset(k, 0)) = 0x3F80u;
    if (warp == 0) {
        tmem_alloc(tslot, C::TMEM_COLS);
        tmem_relinquish();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (tid == 0) LA_TRACE_AT(0, 63, 1);
    // the first two chunks' Q, K, V boxes into L2 while the previous launch on
    // the stream drains: a hint only (L2 is where that launch's writes land, so
    // a line fetched now cannot be stale when the loads below read it).
    // Measured at D = M = 64: 38.2 -> 37.4 us with one chunk, 36.8 with two,
    // 37.2 with three, 37.8 with four (the early traffic then delays the
    // previous grid's completion)
    if (C::DS && !VAR && tid == 0)
        for (int c = 0; c < 2 && c < args.cps && (c_begin + c) * kC < args.N; ++c) {
            const int t0 = (c_begin + c) * kC;
            tma_prefetch_3d(&tm_q, 0, t0, bh);
            tma_prefetch_3d(&tm_k, 0, t0, bh);
            tma_prefetch_3d(&tm_v, 0, t0, bh);
        }
    // everything above read no global memory; from here on the previous
    // launch on the stream has completed and its writes are visible
    pdl_wait_cta();
    if (tid == 0) LA_CTA_AT(1);
    // this head's sequence length (rows past it are read but ignored)
    const int Nseq = args.lens ? max(0, min(args.N, LA_IN_BOUNDS(bh < args.nheads, args.err) ? args.lens[bh / args.H] : 0))
                               : args.N;
    const int nch_total = (Nseq + kC - 1) / kC;
    const int n = max(0, min(nch_total, c_begin + args.cps) - c_begin);

    // Test hook: wait on a barrier that nothing arrives on, then give up.
    if (args.inject_ns && tid == 0) {
        if (!mbar_wait_bounded(never, 0, now_ns() + args.inject_ns, nullptr)) set_abort(abort, args.err);
    }
    __syncthreads();

    constexpr uint32_t ID_16 = idesc_bf16(128, 16, 1, 1);
    const uint32_t ones_a = smem_u32(ones);
    const uint64_t ones_d = ones_desc(ones_a);
    // V read MN-major; with M = 64 its second N-atom is the ones tile
    auto v_base = [&](uint32_t va) { return smem_desc(va, C::O_IN_P ? ones_a - va : (uint32_t)(kC * 128), 1024); };

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0 && !*abort) {
            prefetch_tmap(&tm_q);
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued = 0, issued_v = 0;
            for (int it = 0; it < n; ++it) {
                const int s = it % C::NS, k = it / C::NS;
                if (it >= C::NS && !wait_bar(&empty[s], (k - 1) & 1, abort)) break;
                uint8_t *st = smem + s * C::STAGE;
                const int t0 = (c_begin + it) * kC;
                LA_TRACE_AT(0, it, 0);
                // DPFP rows arrive raw (at most 64 columns, one box each), the
                // feature-map group expands them to the D feature columns
                const int qk_boxes = VAR && args.feat == kFeatDpfp ? 1 : D / 64;
                mbar_arrive_expect_tx(&full[s], 2 * qk_boxes * kC * 128 + (C::SPLITV ? 0 : C::TILE_V));
                for (int j = 0; j < qk_boxes; ++j) tma_load_3d(st + j * kC * 128, &tm_q, &full[s], j * 64, t0, bh);
                for (int j = 0; j < qk_boxes; ++j)
                    tma_load_3d(st + C::TILE_QK + j * kC * 128, &tm_k, &full[s], j * 64, t0, bh);
                ++issued;
                uint64_t *fv = &full[s];
                if (C::SPLITV) {
                    if (it >= C::NS && !wait_bar(&empty_v[s], (k - 1) & 1, abort)) break;
                    fv = &full_v[s];
                    mbar_arrive_expect_tx(fv, C::TILE_V);
                }
#pragma unroll
                for (int j = 0; j < M / 64; ++j)
                    tma_load_3d(st + 2 * C::TILE_QK + j * kC * 128, &tm_v, fv, j * 64, t0, bh);
                ++issued_v;
            }
            if (*abort) {   // let the copies in flight land before the CTA exits
                for (int it = max(0, issued - C::NS); it < issued; ++it)
                    mbar_wait_bounded(&full[it % C::NS], (it / C::NS) & 1, now_ns() + kWaitNs, nullptr);
                if (C::SPLITV)
                    for (int it = max(0, issued_v - C::NS); it < issued_v; ++it)
                        mbar_wait_bounded(&full_v[it % C::NS], (it / C::NS) & 1, now_ns() + kWaitNs, nullptr);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ P issuer
        // P = phi(Q) phi(K)^T for each chunk into its P buffer, as soon as the
        // feature map is applied and the buffer is free; with DS also the state
        // increment dS = phi(K)^T [V | 1] into its buffer
        if (lane == 0 && !*abort) {
            constexpr uint32_t ID_P = idesc_bf16(128, kC, 0, 0);
            constexpr uint32_t ID_DS = idesc_bf16(128, M + 16, 1, 1);
            for (int j = 0; j < n; ++j) {
                const int s = j % C::NS, pb = j % C::NPB, kb = j / C::NPB;
                if (!wait_bar(&phi_done[s], (j / C::NS) & 1, abort)) break;
                LA_TRACE_AT(1, j, 0);
                if (C::O_IN_P) {
                    // O(j - NPB) shares the buffer: it must have been read out
                    if (kb > 0 && !wait_bar(&o_free[pb], (kb - 1) & 1, abort)) break;
                } else if (j > 0 && !wait_bar(&a_ready[0], (j - 1) & 1, abort)) {   // P(j-1) has been read
                    break;
                }
                LA_TRACE_AT(1, j, 1);
                tc_fence_after();
                const uint32_t st = smem_u32(smem + s * C::STAGE);
                const uint64_t dq = kmajor_base(st), dk = kmajor_base(st + C::TILE_QK);
                const uint32_t dp = tmem + C::col_p(pb);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_f16_ss(dp, dq + kmajor_step(ks), dk + kmajor_step(ks), ID_P, ks > 0);
                mma_commit(&p_full[pb]);
                LA_TRACE_AT(1, j, 2);
                if (C::DS) {
                    if (j >= 2 && !wait_bar(&ds_free[j & 1], ((j >> 1) - 1) & 1, abort)) break;
                    if (C::SPLITV && !wait_bar(&full_v[s], (j / C::NS) & 1, abort)) break;   // V landed
                    LA_TRACE_AT(1, j, 3);
                    tc_fence_after();
                    // A = phi(K)^T read MN-major with M-atom stride 0 (rows 64-127 repeat 0-63)
                    const uint64_t dk = smem_desc(st + C::TILE_QK, 0, 1024), dv = v_base(st + 2 * C::TILE_QK);
#pragma unroll
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_f16_ss(tmem + C::col_ds(j), dk + mnmajor_step(ks), dv + mnmajor_step(ks), ID_DS, ks > 0);
                    mma_commit(&ds_full[j & 1]);
                    mma_commit(&empty[s]);
                    if (C::SPLITV) mma_commit(&empty_v[s]);
                    LA_TRACE_AT(1, j, 4);
                }
            }
        }
        if (lane == 0) mma_commit(drain);   // arrives once this thread's MMAs (if any) are done
    } else if (warp == 2) {
        // ------------------------------------------------------ output issuer
        // Per chunk, in this order: (without DS) S += phi(K)^T V and z +=
        // phi(K)^T 1 (the serial chain from chunk to chunk; A = phi(K) read
        // MN-major, 128 rows, accumulator rows >= D never read), then the output
        // MMAs O = A [V | 1] + phi(Q) [S_prev | z_prev].  One commit after the
        // output MMAs covers both, so it releases the stage; s_full after the
        // state update also guarantees that the output MMAs of the previous
        // chunk, which read the snapshot buffer the O group overwrites next,
        // have completed.
        if (lane == 0 && !*abort) {
            constexpr int NV = C::O_IN_P ? M + 16 : M;
            constexpr uint32_t ID_S = idesc_bf16(128, NV, 1, 1);
            constexpr uint32_t ID_O = idesc_bf16(128, M, 0, 1);
            constexpr uint32_t ID_AV = idesc_bf16(128, NV, 0, 1);
            constexpr uint32_t ID_D = idesc_bf16(128, 16, 0, 1);
            constexpr uint32_t ID_I = C::ZMMA ? idesc_bf16(128, M + 16, 0, 1) : ID_O;
            for (int it = 0; it < n; ++it) {
                const int s = it % C::NS, pb = it % C::NPB, kb = it / C::NPB;
                if (!wait_bar(&phi_done[s], (it / C::NS) & 1, abort)) break;
                if (C::SPLITV && !wait_bar(&full_v[s], (it / C::NS) & 1, abort)) break;   // V landed
                if (!snap_wait(it)) break;   // S(it-1) has been read out
                LA_TRACE_AT(4, it, 5);
                tc_fence_after();
                const uint32_t st = smem_u32(smem + s * C::STAGE);
                const uint32_t qa = st, va = st + 2 * C::TILE_QK;
                const uint64_t dv = v_base(va);
                if (!C::DS) {
                    const uint64_t dk = smem_desc(st + C::TILE_QK, kC * 128, 1024);
#pragma unroll
                    for (int ks = 0; ks < kC / 16; ++ks) {
                        mma_f16_ss(tmem + C::COL_S, dk + mnmajor_step(ks), dv + mnmajor_step(ks), ID_S, 1);
                        if (!C::O_IN_P) mma_f16_ss(tmem + C::COL_Z, dk + mnmajor_step(ks), ones_d, ID_16, 1);
                    }
                    mma_commit(s_full);
                }

                if (!wait_bar(&a_ready[pb], kb & 1, abort)) break;
                if (!C::O_IN_P && it > 0 && !wait_bar(&o_free[0], (it - 1) & 1, abort)) break;
                LA_TRACE_AT(4, it, 6);
                tc_fence_after();
                // phi(Q) [S_prev | z]: the z atom is the 16-column window of the ones
                // tile holding snapshot it's z
                const uint32_t sa = smem_u32(snap_buf(it));
                const uint32_t za = ones_a + 2 * (zcol(it) - 1);
                const uint64_t dq = kmajor_base(qa);
                const uint64_t ds = smem_desc(sa, C::ZMMA ? za - sa : (uint32_t)(D * 128), 1024);
                if (C::O_IN_P) {
                    // O = A [V | 1] (numerator and row sums), then O += phi(Q) S_prev
#pragma unroll
                    for (int ks = 0; ks < kC / 16; ++ks)
                        mma_f16_ts(tmem + C::col_o(pb), tmem + C::col_a(pb) + ks * 8, dv + mnmajor_step(ks), ID_AV,
                                   ks > 0);
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_f16_ss(tmem + C::col_o(pb), dq + kmajor_step(ks), ds + mnmajor_step(ks), ID_I, 1);
                } else {
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        mma_f16_ss(tmem + C::col_o(0), dq + kmajor_step(ks), ds + mnmajor_step(ks), ID_I, ks > 0);
                    // O += A V and row sums A 1  (A = masked P as bf16 in TMEM, K = C)
#pragma unroll
                    for (int ks = 0; ks < kC / 16; ++ks) {
                        const uint32_t at = tmem + C::col_a(0) + ks * 8;
                        mma_f16_ts(tmem + C::col_o(0), at, dv + mnmajor_step(ks), ID_O, 1);
                        mma_f16_ts(tmem + C::col_den(0), at, ones_d, ID_D, ks > 0);
                    }
                }
                mma_commit(&o_full[pb]);
                mma_commit(&empty[s]);
                if (C::SPLITV) mma_commit(&empty_v[s]);
                LA_TRACE_AT(4, it, 7);
            }
        }
        if (lane == 0) mma_commit(drain);
    } else if (warp < kWarpO) {
        // ------------------------------------------------------ P group
        // masks P(it), rounds it to bf16 into TMEM (the A operand), and
        // computes phi(Q_r).z_prev for the O group
        const int q4 = warp & 3;                 // TMEM lane quarter this warp may access
        const int r = 32 * q4 + lane;            // chunk row owned by this thread
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        for (int it = 0; it < n; ++it) {
            const int s = it % C::NS, pb = it % C::NPB, kb = it / C::NPB;
            if (tid == 32 * kWarpP) LA_TRACE_AT(2, it, 3);
            bool ok = wait_bar_warp(&p_full[pb], kb & 1, abort);
            // without O_IN_P, A(it-1) must have been consumed before it is overwritten
            if (!C::O_IN_P && it > 0) ok = ok && wait_bar_warp(&o_full[0], (it - 1) & 1, abort);
            if (tid == 32 * kWarpP) LA_TRACE_AT(2, it, 4);
            if (ok) {
                tc_fence_after();
#pragma unroll 1
                for (int c0 = 0; c0 < kC; c0 += 32) {
                    uint32_t a[16];
                    if (c0 > 32 * q4) {          // above the diagonal for every row of this warp
#pragma unroll
                        for (int j = 0; j < 16; ++j) a[j] = 0u;
                    } else {
                        float x[32];
                        tmem_ld32f(tmem + lane_off + C::col_p(pb) + c0, x);
                        if (c0 == 32 * q4) {     // the diagonal block: keep j <= r
#pragma unroll
                            for (int j = 0; j < 16; ++j)
                                a[j] = pack_bf16x2(c0 + 2 * j <= r ? x[2 * j] : 0.f,
                                                   c0 + 2 * j + 1 <= r ? x[2 * j + 1] : 0.f);
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) a[j] = pack_bf16x2(x[2 * j], x[2 * j + 1]);
                        }
                    }
                    tmem_st16(tmem + lane_off + C::col_a(pb) + c0 / 2, a);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&a_ready[pb]);
            if (tid == 32 * kWarpP) LA_TRACE_AT(2, it, 5);
            if (!C::ZMMA) {
                // phi(Q_r) . z_prev into TMEM for the O group; the stage is released
                // once every thread of this group has read its phi(Q) row
                if (__all_sync(0xffffffffu, snap_wait(it))) {
                    uint32_t w[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) w[j] = 0u;
                    w[0] = __float_as_uint(q_dot_z<D>(smem + s * C::STAGE, r, zs_buf(it)));
                    tmem_st16(tmem + lane_off + C::col_dz(it), w);
                    tmem_wait_st();
                }
                tc_fence_before();
                mbar_arrive(&dz_ready[it % C::NDZ]);
                mbar_arrive(&empty[s]);
            }
        }
    } else if (warp < kWarpPhi) {
        // ------------------------------------------------------ O group
        // state snapshots (the B operand of phi(Q) S_prev) and the output rows
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        float *S_h = args.S ? args.S + (size_t)bh * D * M : nullptr;
        float *z_h = args.z ? args.z + (size_t)bh * D : nullptr;
        const float *ws_h = args.seg_ws ? args.seg_ws + (size_t)bh * args.nseg * (D * M + D) : nullptr;
        const bool tracer = tid == 32 * kWarpO + 32 * ((4 - kWarpO % 4) % 4);
        // z of a snapshot as two bf16 parts in the ones tile (ZMMA), or fp32
        auto put_z = [&](int j, int row, float zr) {
            if (C::ZMMA) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(zr);
                const __nv_bfloat16 lo = __float2bfloat16_rn(zr - __bfloat162float(hi));
                *reinterpret_cast<__nv_bfloat16 *>(ones + sw128_offset(row, zcol(j))) = hi;
                *reinterpret_cast<__nv_bfloat16 *>(ones + sw128_offset(row, zcol(j) + 1)) = lo;
            } else {
                zs_buf(j)[row] = zr;
            }
        };
        // fp32 state entering the segment (row `row`, columns c0..c0+31, and z):
        // the carried-in state plus the earlier segments' sums
        auto load_state32 = [&](int row, int c0, float (&v)[32]) {
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.f;
#ifdef LA_CHECKED
            if (args.inject_oob) row += D;   // test hook: caught below
#endif
            // src is the start of a D x M block at element `base` of a buffer of `extent` elements
            auto add = [&](const float *src, long long base, long long extent) {
                if (!LA_IN_BOUNDS(row < D && c0 + 32 <= M && base + (long long)row * M + c0 + 32 <= extent, args.err))
                    return;
#pragma unroll
                for (int j = 0; j < 32; j += 4) {
                    const float4 x = *reinterpret_cast<const float4 *>(src + row * M + c0 + j);
                    v[j] += x.x; v[j + 1] += x.y; v[j + 2] += x.z; v[j + 3] += x.w;
                }
            };
            const long long wsb = (long long)bh * args.nseg * (D * M + D);
            if (ws_h) {
                add(ws_h + (size_t)(args.nseg - 1) * (D * M + D), wsb + (long long)(args.nseg - 1) * (D * M + D),
                    args.ws_floats);
                for (int g = 0; g < seg; ++g)
                    add(ws_h + (size_t)g * (D * M + D), wsb + (long long)g * (D * M + D), args.ws_floats);
            } else if (S_h) {
                add(S_h, (long long)bh * D * M, args.state_elems);
            }
        };
        auto load_z = [&](int row) {
            float zr = 0.f;
            if (!LA_IN_BOUNDS(row < D && bh < args.nheads &&
                                  (!ws_h || ((long long)bh * args.nseg + args.nseg) * (D * M + D) <= args.ws_floats),
                              args.err))
                return zr;
            if (ws_h) {
                zr = ws_h[(size_t)(args.nseg - 1) * (D * M + D) + D * M + row];
                for (int g = 0; g < seg; ++g) zr += ws_h[(size_t)g * (D * M + D) + D * M + row];
            } else if (z_h) {
                zr = z_h[row];
            }
            return zr;
        };
        // output rows of chunk it: num / (row sum + phi(Q).z_prev), either staged
        // in the stage and stored by TMA, or each thread storing its own row;
        // then the P/O buffer is handed back
        const bool leader = tid == 32 * kWarpO;
        if (leader && args.out && C::OUT_TMA) prefetch_tmap(&tm_o);
        auto output_rows = [&](int it) {
            const int pb = it % C::NPB, kb = it / C::NPB;
            const int t = (c_begin + it) * kC + r;
            // the rows are staged in the stage's V tile (SPLITV) or its Q and K tiles
            uint8_t *stage_out = smem + (it % C::NS) * C::STAGE + (C::SPLITV ? 2 * C::TILE_QK : 0);
            bool ok = wait_bar_warp(&o_full[pb], kb & 1, abort);
            if (!C::ZMMA) ok = ok && wait_bar_warp(&dz_ready[it % C::NDZ], (it / C::NDZ) & 1, abort);
            if (tracer) LA_TRACE_AT(4, it, 3);
            if (ok) {
                tc_fence_after();
                uint32_t dv[16];
                tmem_ld16(tmem + lane_off + C::col_den(pb), dv);
                float den;
                if (C::ZMMA) {   // row sum + phi(Q).z_hi + phi(Q).z_lo
                    tmem_wait_ld();
                    den = __uint_as_float(dv[0]) + (__uint_as_float(dv[1]) + __uint_as_float(dv[2]));
                } else {
                    uint32_t zv[16];
                    tmem_ld16(tmem + lane_off + C::col_dz(it), zv);
                    tmem_wait_ld();
                    den = __uint_as_float(dv[0]) + __uint_as_float(zv[0]);
                }
                const float inv = VAR && args.no_den ? 1.f : 1.f / den;
                uint4 *dst = !C::OUT_TMA && args.out && t < Nseq &&
                                     LA_IN_BOUNDS((long long)bh * args.o_hs + (long long)t * args.o_rs + M <= args.out_elems,
                                                  args.err)
                                 ? reinterpret_cast<uint4 *>(args.out + (size_t)bh * args.o_hs + (size_t)t * args.o_rs)
                                 : nullptr;
                // rows of 256-bit stores when the output's base allows them (each
                // store of a warp writes one 32-byte sector of 32 rows)
                const bool v8 = (reinterpret_cast<uintptr_t>(args.out) & 31u) == 0;
#pragma unroll 1
                for (int c0 = 0; c0 < M; c0 += 32) {
                    float o[32];
                    tmem_ld32f(tmem + lane_off + C::col_o(pb) + c0, o);
                    if (args.out) {
                        uint4 w4[4];
#pragma unroll
                        for (int c8 = 0; c8 < 4; ++c8) {
                            const int c = c0 + 8 * c8;
                            uint4 w;
                            w.x = pack_bf16x2(o[8 * c8] * inv, o[8 * c8 + 1] * inv);
                            w.y = pack_bf16x2(o[8 * c8 + 2] * inv, o[8 * c8 + 3] * inv);
                            w.z = pack_bf16x2(o[8 * c8 + 4] * inv, o[8 * c8 + 5] * inv);
                            w.w = pack_bf16x2(o[8 * c8 + 6] * inv, o[8 * c8 + 7] * inv);
                            w4[c8] = w;
                            if (C::OUT_TMA)
                                *reinterpret_cast<uint4 *>(stage_out + (c / 64) * kC * 128 + sw128_offset(r, c % 64)) = w;
                            else if (dst && !v8)
                                dst[c / 8] = w;
                        }
                        if (!C::OUT_TMA && dst && v8) {
                            st_global_v8(dst + c0 / 8, w4[0], w4[1]);
                            st_global_v8(dst + c0 / 8 + 2, w4[2], w4[3]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&o_free[pb]);
            if (C::OUT_TMA) {
                fence_proxy_async();
                o_sync();
                if (leader) {
                    if (ok && args.out) {
#pragma unroll
                        for (int j = 0; j < M / 64; ++j)
                            tma_store_3d(&tm_o, stage_out + j * kC * 128, j * 64, (c_begin + it) * kC, bh);
                        tma_store_commit();
                    }
                    tma_store_wait_read0();
                    mbar_arrive(C::SPLITV ? &empty_v[it % C::NS] : &empty[it % C::NS]);
                }
            }
            if (tracer) LA_TRACE_AT(4, it, 4);
        };

        if (C::DS) {
            // The state lives here in fp32: thread (q4, lane) owns row d of it,
            // columns 32h..32h+31 (h = q4 / 2), and z_d when h = 0.  It reads the
            // same row of each increment from accumulator lane 32 q4 + lane.
            const int d = 32 * (q4 & 1) + lane, h = q4 >> 1;
            float sv[32];
            float zr = 0.f;
            load_state32(d, 32 * h, sv);
            if (h == 0) zr = load_z(d);
            store_snap32<D>(snap_buf(0), d, 32 * h, sv);
            if (h == 0) put_z(0, d, zr);
            fence_proxy_async();
            mbar_arrive(&snap_bar[0]);
            for (int it = 0; it < n; ++it) {
                if (tracer) LA_TRACE_AT(4, it, 0);
                const bool ok = wait_bar_warp(&ds_full[it & 1], (it >> 1) & 1, abort);
                if (tracer) LA_TRACE_AT(4, it, 1);
                if (ok) {
                    tc_fence_after();
                    float dsv[32];
                    tmem_ld32f(tmem + lane_off + C::col_ds(it) + 32 * h, dsv);
                    if (h == 0) {    // warp-uniform: z is column M of the increment
                        uint32_t zv[16];
                        tmem_ld16(tmem + lane_off + C::col_ds(it) + M, zv);
                        tmem_wait_ld();
                        zr += __uint_as_float(zv[0]);
                    }
#pragma unroll
                    for (int j = 0; j < 32; ++j) sv[j] += dsv[j];
                }
                tc_fence_before();
                mbar_arrive(&ds_free[it & 1]);
                if (it + 1 < n) {
                    // the buffer of snapshot it+1 was last read by the output MMAs
                    // of chunk it-1, which completed before output_rows(it-1) ran
                    store_snap32<D>(snap_buf(it + 1), d, 32 * h, sv);
                    if (h == 0) put_z(it + 1, d, zr);
                    fence_proxy_async();
                    mbar_arrive(&snap_bar[(it + 1) & 1]);
                }
                if (tracer) LA_TRACE_AT(4, it, 2);
                output_rows(it);
            }
            if (leader && C::OUT_TMA && args.out) tma_store_wait_all0();
            if (leader) LA_TRACE_AT(0, 63, 2);
            if (leader) LA_CTA_AT(7);
            // state after the last token (last segment only)
            if (S_h && seg == args.nseg - 1 && n > 0 && !*abort &&
                LA_IN_BOUNDS(((long long)bh * D + d) * M + 32 * h + 32 <= args.state_elems, args.err)) {
#pragma unroll
                for (int j = 0; j < 32; j += 4)
                    *reinterpret_cast<float4 *>(S_h + d * M + 32 * h + j) = make_float4(sv[j], sv[j + 1], sv[j + 2], sv[j + 3]);
                if (h == 0 && z_h) z_h[d] = zr;
            }
        } else {
            const bool srow = r < D;                 // owns a state row
            const bool swarp = 32 * q4 < D;          // warp-uniform
            // the state entering the segment into TMEM and snapshot 0
            if (swarp) {
                float zr = 0.f;
                if (srow) {
                    zr = load_z(r);
                    put_z(0, r, zr);
                }
#pragma unroll 1
                for (int c0 = 0; c0 < M; c0 += 32) {
                    float v[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] = 0.f;
                    if (srow) {
                        load_state32(r, c0, v);
                        store_snap32<D>(snap_buf(0), r, c0, v);
                    }
                    tmem_st32f(tmem + lane_off + C::COL_S + c0, v);
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
            mbar_arrive(&snap_bar[0]);

            for (int it = 0; it < n; ++it) {
                const int pb = it % C::NPB, kb = it / C::NPB;
                // ---- snapshot of the state after chunk it, for chunk it+1
                if (tracer) LA_TRACE_AT(4, it, 0);
                bool ok = wait_bar_warp(s_full, it & 1, abort);
                if (!C::DB) ok = ok && wait_bar_warp(&o_full[pb], kb & 1, abort);   // single snapshot: read by O(it)
                if (tracer) LA_TRACE_AT(4, it, 1);
                if (it + 1 < n) {
                    if (ok && swarp) {
                        tc_fence_after();
                        uint8_t *sb = snap_buf(it + 1);
#pragma unroll 1
                        for (int c0 = 0; c0 < M; c0 += 32) {
                            float v[32];
                            tmem_ld32f(tmem + lane_off + C::COL_S + c0, v);
                            if (srow) store_snap32<D>(sb, r, c0, v);
                        }
                        uint32_t zv[16];
                        tmem_ld16(tmem + lane_off + C::COL_Z, zv);
                        tmem_wait_ld();
                        if (srow) put_z(it + 1, r, __uint_as_float(zv[0]));
                    }
                    tc_fence_before();
                    fence_proxy_async();
                    mbar_arrive(&snap_bar[(it + 1) & 1]);
                }
                if (tracer) LA_TRACE_AT(4, it, 2);
                output_rows(it);
            }
            if (leader && C::OUT_TMA && args.out) tma_store_wait_all0();
            // ---- state after the last token (last segment only)
            if (S_h && seg == args.nseg - 1 && n > 0) {
                const bool ok = wait_bar_warp(s_full, (n - 1) & 1, abort);
                if (ok && swarp) {
                    tc_fence_after();
#pragma unroll 1
                    for (int c0 = 0; c0 < M; c0 += 32) {
                        float v[32];
                        tmem_ld32f(tmem + lane_off + C::COL_S + c0, v);
                        if (srow && LA_IN_BOUNDS(((long long)bh * D + r) * M + c0 + 32 <= args.state_elems, args.err))
#pragma unroll
                            for (int j = 0; j < 32; j += 4)
                                *reinterpret_cast<float4 *>(S_h + r * M + c0 + j) =
                                    make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
                    }
                    uint32_t zv[16];
                    tmem_ld16(tmem + lane_off + C::COL_Z, zv);
                    tmem_wait_ld();
                    if (srow && z_h) z_h[r] = __uint_as_float(zv[0]);
                }
            }
        }
    } else {
        // ------------------------------------------------------ feature-map group(s)
        // K rows past the sequence end are zeroed: they must add nothing
        const int grp = (warp - kWarpPhi) / 4;   // 0: Q (and K with one group), 1: K
        const int t = tid - 32 * (kWarpPhi + 4 * grp);
        for (int it = 0; it < n; ++it) {
            const int s = it % C::NS;
            if (t == 0) LA_TRACE_AT(3, it, 3 * grp);
            if (wait_bar(&full[s], (it / C::NS) & 1, abort)) {
                if (t == 0) LA_TRACE_AT(3, it, 3 * grp + 1);
                if (t == 0 && grp == 0 && it == 0) LA_CTA_AT(2);
                if (t == 0 && grp == 0 && it == n - 1) LA_CTA_AT(3);
                uint8_t *st = smem + s * C::STAGE;
                const int kz = min(kC, Nseq - (c_begin + it) * kC);
                if (!VAR || args.feat == kFeatPhi) {
                    if (grp == 0) phi_tile<D>(st, t, kC);
                    if (grp == C::NPHI - 1) phi_tile<D>(st + C::TILE_QK, t, kz);
                } else if constexpr (VAR) {   // a variant's feature map, one row per thread
                    if (grp == 0) feature_row<D>(st, t, kC, args.feat, args.dr, args.nu, args.sum_norm);
                    if (grp == C::NPHI - 1)
                        feature_row<D>(st + C::TILE_QK, t, kz, args.feat, args.dr, args.nu, args.sum_norm);
                }
                if (t == 0) LA_TRACE_AT(3, it, 3 * grp + 2);
            }
            fence_proxy_async();
            mbar_arrive(&phi_done[s]);
        }
    }
    // no MMA may still be running when the CTA frees its TMEM
    if (tid == 0) mbar_wait_bounded(drain, 0, now_ns() + kWaitNs, nullptr);
    if (tid == 0) LA_TRACE_AT(0, 63, 3);
    if (tid == 0) LA_CTA_AT(8);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, C::TMEM_COLS);
    if (tid == 0 && *abort) record_error(args.err, kErrTimeout);
}

// ------------------------------------------------- state reduction kernel
// For each (head, split): S = sum_j phi(K_j) V_j^T and z = sum_j phi(K_j)
// over the split's chunks, in fp32, into ws[bh][split] = (S row-major, z).
// The CTA of split 0 can also copy a carried-in state (or zeros) into slot
// init_slot, so that the causal kernel's segments read their starting state
// from the workspace only.  Two CTAs share an SM.

template <int D, int M>
struct RCfg {
    static constexpr int TILE_K = kC * D * 2;
    static constexpr int TILE_V = kC * M * 2;
    static constexpr int STAGE = TILE_K + TILE_V;
    static constexpr bool VONES = (M == 64);           // V read as [V | ones], z in column M
    static constexpr int ONES = VONES ? kC * 128 : kOnesBytes;
    static constexpr int BUDGET = (int)kSmemMax / 2 - 1024;   // two CTAs per SM
    static constexpr int NS_FIT = (BUDGET - ONES - 256) / STAGE;
    static constexpr int NS = NS_FIT > 4 ? 4 : (NS_FIT < 2 ? 2 : NS_FIT);
    static constexpr int OFF_ONES = NS * STAGE;
    static constexpr int OFF_BAR = OFF_ONES + ONES;
    static constexpr int NBARS = 3 * NS + 2;
    static constexpr int OFF_TSLOT = OFF_BAR + 8 * NBARS;
    static constexpr int SMEM = OFF_TSLOT + 16;
    static constexpr uint32_t TMEM_COLS = 256;
    static constexpr uint32_t COL_S = 0, COL_Z = M;
};

struct ReduceArgs {
    float *ws;               // [BH, nslot, D*M + D]
    const float *S_init;     // [BH, D, M] or null
    const float *z_init;     // [BH, D] or null
    int N;
    int nslot;               // slots per head in ws
    int nred;                // splits reduced per head (CTAs per head)
    int cps;                 // chunks per split
    int init_slot;           // -1: none
    int *err;
    long long ws_floats;     // extents the checked build tests writes against
    long long nheads;
    int inject_oob;          // checked build test hook: slot offset past the workspace
};

template <int D, int M>
__global__ void __launch_bounds__(kThreads, 2)
state_reduce_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                    const ReduceArgs args)
{
    using C = RCfg<D, M>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_TSLOT + 4);
    const int bh = blockIdx.x / args.nred, sp = blockIdx.x % args.nred;
    const int nch_total = (args.N + kC - 1) / kC;
    const int c_begin = sp * args.cps;
    const int n = max(0, min(nch_total, c_begin + args.cps) - c_begin);

    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full = bar, *empty = bar + C::NS, *phi_done = bar + 2 * C::NS;
    uint64_t *done = bar + 3 * C::NS, *init = done + 1;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::OFF_TSLOT);
    uint8_t *ones = smem + C::OFF_ONES;

    if (tid == 0) {
        *abort = (smem_u32(smem) & 1023u) ? 1 : 0;
        if (*abort) record_error(args.err, kErrTimeout);
        for (int s = 0; s < C::NS; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
            mbar_init(&phi_done[s], kGrp);
        }
        mbar_init(done, 1);
        mbar_init(init, kGrp);
        fence_mbar_init();
    }
    // ones operand (MN-major, ones in column 0)
    for (int i = tid; i < C::ONES / 4; i += kThreads) reinterpret_cast<uint32_t *>(ones)[i] = 0u;
    __syncthreads();
    for (int k = tid; k < C::ONES / 128; k += kThreads) *reinterpret_cast<uint16_t *>(ones + sw128_offset(k, 0)) = 0x3F80u;
    if (warp == 0) {
        tmem_alloc(tslot, C::TMEM_COLS);
        tmem_relinquish();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    pdl_wait_cta();   // set-up above touched no global memory

    if (warp == 0) {
        if (lane == 0 && !*abort) {
            prefetch_tmap(&tm_k);
            prefetch_tmap(&tm_v);
            int issued = 0;
            for (int it = 0; it < n; ++it) {
                const int s = it % C::NS, k = it / C::NS;
                if (it >= C::NS && !wait_bar(&empty[s], (k - 1) & 1, abort)) break;
                uint8_t *st = smem + s * C::STAGE;
                const int t0 = (c_begin + it) * kC;
                mbar_arrive_expect_tx(&full[s], C::STAGE);
#pragma unroll
                for (int j = 0; j < D / 64; ++j) tma_load_3d(st + j * kC * 128, &tm_k, &full[s], j * 64, t0, bh);
#pragma unroll
                for (int j = 0; j < M / 64; ++j)
                    tma_load_3d(st + C::TILE_K + j * kC * 128, &tm_v, &full[s], j * 64, t0, bh);
                ++issued;
            }
            if (*abort)
                for (int it = max(0, issued - C::NS); it < issued; ++it)
                    mbar_wait_bounded(&full[it % C::NS], (it / C::NS) & 1, now_ns() + kWaitNs, nullptr);
        }
    } else if (warp == 1) {
        if (lane == 0 && !*abort) {
            constexpr uint32_t ID_S = idesc_bf16(128, C::VONES ? M + 16 : M, 1, 1);
            constexpr uint32_t ID_Z = idesc_bf16(128, 16, 1, 1);
            const uint32_t ones_a = smem_u32(ones);
            bool ok = wait_bar(init, 0, abort);   // accumulators zeroed
            for (int it = 0; ok && it < n; ++it) {
                const int s = it % C::NS;
                if (!(ok = wait_bar(&phi_done[s], (it / C::NS) & 1, abort))) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(smem + s * C::STAGE), va = ka + C::TILE_K;
                const uint64_t dk = smem_desc(ka, kC * 128, 1024);
                const uint64_t dv = smem_desc(va, C::VONES ? ones_a - va : (uint32_t)(kC * 128), 1024);
                const uint64_t dones = ones_desc(ones_a);
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks) {
                    mma_f16_ss(tmem + C::COL_S, dk + mnmajor_step(ks), dv + mnmajor_step(ks), ID_S, 1);
                    if (!C::VONES) mma_f16_ss(tmem + C::COL_Z, dk + mnmajor_step(ks), dones, ID_Z, 1);
                }
                mma_commit(&empty[s]);
            }
            mma_commit(done);
            mbar_wait_bounded(done, 0, now_ns() + kWaitNs, nullptr);
        }
    } else if (warp < 6) {
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const bool swarp = 32 * q4 < D;
        if (swarp) {
            float zero[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) zero[j] = 0.f;
            for (int c0 = 0; c0 < M + 16; c0 += 32) tmem_st32f(tmem + lane_off + c0, zero);
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(init);
        long long base = ((long long)bh * args.nslot + sp) * (D * M + D);
#ifdef LA_CHECKED
        if (args.inject_oob) base += args.ws_floats;   // test hook: one workspace length past, caught below
#endif
        const bool dst_ok = LA_IN_BOUNDS(bh < args.nheads && base + (D * M + D) <= args.ws_floats, args.err);
        float *dst = args.ws + base;
        if (args.init_slot >= 0 && sp == 0 && r < D &&
            LA_IN_BOUNDS(((long long)bh * args.nslot + args.init_slot + 1) * (D * M + D) <= args.ws_floats, args.err)) {
            float *di = args.ws + ((size_t)bh * args.nslot + args.init_slot) * (D * M + D);
            const float *Si = args.S_init ? args.S_init + (size_t)bh * D * M : nullptr;
            for (int c = 0; c < M; c += 4)
                *reinterpret_cast<float4 *>(di + r * M + c) =
                    Si ? *reinterpret_cast<const float4 *>(Si + r * M + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            di[D * M + r] = args.z_init ? args.z_init[(size_t)bh * D + r] : 0.f;
        }
        const bool ok = wait_bar_warp(done, 0, abort);
        // S leaves through the stages (free once every MMA has completed) so
        // that its stores are coalesced
        float *stage = reinterpret_cast<float *>(smem);
        static_assert(D * M * 4 <= C::NS * C::STAGE, "staging area");
        if (ok && swarp) {
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < M; c0 += 32) {
                float v[32];
                tmem_ld32f(tmem + lane_off + C::COL_S + c0, v);
                if (r < D) stage_row32_f32<M>(stage, r, c0, v);
            }
            uint32_t zv[16];
            tmem_ld16(tmem + lane_off + C::COL_Z, zv);
            tmem_wait_ld();
            if (r < D && dst_ok) dst[D * M + r] = __uint_as_float(zv[0]);
        }
        epi_sync();
        if (ok && dst_ok) store_staged_f32<D, M>(dst, stage, r, kGrp);
    } else {
        const int t = tid - 64 - kGrp;
        for (int it = 0; it < n; ++it) {
            const int s = it % C::NS;
            if (wait_bar(&full[s], (it / C::NS) & 1, abort))
                phi_tile<D>(smem + s * C::STAGE, t, min(kC, args.N - (c_begin + it) * kC));
            fence_proxy_async();
            mbar_arrive(&phi_done[s]);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, C::TMEM_COLS);
    if (tid == 0 && *abort) record_error(args.err, kErrTimeout);
}

// ------------------------------------------------ fused non-causal kernel
// Non-causal attention, sec. 3.2 eq. (5), in one launch.  The CTAs of one
// head form a thread-block cluster; CTA g of the cluster owns rows
// [g * cps * C, (g + 1) * cps * C) of the head.
//   phase 1: S_g = sum phi(K_j) V_j^T, z_g = sum phi(K_j) over its rows (fp32,
//            TMEM), written to the workspace slot ws[bh][g];
//   exchange: cluster barrier (release/acquire), then every CTA sums the
//            cluster's G slots into a bf16 snapshot [S | z_hi z_lo];
//   phase 2: for its rows, V'_i = phi(Q_i)^T S / phi(Q_i)^T z by one MMA of
//            N = M + 16 per 128-row tile, divided, staged in the tile's slot
//            and stored by TMA.
// The producer streams the Q tiles of phase 2 into the ring as soon as the
// K, V tiles of phase 1 release it, so the exchange overlaps their loads and
// their feature map.  Warps: 0 producer, 1 MMA issuer, 2-5 epilogue group,
// 6-9 feature-map group.

template <int D, int M>
struct NCfg {
    static constexpr int TILE_K = kC * D * 2;
    static constexpr int TILE_V = kC * M * 2;
    // The ring is made of units of one tile each: a phase-1 item takes two
    // consecutive units (its K tile, then its V tile), a phase-2 item one (its
    // Q tile, then its output tile in place), so that twice as many Q tiles as
    // K/V pairs can be in flight while the partial sums are exchanged.
    static constexpr int UNIT = TILE_K > TILE_V ? TILE_K : TILE_V;
    static constexpr bool VONES = (M == 64);            // V read as [V | ones], z in column M
    static constexpr int ONES = VONES ? kC * 128 : kOnesBytes;
    static constexpr int SNAP = D * M * 2 + D * 128;    // M/64 state atoms then the z atom
    // the ones tile is dead once phase 1's MMAs are done: the snapshot may reuse it
    static constexpr bool SHARE = ONES >= SNAP;
    static constexpr int CTAS_PER_SM = (D == 64 && M == 64) ? 2 : 1;
    static constexpr int BUDGET = (int)kSmemMax / CTAS_PER_SM - 1024;
    // D = M = 64: the partial sums are exchanged through the cluster's shared
    // memory (clusters of 2, 4 or 8): RECV holds, for the D / G rows this CTA
    // owns, every CTA's fp32 partial rows and z entries
    static constexpr bool DSX = (D == 64 && M == 64);
    static constexpr int RECV = DSX ? D * (M + 1) * 4 : 0;
    static constexpr int FIXED = (SHARE ? ONES : ONES + SNAP) + RECV + 256;
    static constexpr int NU_FIT = (BUDGET - FIXED) / UNIT;
    static constexpr int NU = NU_FIT > 8 ? 8 : NU_FIT;
    static_assert(NU >= 4, "pipeline needs two phase-1 items in flight");
    static constexpr int OFF_ONES = NU * UNIT;
    static constexpr int OFF_SNAP = SHARE ? OFF_ONES : OFF_ONES + ONES;
    static constexpr int OFF_RECV = OFF_SNAP + (SHARE ? ONES : SNAP);
    static constexpr int NBARS = 3 * NU + 3 + 3 + 4 + 2;
    static constexpr int OFF_BAR = OFF_RECV + RECV;
    static constexpr int OFF_TSLOT = OFF_BAR + 8 * NBARS;
    static constexpr int SMEM = OFF_TSLOT + 16;
    static_assert(SMEM <= BUDGET + 1024, "shared memory budget");
    // TMEM: the phase-1 accumulator [S | z] at column 0, then (after it has
    // been read out) the phase-2 output buffers of NO columns each
    static constexpr uint32_t TMEM_COLS = CTAS_PER_SM == 2 ? 256 : 512;
    static constexpr uint32_t COL_S = 0, COL_Z = M;
    static constexpr int NO = M + 16;                   // numerator, z_hi, z_lo
    static constexpr int NOBUF = (int)TMEM_COLS / NO >= 3 ? 3 : (int)TMEM_COLS / NO;
    static __device__ __forceinline__ uint32_t col_o(int b) { return (uint32_t)(b * NO); }
};

struct NoncausalArgs {
    float *ws;               // [BH, G, D*M + D]
    int N;
    int G;                   // CTAs per head (cluster size)
    int cps;                 // chunks per CTA
    int *err;
    int feat, dr, nu, sum_norm, no_den;   // a variant's feature map and read-out (VAR only)
    long long ws_floats, nheads;          // extents the checked build tests accesses against
};

// VAR: a variant's feature map and read-out, as in causal_tc_kernel.
template <int D, int M, bool VAR>
__global__ void __launch_bounds__(kThreads, NCfg<D, M>::CTAS_PER_SM)
noncausal_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const NoncausalArgs args)
{
    using C = NCfg<D, M>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int *abort = reinterpret_cast<volatile int *>(smem + C::OFF_TSLOT + 4);
    LA_CTA_BEGIN();
    if (tid == 0) LA_CTA_AT(0);
    if (!VAR) pdl_launch_dependents();   // as in causal_tc_kernel (measured)
    const int bh = blockIdx.x / args.G, g = blockIdx.x % args.G;
    const int nch_total = (args.N + kC - 1) / kC;
    const int c_begin = g * args.cps;
    const int n = max(0, min(nch_total, c_begin + args.cps) - c_begin);
    const int total = 2 * n;                 // ring items: n K/V pairs, then n Q tiles

    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
    uint64_t *full = bar, *empty = bar + C::NU, *phi_done = bar + 2 * C::NU;
    uint64_t *o_full = bar + 3 * C::NU, *o_free = o_full + 3;
    // Units are used in one global sequence u = 0, 1, 2, ...: K/V pair i takes
    // units 2i and 2i + 1, Q tile i unit 2n + i.  Use u of a unit is its
    // (u / NU)-th use, so each of its barriers completes one phase per use.
    auto unit = [&](int u) { return smem + (u % C::NU) * C::UNIT; };
    auto ph = [&](int u) { return (uint32_t)((u / C::NU) & 1); };
    uint64_t *init = o_free + 3, *red_done = init + 1, *snap_bar = red_done + 1, *drain = snap_bar + 1;
    uint64_t *recv_bar = drain + 1, *snapx_bar = recv_bar + 1;   // exchange through shared memory
    // partial sums exchanged through the cluster's shared memory (else
    // through the workspace and L2)
    const bool dsx = C::DSX && (args.G == 2 || args.G == 4 || args.G == 8);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(smem + C::OFF_TSLOT);
    uint8_t *ones = smem + C::OFF_ONES;
    uint8_t *snap = smem + C::OFF_SNAP;

    if (tid == 0) {
        *abort = (smem_u32(smem) & 1023u) ? 1 : 0;
        if (*abort) record_error(args.err, kErrTimeout);
        for (int s = 0; s < C::NU; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);   // phase 1: MMA commit; phase 2: epilogue after the store read the tile
            mbar_init(&phi_done[s], kGrp);
        }
        for (int b = 0; b < 3; ++b) {
            mbar_init(&o_full[b], 1);
            mbar_init(&o_free[b], kGrp);
        }
        mbar_init(init, kGrp);
        mbar_init(red_done, 1);
        mbar_init(snap_bar, kGrp);
        mbar_init(drain, 1);
        mbar_init(recv_bar, 1);
        mbar_init(snapx_bar, 1);
        if (dsx) {
            // every CTA of the cluster (this one included) stores here, by
            // st.async, its fp32 partial rows r with r % G == rank (and their z),
            // then the owners of all D rows store the bf16 snapshot rows
            mbar_arrive_expect_tx(recv_bar, (uint32_t)C::RECV);
            mbar_arrive_expect_tx(snapx_bar, (uint32_t)(D * (M / 8 + 1) * 16));
        }
        fence_mbar_init();
    }
    for (int i = tid; i < C::ONES / 4; i += kThreads) reinterpret_cast<uint32_t *>(ones)[i] = 0u;
    __syncthreads();
    for (int k = tid; k < C::ONES / 128; k += kThreads) *reinterpret_cast<uint16_t *>(ones + sw128_offset(k, 0)) = 0x3F80u;
    if (warp == 0) {
        tmem_alloc(tslot, C::TMEM_COLS);
        tmem_relinquish();
    }
    fence_proxy_async();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (tid == 0) {   // kernel parameters, which no earlier launch writes: may overlap the wait
        // (measured 33.1 -> 32.7 us here; the causal kernel measured slower with it)
        prefetch_tmap(&tm_q);
        prefetch_tmap(&tm_k);
        prefetch_tmap(&tm_v);
        prefetch_tmap(&tm_o);
    }
    // the first two K, V chunks into L2 meanwhile, as in causal_tc_kernel
    // (measured 32.7 -> 32.0 us with one chunk, 31.6 with two)
    if (!VAR && tid == 0)
        for (int c = 0; c < 2 && c < n; ++c) {
            const int t0 = (c_begin + c) * kC;
#pragma unroll
            for (int j = 0; j < D / 64; ++j) tma_prefetch_3d(&tm_k, j * 64, t0, bh);
#pragma unroll
            for (int j = 0; j < M / 64; ++j) tma_prefetch_3d(&tm_v, j * 64, t0, bh);
        }
    pdl_wait_cta();   // set-up above touched no global memory
    if (tid == 0) LA_CTA_AT(1);
    const bool epi = warp >= 2 && warp < 6;
    // Cluster barrier.  Exchange through the workspace: one phase; every
    // thread arrives once, the epilogue group only after its partial sums are
    // in the workspace.  Through shared memory: phase A (every thread now:
    // the barriers above are initialised; the epilogue waits on it before its
    // first store into another CTA) and phase B at the end (no CTA exits while
    // another may still store into it).
    if (dsx || !epi) cluster_arrive_release();

    if (warp == 0) {
        // ------------------------------------------------------ producer
        if (lane == 0 && !*abort) {
            int u = 0;                   // next unit of the sequence
            for (int idx = 0; idx < total; ++idx) {
                const int nun = idx < n ? 2 : 1;
                bool ok = true;
                for (int j = 0; j < nun && ok; ++j)
                    if (u + j >= C::NU) ok = wait_bar(&empty[(u + j) % C::NU], ph(u + j) ^ 1u, abort);
                if (!ok) break;
                // DPFP rows arrive raw (at most 64 columns, one box)
                const int qk_boxes = VAR && args.feat == kFeatDpfp ? 1 : D / 64;
                uint64_t *f0 = &full[u % C::NU];
                if (idx < n) {
                    const int t0 = (c_begin + idx) * kC;
                    uint64_t *f1 = &full[(u + 1) % C::NU];
                    mbar_arrive_expect_tx(f0, qk_boxes * kC * 128);
                    for (int j = 0; j < qk_boxes; ++j) tma_load_3d(unit(u) + j * kC * 128, &tm_k, f0, j * 64, t0, bh);
                    mbar_arrive_expect_tx(f1, C::TILE_V);
#pragma unroll
                    for (int j = 0; j < M / 64; ++j) tma_load_3d(unit(u + 1) + j * kC * 128, &tm_v, f1, j * 64, t0, bh);
                } else {
                    const int t0 = (c_begin + idx - n) * kC;
                    mbar_arrive_expect_tx(f0, qk_boxes * kC * 128);
                    for (int j = 0; j < qk_boxes; ++j) tma_load_3d(unit(u) + j * kC * 128, &tm_q, f0, j * 64, t0, bh);
                }
                u += nun;
            }
            if (*abort)   // let the copies in flight land before the CTA exits
                for (int w = max(0, u - C::NU); w < u; ++w)
                    mbar_wait_bounded(&full[w % C::NU], ph(w), now_ns() + kWaitNs, nullptr);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------ MMA issuer
        if (lane == 0 && !*abort) {
            constexpr uint32_t ID_S = idesc_bf16(128, C::VONES ? M + 16 : M, 1, 1);
            constexpr uint32_t ID_Z = idesc_bf16(128, 16, 1, 1);
            constexpr uint32_t ID_O = idesc_bf16(128, C::NO, 0, 1);
            const uint32_t ones_a = smem_u32(ones);
            bool ok = wait_bar(init, 0, abort);   // accumulator zeroed
            // phase 1: [S | z] += phi(K)^T [V | 1]
            for (int it = 0; ok && it < n; ++it) {
                const int u = 2 * it;    // K unit; V in unit u + 1
                if (!(ok = wait_bar(&phi_done[u % C::NU], ph(u), abort))) break;
                if (!(ok = wait_bar(&full[(u + 1) % C::NU], ph(u + 1), abort))) break;
                tc_fence_after();
                const uint32_t ka = smem_u32(unit(u)), va = smem_u32(unit(u + 1));
                const uint64_t dk = smem_desc(ka, kC * 128, 1024);
                const uint64_t dv = smem_desc(va, C::VONES ? ones_a - va : (uint32_t)(kC * 128), 1024);
                const uint64_t dones = ones_desc(ones_a);
#pragma unroll
                for (int ks = 0; ks < kC / 16; ++ks) {
                    mma_f16_ss(tmem + C::COL_S, dk + mnmajor_step(ks), dv + mnmajor_step(ks), ID_S, 1);
                    if (!C::VONES) mma_f16_ss(tmem + C::COL_Z, dk + mnmajor_step(ks), dones, ID_Z, 1);
                }
                mma_commit(&empty[u % C::NU]);
                mma_commit(&empty[(u + 1) % C::NU]);
            }
            mma_commit(red_done);
            // phase 2: O = phi(Q) [S | z_hi z_lo]
            ok = ok && wait_bar(snap_bar, 0, abort);
            const uint32_t snap_a = smem_u32(snap);
            for (int i = 0; ok && i < n; ++i) {
                const int u = 2 * n + i, ob = i % C::NOBUF, kb = i / C::NOBUF;
                if (!(ok = wait_bar(&phi_done[u % C::NU], ph(u), abort))) break;
                if (kb > 0 && !(ok = wait_bar(&o_free[ob], (kb - 1) & 1, abort))) break;
                tc_fence_after();
                const uint64_t dq = kmajor_base(smem_u32(unit(u)));
                const uint64_t ds = smem_desc(snap_a, D * 128, 1024);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    mma_f16_ss(tmem + C::col_o(ob), dq + kmajor_step(ks), ds + mnmajor_step(ks), ID_O, ks > 0);
                mma_commit(&o_full[ob]);
            }
        }
        if (lane == 0) {
            mma_commit(drain);   // arrives once this thread's MMAs (if any) are done
            mbar_wait_bounded(drain, 0, now_ns() + kWaitNs, nullptr);
        }
    } else if (epi) {
        // ------------------------------------------------------ epilogue group
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const uint32_t lane_off = (uint32_t)(32 * q4) << 16;
        const bool swarp = 32 * q4 < D;
        const bool leader = tid == 64;
        constexpr int W = D * M + D;
        float *slot = args.ws + ((size_t)bh * args.G + g) * W;
        // the head's G slots lie inside the workspace (checked build)
        const bool ws_ok =
            dsx || LA_IN_BOUNDS(bh < args.nheads && ((long long)bh + 1) * args.G * W <= args.ws_floats, args.err);
        if (swarp) {
            float zero[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) zero[j] = 0.f;
            for (int c0 = 0; c0 < M + 16; c0 += 32) tmem_st32f(tmem + lane_off + c0, zero);
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(init);
        const bool ok1 = wait_bar_warp(red_done, 0, abort);
        if (leader) LA_CTA_AT(3);
        if (dsx) {
            // Exchange through shared memory.  Row r of the head's state is owned
            // by the CTA of rank r % G; every CTA stores its fp32 partial of row r
            // (and z_r) into the owner's RECV slot of its own rank, the owner sums
            // the G partials of its D / G rows, rounds them to the bf16 snapshot
            // [S | z_hi z_lo] and stores those snapshot rows into every CTA of the
            // cluster (itself included).  Each store counts its bytes on the
            // receiver's mbarrier.
            const uint32_t rank = cluster_ctarank();
            const int G = args.G, RPO = D / G;
            const uint32_t slot_bytes = (uint32_t)(C::RECV / G);
            const uint32_t recv_a = smem_u32(smem + C::OFF_RECV);
            const uint32_t snap_a = smem_u32(snap);
            cluster_wait_acquire();   // phase A: every CTA's barriers are initialised
            if (ok1 && swarp) {       // thread r holds row r of this CTA's partial
                tc_fence_after();
                const uint32_t owner = (uint32_t)(r % G), i = (uint32_t)(r / G);
                const uint32_t dst = mapa_shared(recv_a + rank * slot_bytes + i * (M * 4), owner);
                const uint32_t dbar = mapa_shared(smem_u32(recv_bar), owner);
#pragma unroll 1
                for (int c0 = 0; c0 < M; c0 += 32) {
                    float v[32];
                    tmem_ld32f(tmem + lane_off + C::COL_S + c0, v);
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        st_async_v4(dst + (uint32_t)(c0 + j) * 4u,
                                    make_uint4(__float_as_uint(v[j]), __float_as_uint(v[j + 1]),
                                               __float_as_uint(v[j + 2]), __float_as_uint(v[j + 3])),
                                    dbar);
                }
                uint32_t zv[16];
                tmem_ld16(tmem + lane_off + C::COL_Z, zv);
                tmem_wait_ld();
                st_async_b32(mapa_shared(recv_a + rank * slot_bytes + (uint32_t)(RPO * M * 4) + i * 4u, owner), zv[0],
                             dbar);
            }
            tc_fence_before();
            if (leader) LA_CTA_AT(4);
            const bool ok2 = ok1 && wait_bar_warp(recv_bar, 0, abort);
            if (leader) LA_CTA_AT(5);
            if (ok2) {
                const int tg = tid - 64;
                const uint8_t *rb = smem + C::OFF_RECV;
                // rows this CTA owns, 8 columns per item: the sum of the G slots
#pragma unroll 1
                for (int it = tg; it < RPO * (M / 8); it += kGrp) {
                    const int i = it / (M / 8), c8 = it % (M / 8);
                    const int row = i * G + (int)rank;
                    float a[8];
#pragma unroll
                    for (int j = 0; j < 8; ++j) a[j] = 0.f;
#pragma unroll 1
                    for (int sl = 0; sl < G; ++sl) {
                        const float4 *pp = reinterpret_cast<const float4 *>(rb + sl * slot_bytes + (i * M + c8 * 8) * 4);
                        const float4 x0 = pp[0], x1 = pp[1];
                        a[0] += x0.x; a[1] += x0.y; a[2] += x0.z; a[3] += x0.w;
                        a[4] += x1.x; a[5] += x1.y; a[6] += x1.z; a[7] += x1.w;
                    }
                    const uint4 w = make_uint4(pack_bf16x2(a[0], a[1]), pack_bf16x2(a[2], a[3]),
                                               pack_bf16x2(a[4], a[5]), pack_bf16x2(a[6], a[7]));
                    const uint32_t off = (uint32_t)((c8 / 8) * D * 128) + sw128_offset(row, (c8 % 8) * 8);
                    for (int t = 0; t < G; ++t)
                        st_async_v4(mapa_shared(snap_a + off, (uint32_t)t), w, mapa_shared(smem_u32(snapx_bar), (uint32_t)t));
                }
                // z of the owned rows as a bf16 pair (hi, lo) in columns 0 and 1
                // of the z atom; its other columns are the ones tile's zeros
                for (int i = tg; i < RPO; i += kGrp) {
                    const int row = i * G + (int)rank;
                    float zr = 0.f;
                    for (int sl = 0; sl < G; ++sl)
                        zr += *reinterpret_cast<const float *>(rb + sl * slot_bytes + RPO * M * 4 + i * 4);
                    const float hi = __bfloat162float(__float2bfloat16_rn(zr));
                    const uint4 w = make_uint4(pack_bf16x2(hi, zr - hi), 0u, 0u, 0u);
                    const uint32_t off = (uint32_t)((M / 64) * D * 128) + sw128_offset(row, 0);
                    for (int t = 0; t < G; ++t)
                        st_async_v4(mapa_shared(snap_a + off, (uint32_t)t), w, mapa_shared(smem_u32(snapx_bar), (uint32_t)t));
                }
            }
            // the snapshot is complete once every owner's rows have landed
            if (ok2) wait_bar_warp(snapx_bar, 0, abort);
        } else {
        // this CTA's partial sums into its workspace slot
        if (ok1 && swarp && ws_ok) {
            tc_fence_after();
#pragma unroll 1
            for (int c0 = 0; c0 < M; c0 += 32) {
                float v[32];
                tmem_ld32f(tmem + lane_off + C::COL_S + c0, v);
                if (r < D)
#pragma unroll
                    for (int j = 0; j < 32; j += 4)
                        *reinterpret_cast<float4 *>(slot + r * M + c0 + j) = make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
            }
            uint32_t zv[16];
            tmem_ld16(tmem + lane_off + C::COL_Z, zv);
            tmem_wait_ld();
            if (r < D) slot[D * M + r] = __uint_as_float(zv[0]);
        }
        tc_fence_before();
        // the slots are read only by this cluster's CTAs: the barrier's
        // cluster-scope release (and the readers' acquire) orders them
        if (leader) LA_CTA_AT(4);
        cluster_arrive_release();
        cluster_wait_acquire();
        if (leader) LA_CTA_AT(5);
        // the head's state: sum of the cluster's slots, as bf16 [S | z_hi z_lo].
        // All 128 threads take 16-column blocks (consecutive threads, consecutive
        // blocks of a row) and load up to four slots' blocks before adding, so
        // that the reads overlap instead of paying one L2 round trip each.
        if (!*abort && ws_ok) {
            const float *src = args.ws + (size_t)bh * args.G * W;
            const int tg = tid - 64;
            // z's slot entries first, so that their loads share the first
            // round trip with the state blocks'
            float zr = 0.f;
            if (r < D)
                for (int j = 0; j < args.G; ++j) zr += __ldcg(src + (size_t)j * W + D * M + r);
            constexpr int BPR = M / 16;                  // 16-column blocks per row
#pragma unroll 1
            for (int b = tg; b < D * BPR; b += kGrp) {
                const int row = b / BPR, c0 = (b % BPR) * 16;
                float v[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = 0.f;
#pragma unroll 1
                for (int j0 = 0; j0 < args.G; j0 += 4) {
                    float4 x[4][4];
#pragma unroll
                    for (int a4 = 0; a4 < 4; ++a4) {
                        const int js = min(j0 + a4, args.G - 1);   // in range; zeroed below if past G
                        const float4 *p = reinterpret_cast<const float4 *>(src + (size_t)js * W + row * M + c0);
#pragma unroll
                        for (int q = 0; q < 4; ++q) x[a4][q] = __ldcg(p + q);   // L2: written by other CTAs
                        if (j0 + a4 >= args.G)
#pragma unroll
                            for (int q = 0; q < 4; ++q) x[a4][q] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
#pragma unroll
                    for (int a4 = 0; a4 < 4; ++a4)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            v[4 * q] += x[a4][q].x; v[4 * q + 1] += x[a4][q].y;
                            v[4 * q + 2] += x[a4][q].z; v[4 * q + 3] += x[a4][q].w;
                        }
                }
#pragma unroll
                for (int c8 = 0; c8 < 2; ++c8) {
                    const int c = c0 + 8 * c8;
                    uint4 w;
                    w.x = pack_bf16x2(v[8 * c8], v[8 * c8 + 1]);
                    w.y = pack_bf16x2(v[8 * c8 + 2], v[8 * c8 + 3]);
                    w.z = pack_bf16x2(v[8 * c8 + 4], v[8 * c8 + 5]);
                    w.w = pack_bf16x2(v[8 * c8 + 6], v[8 * c8 + 7]);
                    *reinterpret_cast<uint4 *>(snap + (c / 64) * D * 128 + sw128_offset(row, c % 64)) = w;
                }
            }
            if (r < D) {
                uint8_t *za = snap + (M / 64) * D * 128;
                for (int c = 0; c < 64; c += 8)
                    *reinterpret_cast<uint4 *>(za + sw128_offset(r, c)) = make_uint4(0u, 0u, 0u, 0u);
                const __nv_bfloat16 hi = __float2bfloat16_rn(zr);
                const __nv_bfloat16 lo = __float2bfloat16_rn(zr - __bfloat162float(hi));
                *reinterpret_cast<__nv_bfloat16 *>(za + sw128_offset(r, 0)) = hi;
                *reinterpret_cast<__nv_bfloat16 *>(za + sw128_offset(r, 1)) = lo;
            }
        }
        }   // exchange through the workspace
        fence_proxy_async();
        mbar_arrive(snap_bar);
        if (leader) LA_CTA_AT(6);
        if (leader) prefetch_tmap(&tm_o);
        // the leader hands a unit back once its output store has read it,
        // checked one tile later so that the store overlaps the next tile
        int pend = -1;
        for (int i = 0; i < n; ++i) {
            const int u = 2 * n + i, ob = i % C::NOBUF, kb = i / C::NOBUF;
            const int t0 = (c_begin + i) * kC;
            uint8_t *tile = unit(u);   // phi(Q) is dead once o_full fires
            const bool ok = wait_bar_warp(&o_full[ob], kb & 1, abort);
            if (ok) {
                tc_fence_after();
                uint32_t dv[16];
                tmem_ld16(tmem + lane_off + C::col_o(ob) + M, dv);
                tmem_wait_ld();
                const float inv = VAR && args.no_den ? 1.f : 1.f / (__uint_as_float(dv[0]) + __uint_as_float(dv[1]));
#pragma unroll 1
                for (int c0 = 0; c0 < M; c0 += 32) {
                    float o[32];
                    tmem_ld32f(tmem + lane_off + C::col_o(ob) + c0, o);
#pragma unroll
                    for (int c8 = 0; c8 < 4; ++c8) {
                        const int c = c0 + 8 * c8;
                        uint4 w;
                        w.x = pack_bf16x2(o[8 * c8] * inv, o[8 * c8 + 1] * inv);
                        w.y = pack_bf16x2(o[8 * c8 + 2] * inv, o[8 * c8 + 3] * inv);
                        w.z = pack_bf16x2(o[8 * c8 + 4] * inv, o[8 * c8 + 5] * inv);
                        w.w = pack_bf16x2(o[8 * c8 + 6] * inv, o[8 * c8 + 7] * inv);
                        *reinterpret_cast<uint4 *>(tile + (c / 64) * kC * 128 + sw128_offset(r, c % 64)) = w;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&o_free[ob]);
            fence_proxy_async();
            epi_sync();
            if (leader) {
                if (ok) {
#pragma unroll
                    for (int j = 0; j < M / 64; ++j) tma_store_3d(&tm_o, tile + j * kC * 128, j * 64, t0, bh);
                    tma_store_commit();
                    tma_store_wait_read1();   // every store but this one has read its tile
                } else {
                    tma_store_wait_read0();
                }
                if (pend >= 0) mbar_arrive(&empty[pend % C::NU]);
                pend = u;
            }
        }
        if (leader) {
            tma_store_wait_read0();
            if (pend >= 0) mbar_arrive(&empty[pend % C::NU]);
            tma_store_wait_all0();
        }
        if (leader) LA_CTA_AT(7);
    } else {
        // ------------------------------------------------------ feature-map group
        // phase 1 K tiles (rows past the sequence end zeroed: they must add
        // nothing), then phase 2 Q tiles
        const int t = tid - 64 - kGrp;
        int u = 0;
        for (int idx = 0; idx < total; ++idx) {
            // the K or Q tile is in unit u; a K/V pair's V unit (u + 1) is the
            // MMA issuer's to wait for, but its phi_done still completes one
            // phase per use
            if (wait_bar(&full[u % C::NU], ph(u), abort)) {
                if (t == 0 && idx == 0) LA_CTA_AT(2);
                const int zf = idx < n ? min(kC, args.N - (c_begin + idx) * kC) : kC;
                if (!VAR || args.feat == kFeatPhi) phi_tile<D, true>(unit(u), t, zf);
                else if constexpr (VAR)   // a variant's feature map, one row per thread
                    feature_row<D>(unit(u), t, zf, args.feat, args.dr, args.nu, args.sum_norm);
            }
            fence_proxy_async();
            // the V unit's arrival first: once the MMA issuer has seen every
            // thread's arrival on the K unit, none is still to arrive on the V
            // unit for this use (a late arrival would land in its next phase)
            if (idx < n) mbar_arrive(&phi_done[(u + 1) % C::NU]);
            mbar_arrive(&phi_done[u % C::NU]);
            u += idx < n ? 2 : 1;
        }
    }
    if (!epi) cluster_wait_acquire();
    if (dsx) {
        // phase B: every CTA has finished storing into the others
        cluster_arrive_release();
        cluster_wait_acquire();
        if (*abort && tid == 0) {   // stores into this CTA that are still in flight land first
            mbar_wait_bounded(recv_bar, 0, now_ns() + 1000000ull, nullptr);
            mbar_wait_bounded(snapx_bar, 0, now_ns() + 1000000ull, nullptr);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid == 0) LA_CTA_AT(8);
    if (warp == 0) tmem_dealloc(tmem, C::TMEM_COLS);
    if (tid == 0 && *abort) record_error(args.err, kErrTimeout);
}

// ---------------------------------------------------------------- launchers

// Segments per head for the causal kernel: enough CTAs to cover the SMs
// (one CTA per SM), at least 8 chunks per segment.
int causal_nseg(long long BH, int N, int sm_count) {
    const long long nch = (N + kC - 1) / kC;
    if (BH >= (long long)sm_count * 3 / 4) return 1;
    long long nseg = std::max(1LL, (long long)sm_count / BH);
    nseg = std::min(nseg, std::max(1LL, nch / 8));
    return (int)nseg;
}

// Tensor map of a [BH][N][cols] tensor, or of a step-major [N][BH][cols] one
// read in the same [BH][N][cols] order.
bool causal_tmap(CUtensorMap *m, const Problem &p, const void *base, int cols) {
    if (!p.step_major) return cached_tmap_bf16_3d(m, base, cols, p.N, p.BH, 64, kC);
    return make_tmap_bf16_3d_strided(m, base, cols, p.N, p.BH, (uint64_t)p.BH * cols * 2, (uint64_t)cols * 2, 64, kC);
}

template <int D, int M>
cudaError_t launch_causal(const Problem &p, const DeviceInfo &dev) {
    using C = Cfg<D, M>;
    CUtensorMap tq, tk, tv;
    // Q, K of a variant with a row feature map arrive raw (dr columns)
    const int qk_cols = p.feat != kFeatPhi ? p.dr : D;
    if (!causal_tmap(&tq, p, p.q, qk_cols) || !causal_tmap(&tk, p, p.k, qk_cols) || !causal_tmap(&tv, p, p.v, M))
        return cudaErrorInvalidValue;
    const int nch = (p.N + kC - 1) / kC;
    // per-sequence lengths, step-major decode inputs or a variant (the
    // segment-sum pre-pass applies elu + 1 and variant calls pass no
    // workspace): no segments
    int nseg = (p.lens || p.step_major || p.feat != kFeatPhi || p.no_den || p.no_segments)
                   ? 1
                   : causal_nseg(p.BH, p.N, dev.sm_count);
    const int cps = (nch + nseg - 1) / nseg;
    nseg = (nch + cps - 1) / cps;
    cudaError_t e;
    if (nseg > 1) {
        if (p.ws_bytes < (size_t)p.BH * nseg * (D * M + D) * sizeof(float)) return cudaErrorInvalidValue;
        ReduceArgs r{(float *)p.ws, p.S, p.z, p.N, nseg, nseg - 1, cps, nseg - 1, dev.err_word,
                     (long long)(p.ws_bytes / sizeof(float)), p.BH, g_inject_bounds};
        if ((e = set_smem(state_reduce_kernel<D, M>, RCfg<D, M>::SMEM)) != cudaSuccess) return e;
        e = launch_pdl(state_reduce_kernel<D, M>, dim3((unsigned)(p.BH * (nseg - 1))), dim3(kThreads),
                       RCfg<D, M>::SMEM, p.stream, 0u, tk, tv, r);
        count_launches(1);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap to;
    if (p.out && !causal_tmap(&to, p, p.out, M)) return cudaErrorInvalidValue;
    if (!p.out) to = tq;   // never used
    CausalArgs a;
    a.out = reinterpret_cast<__nv_bfloat16 *>(p.out);
    a.S = p.S;
    a.z = p.z;
    a.seg_ws = nseg > 1 ? (const float *)p.ws : nullptr;
    a.N = p.N;
    a.nseg = nseg;
    a.cps = cps;
    a.err = dev.err_word;
    a.inject_ns = g_inject_timeout ? (uint64_t)g_inject_limit_us * 1000ull : 0ull;
    a.lens = p.lens;
    a.H = p.H > 0 ? p.H : 1;
    a.o_rs = p.step_major ? p.BH * (long long)M : (long long)M;
    a.o_hs = p.step_major ? (long long)M : (long long)p.N * M;
    a.feat = p.feat;
    a.dr = p.dr;
    a.nu = p.nu;
    a.sum_norm = p.sum_norm ? 1 : 0;
    a.no_den = p.no_den ? 1 : 0;
    a.nheads = p.BH;
    a.state_elems = p.S ? p.BH * D * M : 0;
    a.ws_floats = nseg > 1 ? (long long)(p.ws_bytes / sizeof(float)) : 0;
    a.out_elems = p.out ? p.BH * (long long)p.N * M : 0;
    a.inject_oob = g_inject_bounds;
    const dim3 grid((unsigned)(p.BH * nseg)), block(C::THREADS);
    if (p.feat != kFeatPhi || p.no_den) {
        if ((e = set_smem(causal_tc_kernel<D, M, true>, C::SMEM)) != cudaSuccess) return e;
        e = launch_pdl(causal_tc_kernel<D, M, true>, grid, block, C::SMEM, p.stream, 0u, tq, tk, tv, to, a);
    } else {
        if ((e = set_smem(causal_tc_kernel<D, M, false>, C::SMEM)) != cudaSuccess) return e;
        e = launch_pdl(causal_tc_kernel<D, M, false>, grid, block, C::SMEM, p.stream, 0u, tq, tk, tv, to, a);
    }
    count_launches(1);
    return e;
}

// CTAs per head of the fused non-causal kernel (the cluster size, at most 8)
// and chunks per CTA, sized so that the grid covers the CTA slots once.
void nc_grid(long long BH, int N, int slots, int &G, int &cps) {
    const int nch = (N + kC - 1) / kC;
    const int want = (int)std::max(1LL, (long long)slots / std::max(1LL, BH));
    G = std::max(1, std::min(std::min(want, 8), nch));
    cps = (nch + G - 1) / G;
    G = (nch + cps - 1) / cps;
}

template <int D, int M, bool VAR>
cudaError_t launch_noncausal_v(const Problem &p, const DeviceInfo &dev) {
    using C = NCfg<D, M>;
    CUtensorMap tq, tk, tv, to;
    const int qk_cols = p.feat != kFeatPhi ? p.dr : D;   // raw rows of a variant's feature map
    if (!cached_tmap_bf16_3d(&tq, p.q, qk_cols, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tk, p.k, qk_cols, p.N, p.BH, 64, kC) ||
        !cached_tmap_bf16_3d(&tv, p.v, M, p.N, p.BH, 64, kC) || !cached_tmap_bf16_3d(&to, p.out, M, p.N, p.BH, 64, kC))
        return cudaErrorInvalidValue;
    int G, cps;
    nc_grid(p.BH, p.N, C::CTAS_PER_SM * dev.sm_count, G, cps);
    if (p.ws_bytes < (size_t)p.BH * G * (D * M + D) * sizeof(float)) return cudaErrorInvalidValue;
    cudaError_t e;
    if ((e = set_smem(noncausal_tc_kernel<D, M, VAR>, C::SMEM)) != cudaSuccess) return e;
    const NoncausalArgs a{(float *)p.ws, p.N, G, cps, dev.err_word, p.feat, p.dr, p.nu, p.sum_norm ? 1 : 0,
                          p.no_den ? 1 : 0, (long long)(p.ws_bytes / sizeof(float)), p.BH};
    e = launch_pdl(noncausal_tc_kernel<D, M, VAR>, dim3((unsigned)(p.BH * G)), dim3(kThreads), C::SMEM, p.stream,
                   (unsigned)G, tq, tk, tv, to, a);
    count_launches(1);
    return e;
}

template <int D, int M>
cudaError_t launch_noncausal(const Problem &p, const DeviceInfo &dev) {
    return (p.feat != kFeatPhi || p.no_den) ? launch_noncausal_v<D, M, true>(p, dev)
                                            : launch_noncausal_v<D, M, false>(p, dev);
}

bool tc_dims(const la_shape &s) {
    return s.dtype == LA_DTYPE_BF16 && (s.D == 64 || s.D == 128) && (s.M == 64 || s.M == 128);
}

}  // namespace

// The chunk length is a hint (la.h): every accepted value (0, 64, 128) takes
// the 128-row regrouping here, one tcgen05 M = 128 tile per chunk.
bool tc_causal_supported(const la_shape &s, int) { return tc_dims(s); }

bool tc_variant_route(const la_shape &s, const la_variant &v, Problem &p) {
    // sum update, bf16, feature width 64 or 128; with the denominator elu + 1
    // only (it is then the plain form, run without segments: the variant
    // calls have no workspace)
    if (s.dtype != LA_DTYPE_BF16 || v.update != LA_UPDATE_SUM) return false;
    if (s.M != 64 && s.M != 128) return false;
    const int F = fw_feature_dim(v, s.D);
    if (F != 64 && F != 128) return false;
    if (v.feature_map == LA_FM_ELU1) {
        p.feat = v.norm == LA_NORM_SUM ? kFeatElu1Sum : kFeatPhi;
    } else if (v.feature_map == LA_FM_DPFP) {
        // the raw widths and shifts feature_row instantiates
        const bool ok = F == 128 ? ((s.D == 64 && v.nu == 1) || (s.D == 32 && v.nu == 2) || (s.D == 16 && v.nu == 4))
                                 : ((s.D == 32 && v.nu == 1) || (s.D == 16 && v.nu == 2));
        if (!ok) return false;
        p.feat = kFeatDpfp;
        p.sum_norm = v.norm == LA_NORM_SUM;
    } else {
        return false;
    }
    p.dr = s.D;
    p.nu = v.nu;
    p.no_den = v.norm != LA_NORM_DEN;
    p.no_segments = true;   // a variant call passes no workspace
    p.D = F;
    return true;
}

size_t tc_causal_ws_bytes(const la_shape &s, int) {
    // Sized for the most segments any device picks (one CTA per SM, up to
    // 192 SMs assumed; never more than one segment per 8 chunks).
    const long long BH = (long long)s.B * s.H;
    if (BH <= 0 || s.N <= 0) return 0;
    const long long nch = (s.N + kC - 1) / kC;
    const long long nseg = std::min(std::max(1LL, 192LL / BH), std::max(1LL, nch / 8));
    if (nseg <= 1) return 0;
    return (size_t)BH * nseg * ((size_t)s.D * s.M + s.D) * sizeof(float);
}

// Partial sums sum phi(K_j) [V_j | 1] of `nsplit` consecutive key ranges of
// cps chunks per head, into ws[bh][split] = [S (D x M) | z (D)] fp32: the
// segment-sum pre-pass run over every split (no carried-in slot).
template <int D, int M>
cudaError_t launch_key_sums(const void *k, const void *v, long long BH, int N, int nsplit, int cps, float *ws,
                            size_t ws_bytes, cudaStream_t stream, const DeviceInfo &dev) {
    CUtensorMap tk, tv;
    if (!cached_tmap_bf16_3d(&tk, k, D, N, BH, 64, kC) || !cached_tmap_bf16_3d(&tv, v, M, N, BH, 64, kC))
        return cudaErrorInvalidValue;
    if (ws_bytes < (size_t)BH * nsplit * (D * M + D) * sizeof(float)) return cudaErrorInvalidValue;
    ReduceArgs r{ws, nullptr, nullptr, N, nsplit, nsplit, cps, -1, dev.err_word,
                 (long long)(ws_bytes / sizeof(float)), BH, g_inject_bounds};
    cudaError_t e = set_smem(state_reduce_kernel<D, M>, RCfg<D, M>::SMEM);
    if (e != cudaSuccess) return e;
    e = launch_pdl(state_reduce_kernel<D, M>, dim3((unsigned)(BH * nsplit)), dim3(kThreads), RCfg<D, M>::SMEM, stream,
                   0u, tk, tv, r);
    count_launches(1);
    return e;
}

cudaError_t tc_key_sums(const void *k, const void *v, long long BH, int N, int D, int M, int nsplit, int cps,
                        float *ws, size_t ws_bytes, cudaStream_t stream, const DeviceInfo &dev) {
    if (D == 64 && M == 64) return launch_key_sums<64, 64>(k, v, BH, N, nsplit, cps, ws, ws_bytes, stream, dev);
    if (D == 64 && M == 128) return launch_key_sums<64, 128>(k, v, BH, N, nsplit, cps, ws, ws_bytes, stream, dev);
    if (D == 128 && M == 64) return launch_key_sums<128, 64>(k, v, BH, N, nsplit, cps, ws, ws_bytes, stream, dev);
    if (D == 128 && M == 128) return launch_key_sums<128, 128>(k, v, BH, N, nsplit, cps, ws, ws_bytes, stream, dev);
    return cudaErrorInvalidValue;
}

cudaError_t tc_causal(const Problem &p, const DeviceInfo &dev) {
    if (p.D == 64 && p.M == 64) return launch_causal<64, 64>(p, dev);
    if (p.D == 64 && p.M == 128) return launch_causal<64, 128>(p, dev);
    if (p.D == 128 && p.M == 64) return launch_causal<128, 64>(p, dev);
    if (p.D == 128 && p.M == 128) return launch_causal<128, 128>(p, dev);
    return cudaErrorInvalidValue;
}

bool tc_noncausal_supported(const la_shape &s) { return tc_dims(s); }

size_t tc_noncausal_ws_bytes(const la_shape &s) {
    // the cluster size nc_grid picks on any device (up to 192 SMs, two CTAs each)
    const long long BH = (long long)s.B * s.H;
    if (BH <= 0 || s.N <= 0) return 0;
    const long long nch = (s.N + kC - 1) / kC;
    const long long G = std::min(std::min(std::max(1LL, 2 * 192LL / BH), 8LL), nch);
    return (size_t)BH * G * ((size_t)s.D * s.M + s.D) * sizeof(float);
}

cudaError_t tc_noncausal(const Problem &p, const DeviceInfo &dev) {
    if (p.D == 64 && p.M == 64) return launch_noncausal<64, 64>(p, dev);
    if (p.D == 64 && p.M == 128) return launch_noncausal<64, 128>(p, dev);
    if (p.D == 128 && p.M == 64) return launch_noncausal<128, 64>(p, dev);
    if (p.D == 128 && p.M == 128) return launch_noncausal<128, 128>(p, dev);
    return cudaErrorInvalidValue;
}

}  // namespace la

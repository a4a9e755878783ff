// tc_kernels.cuh - device helpers and constants shared by the tensor-core
// kernels of liblinattn.so (tcgen05 MMA, TMEM, TMA on 128-byte swizzled
// tiles), and the host helper that opts a kernel in to large shared memory.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include <mutex>
#include <utility>
#include <vector>

#include "la_common.cuh"
#include "tc_ptx.cuh"

namespace la {
namespace {

using namespace tc;

constexpr int kC = 128;                          // chunk rows (MMA M)
constexpr int kGrp = 128;                        // threads of one warpgroup
constexpr int kThreads = 64 + 2 * kGrp;          // producer, MMA, epilogue group, phi group
constexpr uint64_t kWaitNs = 2000000000ull;      // 2 s per wait
constexpr uint32_t kSmemMax = 232448;            // 227 KB opt-in per CTA
constexpr int kOnesBytes = 1024;                 // one 8-row swizzle atom of a ones operand

// ---------------------------------------------------------------- helpers

__device__ __forceinline__ uint64_t now_ns() { return globaltimer_ns(); }

// Bounded wait that also gives up as soon as another role has aborted.  A
// wait that gives up raises the CTA's abort flag, so that every role winds
// down; the kernel records LA_ERR_TIMEOUT at its exit.
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort) {
    if (*abort) return false;
    if (mbar_try_wait(bar, parity)) return true;
    if (mbar_wait_bounded(bar, parity, now_ns() + kWaitNs, abort)) return true;
    *abort = 1;
    return false;
}

// Warp-uniform variant: the whole warp proceeds only if every lane's wait succeeded.
__device__ __forceinline__ bool wait_bar_warp(uint64_t *bar, uint32_t parity, volatile int *abort) {
    return __all_sync(0xffffffffu, wait_bar(bar, parity, abort));
}

__device__ __forceinline__ void set_abort(volatile int *abort, int *err) {
    *abort = 1;
    record_error(err, kErrTimeout);
}

// Named barrier for the 128 threads of the epilogue group.
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// phi(x) = elu(x) + 1 (x + 1 for x > 0, e^x otherwise) of two packed bf16
// values.  The exponentials in fp32: each value
// widened (exact), e = 2^(x log2 e) by the MUFU's fp32 exponential, and the
// pair rounded to bf16 once; the rest on the packed pair: max(x, 0) +
// min(e, 1), which is x + 1 rounded once for x > 0 and the rounded e itself
// for x <= 0.  Every feature value is therefore the correctly rounded bf16 of
// phi, up to the exponential's 2^-22.  NaN propagates.
__device__ __forceinline__ uint32_t phi_bf16x2(uint32_t w) {
    float ea, eb;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ea) : "f"(__uint_as_float(w << 16) * 1.4426950408889634f));
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(eb) : "f"(__uint_as_float(w & 0xFFFF0000u) * 1.4426950408889634f));
    const uint32_t e = pack_bf16x2(ea, eb);
    uint32_t m, n, r;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(m) : "r"(w), "r"(0u));
    asm("min.NaN.bf16x2 %0, %1, %2;" : "=r"(n) : "r"(e), "r"(0x3F803F80u));
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(m), "r"(n));
    return r;
}

// Applies phi in place to a C x DD tile (sub-tiles of 64 columns, each C rows
// x 128 bytes); rows >= zero_from are written as zeros.  Each thread handles
// four 16-byte chunks at a time (loads, then 16 independent phi pairs, then
// stores) so that enough exponentials are in flight (eight at a time measured
// slower in the causal kernels: 39.2 -> 41.3 us at D = 64, 310 -> 342 us at
// D = 128).
template <int DD, bool PIPE = false>
__device__ __forceinline__ void phi_tile(uint8_t *tile, int t, int zero_from) {
    constexpr int CHUNKS = kC * DD * 2 / 16;
    constexpr int U = 4;
    constexpr int NIT = CHUNKS / (U * kGrp);
    static_assert(CHUNKS % (U * kGrp) == 0, "whole rounds of four chunks per thread");
    auto store_round = [&](int u0, uint4 (&v)[U]) {
#pragma unroll
        for (int i = 0; i < U; ++i) {
            v[i].x = phi_bf16x2(v[i].x);
            v[i].y = phi_bf16x2(v[i].y);
            v[i].z = phi_bf16x2(v[i].z);
            v[i].w = phi_bf16x2(v[i].w);
        }
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const uint32_t off = (uint32_t)(u0 + i * kGrp) * 16u;
            const int row = (int)((off % (kC * 128u)) >> 7);
            *reinterpret_cast<uint4 *>(tile + off) = row >= zero_from ? make_uint4(0u, 0u, 0u, 0u) : v[i];
        }
    };
    if constexpr (!PIPE) {
#pragma unroll 1
        for (int u0 = t; u0 < CHUNKS; u0 += U * kGrp) {
            uint4 v[U];
#pragma unroll
            for (int i = 0; i < U; ++i) v[i] = *reinterpret_cast<const uint4 *>(tile + (u0 + i * kGrp) * 16);
            store_round(u0, v);
        }
    } else {
        // software pipelined (unrolled): the next round's loads are issued
        // before this round's arithmetic.  Measured: non-causal kernel 28.95 ->
        // 28.55 us; in the causal kernels the same order was slower (37.7 ->
        // 48.7 us at D = M = 64; rolled, 37.7 -> 38.1), so they keep PIPE = 0.
        uint4 v[U], nx[U];
#pragma unroll
        for (int i = 0; i < U; ++i) v[i] = *reinterpret_cast<const uint4 *>(tile + (t + i * kGrp) * 16);
#pragma unroll
        for (int it = 0; it < NIT; ++it) {
            const int u0 = t + it * U * kGrp;
            if (it + 1 < NIT)
#pragma unroll
                for (int i = 0; i < U; ++i) nx[i] = *reinterpret_cast<const uint4 *>(tile + (u0 + (U + i) * kGrp) * 16);
            store_round(u0, v);
            if (it + 1 < NIT)
#pragma unroll
                for (int i = 0; i < U; ++i) v[i] = nx[i];
        }
    }
}

// ------------------------------------------------- feature maps of the variants
// Feature maps computed row by row in place: thread t owns row t of a C x F
// tile (F/64 sub-tiles of C rows x 128 bytes, 128-byte swizzle).  The raw row
// (DR columns) sits in the first DR columns of the tile as TMA left it; the
// features overwrite the whole row, rounded once to bf16.  Rows >= zero_from
// are written as zeros (keys past the end of a sequence).
//   kFeatElu1Sum: elu(x) + 1, divided by its component sum (DR = F).
//   kFeatDpfp:    DPFP-NU ("Linear Transformers Are Secretly Fast Weight
//                 Programmers"): r = [relu(x), relu(-x)], feature
//                 (s-1)*2DR + i = r_i r_{(i+s) mod 2DR}, F = 2 DR NU; divided by
//                 the component sum if SUM.
constexpr int kFeatPhi = 0, kFeatElu1Sum = 1, kFeatDpfp = 2;

template <int DR>
__device__ __forceinline__ void load_raw_row(const uint8_t *tile, int r, uint32_t (&w)[DR / 2]) {
#pragma unroll
    for (int c8 = 0; c8 < DR / 8; ++c8) {
        const uint4 v = *reinterpret_cast<const uint4 *>(tile + (c8 / 8) * kC * 128 + sw128_offset(r, (c8 % 8) * 8));
        w[4 * c8] = v.x;
        w[4 * c8 + 1] = v.y;
        w[4 * c8 + 2] = v.z;
        w[4 * c8 + 3] = v.w;
    }
}

// Packed bf16x2 helpers of the DPFP rows.
__device__ __forceinline__ uint32_t bmax0(uint32_t x) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0u));
    return r;
}
__device__ __forceinline__ uint32_t bmin0(uint32_t x) {
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(x), "r"(0u));
    return r;
}
__device__ __forceinline__ uint32_t bmul(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t badd(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// Word k of the partner values x'_i of shift s for the elements 2k, 2k+1 of
// a raw row w (DR bf16 values, two per word): x'_i = x_{i+s} for i + s < DR,
// else -x_{i+s-DR} (the second half of r = [relu(x), relu(-x)]).  k and s are
// compile-time after unrolling, so the wrap tests fold away.
template <int DR>
__device__ __forceinline__ uint32_t dpfp_partner(const uint32_t (&w)[DR / 2], int k, int s) {
    constexpr int NW = DR / 2;
    auto word = [&](int a) { return a < NW ? w[a] : (w[a - NW] ^ 0x80008000u); };
    if ((s & 1) == 0) return word(k + s / 2);
    const int a = k + (s - 1) / 2;
    return __byte_perm(word(a), word(a + 1), 0x5432);   // high half of word a, low half of word a + 1
}

// DPFP ("Linear Transformers Are Secretly Fast Weight Programmers", sec. 5.2)
// of row r from its raw values, in packed bf16x2 arithmetic: for shift s and
// i < DR the features (s-1)*2DR + i = relu(x_i) relu(x'_i) and
// (s-1)*2DR + DR + i = relu(-x_i) relu(-x'_i) = min(x_i, 0) min(x'_i, 0), each
// product rounded to bf16 once.  With SUM the row is then divided by its
// feature sum (fp32; the two products of an element never both differ from
// zero, so their packed sum is exact) in a second pass over the stored row,
// a second bf16 rounding.  The row's DR/2 raw words stay in registers.
template <int F, int DR, int NU, bool SUM>
__device__ __forceinline__ void dpfp_row(uint8_t *tile, int r, bool zero) {
    static_assert(F == 2 * DR * NU && DR <= 64 && DR % 8 == 0, "DPFP width");
    constexpr int NW = DR / 2;
    uint32_t w[NW];
    load_raw_row<DR>(tile, r, w);
    auto at = [&](int c) { return reinterpret_cast<uint4 *>(tile + (c / 64) * kC * 128 + sw128_offset(r, c % 64)); };
    float s0 = 0.f, s1 = 0.f;
    // all raw words are read before the first feature chunk overwrites them
#pragma unroll
    for (int s = 1; s <= NU; ++s)
#pragma unroll
        for (int k0 = 0; k0 < NW; k0 += 4) {
            uint32_t hi[4], lo[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const uint32_t xp = dpfp_partner<DR>(w, k0 + u, s);
                hi[u] = bmul(bmax0(w[k0 + u]), bmax0(xp));
                lo[u] = bmul(bmin0(w[k0 + u]), bmin0(xp));
                if (SUM) {
                    const uint32_t t = badd(hi[u], lo[u]);
                    s0 += bf16lo(t);
                    s1 += bf16hi(t);
                }
            }
            const int c = (s - 1) * 2 * DR + 2 * k0;
            *at(c) = zero ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(hi[0], hi[1], hi[2], hi[3]);
            *at(c + DR) = zero ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(lo[0], lo[1], lo[2], lo[3]);
        }
    if (SUM && !zero) {
        const float sum = s0 + s1;
        const float sc = sum > 0.f ? 1.f / sum : 0.f;
        const uint32_t scw = pack_bf16x2(sc, sc);
#pragma unroll 4
        for (int c = 0; c < F; c += 8) {
            uint4 v = *at(c);
            v.x = bmul(v.x, scw);
            v.y = bmul(v.y, scw);
            v.z = bmul(v.z, scw);
            v.w = bmul(v.w, scw);
            *at(c) = v;
        }
    }
}

// Elementwise: pass 1 maps each 8-column chunk in place with phi_bf16x2 and
// sums the bf16 results in fp32; pass 2 scales the chunks by 1 / sum (a
// second bf16 rounding).
template <int F>
__device__ __forceinline__ void elu1_sum_row(uint8_t *tile, int r, bool zero) {
    auto at = [&](int c) { return reinterpret_cast<uint4 *>(tile + (c / 64) * kC * 128 + sw128_offset(r, c % 64)); };
    float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
    for (int c = 0; c < F; c += 8) {
        uint4 w = *at(c);
        w.x = phi_bf16x2(w.x);
        w.y = phi_bf16x2(w.y);
        w.z = phi_bf16x2(w.z);
        w.w = phi_bf16x2(w.w);
        s0 += (bf16lo(w.x) + bf16hi(w.x)) + (bf16lo(w.y) + bf16hi(w.y));
        s1 += (bf16lo(w.z) + bf16hi(w.z)) + (bf16lo(w.w) + bf16hi(w.w));
        *at(c) = w;
    }
    const float scale = 1.f / (s0 + s1);
#pragma unroll 4
    for (int c = 0; c < F; c += 8) {
        const uint4 w = *at(c);
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (!zero)
            o = make_uint4(pack_bf16x2(bf16lo(w.x) * scale, bf16hi(w.x) * scale),
                           pack_bf16x2(bf16lo(w.y) * scale, bf16hi(w.y) * scale),
                           pack_bf16x2(bf16lo(w.z) * scale, bf16hi(w.z) * scale),
                           pack_bf16x2(bf16lo(w.w) * scale, bf16hi(w.w) * scale));
        *at(c) = o;
    }
}

// Applies feature map `feat` (kFeatElu1Sum or kFeatDpfp with raw width dr,
// nu shifts, sum normalisation if sum) to row t of an F-wide tile.
template <int F>
__device__ __forceinline__ void feature_row(uint8_t *tile, int t, int zero_from, int feat, int dr, int nu, bool sum) {
    const bool zero = t >= zero_from;
    if (feat == kFeatElu1Sum) {
        elu1_sum_row<F>(tile, t, zero);
        return;
    }
    if constexpr (F == 128) {
        if (dr == 64 && nu == 1) sum ? dpfp_row<F, 64, 1, true>(tile, t, zero) : dpfp_row<F, 64, 1, false>(tile, t, zero);
        else if (dr == 32 && nu == 2) sum ? dpfp_row<F, 32, 2, true>(tile, t, zero) : dpfp_row<F, 32, 2, false>(tile, t, zero);
        else if (dr == 16 && nu == 4) sum ? dpfp_row<F, 16, 4, true>(tile, t, zero) : dpfp_row<F, 16, 4, false>(tile, t, zero);
    } else if constexpr (F == 64) {
        if (dr == 32 && nu == 1) sum ? dpfp_row<F, 32, 1, true>(tile, t, zero) : dpfp_row<F, 32, 1, false>(tile, t, zero);
        else if (dr == 16 && nu == 2) sum ? dpfp_row<F, 16, 2, true>(tile, t, zero) : dpfp_row<F, 16, 2, false>(tile, t, zero);
    }
}

// A D x M fp32 block held one row per thread leaves through shared memory so
// that its global stores are coalesced: stage_row32_f32 puts columns
// [c0, c0+32) of row r into the staging area (16-byte units, unit c4 of row
// r at c4 ^ (r mod M/4): a warp's rows land in distinct banks), and, after a
// barrier over the writing threads, store_staged_f32 copies the block to the
// contiguous D*M floats at dst with 16-byte stores by threads t of nthr.
template <int M>
__device__ __forceinline__ void stage_row32_f32(float *stage, int r, int c0, const float *v) {
    constexpr int R4 = M / 4;
    float4 *row = reinterpret_cast<float4 *>(stage) + r * R4;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        row[(c0 / 4 + j) ^ (r % R4)] = make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]);
}
template <int D, int M>
__device__ __forceinline__ void store_staged_f32(float *dst, const float *stage, int t, int nthr) {
    constexpr int R4 = M / 4;
    const float4 *s4 = reinterpret_cast<const float4 *>(stage);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    for (int f = t; f < D * R4; f += nthr) {
        const int row = f / R4, c4 = f % R4;
        d4[f] = s4[row * R4 + (c4 ^ (row % R4))];
    }
}

// Writes columns [c0, c0+32) of row r of a D x M fp32 state as bf16 into the
// MN-major swizzled snapshot [D rows x M cols] (sub-tiles of 64 columns).
template <int D>
__device__ __forceinline__ void store_snap32(uint8_t *snap, int r, int c0, const float *v) {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        const int c = c0 + c8 * 8;
        uint8_t *dst = snap + (c / 64) * D * 128 + sw128_offset(r, c % 64);
        const float *x = v + c8 * 8;
        uint4 w;
        w.x = pack_bf16x2(x[0], x[1]);
        w.y = pack_bf16x2(x[2], x[3]);
        w.z = pack_bf16x2(x[4], x[5]);
        w.w = pack_bf16x2(x[6], x[7]);
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

// Loads 32 consecutive fp32 TMEM columns of this thread's lane.
__device__ __forceinline__ void tmem_ld32f(uint32_t taddr, float (&v)[32]) {
    uint32_t a[16], b[16];
    tmem_ld16(taddr, a);
    tmem_ld16(taddr + 16, b);
    tmem_wait_ld();
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        v[j] = __uint_as_float(a[j]);
        v[16 + j] = __uint_as_float(b[j]);
    }
}

__device__ __forceinline__ void tmem_st32f(uint32_t taddr, const float (&v)[32]) {
    uint32_t a[16], b[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        a[j] = __float_as_uint(v[j]);
        b[j] = __float_as_uint(v[16 + j]);
    }
    tmem_st16(taddr, a);
    tmem_st16(taddr + 16, b);
}

// A (TMEM) x B (shared memory) MMA, kind::f16.
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Descriptors of the operand tiles (all 128-byte swizzled, 1024-byte aligned).
// A descriptor's start-address field counts 16-byte units in its low bits, so
// a K-step is a constant added to a base descriptor built once per chunk: the
// single thread issuing MMAs must not spend its time on descriptor arithmetic.
// K-major tile with rows of up to 128 elements stored as 64-element sub-tiles
// of kC rows: K-step ks (16 elements) starts 32 bytes further, or in the next
// sub-tile after 4 steps.
__device__ __forceinline__ uint64_t kmajor_base(uint32_t tile) { return smem_desc(tile, 16, 1024); }
__host__ __device__ constexpr uint64_t kmajor_step(int ks, int rows = kC) {
    return (uint64_t)((ks / 4) * rows * 128 / 16 + (ks % 4) * 2);
}
// MN-major: K-step ks covers rows 16ks..16ks+15, 2048 bytes further.
__host__ __device__ constexpr uint64_t mnmajor_step(int ks) { return (uint64_t)(ks * 128); }
// B operand of 16 K-rows made of one 8-row atom read twice (K-group stride 0):
// valid because every row of the ones operand is the same.
__device__ __forceinline__ uint64_t ones_desc(uint32_t tile) { return smem_desc(tile, 1024, 0); }

// Opts a kernel in to `bytes` of dynamic shared memory, once per (kernel,
// device): the memo is keyed by the kernel's address, since all instances
// of a kernel template share one function type.
template <typename K>
cudaError_t set_smem(K kernel, int bytes) {
    static std::mutex mu;
    static std::vector<std::pair<const void *, int>> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
    const void *key = reinterpret_cast<const void *>(kernel);
    std::lock_guard<std::mutex> lock(mu);
    for (const auto &d : done)
        if (d.first == key && d.second == dev) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.emplace_back(key, dev);
    return e;
}

}  // namespace
}  // namespace la

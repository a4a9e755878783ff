// tc_bwd_common.cuh - helpers shared by the tensor-core backward kernels
// (la_tc_bwd_nc.cu, la_tc_bwd_chunk.cu): operand tiles of fp32 sums as bf16
// hi + lo pairs, row loads and stores of 128-row tiles, and the barrier
// idioms of kernels whose phases run one after another in every thread.
#pragma once

#include "la_common.cuh"
#include "tc_kernels.cuh"
#include "tc_ptx.cuh"

namespace la {
namespace tc {

constexpr int kNT = 128;   // threads of the non-causal backward's kernels; one row of a 128-row tile each

// Row-major operand [X_hi | w | X_lo] (X: rows x cols) in 64-column swizzled
// atoms of `rows` rows each.
template <int ROWS, int COLS>
struct XwTile {
    static constexpr int ATOM = ROWS * 128;
    static constexpr int W_ATOM = (COLS / 64) * ATOM;   // byte offset of the w atom
    static constexpr int LO = W_ATOM + ATOM;            // byte offset of X_lo
    static constexpr int BYTES = LO + W_ATOM;
};

// Sum of the head's nsplit fp32 partial slots [X (D x M) | w (D)] (slot stride
// D*M + D floats) into the bf16 operand tile [X_hi | w | X_lo]: thread r < D
// takes row r.
template <int D, int M>
__device__ __forceinline__ void sum_partials_to_tile(const float *slots, int nsplit, uint8_t *tile, int r) {
    constexpr int W = D * M + D;
    if (r >= D) return;
#pragma unroll 1
    for (int c0 = 0; c0 < M; c0 += 32) {
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = 0.f;
        for (int sp = 0; sp < nsplit; ++sp) {
            const float4 *src = reinterpret_cast<const float4 *>(slots + (size_t)sp * W + r * M + c0);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float4 a = __ldcg(src + j);
                x[4 * j] += a.x; x[4 * j + 1] += a.y; x[4 * j + 2] += a.z; x[4 * j + 3] += a.w;
            }
        }
        float lo[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float h = __bfloat162float(__float2bfloat16_rn(x[j]));
            lo[j] = x[j] - h;
            x[j] = h;
        }
        store_snap32<D>(tile, r, c0, x);
        store_snap32<D>(tile + XwTile<D, M>::LO, r, c0, lo);
    }
    float w = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) w += __ldcg(slots + (size_t)sp * W + D * M + r);
    const float hi = __bfloat162float(__float2bfloat16_rn(w));
    const uint32_t hl = pack_bf16x2(hi, w - hi);
    uint8_t *wa = tile + XwTile<D, M>::W_ATOM;
#pragma unroll
    for (int c = 0; c < 64; c += 8)
        *reinterpret_cast<uint4 *>(wa + sw128_offset(r, c)) = make_uint4(c == 0 ? hl : 0u, c == 0 ? hl : 0u, 0u, 0u);
}

// Row r of a bf16 result (n columns, fp32 in x) to global memory: 256-bit
// stores when the row start allows, else 128-bit.
template <int NCOL>
__device__ __forceinline__ void store_row_bf16(__nv_bfloat16 *dst, const float *x) {
    uint4 w[NCOL / 8];
#pragma unroll
    for (int c8 = 0; c8 < NCOL / 8; ++c8)
        w[c8] = make_uint4(pack_bf16x2(x[8 * c8], x[8 * c8 + 1]), pack_bf16x2(x[8 * c8 + 2], x[8 * c8 + 3]),
                           pack_bf16x2(x[8 * c8 + 4], x[8 * c8 + 5]), pack_bf16x2(x[8 * c8 + 6], x[8 * c8 + 7]));
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    if ((reinterpret_cast<uintptr_t>(dst) & 31u) == 0) {
#pragma unroll
        for (int c16 = 0; c16 < NCOL / 16; ++c16) st_global_v8(d + 2 * c16, w[2 * c16], w[2 * c16 + 1]);
    } else {
#pragma unroll
        for (int c8 = 0; c8 < NCOL / 8; ++c8) d[c8] = w[c8];
    }
}

// Columns c0..c0+31 of bf16 row r of a swizzled [kC x cols] tile as fp32.
__device__ __forceinline__ void load_row32(const uint8_t *tile, int r, int c0, float (&x)[32]) {
#pragma unroll
    for (int c8 = 0; c8 < 4; ++c8) {
        const int c = c0 + 8 * c8;
        const uint4 v = *reinterpret_cast<const uint4 *>(tile + (c / 64) * kC * 128 + sw128_offset(r, c % 64));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            x[8 * c8 + 2 * e] = bf16lo(w[e]);
            x[8 * c8 + 2 * e + 1] = bf16hi(w[e]);
        }
    }
}

// psi(x) = phi(x) - 1 = elu(x) (x for x > 0, e^x - 1 otherwise) in place on a
// C x DD bf16 tile (64-column sub-tiles of C rows), rows >= zero_from as
// zeros; thread t of kNT.  Where the inputs are small, phi is close to 1 and
// its bf16 rounding swamps x: a product whose terms cancel along the 1 takes
// psi as its operand and adds the other factor's row sums for the 1 in fp32.
template <int DD>
__device__ __forceinline__ void psi_tile(uint8_t *tile, int t, int zero_from) {
    constexpr int CHUNKS = kC * DD * 2 / 16;
    static_assert(CHUNKS % (4 * kNT) == 0, "whole rounds of four chunks per thread");
#pragma unroll 1
    for (int u0 = t; u0 < CHUNKS; u0 += 4 * kNT) {
        uint4 v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = *reinterpret_cast<const uint4 *>(tile + (u0 + i * kNT) * 16);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float a = bf16lo(w[u]), b = bf16hi(w[u]);
                float ea, eb;
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(ea) : "f"(a * 1.4426950408889634f));
                asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(eb) : "f"(b * 1.4426950408889634f));
                w[u] = pack_bf16x2(a > 0.f ? a : ea - 1.f, b > 0.f ? b : eb - 1.f);
            }
            const uint32_t off = (uint32_t)(u0 + i * kNT) * 16u;
            const int row = (int)((off % (kC * 128u)) >> 7);
            *reinterpret_cast<uint4 *>(tile + off) =
                row >= zero_from ? make_uint4(0u, 0u, 0u, 0u) : make_uint4(w[0], w[1], w[2], w[3]);
        }
    }
}

// fp32 sum of the NCOL bf16 values of row r of a swizzled [kC x NCOL] tile.
template <int NCOL>
__device__ __forceinline__ float row_sum(const uint8_t *tile, int r) {
    float s = 0.f;
#pragma unroll
    for (int c0 = 0; c0 < NCOL; c0 += 32) {
        float x[32];
        load_row32(tile, r, c0, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) s += x[j];
    }
    return s;
}

// Every thread's shared-memory writes and TMEM stores visible to the MMAs
// thread 0 issues next; false (CTA-uniform) if any thread's `mine` is false.
__device__ __forceinline__ bool operands_ready(bool mine) {
    tmem_wait_st();
    fence_proxy_async();
    tc_fence_before();
    const bool all = __syncthreads_and(mine ? 1 : 0) != 0;
    tc_fence_after();
    return all;
}

// Thread 0 commits its MMAs to `bar`; every thread waits for that phase.
__device__ __forceinline__ bool mma_done(uint64_t *bar, uint32_t &phase) {
    if (threadIdx.x == 0) mma_commit(bar);
    const bool got = mbar_wait_bounded(bar, phase, now_ns() + kWaitNs, nullptr);
    phase ^= 1u;
    tc_fence_after();
    return __syncthreads_and(got ? 1 : 0) != 0;
}

}  // namespace tc
}  // namespace la

// tc_host.h - host helpers for the tensor-core path: building TMA tensor
// maps through the driver entry point (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>

namespace la {
namespace tc {

inline PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Tensor map over a row-major bf16 tensor [outer][rows][cols] (cols
// innermost), boxes of box_cols x box_rows x 1 with the 128-byte swizzle.
// Out-of-range rows read as zero on loads and are skipped on stores.
// Requirements checked by the driver: 16-byte aligned base, row pitch a
// multiple of 16 bytes, box_cols * 2 <= 128.
inline bool make_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t outer,
                              uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, rows, outer};
    cuuint64_t strides[2] = {cols * 2, cols * rows * 2};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Tensor map over a bf16 tensor with explicit strides (bytes, multiples of 16):
// element (c, r, o) at base + 2c + r * row_stride + o * outer_stride.  Used for
// step-major decode inputs [T][B*H][cols], read as [B*H][T][cols].
inline bool make_tmap_bf16_3d_strided(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows,
                                      uint64_t outer, uint64_t row_stride, uint64_t outer_stride,
                                      uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[3] = {cols, rows, outer};
    cuuint64_t strides[2] = {row_stride, outer_stride};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Same as make_tmap_bf16_3d, served from a small per-thread cache keyed by
// (base, cols, rows, outer, box): encoding a tensor map costs host time on
// every call, and a caller usually passes the same buffers again and again.
inline bool cached_tmap_bf16_3d(CUtensorMap *map, const void *base, uint64_t cols, uint64_t rows, uint64_t outer,
                                uint32_t box_cols, uint32_t box_rows) {
    struct Entry {
        const void *base;
        uint64_t cols, rows, outer;
        uint32_t box_cols, box_rows;
        CUtensorMap map;
        bool used;
    };
    constexpr int kEntries = 16;
    thread_local Entry cache[kEntries];
    thread_local int next = 0;
    for (int i = 0; i < kEntries; ++i) {
        const Entry &e = cache[i];
        if (e.used && e.base == base && e.cols == cols && e.rows == rows && e.outer == outer &&
            e.box_cols == box_cols && e.box_rows == box_rows) {
            *map = e.map;
            return true;
        }
    }
    if (!make_tmap_bf16_3d(map, base, cols, rows, outer, box_cols, box_rows)) return false;
    Entry &e = cache[next];
    next = (next + 1) % kEntries;
    e = Entry{base, cols, rows, outer, box_cols, box_rows, *map, true};
    return true;
}

}  // namespace tc
}  // namespace la

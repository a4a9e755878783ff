// la_common.cuh - device helpers shared by the kernels of liblinattn.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace la {

// Error codes a kernel may record in the device error word (values of la_status).
constexpr int kErrTimeout = 4;
constexpr int kErrBounds = 5;

// Bounds checks of the checked build (compiled with -DLA_CHECKED, a separate
// library): LA_IN_BOUNDS(cond, err) is true when cond holds; otherwise it
// records LA_ERR_BOUNDS in the error word and is false, and the caller skips
// the access it guards.  In the release build it is `true` and costs nothing.
#ifdef LA_CHECKED
#define LA_IN_BOUNDS(cond, err) ((cond) ? true : (::la::record_error((err), ::la::kErrBounds), false))
#else
#define LA_IN_BOUNDS(cond, err) true
#endif

// phi(x) = elu(x) + 1 with alpha = 1 ("Transformers are RNNs", sec. 3.2.1,
// eq. (7)): x + 1 for x > 0, exp(x) otherwise.  Accurate exp for the SIMT path.
__device__ __forceinline__ float phi_accurate(float x) { return x > 0.f ? x + 1.f : expf(x); }


template <typename T> __device__ __forceinline__ float to_f32(T x);
template <> __device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Records `code` in the error word unless an earlier error is already there.
__device__ __forceinline__ void record_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Programmatic dependent launch: pdl_wait() returns once the grids this
// launch depends on have completed and their writes are visible (at once for
// a launch without such a dependency); pdl_launch_dependents() lets the next
// launch on the stream be scheduled (its own pdl_wait() still waits for this
// grid to complete).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// pdl_wait() for a whole CTA (every thread calls it): one thread waits, the
// others at the barrier; the prerequisite grids' writes are then visible to
// every thread of this grid.
__device__ __forceinline__ void pdl_wait_cta() {
    if (threadIdx.x == 0) pdl_wait();
    __syncthreads();
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

}  // namespace la

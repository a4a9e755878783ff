// la_noalloc.cu - non-causal attention for callers that cannot allocate
// device memory: the partial sums live in a fixed array compiled into the
// library instead of a caller-supplied workspace.
#include <mutex>

#include "la_common.cuh"
#include "la_internal.h"

namespace la {
namespace {

constexpr size_t kScratchBytes = (size_t)8 << 20;   // 8 MiB, held by every device that loads the library

// In host code this name is only a host-side handle for the symbol, not a
// device address; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
float *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached; nullptr on failure.
float *scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return nullptr;
        g_scratch_ptr[dev] = static_cast<float *>(p);
    }
    return g_scratch_ptr[dev];
}

bool dim_ok(int x) { return x == 16 || x == 32 || x == 64 || x == 128; }
bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace la

using namespace la;

extern "C" la_status la_forward_noncausal_noalloc(const void *q, const void *k, const void *v, void *out,
                                                  la_shape s, la_stream_t stream) {
    if (s.B < 0 || s.H < 0 || s.N < 0) return LA_ERR_INVALID_ARG;
    if (s.dtype != LA_DTYPE_F32 && s.dtype != LA_DTYPE_BF16) return LA_ERR_INVALID_ARG;
    if (!dim_ok(s.D) || !dim_ok(s.M)) return LA_ERR_UNSUPPORTED;
    const long long BH = (long long)s.B * s.H;
    if (BH == 0 || s.N == 0) return LA_OK;
    for (const void *p : {q, k, v, (const void *)out})
        if (p == nullptr || !aligned16(p)) return LA_ERR_INVALID_ARG;
    if (out == q || out == k || out == v) return LA_ERR_INVALID_ARG;
    // One split of partial sums needs BH * (D*M + D) floats; at least one must
    // fit.  BH is bounded first, so that the product below cannot wrap.
    const size_t per_head = ((size_t)s.D * s.M + s.D) * sizeof(float);
    if (BH > (long long)(kScratchBytes / per_head)) return LA_ERR_UNSUPPORTED;
    const size_t per_split = (size_t)BH * per_head;
    const int max_splits = (int)(kScratchBytes / per_split);
    const DeviceInfo *dev = device_info();
    float *scratch = scratch_on_current_device();
    if (!dev || !scratch) return LA_ERR_CUDA;
    Problem p{q, k, v, out, nullptr, nullptr, BH, s.N, s.D, s.M, s.dtype, 0, scratch, kScratchBytes,
              (cudaStream_t)stream};
    return simt_noncausal_capped(p, *dev, max_splits) == cudaSuccess ? LA_OK : LA_ERR_CUDA;
}

// la_api.cu - the extern "C" entry points of liblinattn.so: host-side argument
// checks, dispatch to the kernels, and the per-device error word.
#include <atomic>
#include <mutex>

#include "la_common.cuh"
#include "la_internal.h"

// One error word per device (each device holds its own copy of a __device__
// variable).  Kernels receive its address; la_get_last_error() reads and clears it.
__device__ int g_la_error_word = 0;

namespace la {

volatile int g_inject_timeout = 0;
volatile int g_inject_limit_us = 1000;
volatile int g_inject_bounds = 0;

static std::atomic<unsigned long long> g_launches{0};
void count_launches(int n) { g_launches.fetch_add((unsigned long long)n, std::memory_order_relaxed); }

namespace {

constexpr int kMaxDevices = 64;
DeviceInfo g_dev[kMaxDevices];
bool g_dev_ready[kMaxDevices];
std::mutex g_dev_mu;

bool dim_ok(int x) { return x == 16 || x == 32 || x == 64 || x == 128; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape checks common to every call.  Negative sizes and unknown dtypes are
// invalid arguments; D, M outside {16, 32, 64, 128} are unsupported.
la_status check_shape(const la_shape &s, bool uses_n) {
    if (s.B < 0 || s.H < 0 || (uses_n && s.N < 0)) return LA_ERR_INVALID_ARG;
    if (s.dtype != LA_DTYPE_F32 && s.dtype != LA_DTYPE_BF16) return LA_ERR_INVALID_ARG;
    if (!dim_ok(s.D) || !dim_ok(s.M)) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

la_status check_ptr(const void *p, bool needed) {
    if (!needed) return LA_OK;
    if (p == nullptr || !aligned16(p)) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

bool chunk_ok(int chunk) { return chunk == 0 || chunk == 64 || chunk == 128; }

la_status from_cuda(cudaError_t e) { return e == cudaSuccess ? LA_OK : LA_ERR_CUDA; }

}  // namespace

const DeviceInfo *device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_dev_mu);
    if (!g_dev_ready[dev]) {
        DeviceInfo d;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&d.max_smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) !=
                cudaSuccess)
            return nullptr;
        void *addr = nullptr;
        if (cudaGetSymbolAddress(&addr, g_la_error_word) != cudaSuccess) return nullptr;
        d.err_word = static_cast<int *>(addr);
        g_dev[dev] = d;
        g_dev_ready[dev] = true;
    }
    return &g_dev[dev];
}

}  // namespace la

using namespace la;

extern "C" {

int la_version(void) { return 10000; }

unsigned long long la_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *la_status_string(la_status st) {
    switch (st) {
        case LA_OK: return "ok";
        case LA_ERR_INVALID_ARG: return "invalid argument";
        case LA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case LA_ERR_CUDA: return "CUDA error";
        case LA_ERR_TIMEOUT: return "a kernel gave up a bounded wait";
        case LA_ERR_BOUNDS: return "a checked build found an access outside a buffer";
    }
    return "unknown status";
}

void la_debug_inject_timeout(int enable, int limit_us) {
    g_inject_limit_us = limit_us > 0 ? limit_us : 1;
    g_inject_timeout = enable ? 1 : 0;
}

int la_checked_build(void) {
#ifdef LA_CHECKED
    return 1;
#else
    return 0;
#endif
}

void la_debug_inject_bounds(int enable) {
#ifdef LA_CHECKED
    g_inject_bounds = enable ? 1 : 0;
#else
    (void)enable;   // the release build has no bounds checks to catch it
#endif
}

size_t la_workspace_bytes(la_op op, la_shape s, int chunk) {
    if (check_shape(s, op != LA_OP_DECODE) != LA_OK) return (size_t)-1;
    switch (op) {
        case LA_OP_NONCAUSAL:
            if (tc_noncausal_supported(s)) return tc_noncausal_ws_bytes(s);
            return simt_noncausal_ws_bytes(s);
        case LA_OP_CAUSAL:
            if (!chunk_ok(chunk)) return (size_t)-1;
            if (tc_causal_supported(s, chunk)) return tc_causal_ws_bytes(s, chunk);
            return 0;
        case LA_OP_DECODE: return 0;
        case LA_OP_NONCAUSAL_BWD: return noncausal_bwd_ws_bytes(s);
        case LA_OP_CAUSAL_BWD: return causal_bwd_ws_bytes(s);
    }
    return (size_t)-1;
}

namespace {

// Checks common to both backward calls; fills the device-side problem.
la_status check_backward(const void *q, const void *k, const void *v, const void *dout, void *dq, void *dk,
                         void *dv, const la_shape &s, la_op op, void *workspace, size_t ws_bytes, bool &work) {
    la_status st = check_shape(s, true);
    if (st != LA_OK) return st;
    const long long BH = (long long)s.B * s.H;
    work = BH > 0 && s.N > 0;
    if ((st = check_ptr(q, work)) || (st = check_ptr(k, work)) || (st = check_ptr(v, work)) ||
        (st = check_ptr(dout, work)) || (st = check_ptr(dq, work)) || (st = check_ptr(dk, work)) ||
        (st = check_ptr(dv, work)))
        return st;
    if (!work) return LA_OK;
    // the gradients must not overlap the inputs or each other
    const void *ins[4] = {q, k, v, dout};
    const void *outs[3] = {dq, dk, dv};
    for (const void *o : outs)
        for (const void *i : ins)
            if (o == i) return LA_ERR_INVALID_ARG;
    if (dq == dk || dq == dv || dk == dv) return LA_ERR_INVALID_ARG;
    const size_t need = la_workspace_bytes(op, s, 0);
    if (ws_bytes < need || (need > 0 && check_ptr(workspace, true) != LA_OK)) return LA_ERR_INVALID_ARG;
    return LA_OK;
}

}  // namespace

la_status la_backward_noncausal(const void *q, const void *k, const void *v, const void *dout, void *dq,
                                void *dk, void *dv, la_shape s, void *workspace, size_t ws_bytes,
                                la_stream_t stream) {
    bool work = false;
    la_status st = check_backward(q, k, v, dout, dq, dk, dv, s, LA_OP_NONCAUSAL_BWD, workspace, ws_bytes, work);
    if (st != LA_OK || !work) return st;
    const DeviceInfo *dev = device_info();
    if (!dev) return LA_ERR_CUDA;
    BwdProblem p{q, k, v, dout, dq, dk, dv, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
                 (long long)s.B * s.H, s.N, s.D, s.M, s.dtype, workspace, ws_bytes, (cudaStream_t)stream};
    if (tc_nc_backward_supported(s)) return from_cuda(tc_noncausal_backward(p, *dev));
    return from_cuda(noncausal_backward(p, *dev));
}

la_status la_backward_causal(const void *q, const void *k, const void *v, const void *dout, void *dq,
                             void *dk, void *dv, la_shape s, const float *S0, const float *z0,
                             const float *dSN, const float *dzN, float *dS0, float *dz0, void *workspace,
                             size_t ws_bytes, la_stream_t stream) {
    if ((S0 == nullptr) != (z0 == nullptr) || (dSN == nullptr) != (dzN == nullptr) ||
        (dS0 == nullptr) != (dz0 == nullptr))
        return LA_ERR_INVALID_ARG;
    bool work = false;
    la_status st = check_backward(q, k, v, dout, dq, dk, dv, s, LA_OP_CAUSAL_BWD, workspace, ws_bytes, work);
    if (st != LA_OK) return st;
    const long long BH = (long long)s.B * s.H;
    for (const void *p : {(const void *)S0, (const void *)z0, (const void *)dSN, (const void *)dzN,
                          (const void *)dS0, (const void *)dz0})
        if ((st = check_ptr(p, p != nullptr && BH > 0)) != LA_OK) return st;
    if (!work) {
        // an empty sequence passes the final-state gradient straight through
        if (dS0 && BH > 0) {
            const size_t nS = (size_t)BH * s.D * s.M * sizeof(float), nz = (size_t)BH * s.D * sizeof(float);
            cudaStream_t cs = (cudaStream_t)stream;
            cudaError_t e = dSN ? cudaMemcpyAsync(dS0, dSN, nS, cudaMemcpyDeviceToDevice, cs)
                                : cudaMemsetAsync(dS0, 0, nS, cs);
            if (e == cudaSuccess)
                e = dzN ? cudaMemcpyAsync(dz0, dzN, nz, cudaMemcpyDeviceToDevice, cs) : cudaMemsetAsync(dz0, 0, nz, cs);
            return from_cuda(e);
        }
        return LA_OK;
    }
    const DeviceInfo *dev = device_info();
    if (!dev) return LA_ERR_CUDA;
    BwdProblem p{q, k, v, dout, dq, dk, dv, S0, z0, dSN, dzN, dS0, dz0,
                 BH, s.N, s.D, s.M, s.dtype, workspace, ws_bytes, (cudaStream_t)stream};
    if (tc_backward_supported(s)) return from_cuda(tc_causal_backward(p, *dev));
    if (tc_chunk_backward_supported(s)) return from_cuda(tc_chunk_causal_backward(p, *dev));
    return from_cuda(causal_backward(p, *dev));
}

la_status la_forward_noncausal(const void *q, const void *k, const void *v, void *out, la_shape s,
                               void *workspace, size_t ws_bytes, la_stream_t stream) {
    la_status st = check_shape(s, true);
    if (st != LA_OK) return st;
    const long long BH = (long long)s.B * s.H;
    const bool work = BH > 0 && s.N > 0;
    if ((st = check_ptr(q, work)) || (st = check_ptr(k, work)) || (st = check_ptr(v, work)) ||
        (st = check_ptr(out, work)))
        return st;
    if (!work) return LA_OK;
    const size_t need = la_workspace_bytes(LA_OP_NONCAUSAL, s, 0);
    if (ws_bytes < need || (need > 0 && check_ptr(workspace, true) != LA_OK)) return LA_ERR_INVALID_ARG;
    if (out == q || out == k || out == v) return LA_ERR_INVALID_ARG;
    const DeviceInfo *dev = device_info();
    if (!dev) return LA_ERR_CUDA;
    Problem p{q, k, v, out, nullptr, nullptr, BH, s.N, s.D, s.M, s.dtype, 0, workspace, ws_bytes,
              (cudaStream_t)stream};
    if (tc_noncausal_supported(s)) return from_cuda(tc_noncausal(p, *dev));
    return from_cuda(simt_noncausal(p, *dev));
}

la_status la_forward_causal(const void *q, const void *k, const void *v, void *out, la_shape s,
                            int chunk, float *S, float *z, void *workspace, size_t ws_bytes,
                            la_stream_t stream) {
    la_status st = check_shape(s, true);
    if (st != LA_OK) return st;
    if (!chunk_ok(chunk)) return LA_ERR_UNSUPPORTED;
    if ((S == nullptr) != (z == nullptr)) return LA_ERR_INVALID_ARG;
    const long long BH = (long long)s.B * s.H;
    const bool work = BH > 0 && s.N > 0;
    if ((st = check_ptr(S, S != nullptr && BH > 0)) || (st = check_ptr(z, z != nullptr && BH > 0)))
        return st;
    if ((st = check_ptr(q, work)) || (st = check_ptr(k, work)) || (st = check_ptr(v, work)) ||
        (st = check_ptr(out, work && out != nullptr)))
        return st;
    if (!work) return LA_OK;   // an empty sequence leaves the state as it is
    if (out != nullptr && (out == q || out == k || out == v)) return LA_ERR_INVALID_ARG;
    const size_t need = la_workspace_bytes(LA_OP_CAUSAL, s, chunk);
    if (ws_bytes < need || (need > 0 && check_ptr(workspace, true) != LA_OK)) return LA_ERR_INVALID_ARG;
    const DeviceInfo *dev = device_info();
    if (!dev) return LA_ERR_CUDA;
    Problem p{q, k, v, out, S, z, BH, s.N, s.D, s.M, s.dtype, chunk, workspace, ws_bytes,
              (cudaStream_t)stream};
    if (tc_causal_supported(s, chunk)) return from_cuda(tc_causal(p, *dev));
    return from_cuda(simt_causal(p, *dev));
}

la_status la_forward_causal_varlen(const void *q, const void *k, const void *v, void *out, const int *lens,
                                   la_shape s, float *S, float *z, void *workspace, size_t ws_bytes,
                                   la_stream_t stream) {
    la_status st = check_shape(s, true);
    if (st != LA_OK) return st;
    if ((S == nullptr) != (z == nullptr)) return LA_ERR_INVALID_ARG;
    const long long BH = (long long)s.B * s.H;
    const bool work = BH > 0 && s.N > 0;
    if ((st = check_ptr(S, S != nullptr && BH > 0)) || (st = check_ptr(z, z != nullptr && BH > 0)))
        return st;
    if ((st = check_ptr(q, work)) || (st = check_ptr(k, work)) || (st = check_ptr(v, work)) ||
        (st = check_ptr(out, work && out != nullptr)))
        return st;
    if (!work) return LA_OK;
    if (lens == nullptr || (reinterpret_cast<uintptr_t>(lens) & 3u) != 0) return LA_ERR_INVALID_ARG;
    if (out != nullptr && (out == q || out == k || out == v)) return LA_ERR_INVALID_ARG;
    const size_t need = la_workspace_bytes(LA_OP_CAUSAL, s, 0);
    if (ws_bytes < need || (need > 0 && check_ptr(workspace, true) != LA_OK)) return LA_ERR_INVALID_ARG;
    const DeviceInfo *dev = device_info();
    if (!dev) return LA_ERR_CUDA;
    Problem p{q, k, v, out, S, z, BH, s.N, s.D, s.M, s.dtype, 0, workspace, ws_bytes, (cudaStream_t)stream};
    p.lens = lens;
    p.H = s.H;
    if (tc_causal_supported(s, 0)) return from_cuda(tc_causal(p, *dev));
    return from_cuda(simt_causal(p, *dev));
}

la_status la_decode_steps(const void *q, const void *k, const void *v, void *y, float *S, float *z,
                          const int *steps, int T, la_shape s, la_stream_t stream) {
    la_status st = check_shape(s, false);
    if (st != LA_OK) return st;
    if (T < 0) return LA_ERR_INVALID_ARG;
    const long long BH = (long long)s.B * s.H;
    const bool work = BH > 0 && T > 0;
    if ((st = check_ptr(q, work)) || (st = check_ptr(k, work)) || (st = check_ptr(v, work)) ||
        (st = check_ptr(y, work)) || (st = check_ptr(S, work)) || (st = check_ptr(z, work)))
        return st;
    if (!work) return LA_OK;
    if (steps != nullptr && (reinterpret_cast<uintptr_t>(steps) & 3u) != 0) return LA_ERR_INVALID_ARG;
    if (BH > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    const DeviceInfo *dev = device_info();
    if (!dev) return LA_ERR_CUDA;
    Problem p{q, k, v, y, S, z, BH, T, s.D, s.M, s.dtype, 0, nullptr, 0, (cudaStream_t)stream};
    p.H = s.H;
    p.lens = steps;
    // several steps with known inputs are the causal form over those tokens,
    // starting from the state: the tensor-core kernel reads the step-major
    // tensors through strided tensor maps
    if (tc_causal_supported(s, 0)) {
        p.step_major = true;
        return from_cuda(tc_causal(p, *dev));
    }
    p.lens = nullptr;
    return from_cuda(decode_steps(p, steps, T));
}

la_status la_decode_step(const void *q, const void *k, const void *v, void *y, float *S, float *z,
                         la_shape s, la_stream_t stream) {
    la_status st = check_shape(s, false);
    if (st != LA_OK) return st;
    const long long BH = (long long)s.B * s.H;
    const bool work = BH > 0;
    if ((st = check_ptr(q, work)) || (st = check_ptr(k, work)) || (st = check_ptr(v, work)) ||
        (st = check_ptr(y, work)) || (st = check_ptr(S, work)) || (st = check_ptr(z, work)))
        return st;
    if (!work) return LA_OK;
    if (BH > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    const DeviceInfo *dev = device_info();
    if (!dev) return LA_ERR_CUDA;
    Problem p{q, k, v, y, S, z, BH, 1, s.D, s.M, s.dtype, 0, nullptr, 0, (cudaStream_t)stream};
    return from_cuda(decode_step(p, *dev));
}

int la_feature_dim(la_variant var, int D) {
    if (fw_check_variant(var, D) == LA_ERR_INVALID_ARG) return 0;
    return fw_feature_dim(var, D);
}

size_t la_variant_workspace_bytes(la_op op, la_shape s, la_variant var) {
    if (check_shape(s, op != LA_OP_DECODE) != LA_OK || fw_check_variant(var, s.D) != LA_OK) return (size_t)-1;
    switch (op) {
        case LA_OP_NONCAUSAL: {
            if (var.update != LA_UPDATE_SUM) return (size_t)-1;
            Problem p{};
            if (tc_variant_route(s, var, p)) {   // the tensor-core kernel's exchange slots, feature width F
                la_shape sf = s;
                sf.D = p.D;
                return tc_noncausal_ws_bytes(sf);
            }
            return fw_noncausal_ws_bytes(s, var);
        }
        case LA_OP_CAUSAL:
        case LA_OP_DECODE: return 0;
        default: return (size_t)-1;
    }
}

namespace {

// Checks shared by the causal and decode variants: the variant, the state
// pointers (z only with the denominator) and beta (delta rule).
la_status check_variant_state(const la_shape &s, const la_variant &var, const void *beta, const float *S,
                              const float *z, bool work, bool state_required) {
    la_status st = fw_check_variant(var, s.D);
    if (st != LA_OK) return st;
    const long long BH = (long long)s.B * s.H;
    if (var.norm == LA_NORM_DEN) {
        if ((S == nullptr) != (z == nullptr)) return LA_ERR_INVALID_ARG;
    } else if (z != nullptr) {
        return LA_ERR_INVALID_ARG;
    }
    if (state_required && BH > 0 && S == nullptr) return LA_ERR_INVALID_ARG;
    if ((st = check_ptr(S, S != nullptr && BH > 0)) || (st = check_ptr(z, z != nullptr && BH > 0))) return st;
    if (var.update == LA_UPDATE_DELTA && (st = check_ptr(beta, work)) != LA_OK) return st;
    if (BH > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    return LA_OK;
}

}  // namespace

la_status la_forward_causal_variant(const void *q, const void *k, const void *v, const void *beta, void *out,
                                    la_shape s, la_variant var, float *S, float *z, la_stream_t stream) {
    la_status st = check_shape(s, true);
    if (st != LA_OK) return st;
    const long long BH = (long long)s.B * s.H;
    const bool work = BH > 0 && s.N > 0;
    if ((st = check_variant_state(s, var, beta, S, z, work, false)) != LA_OK) return st;
    if ((st = check_ptr(q, work)) || (st = check_ptr(k, work)) || (st = check_ptr(v, work)) ||
        (st = check_ptr(out, work && out != nullptr)))
        return st;
    if (!work) return LA_OK;   // an empty sequence leaves the state as it is
    if (out != nullptr && (out == q || out == k || out == v || out == beta)) return LA_ERR_INVALID_ARG;
    Problem p{q, k, v, out, S, z, BH, s.N, s.D, s.M, s.dtype, 0, nullptr, 0, (cudaStream_t)stream};
    if (tc_variant_route(s, var, p)) {
        // bf16, sum update, no denominator, F in {64, 128}: the chunked
        // tensor-core kernel with the feature map applied row by row on chip
        const DeviceInfo *dev = device_info();
        if (!dev) return LA_ERR_CUDA;
        return from_cuda(tc_causal(p, *dev));
    }
    if (tc_delta_supported(s, var)) {
        // bf16 delta rule, F = M = 64: chunks of 128 tokens on tensor cores with
        // the triangular solve for the pseudo-values on CUDA cores
        const DeviceInfo *dev = device_info();
        if (!dev) return LA_ERR_CUDA;
        return from_cuda(tc_delta(p, beta, var, *dev));
    }
    return from_cuda(fw_causal(p, var.update == LA_UPDATE_DELTA ? beta : nullptr, var));
}

la_status la_forward_noncausal_variant(const void *q, const void *k, const void *v, void *out, la_shape s,
                                       la_variant var, void *workspace, size_t ws_bytes, la_stream_t stream) {
    la_status st = check_shape(s, true);
    if (st != LA_OK) return st;
    if ((st = fw_check_variant(var, s.D)) != LA_OK) return st;
    if (var.update != LA_UPDATE_SUM) return LA_ERR_UNSUPPORTED;
    const long long BH = (long long)s.B * s.H;
    const bool work = BH > 0 && s.N > 0;
    if ((st = check_ptr(q, work)) || (st = check_ptr(k, work)) || (st = check_ptr(v, work)) ||
        (st = check_ptr(out, work)))
        return st;
    if (!work) return LA_OK;
    if (BH > 0x7fffffffLL) return LA_ERR_UNSUPPORTED;
    if (out == q || out == k || out == v) return LA_ERR_INVALID_ARG;
    const size_t need = la_variant_workspace_bytes(LA_OP_NONCAUSAL, s, var);
    if (ws_bytes < need || (need > 0 && check_ptr(workspace, true) != LA_OK)) return LA_ERR_INVALID_ARG;
    const DeviceInfo *dev = device_info();
    if (!dev) return LA_ERR_CUDA;
    Problem p{q, k, v, out, nullptr, nullptr, BH, s.N, s.D, s.M, s.dtype, 0, workspace, ws_bytes,
              (cudaStream_t)stream};
    // bf16, no denominator, F in {64, 128}: the one-launch tensor-core kernel
    // with the feature map applied row by row on chip
    if (tc_variant_route(s, var, p)) return from_cuda(tc_noncausal(p, *dev));
    return from_cuda(fw_noncausal(p, var, *dev));
}

la_status la_decode_step_variant(const void *q, const void *k, const void *v, const void *beta, void *y,
                                 float *S, float *z, la_shape s, la_variant var, la_stream_t stream) {
    la_status st = check_shape(s, false);
    if (st != LA_OK) return st;
    const long long BH = (long long)s.B * s.H;
    const bool work = BH > 0;
    if ((st = check_variant_state(s, var, beta, S, z, work, true)) != LA_OK) return st;
    if ((st = check_ptr(q, work)) || (st = check_ptr(k, work)) || (st = check_ptr(v, work)) ||
        (st = check_ptr(y, work)))
        return st;
    if (!work) return LA_OK;
    if (y == q || y == k || y == v || y == beta) return LA_ERR_INVALID_ARG;
    // one step is the causal form over a single token, started from (S, z)
    Problem p{q, k, v, y, S, z, BH, 1, s.D, s.M, s.dtype, 0, nullptr, 0, (cudaStream_t)stream};
    return from_cuda(fw_causal(p, var.update == LA_UPDATE_DELTA ? beta : nullptr, var));
}

la_status la_get_last_error(la_stream_t stream) {
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return LA_ERR_CUDA;
    if (cudaGetLastError() != cudaSuccess) return LA_ERR_CUDA;
    int word = 0;
    if (cudaMemcpyFromSymbol(&word, g_la_error_word, sizeof(int)) != cudaSuccess) return LA_ERR_CUDA;
    if (word != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_la_error_word, &zero, sizeof(int)) != cudaSuccess) return LA_ERR_CUDA;
    }
    return (la_status)word;
}

}  // extern "C"

// la_internal.h - host-side declarations shared by the translation units of
// liblinattn.so (argument checking lives in la_api.cu, kernels elsewhere).
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/la.h"

namespace la {

// Cached per-device facts.
struct DeviceInfo {
    int sm_count = 0;
    int cc_major = 0, cc_minor = 0;
    int max_smem_optin = 0;
    int *err_word = nullptr;   // device address of this device's error word
};

// Returns nullptr if the current device cannot be queried.
const DeviceInfo *device_info();

// Problem description shared by the launchers (all sizes already validated).
struct Problem {
    const void *q, *k, *v;
    void *out;                 // may be null (causal: state only)
    float *S, *z;              // causal carry / decode state, may be null (causal)
    long long BH;              // B * H
    int N, D, M;
    la_dtype dtype;
    int chunk;
    void *ws;
    size_t ws_bytes;
    cudaStream_t stream;
    const int *lens = nullptr;   // causal: per-batch sequence lengths (device, [B]) or null
    int H = 1;                   // heads per batch entry (to index lens)
    bool step_major = false;     // causal: q, k, v, out laid out [N][B*H][.] (decode steps)
    // variants on the tensor-core causal kernel (D above is then the feature width F)
    int feat = 0;                // 0: elu + 1; 1: elu + 1 sum-normalised; 2: DPFP (row feature maps)
    int dr = 0, nu = 0;          // raw width of q, k rows and DPFP shifts (feat != 0)
    bool sum_norm = false;       // DPFP: rows divided by their sums
    bool no_den = false;         // output = numerator (no denominator)
    bool no_segments = false;    // causal: one CTA per head (the call has no workspace)
};

// Backward-pass problem (sizes already validated).
struct BwdProblem {
    const void *q, *k, *v, *dout;
    void *dq, *dk, *dv;
    const float *S0, *z0;      // carried-in state of the forward (causal), may be null
    const float *dSN, *dzN;    // gradient reaching the final state (causal), may be null
    float *dS0, *dz0;          // gradient of the carried-in state (causal), may be null
    long long BH;
    int N, D, M;
    la_dtype dtype;
    void *ws;
    size_t ws_bytes;
    cudaStream_t stream;
};

// ---- backward (la_bwd.cu): CUDA cores, any D, M in {16,32,64,128}, fp32 or bf16.
size_t causal_bwd_ws_bytes(const la_shape &s);
size_t noncausal_bwd_ws_bytes(const la_shape &s);
cudaError_t causal_backward(const BwdProblem &p, const DeviceInfo &dev);
cudaError_t noncausal_backward(const BwdProblem &p, const DeviceInfo &dev);
// tensor-core causal backward (la_tc_bwd.cu): bf16, D = M = 64
bool tc_backward_supported(const la_shape &s);
// per-split key sums [S | z] on tensor cores (la_tc.cu), bf16, D, M in {64, 128}
cudaError_t tc_key_sums(const void *k, const void *v, long long BH, int N, int D, int M, int nsplit, int cps,
                        float *ws, size_t ws_bytes, cudaStream_t stream, const DeviceInfo &dev);
// tensor-core non-causal backward (la_tc_bwd_nc.cu): bf16, D, M in {64, 128}
bool tc_nc_backward_supported(const la_shape &s);
size_t tc_nc_backward_ws_bytes(const la_shape &s);
// chunk-parallel tensor-core causal backward (la_tc_bwd_chunk.cu): bf16,
// D, M in {64, 128} other than D = M = 64
bool tc_chunk_backward_supported(const la_shape &s);
size_t tc_chunk_backward_ws_bytes(const la_shape &s);
cudaError_t tc_chunk_causal_backward(const BwdProblem &p, const DeviceInfo &dev);
cudaError_t tc_noncausal_backward(const BwdProblem &p, const DeviceInfo &dev);
cudaError_t tc_causal_backward(const BwdProblem &p, const DeviceInfo &dev);

// ---- SIMT kernels (la_simt.cu): any D, M in {16,32,64,128}, fp32 or bf16.
size_t simt_noncausal_ws_bytes(const la_shape &s);
cudaError_t simt_noncausal(const Problem &p, const DeviceInfo &dev);
cudaError_t simt_causal(const Problem &p, const DeviceInfo &dev);
cudaError_t decode_step(const Problem &p, const DeviceInfo &dev);
// T recurrent steps in one launch, the state held on chip (inputs [T, B*H, .]);
// steps: per-batch step counts (device, [B]) or null (all T)
cudaError_t decode_steps(const Problem &p, const int *steps, int T);
// Same two kernels as simt_noncausal with at most max_splits partial sums in p.ws.
cudaError_t simt_noncausal_capped(const Problem &p, const DeviceInfo &dev, int max_splits);

// ---- tensor-core (tcgen05) kernels (la_tc.cu): bf16, D, M in {64, 128}.
bool tc_causal_supported(const la_shape &s, int chunk);
size_t tc_causal_ws_bytes(const la_shape &s, int chunk);
cudaError_t tc_causal(const Problem &p, const DeviceInfo &dev);
bool tc_noncausal_supported(const la_shape &s);
size_t tc_noncausal_ws_bytes(const la_shape &s);
cudaError_t tc_noncausal(const Problem &p, const DeviceInfo &dev);

// ---- variants (la_fw.cu): feature maps, sum normalisation, delta rule; CUDA cores.
constexpr int kFwMaxFeatures = 512;          // largest feature width F
int fw_feature_dim(const la_variant &v, int D);
la_status fw_check_variant(const la_variant &v, int D);
size_t fw_noncausal_ws_bytes(const la_shape &s, const la_variant &v);
// causal form (also one decode step with N = 1); beta [BH, N] for the delta rule
cudaError_t fw_causal(const Problem &p, const void *beta, const la_variant &v);
cudaError_t fw_noncausal(const Problem &p, const la_variant &v, const DeviceInfo &dev);

// tensor-core route of a sum-update variant, if it has one: fills p.feat, dr,
// nu, sum_norm, no_den and sets p.D to the feature width; false otherwise
bool tc_variant_route(const la_shape &s, const la_variant &v, Problem &p);

// chunked delta rule on tensor cores (la_tc_delta.cu): bf16, sum-normalised
// features of width 64 (elu + 1 at D = 64, DPFP at D = 32 / nu = 1 or
// D = 16 / nu = 2), M = 64
bool tc_delta_supported(const la_shape &s, const la_variant &v);
cudaError_t tc_delta(const Problem &p, const void *beta, const la_variant &v, const DeviceInfo &dev);

// Launches `kernel` with programmatic stream serialization: it may start as
// soon as the previous launch on the stream triggers (explicitly, or
// implicitly as its CTAs exit), its set-up overlapping that launch's tail;
// every such kernel calls pdl_wait_cta() before its first global-memory
// access.  cluster_x
// > 0 also sets a cluster shape (cluster_x, 1, 1) (a cluster kernel keeps its
// cluster launch even at one CTA per cluster).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       unsigned cluster_x, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.numAttrs = 1;
    if (cluster_x > 0) {
        attr[1].id = cudaLaunchAttributeClusterDimension;
        attr[1].val.clusterDim.x = cluster_x;
        attr[1].val.clusterDim.y = 1;
        attr[1].val.clusterDim.z = 1;
        cfg.numAttrs = 2;
    }
    cfg.attrs = attr;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args &&>(args)...);
}

// Counts kernel launches made through the library (la_api.cu).
void count_launches(int n);

// Test hook state (la_api.cu).
extern volatile int g_inject_timeout;
extern volatile int g_inject_limit_us;
// checked build only: the next causal tensor-core launches offset the row of
// their state loads past the state (caught by the bounds checks)
extern volatile int g_inject_bounds;

}  // namespace la

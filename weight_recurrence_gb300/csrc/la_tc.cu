// la_tc.cu - tensor-core (tcgen05) kernels of liblinattn.so.
#include "la_common.cuh"
#include "la_internal.h"

namespace la {

bool tc_causal_supported(const la_shape &, int) { return false; }
size_t tc_causal_ws_bytes(const la_shape &, int) { return 0; }
cudaError_t tc_causal(const Problem &, const DeviceInfo &) { return cudaErrorNotSupported; }
bool tc_noncausal_supported(const la_shape &) { return false; }
size_t tc_noncausal_ws_bytes(const la_shape &) { return 0; }
cudaError_t tc_noncausal(const Problem &, const DeviceInfo &) { return cudaErrorNotSupported; }

}  // namespace la

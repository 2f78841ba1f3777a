// FP8-KV variant of the forward (656-byte rows).  Placeholder until the
// dequantising kernel lands: reports no capacity, so the API returns
// DSA_ERR_UNSUPPORTED for the FP8 entry point.
#include <cuda_runtime.h>

#include "dsa_internal.h"

namespace dsa {
int fwd_fp8_max_active_pairs() { return 0; }
cudaError_t launch_fwd_fp8(const FwdParams&, cudaStream_t) { return cudaErrorNotSupported; }
}  // namespace dsa

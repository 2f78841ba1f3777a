// bf16-KV instantiation of the sparse MLA forward (see dsa_fwd_impl.cuh).
#include "dsa_fwd_impl.cuh"

namespace dsa {
int fwd_max_active_pairs() { return max_active_pairs_impl<fwd::kFmtBf16>(); }
cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream) { return launch_impl<fwd::kFmtBf16>(p, stream); }
}  // namespace dsa

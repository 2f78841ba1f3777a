// FP8-KV instantiation of the sparse MLA forward (see dsa_fwd_impl.cuh): 656-byte
// rows of 512 e4m3 latent codes, 4 fp32 scales and 64 bf16 rope values.
#include "dsa_fwd_impl.cuh"

namespace dsa {
int fwd_fp8_max_active_pairs() { return max_active_pairs_impl<fwd::kFmtFp8>(); }
cudaError_t launch_fwd_fp8(const FwdParams& p, cudaStream_t stream) { return launch_impl<fwd::kFmtFp8>(p, stream); }
}  // namespace dsa

// FP4-KV instantiation of the sparse MLA forward (see dsa_fwd_impl.cuh): 448-byte
// rows of 512 e2m1 latent codes (two per byte), 16 fp32 scales and 64 bf16 rope values.
#include "dsa_fwd_impl.cuh"

namespace dsa {
int fwd_fp4_max_active_pairs() { return max_active_pairs_impl<fwd::kFmtFp4>(); }
cudaError_t launch_fwd_fp4(const FwdParams& p, cudaStream_t stream) { return launch_impl<fwd::kFmtFp4>(p, stream); }
}  // namespace dsa

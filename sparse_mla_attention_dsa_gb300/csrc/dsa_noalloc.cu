// An allocation-free variant of the bf16 forward for callers that cannot
// allocate device memory: code running where cudaMalloc is unavailable or not
// allowed (inside an allocator of its own, a plugin handed only input and
// output buffers, a process whose memory is pinned in advance).  Instead of a
// caller workspace it uses one scratch array compiled into this library.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/dsa.h"
#include "dsa_internal.h"

namespace dsa {

// Limits of the built-in scratch: up to 8192 query tokens, 128 heads and 80 SM
// pairs (a GB300 has 76).  The split-token partial outputs dominate its size
// (about 43 MiB); every GPU that loads the library keeps it until the process exits.
constexpr int kNoAllocMaxTokens = 8192;
constexpr int kNoAllocMaxPairs = 80;
constexpr size_t kNoAllocScratchBytes = workspace_layout(kNoAllocMaxTokens, kMaxHeads, kNoAllocMaxPairs).total;

// One copy per device.  In host code this name stands for the array, it is not
// its device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
static void* g_scratch_addr[kMaxDevices] = {};
static std::mutex g_scratch_mutex;

// Device address of the scratch array on the current device, looked up once per device.
static void* scratch_address(int dev) {
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_scratch_addr[dev] = ptr;
  }
  return g_scratch_addr[dev];
}

}  // namespace dsa

extern "C" dsa_status dsa_sparse_attn_fwd_noalloc(const void* q, const void* kv, const int32_t* indices, int s_q,
                                                  int h_q, int s_kv, int topk, float sm_scale, void* out, float* lse,
                                                  cudaStream_t stream) {
  if (s_q < 0 || h_q < 1 || h_q > dsa::kMaxHeads || s_kv < 0 || topk < 1) return DSA_ERR_INVALID_ARG;
  if (s_q == 0) return DSA_OK;
  if (s_q > dsa::kNoAllocMaxTokens) return DSA_ERR_WORKSPACE;
  const size_t need = dsa_sparse_attn_fwd_workspace_size(s_q, h_q, topk, DSA_KV_BF16);
  if (need == 0) return DSA_ERR_UNSUPPORTED;
  if (need > dsa::kNoAllocScratchBytes) return DSA_ERR_WORKSPACE;  // more SM pairs than the array covers
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= dsa::kMaxDevices) return DSA_ERR_CUDA;
  void* scratch = dsa::scratch_address(dev);
  if (scratch == nullptr) return DSA_ERR_CUDA;
  return dsa_sparse_attn_fwd(q, kv, indices, s_q, h_q, s_kv, topk, sm_scale, out, lse, scratch,
                             dsa::kNoAllocScratchBytes, stream);
}

// Output projection with residual after the attention: y = O . W_o + x
// ("FlashMLA算子Ascend 950移植：从tiling到访存优化全解读", section 3.4, 输出投影与残差合并).
//
// O of a token is the head-major concatenation of its attention output (h_q * 512 bf16 values), W_o is
// [h_q * 512, d_model] and x, y are [s_q, d_model], all row-major bf16.  Over a batch of tokens this is
// one dense GEMM (M = s_q, K = h_q * 512, N = d_model) with the residual as its C operand, run by
// cuBLASLt on the caller's stream right after the attention kernels.  The page keeps O on chip and
// multiplies it there; with all heads of one token on an SM pair that product would be a GEMV per
// token that streams all of W_o (h_q * 512 * d_model values) once per token, so the batched GEMM over
// tokens is the form that reaches the tensor cores; O makes one round trip through memory.
#include <cublasLt.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <vector>

#include "../../include/dsa.h"

namespace {

constexpr size_t kLtWorkspace = 32u << 20;  // cuBLASLt workspace handed to every call
constexpr int kMaxDevices = 64;
constexpr size_t kMaxCachedAlgos = 256;  // distinct (device, shape) entries kept

std::mutex g_mu;
cublasLtHandle_t g_handle[kMaxDevices] = {};

struct AlgoEntry {
  int dev, m, n, k;
  bool residual;
  size_t ws;
  cublasLtMatmulAlgo_t algo;
};
std::vector<AlgoEntry> g_algos;

cublasLtHandle_t handle_for(int dev) {
  std::lock_guard<std::mutex> lk(g_mu);
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  if (!g_handle[dev] && cublasLtCreate(&g_handle[dev]) != CUBLAS_STATUS_SUCCESS) g_handle[dev] = nullptr;
  return g_handle[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// RAII holders for the cuBLASLt descriptors of one call.
struct Descs {
  cublasLtMatmulDesc_t op = nullptr;
  cublasLtMatrixLayout_t a = nullptr, b = nullptr, cd = nullptr;
  cublasLtMatmulPreference_t pref = nullptr;
  ~Descs() {
    if (pref) cublasLtMatmulPreferenceDestroy(pref);
    if (cd) cublasLtMatrixLayoutDestroy(cd);
    if (b) cublasLtMatrixLayoutDestroy(b);
    if (a) cublasLtMatrixLayoutDestroy(a);
    if (op) cublasLtMatmulDescDestroy(op);
  }
};

}  // namespace

extern "C" {

size_t dsa_out_proj_workspace_size(void) { return kLtWorkspace; }

dsa_status dsa_out_proj(const void* o, const void* w_o, const void* x, int s_q, int h_q, int d_model, void* y,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  if (s_q < 0 || h_q < 1 || h_q > DSA_MAX_HEADS || d_model < 8 || (d_model % 8) != 0) return DSA_ERR_INVALID_ARG;
  if (s_q == 0) return DSA_OK;
  if (!o || !w_o || !y) return DSA_ERR_INVALID_ARG;
  if (!aligned16(o) || !aligned16(w_o) || !aligned16(y) || (x && !aligned16(x))) return DSA_ERR_MISALIGNED;
  if (!workspace || workspace_bytes < kLtWorkspace || !aligned16(workspace)) return DSA_ERR_WORKSPACE;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
  cublasLtHandle_t h = handle_for(dev);
  if (!h) return DSA_ERR_UNSUPPORTED;

  // Column-major view of the row-major problem: Y^T [d_model, s_q] = W_o^T [d_model, K] . O^T [K, s_q] + X^T.
  const int m = d_model, n = s_q, k = h_q * DSA_D_V;
  const bool residual = x != nullptr;
  Descs d;
  if (cublasLtMatmulDescCreate(&d.op, CUBLAS_COMPUTE_32F, CUDA_R_32F) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&d.a, CUDA_R_16BF, m, k, m) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&d.b, CUDA_R_16BF, k, n, k) != CUBLAS_STATUS_SUCCESS ||
      cublasLtMatrixLayoutCreate(&d.cd, CUDA_R_16BF, m, n, m) != CUBLAS_STATUS_SUCCESS)
    return DSA_ERR_UNSUPPORTED;

  cublasLtMatmulAlgo_t algo{};
  bool have = false;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    for (const AlgoEntry& e : g_algos)
      if (e.dev == dev && e.m == m && e.n == n && e.k == k && e.residual == residual && e.ws == kLtWorkspace) {
        algo = e.algo;
        have = true;
        break;
      }
  }
  if (!have) {
    if (cublasLtMatmulPreferenceCreate(&d.pref) != CUBLAS_STATUS_SUCCESS) return DSA_ERR_UNSUPPORTED;
    const size_t ws = kLtWorkspace;
    cublasLtMatmulPreferenceSetAttribute(d.pref, CUBLASLT_MATMUL_PREF_MAX_WORKSPACE_BYTES, &ws, sizeof(ws));
    cublasLtMatmulHeuristicResult_t res{};
    int found = 0;
    if (cublasLtMatmulAlgoGetHeuristic(h, d.op, d.a, d.b, d.cd, d.cd, d.pref, 1, &res, &found) !=
            CUBLAS_STATUS_SUCCESS || found < 1)
      return DSA_ERR_UNSUPPORTED;
    algo = res.algo;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_algos.size() >= kMaxCachedAlgos) g_algos.erase(g_algos.begin());  // bounded: oldest shape goes
    g_algos.push_back(AlgoEntry{dev, m, n, k, residual, kLtWorkspace, algo});
  }
  const float alpha = 1.f, beta = residual ? 1.f : 0.f;
  const cublasStatus_t st = cublasLtMatmul(h, d.op, &alpha, w_o, d.a, o, d.b, &beta, residual ? x : y, d.cd, y, d.cd,
                                           &algo, workspace, kLtWorkspace, stream);
  return st == CUBLAS_STATUS_SUCCESS ? DSA_OK : DSA_ERR_CUDA;
}

size_t dsa_sparse_attn_fwd_oproj_workspace_size(int s_q, int h_q, int topk, int kv_format) {
  const size_t attn = dsa_sparse_attn_fwd_workspace_size(s_q, h_q, topk, kv_format);
  if (attn == 0) return 0;
  return (attn + 255) / 256 * 256 + kLtWorkspace;
}

dsa_status dsa_sparse_attn_fwd_oproj(int kv_format, const void* q, const void* kv, const int32_t* indices, int s_q,
                                     int h_q, int s_kv, int topk, float sm_scale, const void* w_o, const void* x,
                                     int d_model, void* out, float* lse, void* y, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream) {
  if (kv_format != DSA_KV_BF16 && kv_format != DSA_KV_FP8 && kv_format != DSA_KV_FP4) return DSA_ERR_INVALID_ARG;
  if (d_model < 8 || (d_model % 8) != 0 || (s_q > 0 && (!w_o || !y))) return DSA_ERR_INVALID_ARG;
  if (s_q == 0) return DSA_OK;
  const size_t attn = dsa_sparse_attn_fwd_workspace_size(s_q, h_q, topk, kv_format);
  if (attn == 0) return h_q < 1 || h_q > DSA_MAX_HEADS || topk < 1 || s_q < 0 ? DSA_ERR_INVALID_ARG : DSA_ERR_UNSUPPORTED;
  const size_t attn_al = (attn + 255) / 256 * 256;
  if (!workspace || workspace_bytes < attn_al + kLtWorkspace) return DSA_ERR_WORKSPACE;
  dsa_status st;
  if (kv_format == DSA_KV_BF16)
    st = dsa_sparse_attn_fwd(q, kv, indices, s_q, h_q, s_kv, topk, sm_scale, out, lse, workspace, attn, stream);
  else if (kv_format == DSA_KV_FP8)
    st = dsa_sparse_attn_fwd_fp8kv(q, kv, indices, s_q, h_q, s_kv, topk, sm_scale, out, lse, workspace, attn, stream);
  else
    st = dsa_sparse_attn_fwd_fp4kv(q, kv, indices, s_q, h_q, s_kv, topk, sm_scale, out, lse, workspace, attn, stream);
  if (st != DSA_OK) return st;
  return dsa_out_proj(out, w_o, x, s_q, h_q, d_model, y, static_cast<uint8_t*>(workspace) + attn_al, kLtWorkspace,
                      stream);
}

}  // extern "C"

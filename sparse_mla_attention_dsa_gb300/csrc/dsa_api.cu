// C ABI of the sparse MLA forward (see include/dsa.h), the scheduling kernel
// that counts valid index slots and lays out the work sequence, and the kernel
// that merges the pieces of tokens split across CTA pairs.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/dsa.h"
#include "dsa_internal.h"

namespace dsa {

int fwd_max_active_pairs();
cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream);
int fwd_fp8_max_active_pairs();
cudaError_t launch_fwd_fp8(const FwdParams& p, cudaStream_t stream);
int fwd_fp4_max_active_pairs();
cudaError_t launch_fwd_fp4(const FwdParams& p, cudaStream_t stream);

// ----------------------------------------------------------------------------
// Scheduling: n_valid per token, then (by the last CTA to finish) the prefix
// sum of index blocks per token, max(1, ceil(n_valid / 128)).  A token with no
// valid slot still owns one (fully masked) block, which writes out = 0 and
// lse = -inf.  Per-CTA load balance follows the weight idea of
// "Flash Attention Infer算子性能优化", section "优化多核负载均衡": work is
// weighted by valid blocks.  With few tokens per SM pair the pairs take equal
// contiguous shares of the block sequence; with many, they take whole tokens
// from a shared counter, and this kernel clears the per-pair token records.
// ----------------------------------------------------------------------------
constexpr int kPrepWarps = 8;

__global__ void __launch_bounds__(kPrepWarps * 32) dsa_prep_kernel(const FwdParams p) {
  __shared__ int is_last;
  __shared__ int part[kPrepWarps * 32];
  const int s_q = p.s_q, topk = p.topk;
  int* nvalid = p.nvalid;
  int* cum = p.cum;
  int* ctrl = p.ctrl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kPrepWarps + warp;
  if (t < s_q) {
    const int32_t* row = p.indices + (size_t)t * topk;
    int c = 0;
    if (p.pg.block_table == nullptr) {  // flat layout: a row id is valid inside [0, s_kv)
      const int s_kv = p.s_kv;
#pragma unroll 4
      for (int i = lane; i < topk; i += 32) {
        const int v = __ldg(row + i);
        c += (v >= 0 && v < s_kv) ? 1 : 0;
      }
    } else {
      const int seq = token_seq(p, t);
      for (int i = lane; i < topk; i += 32) c += resolve_row(p, seq, __ldg(row + i)) >= 0 ? 1 : 0;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if (lane == 0) nvalid[t] = c;
  }
  if (p.dyn) {  // the per-pair token records start empty
    const size_t n = (size_t)p.npairs * (size_t)(s_q + 1);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
      p.seq[i] = 0;
  }
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) is_last = (atomicAdd(&ctrl[kCtrlTicket], 1) == (int)gridDim.x - 1);
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  // exclusive scan of blocks-per-token over all tokens (one CTA)
  const int nthr = blockDim.x;
  const int per = (s_q + nthr - 1) / nthr;
  const int t0 = threadIdx.x * per, t1 = min(s_q, t0 + per);
  int local = 0;
  for (int i = t0; i < t1; ++i) {
    const int nv = __ldcg(nvalid + i);
    local += max(1, (nv + kBT - 1) / kBT);
  }
  part[threadIdx.x] = local;
  __syncthreads();
  for (int off = 1; off < nthr; off <<= 1) {
    const int v = threadIdx.x >= off ? part[threadIdx.x - off] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int run = part[threadIdx.x] - local;  // exclusive prefix
  for (int i = t0; i < t1; ++i) {
    cum[i] = run;
    const int nv = __ldcg(nvalid + i);
    run += max(1, (nv + kBT - 1) / kBT);
  }
  if (threadIdx.x == nthr - 1) {
    cum[s_q] = part[nthr - 1];
    ctrl[kCtrlTotalBlocks] = part[nthr - 1];
  }
}

// ----------------------------------------------------------------------------
// Merge of split tokens.  Each piece j of a token holds out_j = O_j / Z_j
// (normalised over its own blocks) and lse_j = ln Z_j (plus its max); then
//   lse = ln sum_j exp(lse_j),   out = sum_j exp(lse_j - lse) * out_j.
// This step is not on the pages; it makes the blockwise result of several
// pair ranges equal to the result of one range (same exact value).
// CTA (p, y) handles heads [8y, 8y + 8) of the token containing boundary
// b_p = p*T/P when b_p is the first boundary strictly inside it; one warp per
// head, 16 output columns per lane.
// ----------------------------------------------------------------------------
__device__ __forceinline__ long long boundary(int p, long long T, int P) { return (long long)p * T / P; }

constexpr int kCombineWarps = 8;

// Largest t in [0, s_q) with cum[t] <= key (cum ascending, cum[0] = 0 <= key): 32-way search by one warp.
__device__ int find_token(const int* cum, int s_q, long long key, int lane) {
  int lo = 0, hi = s_q - 1;  // answer in [lo, hi]
  while (hi > lo) {
    const int span = hi - lo;
    const int step = (span + 31) / 32;
    const int pos = lo + lane * step;
    const bool le = pos <= hi && (long long)__ldg(cum + pos) <= key;
    const unsigned m = __ballot_sync(0xffffffffu, le);
    const int last = 31 - __clz(m);                  // lane 0 always qualifies (pos = lo)
    lo = lo + last * step;
    hi = min(hi, lo + step - 1);
  }
  return lo;
}

__global__ void __launch_bounds__(kCombineWarps * 32) dsa_combine_kernel(const int* __restrict__ cum,
                                                                         const int* __restrict__ ctrl, int s_q, int h_q,
                                                                         int npairs, const float* __restrict__ part_lse,
                                                                         const float* __restrict__ part_o, uint16_t* out,
                                                                         float* lse, int dyn) {
  if (dyn) return;  // whole tokens only: nothing was split
  __shared__ int tok_s;
  __shared__ long long c0_s, c1_s;
  const int p = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long T = ctrl[kCtrlTotalBlocks];
  if (warp == 0) {
    int tok = -1;
    long long c0 = 0, c1 = 0;
    const long long bp = boundary(p, T, npairs);
    if (p > 0 && bp < T) {
      const int t = find_token(cum, s_q, bp, lane);
      c0 = cum[t];
      c1 = cum[t + 1];
      // split at bp, and bp is the first boundary inside t
      if (bp != c0 && boundary(p - 1, T, npairs) <= c0) tok = t;
    }
    if (lane == 0) { tok_s = tok; c0_s = c0; c1_s = c1; }
  }
  __syncthreads();
  const int t = tok_s;
  const int h = blockIdx.y * kCombineWarps + warp;
  if (t < 0 || h >= h_q) return;
  const long long c0 = c0_s, c1 = c1_s;
  // pairs covering blocks c0 .. c1-1: pair(g) = ((g + 1) * P - 1) / T; a pair whose range starts inside t
  // holds t as its first piece (slot 2q), otherwise as its second (slot 2q + 1)
  const int pfirst = (int)(((c0 + 1) * npairs - 1) / T);
  const int plast = (int)((c1 * npairs - 1) / T);
  auto slot_lse = [&](int q, int& slot) -> float {
    const long long bq = boundary(q, T, npairs), bq1 = boundary(q + 1, T, npairs);
    if (bq1 <= bq) { slot = -1; return -INFINITY; }  // empty range
    slot = (bq >= c0) ? 2 * q : 2 * q + 1;
    return __ldg(part_lse + (size_t)slot * h_q + h);
  };
  float m = -INFINITY;
  for (int q = pfirst + lane; q <= plast; q += 32) {
    int sl;
    m = fmaxf(m, slot_lse(q, sl));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float wsum = 0.f;
  float4 acc[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
  const int d0 = lane * 16;
  for (int q = pfirst; q <= plast; ++q) {
    int sl;
    const float l = slot_lse(q, sl);
    if (sl < 0 || m == -INFINITY) continue;
    const float w = expf(l - m);
    wsum += w;
    const float4* src = reinterpret_cast<const float4*>(part_o + ((size_t)sl * h_q + h) * kDV + d0);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float4 v = __ldg(src + u);
      acc[u].x += w * v.x; acc[u].y += w * v.y; acc[u].z += w * v.z; acc[u].w += w * v.w;
    }
  }
  const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
  uint32_t pk[8];
#pragma unroll
  for (int u = 0; u < 4; ++u) {
    pk[2 * u] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[u].x * inv)) |
                ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[u].y * inv)) << 16);
    pk[2 * u + 1] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[u].z * inv)) |
                    ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(acc[u].w * inv)) << 16);
  }
  uint4* dst = reinterpret_cast<uint4*>(out + ((size_t)t * h_q + h) * kDV + d0);
  dst[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
  dst[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
  if (lane == 0) lse[(size_t)t * h_q + h] = (wsum > 0.f) ? m + logf(wsum) : -INFINITY;
}

// Output for s_kv == 0: no row can be valid.
__global__ void dsa_fill_empty_kernel(uint16_t* out, float* lse, size_t n_out, size_t n_lse) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  for (size_t k = i; k < n_out; k += stride) out[k] = 0;
  for (size_t k = i; k < n_lse; k += stride) lse[k] = -INFINITY;
}

static bool device_ok() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  return major == 10 && minor == 3;
}

static int pairs_for(int kv_format) {
  return kv_format == DSA_KV_FP8 ? fwd_fp8_max_active_pairs()
         : kv_format == DSA_KV_FP4 ? fwd_fp4_max_active_pairs()
                                   : fwd_max_active_pairs();
}

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

static cudaEvent_t g_ev_before = nullptr, g_ev_after = nullptr;

static dsa_status forward(int kv_format, const void* q, const void* kv, const int32_t* indices, int s_q, int h_q,
                          int s_kv, int topk, float sm_scale, void* out, float* lse, void* workspace,
                          size_t workspace_bytes, cudaStream_t stream, const PagedView* pg = nullptr) {
  if (s_q < 0 || h_q < 1 || h_q > kMaxHeads || s_kv < 0 || topk < 1 || !std::isfinite(sm_scale))
    return DSA_ERR_INVALID_ARG;
  if (s_q == 0) return DSA_OK;
  if (!q || !indices || !out || !lse || (s_kv > 0 && !kv)) return DSA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(out) || !aligned16(lse) || !aligned16(indices) || (kv && !aligned16(kv)))
    return DSA_ERR_MISALIGNED;
  if (!device_ok()) return DSA_ERR_UNSUPPORTED;
  const int npairs = pairs_for(kv_format);
  if (npairs <= 0) return DSA_ERR_UNSUPPORTED;
  const WorkspaceLayout L = workspace_layout(s_q, h_q, npairs);
  if (!workspace || workspace_bytes < L.total || !aligned16(workspace)) return DSA_ERR_WORKSPACE;
  if (s_kv == 0) {
    if (cudaMemsetAsync(workspace, 0, 256, stream) != cudaSuccess) return DSA_ERR_CUDA;
    const size_t n_out = (size_t)s_q * h_q * kDV, n_lse = (size_t)s_q * h_q;
    dsa_fill_empty_kernel<<<256, 256, 0, stream>>>((uint16_t*)out, lse, n_out, n_lse);
    return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
  }

  uint8_t* ws = (uint8_t*)workspace;
  FwdParams p;
  p.q = (const uint16_t*)q;
  p.kv = (const uint8_t*)kv;
  p.indices = indices;
  p.out = (uint16_t*)out;
  p.lse = lse;
  p.s_q = s_q;
  p.h_q = h_q;
  p.s_kv = s_kv;
  p.topk = topk;
  p.scale_log2 = sm_scale * 1.4426950408889634f;
  p.pg = pg ? *pg : PagedView{nullptr, nullptr, 1, 1, 1};
  p.ctrl = (int*)(ws + L.ctrl);
  p.nvalid = (int*)(ws + L.nvalid);
  p.cum = (int*)(ws + L.cum);
  p.seq = (int*)(ws + L.seq);
  p.dyn = s_q >= kDynTokensPerPair * npairs ? 1 : 0;
  p.part_lse = (float*)(ws + L.part_lse);
  p.part_o = (float*)(ws + L.part_o);
  p.npairs = npairs;

  if (cudaMemsetAsync(p.ctrl, 0, 256, stream) != cudaSuccess) return DSA_ERR_CUDA;
  const int prep_blocks = (s_q + kPrepWarps - 1) / kPrepWarps;
  dsa_prep_kernel<<<prep_blocks, kPrepWarps * 32, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return DSA_ERR_CUDA;

  cudaError_t e;
  const bool timed = g_ev_before != nullptr && g_ev_after != nullptr;
  if (timed) cudaEventRecord(g_ev_before, stream);
  e = (kv_format == DSA_KV_BF16)  ? launch_fwd_bf16(p, stream)
      : (kv_format == DSA_KV_FP8) ? launch_fwd_fp8(p, stream)
                                  : launch_fwd_fp4(p, stream);
  if (timed) cudaEventRecord(g_ev_after, stream);
  if (e != cudaSuccess) return DSA_ERR_CUDA;
  const dim3 cgrid((unsigned)npairs, (unsigned)((h_q + kCombineWarps - 1) / kCombineWarps));
  dsa_combine_kernel<<<cgrid, kCombineWarps * 32, 0, stream>>>(p.cum, p.ctrl, s_q, h_q, npairs, p.part_lse, p.part_o,
                                                               (uint16_t*)out, lse, p.dyn);
  return cudaGetLastError() == cudaSuccess ? DSA_OK : DSA_ERR_CUDA;
}

}  // namespace dsa

extern "C" {

size_t dsa_sparse_attn_fwd_workspace_size(int s_q, int h_q, int topk, int kv_format) {
  if (s_q < 0 || h_q < 1 || h_q > dsa::kMaxHeads || topk < 1) return 0;
  if (kv_format != DSA_KV_BF16 && kv_format != DSA_KV_FP8 && kv_format != DSA_KV_FP4) return 0;
  const int npairs = dsa::pairs_for(kv_format);
  if (npairs <= 0) return 0;
  return dsa::workspace_layout(s_q, h_q, npairs).total;
}

dsa_status dsa_sparse_attn_fwd(const void* q, const void* kv, const int32_t* indices, int s_q, int h_q, int s_kv,
                               int topk, float sm_scale, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream) {
  return dsa::forward(DSA_KV_BF16, q, kv, indices, s_q, h_q, s_kv, topk, sm_scale, out, lse, workspace,
                      workspace_bytes, stream);
}

dsa_status dsa_sparse_attn_fwd_fp8kv(const void* q, const void* kv_fp8, const int32_t* indices, int s_q, int h_q,
                                     int s_kv, int topk, float sm_scale, void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream) {
  return dsa::forward(DSA_KV_FP8, q, kv_fp8, indices, s_q, h_q, s_kv, topk, sm_scale, out, lse, workspace,
                      workspace_bytes, stream);
}

dsa_status dsa_sparse_attn_fwd_paged(int kv_format, const void* q, const void* kv_pool, const int32_t* indices,
                                     const int32_t* seq_of_token, const int32_t* block_table, int s_q, int h_q,
                                     int n_rows, int topk, int n_seq, int max_pages, int page_size, float sm_scale,
                                     void* out, float* lse, void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream) {
  if (kv_format != DSA_KV_BF16 && kv_format != DSA_KV_FP8 && kv_format != DSA_KV_FP4) return DSA_ERR_INVALID_ARG;
  if (n_seq < 1 || max_pages < 1 || page_size < 1 || (long long)n_seq * max_pages > 0x7fffffffLL)
    return DSA_ERR_INVALID_ARG;
  if (s_q > 0 && (!seq_of_token || !block_table)) return DSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(seq_of_token) & 3u) || (reinterpret_cast<uintptr_t>(block_table) & 3u))
    return DSA_ERR_MISALIGNED;
  const dsa::PagedView pg{block_table, seq_of_token, page_size, max_pages, n_seq};
  return dsa::forward(kv_format, q, kv_pool, indices, s_q, h_q, n_rows, topk, sm_scale, out, lse, workspace,
                      workspace_bytes, stream, &pg);
}

dsa_status dsa_sparse_attn_fwd_fp4kv(const void* q, const void* kv_fp4, const int32_t* indices, int s_q, int h_q,
                                     int s_kv, int topk, float sm_scale, void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream) {
  return dsa::forward(DSA_KV_FP4, q, kv_fp4, indices, s_q, h_q, s_kv, topk, sm_scale, out, lse, workspace,
                      workspace_bytes, stream);
}

dsa_status dsa_read_device_status(const void* workspace, cudaStream_t stream) {
  if (!workspace) return DSA_ERR_WORKSPACE;
  int st = 0;
  if (cudaMemcpyAsync(&st, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return DSA_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DSA_ERR_CUDA;
  return (dsa_status)st;
}

const char* dsa_status_string(dsa_status s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED";
    case DSA_ERR_MISALIGNED: return "DSA_ERR_MISALIGNED";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_TIMEOUT: return "DSA_ERR_DEVICE_TIMEOUT";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
  }
  return "DSA_ERR_UNKNOWN";
}

int dsa_kernels_per_call(void) { return 3; }

void dsa_set_timing_events(cudaEvent_t before, cudaEvent_t after) {
  dsa::g_ev_before = before;
  dsa::g_ev_after = after;
}

}  // extern "C"

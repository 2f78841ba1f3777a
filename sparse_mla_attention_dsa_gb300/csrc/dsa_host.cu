// Forward from host buffers: the query tokens go through the GPU in chunks, with the host-to-device
// copy of chunk i+1, the forward of chunk i and the device-to-host copy of chunk i-1 in flight at once
// (two copy streams beside the caller's stream, two sets of chunk buffers in the caller's device
// buffer).  This is runtime plumbing around the forward, not part of the method: the pages compute on
// device memory only.
#include <cuda_runtime.h>

#include <cstdint>
#include <utility>
#include <vector>

#include "../../include/dsa.h"

namespace {

constexpr size_t kAlign = 256;
size_t up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

size_t row_bytes(int kv_format) {
  return kv_format == DSA_KV_BF16 ? 2u * DSA_D_QK : kv_format == DSA_KV_FP8 ? DSA_FP8_ROW_BYTES : DSA_FP4_ROW_BYTES;
}

struct HostLayout {
  size_t status, ws, ws_bytes, kv, q[2], idx[2], out[2], lse[2], total;
};

// Token ranges of the chunks: the first and the last chunk are half size, so that the upload before the
// first forward and the download after the last one (the parts no compute hides) are short; the rest are
// `chunk` tokens.  One chunk when s_q <= chunk.
std::vector<std::pair<int, int>> chunk_plan(int s_q, int chunk) {
  std::vector<std::pair<int, int>> v;
  if (s_q <= chunk) {
    v.emplace_back(0, s_q);
    return v;
  }
  const int half = chunk / 2 > 0 ? chunk / 2 : 1;
  int t = 0;
  v.emplace_back(t, half);
  t += half;
  while (s_q - t > chunk + half) {
    v.emplace_back(t, chunk);
    t += chunk;
  }
  const int rest = s_q - t;  // in (0, chunk + half]
  if (rest > half) {
    v.emplace_back(t, rest - half);
    t += rest - half;
    v.emplace_back(t, half);
  } else {
    v.emplace_back(t, rest);
  }
  return v;
}

// Device buffer: one status word per chunk, the forward workspace, the whole KV, then two sets of chunk
// buffers (q, indices, out, lse).  Every region starts on a 256-byte boundary.
HostLayout host_layout(int kv_format, int s_q, int h_q, int s_kv, int topk, int chunk) {
  HostLayout L{};
  const int nchunks = (int)chunk_plan(s_q, chunk).size();
  size_t off = 0;
  L.status = off; off += up(sizeof(int) * (size_t)nchunks);
  L.ws = off;
  L.ws_bytes = dsa_sparse_attn_fwd_workspace_size(chunk, h_q, topk, kv_format);
  off += up(L.ws_bytes);
  L.kv = off;     off += up((size_t)s_kv * row_bytes(kv_format));
  for (int b = 0; b < 2; ++b) {
    L.q[b] = off;   off += up((size_t)chunk * h_q * DSA_D_QK * 2);
    L.idx[b] = off; off += up((size_t)chunk * topk * sizeof(int32_t));
    L.out[b] = off; off += up((size_t)chunk * h_q * DSA_D_V * 2);
    L.lse[b] = off; off += up((size_t)chunk * h_q * sizeof(float));
  }
  L.total = L.ws_bytes ? off : 0;
  return L;
}

dsa_status forward_chunk(int kv_format, const void* q, const void* kv, const int32_t* idx, int n, int h_q, int s_kv,
                         int topk, float sm_scale, void* out, float* lse, void* ws, size_t ws_bytes,
                         cudaStream_t stream) {
  if (kv_format == DSA_KV_BF16)
    return dsa_sparse_attn_fwd(q, kv, idx, n, h_q, s_kv, topk, sm_scale, out, lse, ws, ws_bytes, stream);
  if (kv_format == DSA_KV_FP8)
    return dsa_sparse_attn_fwd_fp8kv(q, kv, idx, n, h_q, s_kv, topk, sm_scale, out, lse, ws, ws_bytes, stream);
  return dsa_sparse_attn_fwd_fp4kv(q, kv, idx, n, h_q, s_kv, topk, sm_scale, out, lse, ws, ws_bytes, stream);
}

// The copy streams and events of one call.  The call synchronises before it returns, so they are idle
// when released.
struct Pipe {
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t start = nullptr, kv = nullptr, in[2] = {}, comp[2] = {}, out[2] = {};
  bool ok = true;
  Pipe() {
    ok &= cudaStreamCreateWithFlags(&h2d, cudaStreamNonBlocking) == cudaSuccess;
    ok &= cudaStreamCreateWithFlags(&d2h, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t* e : {&start, &kv, &in[0], &in[1], &comp[0], &comp[1], &out[0], &out[1]})
      ok &= cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
  }
  ~Pipe() {
    for (cudaEvent_t e : {start, kv, in[0], in[1], comp[0], comp[1], out[0], out[1]})
      if (e) cudaEventDestroy(e);
    if (h2d) cudaStreamDestroy(h2d);
    if (d2h) cudaStreamDestroy(d2h);
  }
  // waits for everything this call queued; false if any of it failed
  bool drain(cudaStream_t stream) const {
    bool good = true;
    if (h2d) good &= cudaStreamSynchronize(h2d) == cudaSuccess;
    if (d2h) good &= cudaStreamSynchronize(d2h) == cudaSuccess;
    good &= cudaStreamSynchronize(stream) == cudaSuccess;
    return good;
  }
};

}  // namespace

extern "C" {

size_t dsa_sparse_attn_fwd_host_device_bytes(int kv_format, int s_q, int h_q, int s_kv, int topk, int chunk_tokens) {
  if (kv_format != DSA_KV_BF16 && kv_format != DSA_KV_FP8 && kv_format != DSA_KV_FP4) return 0;
  if (s_q < 1 || h_q < 1 || h_q > DSA_MAX_HEADS || s_kv < 0 || topk < 1 || chunk_tokens < 1) return 0;
  const int chunk = chunk_tokens < s_q ? chunk_tokens : s_q;
  return host_layout(kv_format, s_q, h_q, s_kv, topk, chunk).total;
}

dsa_status dsa_sparse_attn_fwd_host(int kv_format, const void* q_host, const void* kv_host,
                                    const int32_t* indices_host, int s_q, int h_q, int s_kv, int topk, float sm_scale,
                                    void* out_host, float* lse_host, void* device_buffer, size_t device_bytes,
                                    int chunk_tokens, cudaStream_t stream) {
  if (kv_format != DSA_KV_BF16 && kv_format != DSA_KV_FP8 && kv_format != DSA_KV_FP4) return DSA_ERR_INVALID_ARG;
  if (s_q < 0 || h_q < 1 || h_q > DSA_MAX_HEADS || s_kv < 0 || topk < 1 || chunk_tokens < 1 || !(sm_scale == sm_scale))
    return DSA_ERR_INVALID_ARG;
  if (s_q == 0) return DSA_OK;
  if (!q_host || !indices_host || !out_host || !lse_host || (s_kv > 0 && !kv_host)) return DSA_ERR_INVALID_ARG;
  const int chunk = chunk_tokens < s_q ? chunk_tokens : s_q;
  const HostLayout L = host_layout(kv_format, s_q, h_q, s_kv, topk, chunk);
  if (L.total == 0) return DSA_ERR_UNSUPPORTED;
  if (!device_buffer || device_bytes < L.total || (reinterpret_cast<uintptr_t>(device_buffer) & 15u))
    return DSA_ERR_WORKSPACE;

  Pipe pp;
  if (!pp.ok) return DSA_ERR_CUDA;
  uint8_t* dev = static_cast<uint8_t*>(device_buffer);
  int* status_dev = reinterpret_cast<int*>(dev + L.status);
  const size_t q_tok = (size_t)h_q * DSA_D_QK * 2, idx_tok = (size_t)topk * sizeof(int32_t),
               out_tok = (size_t)h_q * DSA_D_V * 2, lse_tok = (size_t)h_q * sizeof(float);
  const std::vector<std::pair<int, int>> plan = chunk_plan(s_q, chunk);
  const int nchunks = (int)plan.size();
  auto ck = [](cudaError_t e) { return e == cudaSuccess; };
  dsa_status result = DSA_OK;
  bool ok = true;

  // the copies start after the work already queued on the caller's stream (an earlier use of the buffer)
  ok &= ck(cudaEventRecord(pp.start, stream));
  ok &= ck(cudaStreamWaitEvent(pp.h2d, pp.start, 0)) && ck(cudaStreamWaitEvent(pp.d2h, pp.start, 0));
  if (ok && s_kv > 0)
    ok &= ck(cudaMemcpyAsync(dev + L.kv, kv_host, (size_t)s_kv * row_bytes(kv_format), cudaMemcpyHostToDevice, pp.h2d));
  ok &= ck(cudaEventRecord(pp.kv, pp.h2d));
  ok &= ck(cudaStreamWaitEvent(stream, pp.kv, 0));
  for (int i = 0; i < nchunks && ok; ++i) {
    const int b = i & 1, t0 = plan[(size_t)i].first, n = plan[(size_t)i].second;
    // inputs of chunk i into buffer set b once chunk i-2's forward has read it
    if (i >= 2) ok &= ck(cudaStreamWaitEvent(pp.h2d, pp.comp[b], 0));
    ok &= ck(cudaMemcpyAsync(dev + L.q[b], static_cast<const uint8_t*>(q_host) + t0 * q_tok, n * q_tok,
                             cudaMemcpyHostToDevice, pp.h2d));
    ok &= ck(cudaMemcpyAsync(dev + L.idx[b], reinterpret_cast<const uint8_t*>(indices_host) + t0 * idx_tok,
                             n * idx_tok, cudaMemcpyHostToDevice, pp.h2d));
    ok &= ck(cudaEventRecord(pp.in[b], pp.h2d));
    // forward of chunk i once its inputs are in and chunk i-2's outputs have left buffer set b
    ok &= ck(cudaStreamWaitEvent(stream, pp.in[b], 0));
    if (i >= 2) ok &= ck(cudaStreamWaitEvent(stream, pp.out[b], 0));
    if (!ok) break;
    result = forward_chunk(kv_format, dev + L.q[b], dev + L.kv, reinterpret_cast<const int32_t*>(dev + L.idx[b]), n,
                           h_q, s_kv, topk, sm_scale, dev + L.out[b], reinterpret_cast<float*>(dev + L.lse[b]),
                           dev + L.ws, L.ws_bytes, stream);
    if (result != DSA_OK) break;
    // the device status this chunk's forward left in the workspace (the next forward resets it)
    ok &= ck(cudaMemcpyAsync(status_dev + i, dev + L.ws, sizeof(int), cudaMemcpyDeviceToDevice, stream));
    ok &= ck(cudaEventRecord(pp.comp[b], stream));
    // outputs of chunk i back to the host
    ok &= ck(cudaStreamWaitEvent(pp.d2h, pp.comp[b], 0));
    ok &= ck(cudaMemcpyAsync(static_cast<uint8_t*>(out_host) + t0 * out_tok, dev + L.out[b], n * out_tok,
                             cudaMemcpyDeviceToHost, pp.d2h));
    ok &= ck(cudaMemcpyAsync(reinterpret_cast<uint8_t*>(lse_host) + t0 * lse_tok, dev + L.lse[b], n * lse_tok,
                             cudaMemcpyDeviceToHost, pp.d2h));
    ok &= ck(cudaEventRecord(pp.out[b], pp.d2h));
  }
  // the caller's stream passes this call only after the last copies back
  for (int b = 0; b < 2 && b < nchunks; ++b) ok &= ck(cudaStreamWaitEvent(stream, pp.out[b], 0));
  if (!pp.drain(stream)) ok = false;
  if (result != DSA_OK) return result;
  if (!ok) return DSA_ERR_CUDA;
  std::vector<int> st((size_t)nchunks, 0);
  if (cudaMemcpy(st.data(), status_dev, sizeof(int) * (size_t)nchunks, cudaMemcpyDeviceToHost) != cudaSuccess)
    return DSA_ERR_CUDA;
  for (int s : st)
    if (s != DSA_OK) return (dsa_status)s;
  return DSA_OK;
}

}  // extern "C"

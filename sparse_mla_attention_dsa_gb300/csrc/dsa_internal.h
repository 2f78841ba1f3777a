// Internal definitions shared by the host API and the kernels of the sparse MLA
// forward (not part of the public C ABI).
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace dsa {

constexpr int kDQK = 576;        // latent 512 + rope 64
constexpr int kDV = 512;         // output channels (first 512 KV columns)
constexpr int kBT = 128;         // B_TOPK: index block processed per step
constexpr int kMaxHeads = 128;   // the MMA M dimension; smaller h_q is padded
constexpr int kFp8RowBytes = 656;

// Workspace layout.  ctrl[] words:
enum CtrlWord { kCtrlStatus = 0, kCtrlTicket = 1, kCtrlTotalBlocks = 2, kCtrlWords = 64 };

struct WorkspaceLayout {
  size_t ctrl, nvalid, cum, part_lse, part_o, total;
};

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr WorkspaceLayout workspace_layout(int s_q, int h_q, int npairs) {
  WorkspaceLayout L{};
  size_t off = 0;
  L.ctrl = off;     off += 256;
  L.nvalid = off;   off += align_up(sizeof(int) * (size_t)(s_q > 0 ? s_q : 1), 256);
  L.cum = off;      off += align_up(sizeof(int) * (size_t)(s_q + 1), 256);
  L.part_lse = off; off += align_up(sizeof(float) * 2 * (size_t)npairs * h_q, 256);
  L.part_o = off;   off += align_up(sizeof(float) * 2 * (size_t)npairs * h_q * kDV, 256);
  L.total = off;
  return L;
}

// Everything a forward launch needs (device pointers).
struct FwdParams {
  const uint16_t* q;         // bf16 bits [s_q, h_q, 576]
  const uint8_t* kv;         // bf16 rows [s_kv, 576] or fp8 rows [s_kv, 656]
  const int32_t* indices;    // [s_q, topk]
  uint16_t* out;             // bf16 bits [s_q, h_q, 512]
  float* lse;                // [s_q, h_q]
  int s_q, h_q, s_kv, topk;
  float scale_log2;          // sm_scale * log2(e)
  int* ctrl;
  int* nvalid;               // [s_q] valid slots per token
  int* cum;                  // [s_q + 1] prefix sum of index blocks per token
  float* part_lse;           // [2 * npairs, h_q]
  float* part_o;             // [2 * npairs, h_q, 512]
  int npairs;
};

// Wait limit for every bounded wait inside the kernels.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s

}  // namespace dsa

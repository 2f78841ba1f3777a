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
enum CtrlWord { kCtrlStatus = 0, kCtrlTicket = 1, kCtrlTotalBlocks = 2, kCtrlNextToken = 3, kCtrlWords = 64 };

struct WorkspaceLayout {
  size_t ctrl, nvalid, cum, seq, part_lse, part_o, total;
};

// Token scheduling: with at least this many tokens per SM pair, pairs take whole tokens from a shared
// counter as they go (so a pair on a slower SM takes fewer); below it, each pair gets an equal static
// share of the index blocks and tokens cut by a share boundary are merged afterwards.
constexpr int kDynTokensPerPair = 8;

constexpr size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

constexpr WorkspaceLayout workspace_layout(int s_q, int h_q, int npairs) {
  WorkspaceLayout L{};
  size_t off = 0;
  L.ctrl = off;     off += 256;
  L.nvalid = off;   off += align_up(sizeof(int) * (size_t)(s_q > 0 ? s_q : 1), 256);
  L.cum = off;      off += align_up(sizeof(int) * (size_t)(s_q + 1), 256);
  L.seq = off;      off += align_up(sizeof(int) * (size_t)npairs * (size_t)(s_q + 1), 256);
  L.part_lse = off; off += align_up(sizeof(float) * 2 * (size_t)npairs * h_q, 256);
  L.part_o = off;   off += align_up(sizeof(float) * 2 * (size_t)npairs * h_q * kDV, 256);
  L.total = off;
  return L;
}

// Paged KV cache ("Flash Attention Infer算子性能优化", section "优化Paged Attention路径"):
// indices are logical positions of the token's sequence, reached through a
// block table of physical pages of the row pool.  block_table == nullptr means
// the flat layout (indices are pool rows).
struct PagedView {
  const int32_t* block_table;   // [n_seq, max_pages] physical page of each logical page, < 0 = unmapped
  const int32_t* seq_of_token;  // [s_q] sequence of each query token
  int page_size, max_pages, n_seq;
};

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
  int* seq;                  // [npairs][s_q + 1] tokens each pair took, in order, as t + 1; -1 = none left
  int dyn;                   // 1: pairs take whole tokens from ctrl[kCtrlNextToken]; 0: static shares
  float* part_lse;           // [2 * npairs, h_q]
  float* part_o;             // [2 * npairs, h_q, 512]
  int npairs;
  PagedView pg;
};

#ifdef __CUDACC__
// Sequence of token t for the paged layout (-1 when outside [0, n_seq)); 0 for the flat layout.
__device__ __forceinline__ int token_seq(const FwdParams& p, int t) {
  if (p.pg.block_table == nullptr) return 0;
  const int s = __ldg(p.pg.seq_of_token + t);
  return (s >= 0 && s < p.pg.n_seq) ? s : -1;
}

// Pool row of index v of a token of sequence `seq`, or -1 when v names no row: outside [0, s_kv) in the
// flat layout; negative, past the block table, on an unmapped page, in an unknown sequence or outside the
// pool in the paged layout (row = table[seq][v / page_size] * page_size + v % page_size).
__device__ __forceinline__ int resolve_row(const FwdParams& p, int seq, int v) {
  if (p.pg.block_table == nullptr) return (v >= 0 && v < p.s_kv) ? v : -1;
  if (v < 0 || seq < 0) return -1;
  const int lp = v / p.pg.page_size;
  if (lp >= p.pg.max_pages) return -1;
  const int ph = __ldg(p.pg.block_table + (size_t)seq * p.pg.max_pages + lp);
  if (ph < 0) return -1;
  const long long row = (long long)ph * p.pg.page_size + (v - lp * p.pg.page_size);
  return row < (long long)p.s_kv ? (int)row : -1;
}
#endif

// Wait limit for every bounded wait inside the kernels.
constexpr unsigned long long kWaitLimitNs = 4000000000ull;  // 4 s

}  // namespace dsa

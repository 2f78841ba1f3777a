// The sparse MLA forward kernel for sm_103a, templated on the KV format: bf16
// rows of 576 values, FP8 rows of 512 e4m3 + 4 fp32 scales + 64 bf16, or FP4
// rows of 512 e2m1 + 16 fp32 scales + 64 bf16.
//
// Method: "Ascend Sparse Attention Forward 算法与优化技术简析", sections
// "数学建模" (what is computed) and "计算流程" (blockwise online softmax with
// skip-scale).  The page's delayed P@V order (section "流水线") survives as
// a pipeline across two SMs; its index prefetch / multi-stage gather idea
// survives as rings of gathered rows; its FP8 decoding (section
// "能不能用 1C1V": KV dequantised to bf16 before the matrix unit) is done by
// the gather warps on their way into the swizzled operand layouts.
//
// Mapping onto a GB300 SM pair (one 2-CTA cluster per unit of work):
//   * 128 heads x 512 fp32 output columns fill one SM's whole tensor memory,
//     and all 128 heads x 576 Q columns must sit beside the logits of any SM
//     that forms them, so the two jobs go to different SMs:
//       CTA 0 ("QK side") holds Q in tensor memory (latent 512 columns as the
//       MMA A operand, rope 64 columns in shared memory), computes the logits
//       of each 128-index block into one of two TMEM tiles, runs the online
//       softmax with skip-scale on 8 warps and sends the bf16 P tile plus the
//       per-row rescale factors to its peer with one bulk DSMEM copy.
//       CTA 1 ("PV side") holds O[128, 512] in tensor memory, applies the
//       rescale factors, multiplies P by V and writes the normalised output.
//     Tensor work per block is 576 vs 512 column-units, so the pair is
//     balanced; only bf16 P crosses between the SMs (one way).
//   * Gathers, bf16: one bulk copy per row lands the 1 KB latent part of 8 rows
//     as an 8 KB unit, which one warp transposes in place into eight
//     128-byte-swizzled atoms: the K-major operand of the QK side and the
//     MN-major operand of the PV side are the same unit layout.  The rope part
//     comes by cp.async straight into its swizzled atom.
//     Quantised rows: cp.async (16 bytes per thread) into a small raw ring,
//     dequantised by the same warps into 16 KB chunks of 128 rows x 64 columns
//     (K-major, QK side) and 16-row groups of 512 columns (MN-major, PV side).
//   * Work: with at least 8 tokens per pair, pairs take whole tokens from a
//     shared counter as they go, so that pairs on slower SMs take fewer.  With
//     fewer tokens (decode), the index blocks of all tokens form one sequence and
//     pair p takes the contiguous range [p*T/P, (p+1)*T/P); a token cut by a range
//     boundary is written as normalised partials and merged by the combine kernel.
//
// Warp roles (512 threads, both CTAs): warp 0 compacts the valid indices of
// each block into a small ring of index lists; warp 2 issues tcgen05.mma;
// warp 3 allocates TMEM.  QK side: warps 4-11 run the softmax (warp w serves
// TMEM lane quarter w % 4 and column half (w - 4) / 4).  PV side: warps 4-7
// rescale O and run the epilogue (one TMEM lane quarter each), warp 3 returns
// P slots to the QK side.  The gather: bf16 rows come by one bulk copy per row
// (QK: warps 12-15 issue, warps 1 and 3 transpose; PV: warps 8-13 issue,
// warps 1, 14, 15 transpose); quantised rows come by cp.async and are
// dequantised by the same warps (QK: 1, 3, 12-15; PV: 1, 8-15).  Gathering
// gets many warps because a GB300 SM ingests random row pieces at only a few
// tens of bytes per clock.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {

namespace fwd {

// KV formats of the kernel template: bf16 rows, or quantised rows (FP8 / FP4) that are staged raw and
// dequantised to bf16 before the tensor cores.
constexpr int kFmtBf16 = 0, kFmtFp8 = 1, kFmtFp4 = 2;

constexpr int kThreads = 512;
constexpr int kSoftmaxWarps = 8;                 // QK side, warps 4..11
constexpr int kEpiWarps = 4;                     // PV side, warps 4..7
constexpr int kGatherWarpsA = 6;                 // FP8, QK side: warps 1, 3, 12..15
constexpr int kGatherWarpsB = 9;                 // FP8, PV side: warps 1, 8..15
// bf16 rows: bulk-copy issuers and in-place transposers
constexpr int kIssuersA = 4;                     // QK side: warps 12..15
constexpr int kTransA = 2;                       // QK side: warps 1, 3
constexpr int kIssuersB = 6;                     // PV side: warps 8..13
constexpr int kTransB = 3;                       // PV side: warps 1, 14, 15
constexpr int kIdxSlots = 4;                     // ring of per-block index lists
constexpr int kIdxSlotInts = kBT + 4;            // 128 row ids + count

// ---- operand tiles and the P message
constexpr int kKChunkBytes = 128 * 128;          // 128 rows x 64 bf16 columns, SW128 K-major
constexpr int kChunksPerBlock = 9;               // 576 / 64
constexpr int kMsgPBytes = 2 * kKChunkBytes;     // P[128 rows, 128 cols] bf16 = two SW128 chunks
constexpr int kMsgTrailer = 3 * 128 * 4 + 16;    // alpha[128], inv_se[128], lse[128], flags
constexpr int kMsgBytes = kMsgPBytes + kMsgTrailer;
constexpr int kMsgSlot = 34816;                  // 34 KB, 1024-aligned slots
static_assert(kMsgBytes <= kMsgSlot && kMsgBytes % 16 == 0, "message layout");
constexpr int kVGroupRows = 16;
constexpr int kVGroupBytes = kVGroupRows * 1024; // 16 rows x 512 columns bf16 = 8 chunks x 2 KB
constexpr int kGroupsPerBlock = 128 / kVGroupRows;
constexpr int kIdxRing = 256;
constexpr int kMaxKSlots = 8, kMaxVSlots = 9;
// bf16 QK side: the K operand of a block as two halves of 64 rows (N = 64 MMAs), each half 8 groups of
// 8 rows; a group's latent part is 8 SW128 atoms (one per 64-column chunk, 8 KB), its rope part one atom
constexpr int kUnitBytes = 8 * 1024;             // 8 rows x 512 latent columns after the in-place transpose
constexpr int kHalfLatBytes = 8 * kUnitBytes;    // 64 KB
constexpr int kHalfRopeBytes = 8 * 1024;         // 8 KB
constexpr int kGroupsPerHalf = 8;
// Share of rows fetched by bulk copies (then transposed) versus cp.async straight into the swizzled
// layout.  A GB300 SM's copy engine takes one 1 KB bulk copy per ~37 cycles and cp.async runs beside it,
// but inside this pipeline cp.async rows land later than bulk rows and lengthen the fill of a buffer, so
// measured on GB300 all-bulk is fastest (prefill 4.19 ms vs 4.46 ms with 3/8 of the rows by cp.async).
constexpr int kBulkGroupsA = 8;                  // QK side: groups [0, kBulkGroupsA) of each half by bulk copy
constexpr int kBulkUnit1B = 8;                   // PV side: unit 1 of slot groups [0, kBulkUnit1B) by bulk copy

// cp.async of 8 rows' latent 1024 bytes straight into 8 SW128 atoms (one warp, 16 pieces per lane; a warp
// instruction covers 4 rows x 128 bytes of one atom).
__device__ __forceinline__ void cp_async_unit(uint32_t dst, const uint8_t* kv, const int* rows, int lane);
// FP8 rows: raw units staged before dequantisation
constexpr int kRawSlots = 4;
constexpr int kRawASlot = 128 * 64;              // QK side unit: 128 rows x 64 bytes (64 e4m3 or 32 bf16)
// Quantised rows: [latent codes | fp32 scales | 64 bf16 rope]
//   FP8: 512 e4m3 (512 B) | 4 scales, one per 128 channels (16 B) | rope (128 B) = 656 B
//   FP4: 512 e2m1 two per byte, low nibble = even channel (256 B) | 16 scales, one per 32 channels (64 B) |
//        rope (128 B) = 448 B
template <int kFmt>
struct QRow {
  static constexpr bool kF4 = kFmt == 2;
  static constexpr int kBytes = kF4 ? 448 : 656;
  static constexpr int kScaleOff = kF4 ? 256 : 512;     // = latent code bytes
  static constexpr int kScaleBytes = kF4 ? 64 : 16;
  static constexpr int kRopeOff = kScaleOff + kScaleBytes;
  static constexpr int kLatUnits = kF4 ? 4 : 8;         // QK raw units of 64 code bytes per row: 128 | 64 channels
  static constexpr int kUnits = kLatUnits + 2;           // + the two 64-byte rope halves
  static constexpr int kRawBRow = kRopeOff;              // PV side stages codes + scales of each row
  static constexpr int kRawBSlot = kVGroupRows * kRawBRow;
  static constexpr int kScaleSlot = 128 * kScaleBytes;   // QK side: the scales of each of 128 rows
};

__host__ __device__ constexpr int align1k(int x) { return (x + 1023) / 1024 * 1024; }

// Shared-memory layout of each side for one KV format.
template <int kFmt>
struct Lay {
  static constexpr bool kQuant = kFmt != kFmtBf16;
  using R = QRow<kFmt == kFmtBf16 ? kFmtFp8 : kFmt>;
  static constexpr int kKSlots = kQuant ? 6 : 0;   // FP8: ring of 128-row x 64-column chunks
  static constexpr int kVSlots = kQuant ? 7 : 9;
  // QK side (cluster rank 0).  bf16: latent halves [2][8 groups][8 atoms], then rope atoms [2][8 groups].
  static constexpr int A_OffK = 0;
  static constexpr int A_OffKR = A_OffK + (kQuant ? 0 : 2 * kHalfLatBytes);
  static constexpr int A_OffRaw = kQuant ? A_OffK + kKSlots * kKChunkBytes : A_OffKR + 2 * kHalfRopeBytes;
  static constexpr int A_OffScales = A_OffRaw + (kQuant ? kRawSlots * kRawASlot : 0);
  static constexpr int A_OffQRope = A_OffScales + (kQuant ? 2 * R::kScaleSlot : 0);
  static constexpr int A_OffMsg = align1k(A_OffQRope + kKChunkBytes);  // one outgoing message buffer
  static constexpr int A_OffMax = A_OffMsg + kMsgSlot;  // [2 halves][128] float
  static constexpr int A_OffSe = A_OffMax + 2 * 128 * 4;
  static constexpr int A_End = A_OffSe + 2 * 128 * 4;
  // PV side (cluster rank 1)
  static constexpr int B_OffV = 0;
  static constexpr int B_OffRaw = B_OffV + kVSlots * kVGroupBytes;
  static constexpr int B_OffMsg = align1k(B_OffRaw + (kQuant ? kRawSlots * R::kRawBSlot : 0));
  static constexpr int B_End = B_OffMsg + 2 * kMsgSlot;
  // common tail: compaction ring, per-block index lists, barriers, misc
  static constexpr int OffCommon = (A_End > B_End ? A_End : B_End);
  static constexpr int OffRing = (OffCommon + 127) / 128 * 128;
  static constexpr int OffIdx = OffRing + kIdxRing * 4;
  static constexpr int OffBar = OffIdx + kIdxSlots * kIdxSlotInts * 4;
  static constexpr int NumBars = 56;
  static constexpr int OffMisc = OffBar + NumBars * 8;
  static constexpr int SmemUsed = OffMisc + 64;
  static constexpr int SmemAlloc = SmemUsed + 1024;
  static_assert(SmemAlloc <= 232448, "shared memory budget");
};

// barrier slots
enum BarCommon {
  IDX_FULL = 0, IDX_EMPTY = IDX_FULL + kIdxSlots, RAW_FULL = IDX_EMPTY + kIdxSlots, RAW_EMPTY = RAW_FULL + kRawSlots,
  BAR_COMMON_END = RAW_EMPTY + kRawSlots
};
enum BarA {
  A_K_FULL = BAR_COMMON_END, A_K_EMPTY = A_K_FULL + kMaxKSlots, A_S_FULL = A_K_EMPTY + kMaxKSlots,
  A_S_EMPTY = A_S_FULL + 2, A_Q_FULL = A_S_EMPTY + 2, A_Q_FREE, A_POUT_EMPTY, A_SMX_SYNC = A_POUT_EMPTY + 2, A_DRAIN,
  A_KH_FULL, A_KH_EMPTY = A_KH_FULL + 2, A_MSG_FREE = A_KH_EMPTY + 2, A_NUM,
  A_LAND = A_K_FULL  // bf16: landing barriers of the 16 groups of a block (spans the FP8 K_FULL/K_EMPTY slots)
};
enum BarB {
  B_V_FULL = BAR_COMMON_END, B_V_EMPTY = B_V_FULL + kMaxVSlots, B_PIN_FULL = B_V_EMPTY + kMaxVSlots,
  B_RESC_DONE = B_PIN_FULL + 2, B_PV_DONE = B_RESC_DONE + 2, B_O_FULL = B_PV_DONE + 2, B_O_FREE, B_DRAIN,
  B_V_LAND, B_NUM = B_V_LAND + kMaxVSlots
};
static_assert((int)A_LAND + 16 <= (int)A_S_FULL, "bf16 landing barriers fit in the K slots");
static_assert((int)A_NUM <= 56 && (int)B_NUM <= 56, "barrier slots");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmQ = 0;     // QK side: Q latent [0, 256) (bf16 pairs), S tiles [256, 384) and [384, 512)
constexpr uint32_t kTmS = 256;
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kBT, 0, 0);
constexpr uint32_t kIdescQK64 = idesc_bf16_f32(128, 64, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);

constexpr float kThresLog2 = 6.0f * 1.4426950408889634f;  // RESCALE_THRES = 6 (natural log) in log2 units
constexpr float kLn2 = 0.6931471805599453f;

// One contiguous run of index blocks of one token.
struct Piece {
  int t, lb0, lb1;   // token, first and one-past-last block (within the token)
  bool full;         // covers all blocks of the token
  int slot;          // partial-output slot when !full
};

// Iterates the pieces of pair p's range [p*T/P, (p+1)*T/P) of the global block sequence.
struct PieceIter {
  const int* cum;
  int s_q, g, g1, t, idx, pair;
  __device__ void init(const int* cum_, int s_q_, int p, int npairs) {
    cum = cum_;
    s_q = s_q_;
    pair = p;
    const long long T = cum[s_q];
    g = (int)((long long)p * T / npairs);
    g1 = (int)((long long)(p + 1) * T / npairs);
    idx = 0;
    int lo = 0, hi = s_q - 1;  // largest t with cum[t] <= g
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (cum[mid] <= g) lo = mid; else hi = mid - 1;
    }
    t = lo;
  }
  __device__ bool next(Piece& pc) {
    if (g >= g1) return false;
    const int c0 = cum[t], c1 = cum[t + 1];
    pc.t = t;
    pc.lb0 = g - c0;
    pc.lb1 = min(c1, g1) - c0;
    pc.full = (pc.lb0 == 0) && (pc.lb1 == c1 - c0);
    pc.slot = 2 * pair + (idx == 0 ? 0 : 1);
    g = c0 + pc.lb1;
    ++t;
    ++idx;
    return true;
  }
};

__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk16) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((chunk16 ^ (row & 7)) << 4);
}

// In-place re-layout of one 8-row unit at shared address `un`: 8 rows of 512 bf16 landed as plain rows
// (row r at r*1024) become 8 SW128 atoms (64-column chunk c at c*1024, row r at r*128 inside it, 16-byte
// pieces XOR-swizzled by r).  As 128-byte segments this is an 8x8 transpose; the segments with (r + c)
// even and with (r + c) odd are each closed under it and disjoint, so a warp moves one class through
// registers (8 pieces per lane), then the other, with one sync between the reads and the writes of each.
// A warp instruction touches 4 whole 128-byte segments, so neither side has bank conflicts.
__device__ __forceinline__ uint4 lds128(uint32_t a) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
  return v;
}
__device__ __forceinline__ void sts128(uint32_t a, uint4 v) {
  asm volatile("st.shared.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(a), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}
__device__ __forceinline__ void transpose_unit(uint32_t un, int lane) {
  const int k = lane & 7, cb = 2 * (lane >> 3);
#pragma unroll
  for (int ph = 0; ph < 2; ++ph) {
    uint4 v[8];
#pragma unroll
    for (int r = 0; r < 8; ++r) v[r] = lds128(un + (uint32_t)(r * 1024 + (cb + ((r + ph) & 1)) * 128 + k * 16));
    __syncwarp();
#pragma unroll
    for (int r = 0; r < 8; ++r)
      sts128(un + (uint32_t)((cb + ((r + ph) & 1)) * 1024) + sw128_off((uint32_t)r, (uint32_t)k), v[r]);
  }
  __syncwarp();
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_unit(uint32_t dst, const uint8_t* kv, const int* rows, int lane) {
#pragma unroll 4
  for (int j = 0; j < 16; ++j) {
    const int q = j * 32 + lane;
    const int ch = q >> 6, r = (q >> 3) & 7, k = q & 7;
    cp_async16(dst + (uint32_t)(ch * 1024) + sw128_off((uint32_t)r, (uint32_t)k),
               kv + (size_t)rows[r] * (kDQK * 2) + ch * 128 + k * 16);
  }
}
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void bulk_s2cluster(uint32_t dst_cluster, uint32_t src_cta, uint32_t bytes,
                                               uint32_t remote_bar) {
  asm volatile("cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   dst_cluster),
               "r"(src_cta), "r"(bytes), "r"(remote_bar)
               : "memory");
}

// 16 e4m3 codes (one 16-byte piece, code i in byte i) times `scale`, rounded to
// bf16: two 16-byte pieces of 8 bf16 each, element order kept.
__device__ __forceinline__ void dequant16(const uint4 w, float scale, uint4& o0, uint4& o1) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2_raw h01 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(in[i] & 0xFFFFu), __NV_E4M3);
    const __half2_raw h23 = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(in[i] >> 16), __NV_E4M3);
    const float2 f01 = __half22float2(__half2(h01));
    const float2 f23 = __half22float2(__half2(h23));
    out[2 * i] = pack_bf16x2(f01.x * scale, f01.y * scale);
    out[2 * i + 1] = pack_bf16x2(f23.x * scale, f23.y * scale);
  }
  o0 = make_uint4(out[0], out[1], out[2], out[3]);
  o1 = make_uint4(out[4], out[5], out[6], out[7]);
}

// 32 e2m1 codes (one 16-byte piece; byte i holds channel 2i in its low nibble and 2i + 1 in its high
// nibble) times `scale`, rounded to bf16: four 16-byte pieces of 8 bf16 each, channel order kept.
__device__ __forceinline__ void dequant32_fp4(const uint4 w, float scale, uint4 (&o)[4]) {
  const uint32_t in[4] = {w.x, w.y, w.z, w.w};
  uint32_t out[16];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)((in[i] >> (8 * j)) & 0xFFu), __NV_E2M1);
      const float2 f = __half22float2(__half2(h));
      out[4 * i + j] = pack_bf16x2(f.x * scale, f.y * scale);
    }
  }
#pragma unroll
  for (int k = 0; k < 4; ++k) o[k] = make_uint4(out[4 * k], out[4 * k + 1], out[4 * k + 2], out[4 * k + 3]);
}

struct Ctx {
  uint8_t* smem;
  uint32_t sbase, bars, tmem, rank, peer, peer_abort;
  volatile int* abort_flag;
  int* status;
  int warp, lane, pair;
  __device__ uint32_t bar(int i) const { return bars + 8u * (uint32_t)i; }
};

__device__ __forceinline__ void set_abort(const Ctx& c) {
  if (!*c.abort_flag) {
    *c.abort_flag = 1;
    atomicCAS(c.status, 0, 5 /* DSA_ERR_DEVICE_TIMEOUT */);
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(c.peer_abort), "r"(1) : "memory");
  }
}

__device__ __forceinline__ bool wait(const Ctx& c, int b, uint32_t parity, bool cluster = false) {
  return mbar_wait(c.bar(b), parity, kWaitLimitNs, c.abort_flag, cluster);
}

// Bounded barrier among the 8 softmax warps (an mbarrier, so that a warp that
// gave up cannot leave the others blocked forever).  `n` counts uses.
__device__ __forceinline__ bool group_sync(const Ctx& c, uint32_t& n) {
  __syncwarp();
  if (c.lane == 0) mbar_arrive(c.bar(A_SMX_SYNC));
  const bool ok = wait(c, A_SMX_SYNC, n & 1u);
  ++n;
  return ok;
}

// Index compaction into a ring: the valid slots of one token, in order.
struct IndexRing {
  int* ring;
  const int32_t* idx_t;
  const FwdParams* prm;
  int topk, seq, head, tail, rp;
  __device__ void reset(int* r, const FwdParams& p, int t) {
    ring = r; prm = &p; idx_t = p.indices + (size_t)t * p.topk; topk = p.topk; seq = token_seq(p, t);
    head = tail = rp = 0;
  }
  // ensure >= kBT entries (or the token's end) are buffered; returns the count for this block
  __device__ int fill(int lane) {
    while (tail - head < kBT && rp < topk) {
      int v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int i = rp + q * 32 + lane;
        v[q] = (i < topk) ? __ldg(idx_t + i) : -1;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) v[q] = resolve_row(*prm, seq, v[q]);  // pool row or -1
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const bool ok = v[q] >= 0;
        const uint32_t m = __ballot_sync(0xffffffffu, ok);
        if (ok) ring[(tail + __popc(m & ((1u << lane) - 1u))) & (kIdxRing - 1)] = v[q];
        tail += __popc(m);
      }
      rp += 128;
      __syncwarp();
    }
    return min(kBT, tail - head);
  }
  __device__ int at(int i) const { return ring[(head + i) & (kIdxRing - 1)]; }
  __device__ void pop(int cnt) {
    head += cnt;
    __syncwarp();
  }
};

// Index blocks of pair `pair`: its share [pair*T/P, (pair+1)*T/P) of the block sequence.
__device__ __forceinline__ uint32_t blocks_of_pair(const FwdParams& p, int pair) {
  const long long T = p.cum[p.s_q];
  return (uint32_t)((long long)(pair + 1) * T / p.npairs - (long long)pair * T / p.npairs);
}

// Index blocks of token t (at least one, so that a token without valid slots still gets its output).
__device__ __forceinline__ int blocks_of_token(const FwdParams& p, int t) {
  const int nv = p.nvalid[t];
  return nv > 0 ? (nv + kBT - 1) / kBT : 1;
}

// Dynamic token scheduling (p.dyn): the pair's i-th token is taken from the shared counter by the first
// role that needs it, the QK side's index compactor, and recorded in seq[pair][i] (t + 1, or -1 when none
// is left); every other role of both CTAs reads the record, waiting (bounded) until it is written.
__device__ __forceinline__ int ld_acquire_gpu(const int* a) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(a) : "memory");
  return v;
}
__device__ __forceinline__ void st_release_gpu(int* a, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(a), "r"(v) : "memory");
}
// Record i of this pair: t + 1, -1 (no more tokens) or 0 (the wait gave up).  One thread.
__device__ __forceinline__ int token_record(const Ctx& c, const FwdParams& p, int i, bool take) {
  int* e = p.seq + (size_t)c.pair * (size_t)(p.s_q + 1) + i;
  if (take) {
    const int t = atomicAdd(p.ctrl + kCtrlNextToken, 1);
    const int v = t < p.s_q ? t + 1 : -1;
    st_release_gpu(e, v);
    return v;
  }
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    const int v = ld_acquire_gpu(e);
    if (v != 0) return v;
    if ((it & 63u) == 0 && (*c.abort_flag || globaltimer_ns() - t0 > kWaitLimitNs)) return 0;
  }
}

// The pieces of a pair: its static share, or whole tokens taken one by one.  next() runs on one thread;
// next_warp() is called by all 32 lanes together: lane 0 takes or reads the record and the warp gets its
// value by a shuffle, so every lane sees the same sequence even when a wait gives up.  `err` is set when
// a wait gave up.
struct WorkIter {
  PieceIter st;
  int i;
  bool dyn, take;
  __device__ void init(const Ctx& c, const FwdParams& p, bool taker) {
    dyn = p.dyn != 0;
    take = taker && c.rank == 0;
    i = 0;
    if (!dyn) st.init(p.cum, p.s_q, c.pair, p.npairs);
  }
  __device__ bool from_record(const FwdParams& p, int v, Piece& pc, bool& err) {
    if (v == 0) {
      err = true;
      return false;
    }
    if (v < 0) return false;
    pc.t = v - 1;
    pc.lb0 = 0;
    pc.lb1 = blocks_of_token(p, pc.t);
    pc.full = true;
    pc.slot = 0;
    return true;
  }
  __device__ bool next(const Ctx& c, const FwdParams& p, Piece& pc, bool& err) {
    if (!dyn) return st.next(pc);
    return from_record(p, token_record(c, p, i++, take), pc, err);
  }
  __device__ bool next_warp(const Ctx& c, const FwdParams& p, Piece& pc, bool& err) {
    if (!dyn) return st.next(pc);
    int v = 0;
    if (c.lane == 0) v = token_record(c, p, i, take);
    v = __shfl_sync(0xffffffffu, v, 0);
    ++i;
    return from_record(p, v, pc, err);
  }
};

// Whether block b of the pair exists, for the roles that walk blocks rather than tokens.  Static: b is
// below the share's count.  Dynamic: the count grows as token records are read.  With `whole_warp`, all
// 32 lanes call has() together and lane 0 reads each record for the warp (one shuffle per record).
struct BlockCount {
  uint32_t known;
  int i;
  bool more, warp;
  __device__ void init(const Ctx& c, const FwdParams& p, bool whole_warp) {
    more = p.dyn != 0;
    warp = whole_warp;
    i = 0;
    known = more ? 0u : blocks_of_pair(p, c.pair);
  }
  __device__ bool has(const Ctx& c, const FwdParams& p, uint32_t b, bool& err) {
    while (b >= known && more) {
      int v;
      if (warp) {
        v = 0;
        if (c.lane == 0) v = token_record(c, p, i, false);
        v = __shfl_sync(0xffffffffu, v, 0);
        ++i;
      } else {
        v = token_record(c, p, i++, false);
      }
      if (v <= 0) {
        more = false;
        if (v == 0) err = true;
        break;
      }
      known += (uint32_t)blocks_of_token(p, v - 1);
    }
    return b < known;
  }
};


// ============================================================================ both sides: index lists
// Warp 0: walks this pair's pieces, compacts the valid slots of each block in
// order and publishes them (row ids + count) in a ring of kIdxSlots lists.
template <int kFmt>
__device__ void index_compactor(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmt>;
  IndexRing ir;
  int* lists = (int*)(c.smem + Y::OffIdx);
  WorkIter it;
  it.init(c, p, true);
  Piece pc;
  uint32_t b = 0;
  bool ok = true, err = false;
  while (ok && it.next_warp(c, p, pc, err)) {
    ir.reset((int*)(c.smem + Y::OffRing), p, pc.t);
    for (int jb = 0; jb < pc.lb1; ++jb) {
      const int cnt = ir.fill(c.lane);
      if (jb >= pc.lb0) {
        const int slot = (int)(b % kIdxSlots);
        if (!wait(c, IDX_EMPTY + slot, ((b / kIdxSlots) & 1u) ^ 1u)) { ok = false; break; }
        int* l = lists + slot * kIdxSlotInts;
#pragma unroll
        for (int q = 0; q < kBT / 32; ++q) {
          const int i = q * 32 + c.lane;
          l[i] = i < cnt ? ir.at(i) : 0;  // padding rows read row 0 and are masked by the softmax
        }
        if (c.lane == 0) l[kBT] = cnt;
        __syncwarp();
        if (c.lane == 0) mbar_arrive(c.bar(IDX_FULL + slot));
        ++b;
      }
      ir.pop(cnt);
    }
  }
  if (!ok || err) set_abort(c);
}

// ============================================================================ QK side
// Quantised rows (FP8 / FP4): cp.async into a raw ring, dequantised by the same warps into the K chunk ring.
template <int kFmt>
static __device__ void qk_gather_q(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmt>;
  using R = QRow<kFmt>;
  uint8_t* smem = c.smem;
  const int warp = c.warp, lane = c.lane;
  const int gw = (warp == 1) ? 0 : (warp == 3) ? 5 : warp - 11;  // 0..5
  const int gt = gw * 32 + lane;
  constexpr int kGT = kGatherWarpsA * 32;
  const int* lists = (const int*)(smem + Y::OffIdx);
  BlockCount bc;
  bc.init(c, p, true);
  bool ok = true, err = false;
  {
    // Per block R::kUnits raw units of 128 rows x 64 bytes: latent code units (one 64-channel chunk of
    // e4m3, or two of e2m1) and the two rope halves (bf16); the block's scales ride with unit 0.  Units
    // are staged in a 4-slot ring two units ahead, then dequantised (latent) or copied (rope) into the
    // swizzled K chunk ring.
    auto exists = [&](uint32_t u) -> bool { return bc.has(c, p, u / (uint32_t)R::kUnits, err); };
    auto issue = [&](uint32_t u) -> bool {
      const uint32_t b = u / (uint32_t)R::kUnits;
      const int k = (int)(u % (uint32_t)R::kUnits), rs = (int)(u % kRawSlots);
      if (!wait(c, RAW_EMPTY + rs, ((u / kRawSlots) & 1u) ^ 1u)) return false;
      if (k == 0 && !wait(c, IDX_FULL + (int)(b % kIdxSlots), (b / kIdxSlots) & 1u)) return false;
      const int* l = lists + (int)(b % kIdxSlots) * kIdxSlotInts;
      const uint32_t dst = c.sbase + Y::A_OffRaw + (uint32_t)rs * kRawASlot;
      const int src_off = (k < R::kLatUnits) ? 64 * k : R::kRopeOff + 64 * (k - R::kLatUnits);
      for (int q = gt; q < 512; q += kGT)
        cp_async16(dst + (uint32_t)q * 16u, p.kv + (size_t)l[q >> 2] * R::kBytes + src_off + 16 * (q & 3));
      if (k == 0) {
        constexpr int kPer = R::kScaleBytes / 16;  // 16-byte pieces of scales per row
        const uint32_t sd = c.sbase + Y::A_OffScales + (b & 1u) * R::kScaleSlot;
        for (int q = gt; q < 128 * kPer; q += kGT)
          cp_async16(sd + (uint32_t)q * 16u, p.kv + (size_t)l[q / kPer] * R::kBytes + R::kScaleOff + 16 * (q % kPer));
      }
      cp_async_arrive(c.bar(RAW_FULL + rs));
      return true;
    };
    auto consume = [&](uint32_t u) -> bool {
      const uint32_t b = u / (uint32_t)R::kUnits;
      const int k = (int)(u % (uint32_t)R::kUnits), rs = (int)(u % kRawSlots);
      if (!wait(c, RAW_FULL + rs, (u / kRawSlots) & 1u)) return false;
      const uint8_t* raw = smem + Y::A_OffRaw + rs * kRawASlot;
      const float* sc = (const float*)(smem + Y::A_OffScales + (b & 1u) * R::kScaleSlot);
      if (k < R::kLatUnits) {
        if constexpr (!R::kF4) {  // FP8: unit k = latent chunk k
          const uint32_t cs = b * (uint32_t)kChunksPerBlock + (uint32_t)k;
          const int s = (int)(cs % Y::kKSlots);
          if (!wait(c, A_K_EMPTY + s, ((cs / Y::kKSlots) & 1u) ^ 1u)) return false;
          uint8_t* kd = smem + Y::A_OffK + s * kKChunkBytes;
          for (int q = gt; q < 512; q += kGT) {
            const int r = q >> 2, rp = q & 3;
            uint4 o0, o1;
            dequant16(*(const uint4*)(raw + q * 16), sc[r * 4 + (k >> 1)], o0, o1);
            *(uint4*)(kd + sw128_off((uint32_t)r, (uint32_t)(2 * rp))) = o0;
            *(uint4*)(kd + sw128_off((uint32_t)r, (uint32_t)(2 * rp + 1))) = o1;
          }
          mbar_arrive(c.bar(A_K_FULL + s));
        } else {  // FP4: unit k = latent chunks 2k and 2k + 1 (piece rp of a row = 32 channels)
          const uint32_t cs0 = b * (uint32_t)kChunksPerBlock + 2u * (uint32_t)k;
          const int s0 = (int)(cs0 % Y::kKSlots), s1 = (int)((cs0 + 1u) % Y::kKSlots);
          if (!wait(c, A_K_EMPTY + s0, ((cs0 / Y::kKSlots) & 1u) ^ 1u) ||
              !wait(c, A_K_EMPTY + s1, (((cs0 + 1u) / Y::kKSlots) & 1u) ^ 1u))
            return false;
          for (int q = gt; q < 512; q += kGT) {
            const int r = q >> 2, rp = q & 3;
            uint4 o[4];
            dequant32_fp4(*(const uint4*)(raw + q * 16), sc[r * 16 + 4 * k + rp], o);
            uint8_t* kd = smem + Y::A_OffK + (rp < 2 ? s0 : s1) * kKChunkBytes;
#pragma unroll
            for (int j = 0; j < 4; ++j) *(uint4*)(kd + sw128_off((uint32_t)r, (uint32_t)(4 * (rp & 1) + j))) = o[j];
          }
          mbar_arrive(c.bar(A_K_FULL + s0));
          mbar_arrive(c.bar(A_K_FULL + s1));
        }
      } else {  // rope half: 32 bf16 of chunk 8, which completes with the second half
        const int hr = k - R::kLatUnits;
        const uint32_t cs = b * (uint32_t)kChunksPerBlock + 8u;
        const int s = (int)(cs % Y::kKSlots);
        if (hr == 0 && !wait(c, A_K_EMPTY + s, ((cs / Y::kKSlots) & 1u) ^ 1u)) return false;
        uint8_t* kd = smem + Y::A_OffK + s * kKChunkBytes;
        for (int q = gt; q < 512; q += kGT)
          *(uint4*)(kd + sw128_off((uint32_t)(q >> 2), (uint32_t)(4 * hr + (q & 3)))) = *(const uint4*)(raw + q * 16);
        if (hr == 1) mbar_arrive(c.bar(A_K_FULL + s));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(RAW_EMPTY + rs));
      if (k == R::kUnits - 1 && lane == 0) mbar_arrive(c.bar(IDX_EMPTY + (int)(b % kIdxSlots)));
      return true;
    };
    for (uint32_t u = 0; u < 2u && ok && exists(u); ++u) ok = issue(u);
    for (uint32_t u = 0; ok && exists(u); ++u) {
      if (exists(u + 2u)) ok = issue(u + 2u);
      if (ok) ok = consume(u);
    }
    if (!ok || err) set_abort(c);
  }
}

// bf16 rows, issuers (warps 12..15): group g of block b (rows 8g..8g+7) goes to half g / 8.  Lane r < 8
// bulk-copies the 1024 latent bytes of row r as they are (the transposer lays them out afterwards); all
// lanes cp.async the 128 rope bytes of the 8 rows straight into the group's swizzled rope atom.  The
// group's landing barrier completes on the bulk bytes plus one cp.async arrival per lane.
static __device__ void qk_issue_bf16(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmtBf16>;
  const int lane = c.lane, i = c.warp - 12;
  const int* lists = (const int*)(c.smem + Y::OffIdx);
  BlockCount bc;
  bc.init(c, p, true);
  uint32_t issued = 0;
  bool ok = true, err = false;
  for (uint32_t b = 0; ok && bc.has(c, p, b, err); ++b) {
    const int slot = (int)(b % kIdxSlots);
    if (!wait(c, IDX_FULL + slot, (b / kIdxSlots) & 1u)) { ok = false; break; }
    const int* l = lists + slot * kIdxSlotInts;
    for (int g = i; g < 2 * kGroupsPerHalf; g += kIssuersA) {
      const int h = g / kGroupsPerHalf, gg = g % kGroupsPerHalf;
      if (!wait(c, A_KH_EMPTY + h, (b & 1u) ^ 1u)) { ok = false; break; }
      const uint32_t land = c.bar(A_LAND + g);
      const bool bulk = gg < kBulkGroupsA;
      const uint32_t unit = c.sbase + Y::A_OffK + (uint32_t)(h * kHalfLatBytes + gg * kUnitBytes);
      if (lane == 0) mbar_arrive_expect_tx(land, bulk ? (uint32_t)kUnitBytes : 0u);
      __syncwarp();
      if (bulk) {
        if (lane < 8) bulk_g2s(unit + (uint32_t)(lane * 1024), p.kv + (size_t)l[g * 8 + lane] * (kDQK * 2), 1024u, land);
      } else {
        cp_async_unit(unit, p.kv, l + g * 8, lane);
      }
      const uint32_t rope = c.sbase + Y::A_OffKR + (uint32_t)(h * kHalfRopeBytes + gg * 1024);
#pragma unroll
      for (int q = lane; q < 64; q += 32) {
        const int r = q >> 3, k = q & 7;
        cp_async16(rope + sw128_off((uint32_t)r, (uint32_t)k), p.kv + (size_t)l[g * 8 + r] * (kDQK * 2) + 1024 + k * 16);
      }
      cp_async_arrive(land);
    }
    if (!ok) break;
    issued = b + 1;
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(IDX_EMPTY + slot));
  }
  if (!ok || err) set_abort(c);
  // the copies of the last block issued land before the CTA may exit
  if (issued > 0)
    for (int g = i; g < 2 * kGroupsPerHalf; g += kIssuersA)
      mbar_wait(c.bar(A_LAND + g), (issued - 1) & 1u, kWaitLimitNs, nullptr);
}

// bf16 rows, transposers (warps 1 and 3): once a group has landed, turn its latent rows into SW128
// atoms in place and count the group towards its half.
static __device__ void qk_transpose_bf16(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmtBf16>;
  const int lane = c.lane, t = (c.warp == 1) ? 0 : 1;
  BlockCount bc;
  bc.init(c, p, true);
  bool ok = true, err = false;
  for (uint32_t b = 0; ok && bc.has(c, p, b, err); ++b) {
    for (int g = t; g < 2 * kGroupsPerHalf; g += kTransA) {
      const int h = g / kGroupsPerHalf, gg = g % kGroupsPerHalf;
      if (!wait(c, A_LAND + g, b & 1u)) { ok = false; break; }
      if (gg < kBulkGroupsA) transpose_unit(c.sbase + Y::A_OffK + (uint32_t)(h * kHalfLatBytes + gg * kUnitBytes), lane);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(A_KH_FULL + h));
    }
  }
  if (!ok || err) set_abort(c);
}

template <int kFmt>
__device__ void qk_mma(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmt>;
  constexpr bool kQuant = kFmt != kFmtBf16;
  if (c.lane == 0) {
    WorkIter it;
    it.init(c, p, false);
    Piece pc;
    uint32_t cseq = 0, blk = 0, item = 0;
    bool ok = true, err = false;
    const uint32_t qrope = c.sbase + Y::A_OffQRope;
    while (ok && it.next(c, p, pc, err)) {
      const int nb = pc.lb1 - pc.lb0;
      if (!wait(c, A_Q_FULL, item & 1u)) { ok = false; break; }
      for (int j = 0; j < nb && ok; ++j, ++blk) {
        const int sb = (int)(blk & 1u);
        if (!wait(c, A_S_EMPTY + sb, ((blk >> 1) & 1u) ^ 1u)) { ok = false; break; }
        tc_fence_after();
        const uint32_t dS = c.tmem + kTmS + (uint32_t)sb * kBT;
        if constexpr (!kQuant) {
          // bf16: each half of 64 rows as soon as its 8 groups are laid out (N = 64), then free it
          for (int h = 0; h < 2 && ok; ++h) {
            if (!wait(c, A_KH_FULL + h, blk & 1u)) { ok = false; break; }
            fence_proxy_async_smem();  // generic-proxy writes (transposer / cp.async) -> tensor core reads
            tc_fence_after();
            // descriptors built once; a step of 16 columns (32 bytes) or one atom (1 KB) only moves the
            // start-address field (bits 0..13, address / 16, no carry below 256 KB)
            const uint64_t lat = smem_desc(c.sbase + Y::A_OffK + (uint32_t)(h * kHalfLatBytes), 16, kUnitBytes);
            const uint64_t rope = smem_desc(c.sbase + Y::A_OffKR + (uint32_t)(h * kHalfRopeBytes), 16, 1024);
            const uint64_t qr = smem_desc(qrope, 16, 1024);
            const uint32_t dh = dS + (uint32_t)(h * 64), qa = c.tmem + kTmQ;
#pragma unroll
            for (int k = 0; k < 8; ++k)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_ts(dh, qa + (uint32_t)(k * 32 + kk * 8), lat + (uint64_t)(k * 64 + kk * 2), kIdescQK64,
                       (k > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_ss(dh, qr + (uint64_t)(kk * 2), rope + (uint64_t)(kk * 2), kIdescQK64, 1u);
            mma_commit(c.bar(A_KH_EMPTY + h));
          }
        } else {
          // FP8: the ring of 128-row chunks, one chunk of 64 columns at a time (N = 128)
          for (int k = 0; k < kChunksPerBlock; ++k, ++cseq) {
            const int s = (int)(cseq % Y::kKSlots);
            if (!wait(c, A_K_FULL + s, (cseq / Y::kKSlots) & 1u)) { ok = false; break; }
            fence_proxy_async_smem();  // generic-proxy writes (cp.async / dequant) -> tensor core reads
            tc_fence_after();
            const uint32_t chunk = c.sbase + Y::A_OffK + (uint32_t)s * kKChunkBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bdesc = smem_desc(chunk + (uint32_t)kk * 32u, 16, 1024);
              const uint32_t acc = (k > 0 || kk > 0) ? 1u : 0u;
              if (k < 8) mma_ts(dS, c.tmem + kTmQ + (uint32_t)(k * 32 + kk * 8), bdesc, kIdescQK, acc);
              else mma_ss(dS, smem_desc(qrope + (uint32_t)kk * 32u, 16, 1024), bdesc, kIdescQK, acc);
            }
            mma_commit(c.bar(A_K_EMPTY + s));
          }
        }
        if (!ok) break;
        mma_commit(c.bar(A_S_FULL + sb));
      }
      mma_commit(c.bar(A_Q_FREE));
      ++item;
    }
    if (!ok || err) set_abort(c);
    mma_commit(c.bar(A_DRAIN));
    mbar_wait(c.bar(A_DRAIN), 0, kWaitLimitNs, nullptr);
  }
  __syncwarp();
}

template <int kFmt>
__device__ void qk_softmax(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmt>;
  uint8_t* smem = c.smem;
  const int warp = c.warp, lane = c.lane;
  const int sw = warp - 4;
  const int quarter = warp & 3, half = sw >> 2;
  const int r = quarter * 32 + lane;  // head row = TMEM lane
  const uint32_t trow = c.tmem + ((uint32_t)(quarter * 32) << 16);
  float* maxbuf = (float*)(smem + Y::A_OffMax);
  float* sebuf = (float*)(smem + Y::A_OffSe);
  const uint32_t peer_msg = mapa_shared(c.sbase + Y::B_OffMsg, c.peer);
  const uint32_t peer_pin_full = mapa_shared(c.bars + 8u * (uint32_t)B_PIN_FULL, c.peer);
  const float sg = p.scale_log2 < 0.f ? -1.f : 1.f;  // direction the scale preserves
  WorkIter it;
  it.init(c, p, false);
  Piece pc;
  uint32_t blk = 0, item = 0, nsync = 0;
  bool ok = true, err = false;
  while (ok && it.next_warp(c, p, pc, err)) {
    const int nb = pc.lb1 - pc.lb0;
    const int nval = p.nvalid[pc.t];
    // ---- Q for this token: latent columns [256*half, +256) into TMEM, rope (half 0) into smem
    if (!wait(c, A_Q_FREE, (item & 1u) ^ 1u)) { ok = false; break; }
    tc_fence_after();
    {
      // this thread's share of the next token's Q row moves into L2 now, one token of work before the
      // next piece reads it (the Q load at a token switch stalls the QK tensor core)
      if (pc.t + 1 < p.s_q && r < p.h_q) {
        const uint8_t* nq = (const uint8_t*)(p.q + ((size_t)(pc.t + 1) * p.h_q + r) * kDQK);
#pragma unroll
        for (int u = 0; u < 4; ++u) prefetch_l2(nq + half * 512 + u * 128);
        if (half == 0) prefetch_l2(nq + 1024);
      }
      const bool live = r < p.h_q;
      const uint4* qrow = (const uint4*)(p.q + ((size_t)pc.t * p.h_q + (live ? r : 0)) * kDQK);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t v[32];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 w = live ? __ldg(qrow + half * 32 + cc * 8 + u) : make_uint4(0, 0, 0, 0);
          v[4 * u] = w.x; v[4 * u + 1] = w.y; v[4 * u + 2] = w.z; v[4 * u + 3] = w.w;
        }
        tmem_st32(trow + kTmQ + (uint32_t)(half * 128 + cc * 32), v);
      }
      if (half == 0) {
        uint8_t* qr = smem + Y::A_OffQRope;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint4 w = live ? __ldg(qrow + 64 + u) : make_uint4(0, 0, 0, 0);
          *(uint4*)(qr + sw128_off((uint32_t)r, (uint32_t)u)) = w;
        }
        fence_proxy_async_smem();
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(A_Q_FULL));
    }
    float rm = -INFINITY, rmfs = -INFINITY, se = 0.f;
    for (int j = 0; j < nb; ++j, ++blk) {
      const int sb = (int)(blk & 1u);
      float s[64];
      // the one outgoing buffer is free once the previous message has landed in the peer
      if (blk > 0 && !wait(c, A_MSG_FREE, (blk - 1u) & 1u, true)) { ok = false; break; }
      if (!wait(c, A_S_FULL + sb, (blk >> 1) & 1u)) { ok = false; break; }
      tc_fence_after();
      {
        uint32_t v[32];
        tmem_ld32(trow + kTmS + (uint32_t)(sb * kBT + half * 64), v);
        tmem_wait_ld();
        reg_fence(v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(v[i]);
        tmem_ld32(trow + kTmS + (uint32_t)(sb * kBT + half * 64 + 32), v);
        tmem_wait_ld();
        reg_fence(v);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[32 + i] = __uint_as_float(v[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(A_S_EMPTY + sb));
      // ---- row max over both column halves (extreme raw logit in the scale's direction, then scaled)
      const int nv = min(kBT, max(0, nval - kBT * (pc.lb0 + j)));
      const int c0 = half * 64;
      const bool full_blk = (c0 + 64 <= nv);
      float ext = -INFINITY;
      if (full_blk) {
#pragma unroll
        for (int i = 0; i < 64; ++i) ext = fmaxf(ext, sg * s[i]);
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i) ext = (c0 + i < nv) ? fmaxf(ext, sg * s[i]) : ext;
      }
      const float hmax = (ext == -INFINITY) ? -INFINITY : (sg * ext) * p.scale_log2;
      maxbuf[half * 128 + r] = hmax;
      if (!group_sync(c, nsync)) { ok = false; break; }
      const float cmax = fmaxf(hmax, maxbuf[(half ^ 1) * 128 + r]);
      rm = fmaxf(rm, cmax);
      const bool trig = rm > rmfs + kThresLog2;
      float alpha = 1.f;
      if (trig) {
        alpha = ex2_approx(rmfs - rm);
        se *= alpha;
        rmfs = rm;
      }
      // ---- message slot free?  then exponentials straight into the P tile (this half = one SW128 chunk)
      const int pb = (int)(blk & 1u);
      if (!wait(c, A_POUT_EMPTY + pb, ((blk >> 1) & 1u) ^ 1u, true)) { ok = false; break; }
      uint8_t* msg = smem + Y::A_OffMsg;
      uint8_t* prow = msg + half * kKChunkBytes;
      const float nrm = -rmfs;
      float psum = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float e[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int i = q * 8 + u;
          e[u] = (full_blk || c0 + i < nv) ? ex2_approx(fmaf(s[i], p.scale_log2, nrm)) : 0.f;
          psum += e[u];
        }
        *(uint4*)(prow + sw128_off((uint32_t)r, (uint32_t)q)) =
            make_uint4(pack_bf16x2(e[0], e[1]), pack_bf16x2(e[2], e[3]), pack_bf16x2(e[4], e[5]), pack_bf16x2(e[6], e[7]));
      }
      se += psum;
      const bool last = (j == nb - 1);
      float* tr = (float*)(msg + kMsgPBytes);
      if (half == 0) tr[r] = alpha;
      if (last) {  // total normaliser of this piece (both halves)
        sebuf[half * 128 + r] = se;
        if (!group_sync(c, nsync)) { ok = false; break; }
        if (half == 0) {
          const float se_tot = se + sebuf[128 + r];
          const bool has = se_tot > 0.f;
          tr[128 + r] = has ? 1.f / se_tot : 0.f;
          tr[256 + r] = has ? (rmfs + log2f(se_tot)) * kLn2 : -INFINITY;
        }
      }
      fence_proxy_async_smem();
      if (!group_sync(c, nsync)) { ok = false; break; }
      if (sw == 0 && lane == 0)
        bulk_s2cluster(peer_msg + (uint32_t)pb * kMsgSlot, c.sbase + Y::A_OffMsg, kMsgBytes,
                       peer_pin_full + 8u * (uint32_t)pb);
    }
    ++item;
  }
  if ((!ok || err) && lane == 0) set_abort(c);
}

// ============================================================================ PV side
// FP8 rows: cp.async into a raw ring, dequantised by the same warps into the V row-group ring.
template <int kFmt>
static __device__ void pv_gather_q(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmt>;
  using R = QRow<kFmt>;
  uint8_t* smem = c.smem;
  const int warp = c.warp, lane = c.lane;
  const int gw = (warp == 1) ? 0 : warp - 7;  // 0..8
  const int gt = gw * 32 + lane;
  constexpr int kGT = kGatherWarpsB * 32;
  const int* lists = (const int*)(smem + Y::OffIdx);
  BlockCount bc;
  bc.init(c, p, true);
  bool ok = true, err = false;
  {
    // Per 16-row group one raw unit: the codes and scales at the start of each row (528 bytes for FP8,
    // 320 for FP4), staged two units ahead, then dequantised into the MN-major V row-group ring.
    auto exists = [&](uint32_t u) -> bool { return bc.has(c, p, u / (uint32_t)kGroupsPerBlock, err); };
    auto issue = [&](uint32_t u) -> bool {
      const uint32_t b = u / (uint32_t)kGroupsPerBlock;
      const int g = (int)(u % (uint32_t)kGroupsPerBlock), rs = (int)(u % kRawSlots);
      if (!wait(c, RAW_EMPTY + rs, ((u / kRawSlots) & 1u) ^ 1u)) return false;
      if (g == 0 && !wait(c, IDX_FULL + (int)(b % kIdxSlots), (b / kIdxSlots) & 1u)) return false;
      const int* l = lists + (int)(b % kIdxSlots) * kIdxSlotInts + g * kVGroupRows;
      const uint32_t dst = c.sbase + Y::B_OffRaw + (uint32_t)rs * R::kRawBSlot;
      constexpr int kPer = R::kRawBRow / 16;  // 16-byte pieces per row
      for (int q = gt; q < kVGroupRows * kPer; q += kGT) {
        const int rr = q / kPer, pc = q - rr * kPer;
        cp_async16(dst + (uint32_t)q * 16u, p.kv + (size_t)l[rr] * R::kBytes + 16 * pc);
      }
      cp_async_arrive(c.bar(RAW_FULL + rs));
      return true;
    };
    auto consume = [&](uint32_t u) -> bool {
      const uint32_t b = u / (uint32_t)kGroupsPerBlock;
      const int g = (int)(u % (uint32_t)kGroupsPerBlock), rs = (int)(u % kRawSlots);
      if (!wait(c, RAW_FULL + rs, (u / kRawSlots) & 1u)) return false;
      const int s = (int)(u % Y::kVSlots);
      if (!wait(c, B_V_EMPTY + s, ((u / Y::kVSlots) & 1u) ^ 1u)) return false;
      const uint8_t* raw = smem + Y::B_OffRaw + rs * R::kRawBSlot;
      uint8_t* vd = smem + Y::B_OffV + s * kVGroupBytes;
      if constexpr (!R::kF4) {  // FP8: piece pc of a row = 16 channels; scale per 128 channels
        for (int q = gt; q < kVGroupRows * 32; q += kGT) {
          const int rr = q >> 5, pc = q & 31;
          const uint8_t* rrow = raw + rr * R::kRawBRow;
          uint4 o0, o1;
          dequant16(*(const uint4*)(rrow + pc * 16), *(const float*)(rrow + R::kScaleOff + 4 * (pc >> 3)), o0, o1);
          uint8_t* chunk = vd + (pc >> 2) * 2048;
          *(uint4*)(chunk + sw128_off((uint32_t)rr, (uint32_t)(2 * (pc & 3)))) = o0;
          *(uint4*)(chunk + sw128_off((uint32_t)rr, (uint32_t)(2 * (pc & 3) + 1))) = o1;
        }
      } else {  // FP4: piece pc of a row = 32 channels = its own scale group
        for (int q = gt; q < kVGroupRows * 16; q += kGT) {
          const int rr = q >> 4, pc = q & 15;
          const uint8_t* rrow = raw + rr * R::kRawBRow;
          uint4 o[4];
          dequant32_fp4(*(const uint4*)(rrow + pc * 16), *(const float*)(rrow + R::kScaleOff + 4 * pc), o);
          uint8_t* chunk = vd + (pc >> 1) * 2048;
#pragma unroll
          for (int j = 0; j < 4; ++j) *(uint4*)(chunk + sw128_off((uint32_t)rr, (uint32_t)(4 * (pc & 1) + j))) = o[j];
        }
      }
      mbar_arrive(c.bar(B_V_FULL + s));
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(RAW_EMPTY + rs));
      if (g == kGroupsPerBlock - 1 && lane == 0) mbar_arrive(c.bar(IDX_EMPTY + (int)(b % kIdxSlots)));
      return true;
    };
    for (uint32_t u = 0; u < 2u && ok && exists(u); ++u) ok = issue(u);
    for (uint32_t u = 0; ok && exists(u); ++u) {
      if (exists(u + 2u)) ok = issue(u + 2u);
      if (ok) ok = consume(u);
    }
    if (!ok || err) set_abort(c);
  }
}

// bf16 rows, issuers (warps 8..13): slot group g of block b holds rows 16g..16g+15 as two 8-row units;
// lane j < 16 bulk-copies the 1024 latent bytes (= V) of row 16g + j into unit j / 8 as a plain row.
static __device__ void pv_issue_bf16(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmtBf16>;
  const int lane = c.lane, i = c.warp - 8;
  const int* lists = (const int*)(c.smem + Y::OffIdx);
  BlockCount bc;
  bc.init(c, p, true);
  uint32_t done = 0;  // groups of all blocks before the current one
  bool ok = true, err = false;
  for (uint32_t b = 0; ok && bc.has(c, p, b, err); ++b) {
    const int slot = (int)(b % kIdxSlots);
    if (!wait(c, IDX_FULL + slot, (b / kIdxSlots) & 1u)) { ok = false; break; }
    const int* l = lists + slot * kIdxSlotInts;
    for (int g = i; g < kGroupsPerBlock; g += kIssuersB) {
      const uint32_t gs = done + (uint32_t)g;
      const int s = (int)(gs % Y::kVSlots);
      if (!wait(c, B_V_EMPTY + s, ((gs / Y::kVSlots) & 1u) ^ 1u)) { ok = false; break; }
      const uint32_t land = c.bar(B_V_LAND + s);
      const bool bulk1 = g < kBulkUnit1B;
      const uint32_t grp = c.sbase + Y::B_OffV + (uint32_t)(s * kVGroupBytes);
      if (lane == 0) mbar_arrive_expect_tx(land, bulk1 ? (uint32_t)kVGroupBytes : (uint32_t)kUnitBytes);
      __syncwarp();
      if (lane < (bulk1 ? kVGroupRows : 8))
        bulk_g2s(grp + (uint32_t)((lane >> 3) * kUnitBytes + (lane & 7) * 1024),
                 p.kv + (size_t)l[g * kVGroupRows + lane] * (kDQK * 2), 1024u, land);
      if (!bulk1) cp_async_unit(grp + (uint32_t)kUnitBytes, p.kv, l + g * kVGroupRows + 8, lane);
      cp_async_arrive(land);  // one arrival per lane, whether or not it issued cp.async
    }
    if (!ok) break;
    done += (uint32_t)kGroupsPerBlock;
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(IDX_EMPTY + slot));
  }
  if (!ok || err) set_abort(c);
  // the copies of the last ring round land before the CTA may exit
  for (uint32_t gs = done > (uint32_t)Y::kVSlots ? done - Y::kVSlots : 0u; gs < done; ++gs)
    if ((int)(gs % (uint32_t)kGroupsPerBlock) % kIssuersB == i)
      mbar_wait(c.bar(B_V_LAND + (int)(gs % Y::kVSlots)), (gs / Y::kVSlots) & 1u, kWaitLimitNs, nullptr);
}

// bf16 rows, transposers (warps 1, 14, 15): lay out both units of a landed slot group and hand it to the MMA.
static __device__ void pv_transpose_bf16(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmtBf16>;
  const int lane = c.lane, t = (c.warp == 1) ? 0 : c.warp - 13;
  BlockCount bc;
  bc.init(c, p, true);
  bool ok = true, err = false;
  for (uint32_t gs = (uint32_t)t; bc.has(c, p, gs / (uint32_t)kGroupsPerBlock, err); gs += kTransB) {
    const int s = (int)(gs % Y::kVSlots);
    if (!wait(c, B_V_LAND + s, (gs / Y::kVSlots) & 1u)) { ok = false; break; }
    const uint32_t grp = c.sbase + Y::B_OffV + (uint32_t)(s * kVGroupBytes);
    transpose_unit(grp, lane);
    if ((int)(gs % (uint32_t)kGroupsPerBlock) < kBulkUnit1B) transpose_unit(grp + (uint32_t)kUnitBytes, lane);
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(B_V_FULL + s));
  }
  if (!ok || err) set_abort(c);
}

template <int kFmt>
__device__ void pv_mma(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmt>;
  constexpr bool kQuant = kFmt != kFmtBf16;
  if (c.lane == 0) {
    WorkIter it;
    it.init(c, p, false);
    Piece pc;
    uint32_t gseq = 0, blk = 0, item = 0;
    bool ok = true, err = false;
    while (ok && it.next(c, p, pc, err)) {
      const int nb = pc.lb1 - pc.lb0;
      for (int j = 0; j < nb && ok; ++j, ++blk) {
        const int pb = (int)(blk & 1u);
        if (!wait(c, B_PIN_FULL + pb, (blk >> 1) & 1u) || !wait(c, B_RESC_DONE + pb, (blk >> 1) & 1u)) {
          ok = false;
          break;
        }
        if (j == 0 && !wait(c, B_O_FREE, (item & 1u) ^ 1u)) { ok = false; break; }
        tc_fence_after();
        const uint32_t pmsg = c.sbase + Y::B_OffMsg + (uint32_t)pb * kMsgSlot;
        for (int g = 0; g < kGroupsPerBlock; ++g, ++gseq) {
          const int s = (int)(gseq % Y::kVSlots);
          if (!wait(c, B_V_FULL + s, (gseq / Y::kVSlots) & 1u)) { ok = false; break; }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint64_t adesc = smem_desc(pmsg + (uint32_t)(g >> 2) * kKChunkBytes + (uint32_t)(g & 3) * 32u, 16, 1024);
          const uint32_t vs = c.sbase + Y::B_OffV + (uint32_t)s * kVGroupBytes;
          const uint32_t acc = (j > 0 || g > 0) ? 1u : 0u;
          // V of 16 rows, MN-major: 64-column chunks LBO apart, the two 8-row atoms along K SBO apart.
          // bf16 groups are two transposed units (chunk stride 1 KB, unit stride 8 KB); FP8 groups are
          // dequantised chunk-major (chunk stride 2 KB, atom stride 1 KB).
          constexpr uint32_t kLbo = kQuant ? 2048u : 1024u, kSbo = kQuant ? 1024u : (uint32_t)kUnitBytes;
          mma_ss(c.tmem + 0, adesc, smem_desc(vs, kLbo, kSbo), kIdescPV, acc);
          mma_ss(c.tmem + 256, adesc, smem_desc(vs + 4u * kLbo, kLbo, kSbo), kIdescPV, acc);
          mma_commit(c.bar(B_V_EMPTY + s));
        }
        if (!ok) break;
        mma_commit(c.bar(B_PV_DONE + pb));
        if (j == nb - 1) mma_commit(c.bar(B_O_FULL));
      }
      ++item;
    }
    if (!ok || err) set_abort(c);
    mma_commit(c.bar(B_DRAIN));
    mbar_wait(c.bar(B_DRAIN), 0, kWaitLimitNs, nullptr);
  }
  __syncwarp();
}

// Message slots: arm the receive barrier for the next message, then hand the slot back to the QK side.
__device__ __forceinline__ void pv_slot_return(const Ctx& c, const FwdParams& p) {
  if (c.lane == 0) {
    const uint32_t peer_pout_empty = mapa_shared(c.bars + 8u * (uint32_t)A_POUT_EMPTY, c.peer);
    const uint32_t peer_msg_free = mapa_shared(c.bars + 8u * (uint32_t)A_MSG_FREE, c.peer);
    BlockCount bc;
    bc.init(c, p, false);
    bool ok = true, err = false;
    for (uint32_t b = 0; b < 2 && bc.has(c, p, b, err); ++b) mbar_arrive_expect_tx(c.bar(B_PIN_FULL + (int)b), kMsgBytes);
    for (uint32_t b = 0; bc.has(c, p, b, err); ++b) {
      const int pb = (int)(b & 1u);
      if (!wait(c, B_PIN_FULL + pb, (b >> 1) & 1u)) { ok = false; break; }
      mbar_arrive_remote(peer_msg_free);  // the QK side may refill its outgoing buffer
      if (!wait(c, B_PV_DONE + pb, (b >> 1) & 1u)) { ok = false; break; }
      if (bc.has(c, p, b + 2, err)) mbar_arrive_expect_tx(c.bar(B_PIN_FULL + pb), kMsgBytes);
      mbar_arrive_remote(peer_pout_empty + 8u * (uint32_t)pb);
    }
    if (!ok || err) set_abort(c);
  }
  __syncwarp();
}

template <int kFmt>
__device__ void pv_epilogue(const Ctx& c, const FwdParams& p) {
  using Y = Lay<kFmt>;
  uint8_t* smem = c.smem;
  const int lane = c.lane;
  const int quarter = c.warp & 3;
  const int r = quarter * 32 + lane;
  const uint32_t trow = c.tmem + ((uint32_t)(quarter * 32) << 16);
  WorkIter it;
  it.init(c, p, false);
  Piece pc;
  uint32_t blk = 0, item = 0;
  bool ok = true, err = false;
  while (ok && it.next_warp(c, p, pc, err)) {
    const int nb = pc.lb1 - pc.lb0;
    float inv = 0.f, lse_val = -INFINITY;
    for (int j = 0; j < nb; ++j, ++blk) {
      const int pb = (int)(blk & 1u);
      if (!wait(c, B_PIN_FULL + pb, (blk >> 1) & 1u)) { ok = false; break; }
      const float* tr = (const float*)(smem + Y::B_OffMsg + pb * kMsgSlot + kMsgPBytes);
      const float alpha = tr[r];
      if (j == nb - 1) { inv = tr[128 + r]; lse_val = tr[256 + r]; }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
        // O holds earlier blocks of this token: rescale it once the previous P@V is done
        const uint32_t bp = blk - 1u;
        if (!wait(c, B_PV_DONE + (int)(bp & 1u), (bp >> 1) & 1u)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 16; ++cc) {
          uint32_t v[32];
          tmem_ld32(trow + (uint32_t)(cc * 32), v);
          tmem_wait_ld();
          reg_fence(v);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
          tmem_st32(trow + (uint32_t)(cc * 32), v);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(B_RESC_DONE + pb));
    }
    if (!ok) break;
    // ---- epilogue: O / Z -> bf16 (or the normalised fp32 partial of a split token)
    if (!wait(c, B_O_FULL, item & 1u)) { ok = false; break; }
    tc_fence_after();
    const bool live = r < p.h_q;
#pragma unroll 1
    for (int cc = 0; cc < 16; ++cc) {
      uint32_t v[32];
      const int col = cc * 32;
      tmem_ld32(trow + (uint32_t)col, v);
      tmem_wait_ld();
      reg_fence(v);
      if (live) {
        if (pc.full) {
          uint4* dst = (uint4*)(p.out + ((size_t)pc.t * p.h_q + r) * kDV + col);
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint4 w;
            w.x = pack_bf16x2(__uint_as_float(v[8 * u + 0]) * inv, __uint_as_float(v[8 * u + 1]) * inv);
            w.y = pack_bf16x2(__uint_as_float(v[8 * u + 2]) * inv, __uint_as_float(v[8 * u + 3]) * inv);
            w.z = pack_bf16x2(__uint_as_float(v[8 * u + 4]) * inv, __uint_as_float(v[8 * u + 5]) * inv);
            w.w = pack_bf16x2(__uint_as_float(v[8 * u + 6]) * inv, __uint_as_float(v[8 * u + 7]) * inv);
            dst[u] = w;
          }
        } else {
          float4* dst = (float4*)(p.part_o + ((size_t)pc.slot * p.h_q + r) * kDV + col);
#pragma unroll
          for (int u = 0; u < 8; ++u)
            dst[u] = make_float4(__uint_as_float(v[4 * u]) * inv, __uint_as_float(v[4 * u + 1]) * inv,
                                 __uint_as_float(v[4 * u + 2]) * inv, __uint_as_float(v[4 * u + 3]) * inv);
        }
      }
    }
    if (live) {
      if (pc.full) p.lse[(size_t)pc.t * p.h_q + r] = lse_val;
      else p.part_lse[(size_t)pc.slot * p.h_q + r] = lse_val;
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(c.bar(B_O_FREE));
    ++item;
  }
  if ((!ok || err) && lane == 0) set_abort(c);
}

}  // namespace fwd

template <int kFmt>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(fwd::kThreads, 1) dsa_fwd_kernel(const FwdParams p) {
  using namespace fwd;
  using Y = Lay<kFmt>;
  constexpr bool kQuant = kFmt != kFmtBf16;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Ctx c;
  c.smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  c.sbase = smem_u32(c.smem);
  c.bars = c.sbase + Y::OffBar;
  c.warp = threadIdx.x >> 5;
  c.lane = threadIdx.x & 31;
  c.rank = cluster_ctarank();
  c.peer = c.rank ^ 1u;
  c.pair = (int)(blockIdx.x >> 1);
  volatile uint32_t* tmem_base_ptr = (volatile uint32_t*)(c.smem + Y::OffMisc);
  c.abort_flag = (volatile int*)(c.smem + Y::OffMisc + 16);
  c.peer_abort = mapa_shared(smem_u32((const void*)c.abort_flag), c.peer);
  c.status = p.ctrl + kCtrlStatus;

  if (threadIdx.x == 0) {
    const int gwarps = (c.rank == 0) ? kGatherWarpsA : kGatherWarpsB;
    const int list_users = kQuant ? gwarps : (c.rank == 0 ? kIssuersA : kIssuersB);
    for (int q = 0; q < kIdxSlots; ++q) {
      mbar_init(c.bar(IDX_FULL + q), 1);
      mbar_init(c.bar(IDX_EMPTY + q), list_users);
    }
    for (int q = 0; q < kRawSlots; ++q) {
      mbar_init(c.bar(RAW_FULL + q), gwarps * 32);
      mbar_init(c.bar(RAW_EMPTY + q), gwarps);
    }
    if (c.rank == 0) {
      if constexpr (kQuant) {
        for (int s = 0; s < Y::kKSlots; ++s) {
          mbar_init(c.bar(A_K_FULL + s), kGatherWarpsA * 32);
          mbar_init(c.bar(A_K_EMPTY + s), 1);
        }
      } else {
        for (int g = 0; g < 2 * kGroupsPerHalf; ++g) mbar_init(c.bar(A_LAND + g), 1 + 32);  // expect_tx + cp.async
        for (int h = 0; h < 2; ++h) {
          mbar_init(c.bar(A_KH_FULL + h), kGroupsPerHalf);
          mbar_init(c.bar(A_KH_EMPTY + h), 1);
        }
      }
      mbar_init(c.bar(A_MSG_FREE), 1);
      for (int b = 0; b < 2; ++b) {
        mbar_init(c.bar(A_S_FULL + b), 1);
        mbar_init(c.bar(A_S_EMPTY + b), kSoftmaxWarps);
        mbar_init(c.bar(A_POUT_EMPTY + b), 1);
      }
      mbar_init(c.bar(A_Q_FULL), kSoftmaxWarps);
      mbar_init(c.bar(A_Q_FREE), 1);
      mbar_init(c.bar(A_SMX_SYNC), kSoftmaxWarps);
      mbar_init(c.bar(A_DRAIN), 1);
    } else {
      for (int s = 0; s < Y::kVSlots; ++s) {
        mbar_init(c.bar(B_V_FULL + s), kQuant ? kGatherWarpsB * 32 : 1);
        mbar_init(c.bar(B_V_EMPTY + s), 1);
        mbar_init(c.bar(B_V_LAND + s), 1 + 32);  // expect_tx + cp.async
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(c.bar(B_PIN_FULL + b), 1);
        mbar_init(c.bar(B_RESC_DONE + b), kEpiWarps);
        mbar_init(c.bar(B_PV_DONE + b), 1);
      }
      mbar_init(c.bar(B_O_FULL), 1);
      mbar_init(c.bar(B_O_FREE), kEpiWarps);
      mbar_init(c.bar(B_DRAIN), 1);
    }
    *c.abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (c.warp == 3) {
    tmem_alloc(smem_u32((const void*)tmem_base_ptr), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive or copy
  c.tmem = *tmem_base_ptr;

  const int w = c.warp;
  if (w == 0) {
    index_compactor<kFmt>(c, p);
  } else if (w == 2) {
    if (c.rank == 0) qk_mma<kFmt>(c, p);
    else pv_mma<kFmt>(c, p);
  } else if (c.rank == 0) {
    if constexpr (kQuant) {
      if (w == 1 || w == 3 || w >= 12) qk_gather_q<kFmt>(c, p);
      else if (w >= 4) qk_softmax<kFmt>(c, p);
    } else {
      if (w >= 12) qk_issue_bf16(c, p);
      else if (w >= 4) qk_softmax<kFmt>(c, p);
      else qk_transpose_bf16(c, p);  // warps 1, 3
    }
  } else {
    if constexpr (kQuant) {
      if (w == 1 || w >= 8) pv_gather_q<kFmt>(c, p);
      else if (w == 3) pv_slot_return(c, p);
      else if (w >= 4) pv_epilogue<kFmt>(c, p);
    } else {
      if (w >= 8 && w < 14) pv_issue_bf16(c, p);
      else if (w == 1 || w >= 14) pv_transpose_bf16(c, p);
      else if (w == 3) pv_slot_return(c, p);
      else if (w >= 4) pv_epilogue<kFmt>(c, p);
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (c.warp == 3) tmem_dealloc(c.tmem, kTmemCols);
  cluster_sync();  // no remote copy or arrive may target an exited CTA
}

// Largest number of 2-CTA clusters of the kernel that fit at once on the current device.
template <int kFmt>
int max_active_pairs_impl() {
  static int cached = -1;
  static int cached_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cached >= 0 && cached_dev == dev) return cached;
  constexpr int smem = fwd::Lay<kFmt>::SmemAlloc;
  if (cudaFuncSetAttribute(dsa_fwd_kernel<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * sms, 1, 1);
  cfg.blockDim = dim3(fwd::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, dsa_fwd_kernel<kFmt>, &cfg) != cudaSuccess || nclusters <= 0) {
    cudaGetLastError();
    return 0;
  }
  cached = nclusters;
  cached_dev = dev;
  return cached;
}

template <int kFmt>
cudaError_t launch_impl(const FwdParams& p, cudaStream_t stream) {
  constexpr int smem = fwd::Lay<kFmt>::SmemAlloc;
  cudaError_t e = cudaFuncSetAttribute(dsa_fwd_kernel<kFmt>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  dsa_fwd_kernel<kFmt><<<2 * p.npairs, fwd::kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa

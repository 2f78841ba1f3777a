// The sparse MLA forward kernel for sm_103a (bf16 KV cache).
//
// Method: "Ascend Sparse Attention Forward 算法与优化技术简析", sections
// "数学建模" (what is computed) and "计算流程" (blockwise online softmax with
// skip-scale).  The page's delayed P@V order (section "流水线") survives as
// a pipeline across two SMs; its index prefetch / multi-stage gather idea
// survives as chunk rings fed by cp.async.
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
//   * Gathers use cp.async (16 bytes per thread) with the address swizzled on
//     the way in, straight into the 128-byte-swizzled layouts tcgen05.mma
//     reads: 16 KB chunks of 128 rows x 64 columns (K-major) on the QK side,
//     16 KB row groups of 16 rows x 512 columns (MN-major) on the PV side.
//   * Work: the index blocks of all tokens form one sequence; pair p takes the
//     contiguous range [p*T/P, (p+1)*T/P).  A token cut by a range boundary is
//     written as normalised partials and merged by the combine kernel.
//
// Warp roles (384 threads, both CTAs): warps 0-1 gather (index compaction +
// cp.async), warp 2 issues tcgen05.mma, warp 3 owns the TMEM allocation (and,
// on the PV side, returns P slots to the QK side), warps 4-11 run the
// softmax (QK side) or the rescale / epilogue (PV side); warp w of them
// serves TMEM lane quarter w % 4 and column half (w - 4) / 4.
#include <cuda.h>
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {

namespace fwd {

constexpr int kThreads = 384;
constexpr int kProducerWarps = 2;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kSoftmaxWarps = 8;

// ---- QK side (cluster rank 0) shared memory
constexpr int kKChunkBytes = 128 * 128;           // 128 rows x 64 bf16 columns, SW128 K-major
constexpr int kKSlots = 8;                        // ring of KV column chunks
constexpr int kChunksPerBlock = 9;                // 576 / 64
constexpr int kMsgPBytes = 2 * kKChunkBytes;      // P[128 rows, 128 cols] bf16 = two SW128 chunks
constexpr int kMsgTrailer = 3 * 128 * 4 + 16;     // alpha[128], inv_se[128], lse[128], flags
constexpr int kMsgBytes = kMsgPBytes + kMsgTrailer;
constexpr int kMsgSlot = 34816;                   // 34 KB, 1024-aligned slots
static_assert(kMsgBytes <= kMsgSlot && kMsgBytes % 16 == 0, "message layout");
constexpr int kA_OffK = 0;
constexpr int kA_OffQRope = kA_OffK + kKSlots * kKChunkBytes;   // 128 KB
constexpr int kA_OffMsg = kA_OffQRope + kKChunkBytes;           // +16 KB
constexpr int kA_OffMax = kA_OffMsg + 2 * kMsgSlot;             // [2 halves][128] float
constexpr int kA_OffSe = kA_OffMax + 2 * 128 * 4;
constexpr int kA_End = kA_OffSe + 2 * 128 * 4;

// ---- PV side (cluster rank 1) shared memory
constexpr int kVGroupRows = 16;
constexpr int kVGroupBytes = kVGroupRows * 1024;  // 16 rows x 512 columns bf16 = 8 chunks x 2 KB
constexpr int kVSlots = 9;
constexpr int kGroupsPerBlock = 128 / kVGroupRows;
constexpr int kB_OffV = 0;
constexpr int kB_OffMsg = kB_OffV + kVSlots * kVGroupBytes;     // 144 KB
constexpr int kB_End = kB_OffMsg + 2 * kMsgSlot;

// ---- common tail: index rings (one per producer warp), barriers, misc
constexpr int kIdxRing = 256;
constexpr int kOffCommon = (kA_End > kB_End ? kA_End : kB_End);
constexpr int kOffRing = (kOffCommon + 127) / 128 * 128;
constexpr int kOffBar = kOffRing + kProducerWarps * kIdxRing * 4;
constexpr int kNumBars = 48;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 64;
constexpr int kSmemAlloc = kSmemUsed + 1024;
static_assert(kSmemAlloc <= 232448, "shared memory budget");

// barrier slots
enum BarA {
  A_K_FULL = 0, A_K_EMPTY = A_K_FULL + kKSlots, A_S_FULL = A_K_EMPTY + kKSlots, A_S_EMPTY = A_S_FULL + 2,
  A_Q_FULL = A_S_EMPTY + 2, A_Q_FREE, A_POUT_EMPTY, A_SMX_SYNC = A_POUT_EMPTY + 2, A_DRAIN, A_NUM
};
enum BarB {
  B_V_FULL = 0, B_V_EMPTY = B_V_FULL + kVSlots, B_PIN_FULL = B_V_EMPTY + kVSlots, B_RESC_DONE = B_PIN_FULL + 2,
  B_PV_DONE = B_RESC_DONE + 2, B_O_FULL = B_PV_DONE + 2, B_O_FREE, B_DRAIN, B_NUM
};
static_assert((int)A_NUM <= kNumBars && (int)B_NUM <= kNumBars, "barrier slots");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmQ = 0;     // QK side: Q latent [0, 256) (bf16 pairs), S tiles [256, 384) and [384, 512)
constexpr uint32_t kTmS = 256;
constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kBT, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);

constexpr float kThresLog2 = 6.0f * 1.4426950408889634f;  // RESCALE_THRES = 6 (natural log) in log2 units
constexpr float kLn2 = 0.6931471805599453f;

struct Piece {
  int t, lb0, lb1;
  bool full;
  int slot;
};

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
    int lo = 0, hi = s_q - 1;
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
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

// Index compaction into a per-warp ring: valid slots of token t in order.
struct IndexRing {
  int* ring;
  const int32_t* idx_t;
  int topk, s_kv, head, tail, rp;
  __device__ void reset(int* r, const int32_t* p, int tk, int skv) {
    ring = r; idx_t = p; topk = tk; s_kv = skv; head = tail = rp = 0;
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
      for (int q = 0; q < 4; ++q) {
        const bool ok = (v[q] >= 0) && (v[q] < s_kv);
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

// ============================================================================ QK side
__device__ void qk_side(const Ctx& c, const FwdParams& p) {
  uint8_t* smem = c.smem;
  const int warp = c.warp, lane = c.lane;
  if (warp < kProducerWarps) {
    // ---------------------------------------------------------------- gather K chunks
    IndexRing ir;
    const int pt = warp * 32 + lane;  // 0..63
    const int piece16 = pt & 7, rsub = pt >> 3;
    PieceIter it;
    it.init(p.cum, p.s_q, c.pair, p.npairs);
    Piece pc;
    uint32_t cseq = 0;
    bool ok = true;
    while (ok && it.next(pc)) {
      ir.reset((int*)(smem + kOffRing) + warp * kIdxRing, p.indices + (size_t)pc.t * p.topk, p.topk, p.s_kv);
      for (int jb = 0; jb < pc.lb1 && ok; ++jb) {
        const int cnt = ir.fill(lane);
        if (jb >= pc.lb0) {
          // row base pointers of this thread's 16 rows (r = rsub + 8 i)
          const uint8_t* rowp[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int r = rsub + 8 * i;
            rowp[i] = p.kv + (size_t)(r < cnt ? ir.at(r) : 0) * (kDQK * 2) + piece16 * 16;
          }
          for (int k = 0; k < kChunksPerBlock; ++k, ++cseq) {
            const int s = (int)(cseq % kKSlots);
            if (!wait(c, A_K_EMPTY + s, ((cseq / kKSlots) & 1u) ^ 1u)) { ok = false; break; }
            const uint32_t dst = c.sbase + kA_OffK + (uint32_t)s * kKChunkBytes;
#pragma unroll
            for (int i = 0; i < 16; ++i) cp_async16(dst + sw128_off(rsub + 8 * i, piece16), rowp[i] + k * 128);
            cp_async_arrive(c.bar(A_K_FULL + s));
          }
        }
        ir.pop(cnt);
      }
    }
    if (!ok) set_abort(c);
    // all issued copies land before exit
    const uint32_t first = cseq > (uint32_t)kKSlots ? cseq - kKSlots : 0u;
    for (uint32_t q = first; q < cseq; ++q) mbar_wait(c.bar(A_K_FULL + (int)(q % kKSlots)), (q / kKSlots) & 1u, kWaitLimitNs, nullptr);
  } else if (warp == 2) {
    // ---------------------------------------------------------------- MMA issuer (QK)
    if (lane == 0) {
      PieceIter it;
      it.init(p.cum, p.s_q, c.pair, p.npairs);
      Piece pc;
      uint32_t cseq = 0, blk = 0, item = 0;
      bool ok = true;
      const uint32_t qrope = c.sbase + kA_OffQRope;
      while (ok && it.next(pc)) {
        const int nb = pc.lb1 - pc.lb0;
        if (!wait(c, A_Q_FULL, item & 1u)) { ok = false; break; }
        for (int j = 0; j < nb && ok; ++j, ++blk) {
          const int sb = (int)(blk & 1u);
          if (!wait(c, A_S_EMPTY + sb, ((blk >> 1) & 1u) ^ 1u)) { ok = false; break; }
          tc_fence_after();
          const uint32_t dS = c.tmem + kTmS + (uint32_t)sb * kBT;
          for (int k = 0; k < kChunksPerBlock; ++k, ++cseq) {
            const int s = (int)(cseq % kKSlots);
            if (!wait(c, A_K_FULL + s, (cseq / kKSlots) & 1u)) { ok = false; break; }
            fence_proxy_async_smem();  // cp.async (generic proxy) data -> tensor core reads
            tc_fence_after();
            const uint32_t chunk = c.sbase + kA_OffK + (uint32_t)s * kKChunkBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bdesc = smem_desc(chunk + (uint32_t)kk * 32u, 16, 1024);
              const uint32_t acc = (k > 0 || kk > 0) ? 1u : 0u;
              if (k < 8) mma_ts(dS, c.tmem + kTmQ + (uint32_t)(k * 32 + kk * 8), bdesc, kIdescQK, acc);
              else mma_ss(dS, smem_desc(qrope + (uint32_t)kk * 32u, 16, 1024), bdesc, kIdescQK, acc);
            }
            mma_commit(c.bar(A_K_EMPTY + s));
          }
          if (!ok) break;
          mma_commit(c.bar(A_S_FULL + sb));
        }
        mma_commit(c.bar(A_Q_FREE));
        ++item;
      }
      if (!ok) set_abort(c);
      mma_commit(c.bar(A_DRAIN));
      mbar_wait(c.bar(A_DRAIN), 0, kWaitLimitNs, nullptr);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- softmax (8 warps)
    const int sw = warp - 4;
    const int quarter = warp & 3, half = sw >> 2;
    const int r = quarter * 32 + lane;  // head row = TMEM lane
    const uint32_t trow = c.tmem + ((uint32_t)(quarter * 32) << 16);
    float* maxbuf = (float*)(smem + kA_OffMax);
    float* sebuf = (float*)(smem + kA_OffSe);
    const uint32_t peer_msg = mapa_shared(c.sbase + kB_OffMsg, c.peer);
    const uint32_t peer_pin_full = mapa_shared(c.bars + 8u * (uint32_t)B_PIN_FULL, c.peer);
    PieceIter it;
    it.init(p.cum, p.s_q, c.pair, p.npairs);
    Piece pc;
    uint32_t blk = 0, item = 0, nsync = 0;
    bool ok = true;
    while (ok && it.next(pc)) {
      const int nb = pc.lb1 - pc.lb0;
      const int nval = p.nvalid[pc.t];
      // ---- Q for this token: latent columns [256*half, +256) into TMEM, rope (half 0) into smem
      if (!wait(c, A_Q_FREE, (item & 1u) ^ 1u)) { ok = false; break; }
      tc_fence_after();
      {
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
          uint8_t* qr = smem + kA_OffQRope;
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
        // ---- row max over both column halves
        const int nv = min(kBT, max(0, nval - kBT * (pc.lb0 + j)));
        const int c0 = half * 64;
        float hmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i) {
          s[i] = (c0 + i < nv) ? s[i] * p.scale_log2 : -INFINITY;
          hmax = fmaxf(hmax, s[i]);
        }
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
        float psum = 0.f;
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float e0 = (c0 + i < nv) ? ex2_approx(s[i] - rmfs) : 0.f;
          const float e1 = (c0 + i + 1 < nv) ? ex2_approx(s[i + 1] - rmfs) : 0.f;
          psum += e0 + e1;
          pk[i / 2] = pack_bf16x2(e0, e1);
        }
        se += psum;
        const bool last = (j == nb - 1);
        float se_tot = 0.f;
        if (last) {  // total normaliser of this piece (both halves)
          sebuf[half * 128 + r] = se;
          if (!group_sync(c, nsync)) { ok = false; break; }
          se_tot = se + sebuf[(half ^ 1) * 128 + r];
        }
        // ---- message: P tile (this half = one SW128 chunk) + trailer
        const int pb = (int)(blk & 1u);
        if (!wait(c, A_POUT_EMPTY + pb, ((blk >> 1) & 1u) ^ 1u, true)) { ok = false; break; }
        uint8_t* msg = smem + kA_OffMsg + pb * kMsgSlot;
        {
          uint8_t* prow = msg + half * kKChunkBytes;
#pragma unroll
          for (int q = 0; q < 8; ++q)
            *(uint4*)(prow + sw128_off((uint32_t)r, (uint32_t)q)) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
          float* tr = (float*)(msg + kMsgPBytes);
          if (half == 0) {
            tr[r] = alpha;
            if (last) {
              const bool has = se_tot > 0.f;
              tr[128 + r] = has ? 1.f / se_tot : 0.f;
              tr[256 + r] = has ? (rmfs + log2f(se_tot)) * kLn2 : -INFINITY;
            }
          }
        }
        fence_proxy_async_smem();
        if (!group_sync(c, nsync)) { ok = false; break; }
        if (sw == 0 && lane == 0)
          bulk_s2cluster(peer_msg + (uint32_t)pb * kMsgSlot, c.sbase + kA_OffMsg + (uint32_t)pb * kMsgSlot, kMsgBytes,
                         peer_pin_full + 8u * (uint32_t)pb);
      }
      ++item;
    }
    if (!ok && lane == 0) set_abort(c);
  }
}

// ============================================================================ PV side
__device__ void pv_side(const Ctx& c, const FwdParams& p) {
  uint8_t* smem = c.smem;
  const int warp = c.warp, lane = c.lane;
  if (warp < kProducerWarps) {
    // ---------------------------------------------------------------- gather V row groups (columns 0..511)
    IndexRing ir;
    const int pt = warp * 32 + lane;
    const int piece16 = pt & 7, chunk = pt >> 3;  // chunk 0..7 of 64 columns
    PieceIter it;
    it.init(p.cum, p.s_q, c.pair, p.npairs);
    Piece pc;
    uint32_t gseq = 0;
    bool ok = true;
    while (ok && it.next(pc)) {
      ir.reset((int*)(smem + kOffRing) + warp * kIdxRing, p.indices + (size_t)pc.t * p.topk, p.topk, p.s_kv);
      for (int jb = 0; jb < pc.lb1 && ok; ++jb) {
        const int cnt = ir.fill(lane);
        if (jb >= pc.lb0) {
          for (int g = 0; g < kGroupsPerBlock; ++g, ++gseq) {
            const int s = (int)(gseq % kVSlots);
            if (!wait(c, B_V_EMPTY + s, ((gseq / kVSlots) & 1u) ^ 1u)) { ok = false; break; }
            const uint32_t dst = c.sbase + kB_OffV + (uint32_t)s * kVGroupBytes + (uint32_t)chunk * 2048u;
#pragma unroll
            for (int rr = 0; rr < kVGroupRows; ++rr) {
              const int row = g * kVGroupRows + rr;
              const uint8_t* src = p.kv + (size_t)(row < cnt ? ir.at(row) : 0) * (kDQK * 2) + chunk * 128 + piece16 * 16;
              cp_async16(dst + sw128_off((uint32_t)rr, (uint32_t)piece16), src);
            }
            cp_async_arrive(c.bar(B_V_FULL + s));
          }
        }
        ir.pop(cnt);
      }
    }
    if (!ok) set_abort(c);
    const uint32_t first = gseq > (uint32_t)kVSlots ? gseq - kVSlots : 0u;
    for (uint32_t q = first; q < gseq; ++q) mbar_wait(c.bar(B_V_FULL + (int)(q % kVSlots)), (q / kVSlots) & 1u, kWaitLimitNs, nullptr);
  } else if (warp == 2) {
    // ---------------------------------------------------------------- MMA issuer (PV)
    if (lane == 0) {
      PieceIter it;
      it.init(p.cum, p.s_q, c.pair, p.npairs);
      Piece pc;
      uint32_t gseq = 0, blk = 0, item = 0;
      bool ok = true;
      while (ok && it.next(pc)) {
        const int nb = pc.lb1 - pc.lb0;
        for (int j = 0; j < nb && ok; ++j, ++blk) {
          const int pb = (int)(blk & 1u);
          if (!wait(c, B_PIN_FULL + pb, (blk >> 1) & 1u) || !wait(c, B_RESC_DONE + pb, (blk >> 1) & 1u)) { ok = false; break; }
          if (j == 0 && !wait(c, B_O_FREE, (item & 1u) ^ 1u)) { ok = false; break; }
          tc_fence_after();
          const uint32_t pmsg = c.sbase + kB_OffMsg + (uint32_t)pb * kMsgSlot;
          for (int g = 0; g < kGroupsPerBlock; ++g, ++gseq) {
            const int s = (int)(gseq % kVSlots);
            if (!wait(c, B_V_FULL + s, (gseq / kVSlots) & 1u)) { ok = false; break; }
            fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t adesc = smem_desc(pmsg + (uint32_t)(g >> 2) * kKChunkBytes + (uint32_t)(g & 3) * 32u, 16, 1024);
            const uint32_t vs = c.sbase + kB_OffV + (uint32_t)s * kVGroupBytes;
            const uint32_t acc = (j > 0 || g > 0) ? 1u : 0u;
            mma_ss(c.tmem + 0, adesc, smem_desc(vs, 2048, 1024), kIdescPV, acc);
            mma_ss(c.tmem + 256, adesc, smem_desc(vs + 4u * 2048u, 2048, 1024), kIdescPV, acc);
            mma_commit(c.bar(B_V_EMPTY + s));
          }
          if (!ok) break;
          mma_commit(c.bar(B_PV_DONE + pb));
          if (j == nb - 1) mma_commit(c.bar(B_O_FULL));
        }
        ++item;
      }
      if (!ok) set_abort(c);
      mma_commit(c.bar(B_DRAIN));
      mbar_wait(c.bar(B_DRAIN), 0, kWaitLimitNs, nullptr);
    }
    __syncwarp();
  } else if (warp == 3) {
    // ---------------------------------------------------------------- message slots: arm, then hand back
    if (lane == 0) {
      const uint32_t peer_pout_empty = mapa_shared(c.bars + 8u * (uint32_t)A_POUT_EMPTY, c.peer);
      PieceIter it;
      it.init(p.cum, p.s_q, c.pair, p.npairs);
      Piece pc;
      uint32_t nblk = 0;
      while (it.next(pc)) nblk += (uint32_t)(pc.lb1 - pc.lb0);
      bool ok = true;
      for (uint32_t b = 0; b < nblk && b < 2; ++b) mbar_arrive_expect_tx(c.bar(B_PIN_FULL + (int)b), kMsgBytes);
      for (uint32_t b = 0; b < nblk; ++b) {
        const int pb = (int)(b & 1u);
        if (!wait(c, B_PV_DONE + pb, (b >> 1) & 1u)) { ok = false; break; }
        if (b + 2 < nblk) mbar_arrive_expect_tx(c.bar(B_PIN_FULL + pb), kMsgBytes);
        mbar_arrive_remote(peer_pout_empty + 8u * (uint32_t)pb);
      }
      if (!ok) set_abort(c);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ---------------------------------------------------------------- rescale + epilogue (8 warps)
    const int sw = warp - 4;
    const int quarter = warp & 3, half = sw >> 2;
    const int r = quarter * 32 + lane;
    const uint32_t trow = c.tmem + ((uint32_t)(quarter * 32) << 16);
    PieceIter it;
    it.init(p.cum, p.s_q, c.pair, p.npairs);
    Piece pc;
    uint32_t blk = 0, item = 0;
    bool ok = true;
    while (ok && it.next(pc)) {
      const int nb = pc.lb1 - pc.lb0;
      float inv = 0.f, lse_val = -INFINITY;
      for (int j = 0; j < nb; ++j, ++blk) {
        const int pb = (int)(blk & 1u);
        if (!wait(c, B_PIN_FULL + pb, (blk >> 1) & 1u)) { ok = false; break; }
        const float* tr = (const float*)(smem + kB_OffMsg + pb * kMsgSlot + kMsgPBytes);
        const float alpha = tr[r];
        if (j == nb - 1) { inv = tr[128 + r]; lse_val = tr[256 + r]; }
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
          const uint32_t bp = blk - 1u;
          if (!wait(c, B_PV_DONE + (int)(bp & 1u), (bp >> 1) & 1u)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t v[32];
            const uint32_t col = (uint32_t)(half * 256 + cc * 32);
            tmem_ld32(trow + col, v);
            tmem_wait_ld();
            reg_fence(v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(trow + col, v);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(c.bar(B_RESC_DONE + pb));
      }
      if (!ok) break;
      // ---- epilogue: O[:, 256*half : +256] / Z -> bf16 (or normalised fp32 partial)
      if (!wait(c, B_O_FULL, item & 1u)) { ok = false; break; }
      tc_fence_after();
      const bool live = r < p.h_q;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t v[32];
        const int col = half * 256 + cc * 32;
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
      if (live && half == 0) {
        if (pc.full) p.lse[(size_t)pc.t * p.h_q + r] = lse_val;
        else p.part_lse[(size_t)pc.slot * p.h_q + r] = lse_val;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(c.bar(B_O_FREE));
      ++item;
    }
    if (!ok && lane == 0) set_abort(c);
  }
}

}  // namespace fwd

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(fwd::kThreads, 1)
    dsa_fwd_bf16_kernel(const FwdParams p) {
  using namespace fwd;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  Ctx c;
  c.smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  c.sbase = smem_u32(c.smem);
  c.bars = c.sbase + kOffBar;
  c.warp = threadIdx.x >> 5;
  c.lane = threadIdx.x & 31;
  c.rank = cluster_ctarank();
  c.peer = c.rank ^ 1u;
  c.pair = (int)(blockIdx.x >> 1);
  volatile uint32_t* tmem_base_ptr = (volatile uint32_t*)(c.smem + kOffMisc);
  c.abort_flag = (volatile int*)(c.smem + kOffMisc + 16);
  c.peer_abort = mapa_shared(smem_u32((const void*)c.abort_flag), c.peer);
  c.status = p.ctrl + kCtrlStatus;

  if (threadIdx.x == 0) {
    if (c.rank == 0) {
      for (int s = 0; s < kKSlots; ++s) {
        mbar_init(c.bar(A_K_FULL + s), kProducerThreads);
        mbar_init(c.bar(A_K_EMPTY + s), 1);
      }
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
      for (int s = 0; s < kVSlots; ++s) {
        mbar_init(c.bar(B_V_FULL + s), kProducerThreads);
        mbar_init(c.bar(B_V_EMPTY + s), 1);
      }
      for (int b = 0; b < 2; ++b) {
        mbar_init(c.bar(B_PIN_FULL + b), 1);
        mbar_init(c.bar(B_RESC_DONE + b), kSoftmaxWarps);
        mbar_init(c.bar(B_PV_DONE + b), 1);
      }
      mbar_init(c.bar(B_O_FULL), 1);
      mbar_init(c.bar(B_O_FREE), kSoftmaxWarps);
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

  if (c.rank == 0) qk_side(c, p);
  else pv_side(c, p);

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (c.warp == 3) tmem_dealloc(c.tmem, kTmemCols);
  cluster_sync();  // no remote copy or arrive may target an exited CTA
}

int fwd_max_active_pairs() {
  static int cached = -1;
  static int cached_dev = -1;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cached >= 0 && cached_dev == dev) return cached;
  if (cudaFuncSetAttribute(dsa_fwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::kSmemAlloc) !=
      cudaSuccess)
    return 0;
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * sms, 1, 1);
  cfg.blockDim = dim3(fwd::kThreads, 1, 1);
  cfg.dynamicSmemBytes = fwd::kSmemAlloc;
  int nclusters = 0;
  if (cudaOccupancyMaxActiveClusters(&nclusters, dsa_fwd_bf16_kernel, &cfg) != cudaSuccess || nclusters <= 0) {
    cudaGetLastError();
    return 0;
  }
  cached = nclusters;
  cached_dev = dev;
  return cached;
}

cudaError_t launch_fwd_bf16(const FwdParams& p, cudaStream_t stream) {
  cudaError_t e =
      cudaFuncSetAttribute(dsa_fwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::kSmemAlloc);
  if (e != cudaSuccess) return e;
  dsa_fwd_bf16_kernel<<<2 * p.npairs, fwd::kThreads, fwd::kSmemAlloc, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dsa

// The sparse MLA forward kernel for sm_103a (bf16 KV cache).
//
// Method: "Ascend Sparse Attention Forward 算法与优化技术简析", sections
// "数学建模" (what is computed) and "计算流程" (blockwise online softmax with
// skip-scale).  The schedule keeps the page's delayed P@V order (section
// "流水线": the QK product of block i+1 is issued before the PV product of
// block i so the softmax of block i overlaps the tensor cores) and its index
// prefetch / multi-stage gather idea; the hardware mapping is new.
//
// Mapping onto a GB300 SM pair (one 2-CTA cluster per unit of work):
//   * 128 heads x 512 fp32 output columns would fill one SM's whole tensor
//     memory, so the pair splits the output: CTA r keeps O[:, 256r : 256r+256].
//   * The QK product is split along d_qk: CTA 0 multiplies columns [0, 288),
//     CTA 1 columns [288, 576).  Each holds its 288 Q columns in tensor memory
//     (the MMA A operand) for the whole token.  The two partial logit tiles are
//     exchanged through distributed shared memory, so both CTAs hold the same
//     float32 logits and take the same softmax decisions.
//   * Each CTA gathers only the 64-column chunks it needs: CTA 0 chunks 0-4
//     (columns 0..319), CTA 1 chunks 4-8 (columns 256..575), with TMA gather4
//     straight into the 128-byte-swizzled layout the MMA reads.  Chunks 0-3 of
//     a stage are then the V operand (MN-major) of the CTA's PV product.
//   * Work: the index blocks of all tokens form one sequence; pair p takes the
//     contiguous range [p*T/P, (p+1)*T/P).  A token cut by a range boundary is
//     written as normalised partials and merged by the combine kernel.
//
// Warp roles (256 threads): warp 0 gathers (index compaction + TMA), warp 1
// issues tcgen05.mma, warp 2 owns the tensor-memory allocation, warps 4-7
// run the softmax (thread = head row = TMEM lane) and the epilogue.
#include <cuda.h>
#include <cuda_runtime.h>

#include "dsa_internal.h"
#include "ptx.cuh"

namespace dsa {

namespace fwd {

constexpr int kStages = 3;
constexpr int kChunks = 5;                       // 64-column chunks gathered per CTA
constexpr int kQkSteps = 18;                     // 16-column K steps of the QK product per CTA
constexpr int kChunkBytes = kBT * 128;           // 64 rows x 128 bytes
constexpr int kStageBytes = kChunks * kChunkBytes;
constexpr int kPBytes = 128 * 128;               // 128 rows x 64 bf16
constexpr int kXBytes = 128 * kBT * 4;           // 128 rows x 64 fp32
constexpr int kOffStage = 0;
constexpr int kOffP = kOffStage + kStages * kStageBytes;
constexpr int kOffX = kOffP + 2 * kPBytes;
constexpr int kOffRing = kOffX + 2 * kXBytes;
constexpr int kRing = 128;
constexpr int kOffBar = kOffRing + kRing * 4;
constexpr int kNumBars = 20;
constexpr int kOffMisc = kOffBar + kNumBars * 8;
constexpr int kSmemUsed = kOffMisc + 64;
constexpr int kSmemAlloc = kSmemUsed + 1024;

enum Bar {
  KV_FULL = 0, KV_EMPTY = kStages, S_FULL = 2 * kStages, S_EMPTY, P_FULL, P_EMPTY = P_FULL + 2,
  X_FULL = P_EMPTY + 2, X_EMPTY = X_FULL + 2, Q_FULL = X_EMPTY + 2, O_FULL, O_FREE, DRAIN
};
static_assert(DRAIN < kNumBars, "barrier slots");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmO = 0;      // [0, 256)   fp32 output accumulator (this CTA's 256 columns)
constexpr uint32_t kTmQ = 256;    // [256, 400) bf16 Q, 288 columns packed in pairs
constexpr uint32_t kTmS = 400;    // [400, 464) fp32 partial logits of one block

constexpr uint32_t kIdescQK = idesc_bf16_f32(128, kBT, 0, 0);
constexpr uint32_t kIdescPV = idesc_bf16_f32(128, 256, 0, 1);

constexpr float kThresLog2 = 6.0f * 1.4426950408889634f;  // RESCALE_THRES = 6 (natural log) in log2 units
constexpr float kLn2 = 0.6931471805599453f;

// One contiguous run of index blocks of one token.
struct Piece {
  int t, lb0, lb1;   // token, first and one-past-last block (within the token)
  bool full;         // covers all blocks of the token
  int slot;          // partial-output slot when !full
};

// Iterates the pieces of pair p's range [g0, g1) of the global block sequence.
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
    // largest t with cum[t] <= g
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

__device__ __forceinline__ void set_abort(volatile int* abort_flag, int* status, uint32_t peer_abort_addr) {
  if (!*abort_flag) {
    *abort_flag = 1;
    atomicCAS(status, 0, 5 /* DSA_ERR_DEVICE_TIMEOUT */);
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort_addr), "r"(1) : "memory");
  }
}

__device__ __forceinline__ uint32_t sw128_off(uint32_t row, uint32_t chunk16) {
  return (row >> 3) * 1024 + (row & 7) * 128 + ((chunk16 ^ (row & 7)) << 4);
}

}  // namespace fwd

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(256, 1)
    dsa_fwd_bf16_kernel(const __grid_constant__ CUtensorMap tmap_kv, const FwdParams p) {
  using namespace fwd;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = (uint8_t*)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBar;
  auto bar = [&](int i) -> uint32_t { return bars + 8u * (uint32_t)i; };
  volatile uint32_t* tmem_base_ptr = (volatile uint32_t*)(smem + kOffMisc);
  volatile int* abort_flag = (volatile int*)(smem + kOffMisc + 16);
  int* ring = (int*)(smem + kOffRing);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const uint32_t peer = rank ^ 1u;
  const int pair = (int)(blockIdx.x >> 1);
  const uint32_t peer_abort = mapa_shared(smem_u32((const void*)abort_flag), peer);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar(KV_FULL + s), 1);
      mbar_init(bar(KV_EMPTY + s), 1);
    }
    mbar_init(bar(S_FULL), 1);
    mbar_init(bar(S_EMPTY), 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(P_FULL + b), 4);
      mbar_init(bar(P_EMPTY + b), 1);
      mbar_init(bar(X_FULL + b), 128);
      mbar_init(bar(X_EMPTY + b), 128);
    }
    mbar_init(bar(Q_FULL), 4);
    mbar_init(bar(O_FULL), 1);
    mbar_init(bar(O_FREE), 4);
    mbar_init(bar(DRAIN), 1);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 2) {
    tmem_alloc(smem_u32((const void*)tmem_base_ptr), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers are initialised before any remote arrive
  const uint32_t tmem = *tmem_base_ptr;
  int* status = p.ctrl + kCtrlStatus;

  if (warp == 0) {
    // ------------------------------------------------------------------ producer
    if (lane == 0) prefetch_tmap(&tmap_kv);
    const int chunk0 = rank ? 4 : 0;
    PieceIter it;
    it.init(p.cum, p.s_q, pair, p.npairs);
    Piece pc;
    uint32_t n = 0;
    bool ok = true;
    while (ok && it.next(pc)) {
      const int32_t* idx_t = p.indices + (size_t)pc.t * p.topk;
      int head = 0, tail = 0, rp = 0;
      for (int jb = 0; jb < pc.lb1 && ok; ++jb) {
        // compact the next valid indices into the ring until a block is full
        while (tail - head < kBT && rp < p.topk) {
          const int i = rp + lane;
          const int v = (i < p.topk) ? __ldg(idx_t + i) : -1;
          const bool valid = (v >= 0) && (v < p.s_kv);
          const uint32_t m = __ballot_sync(0xffffffffu, valid);
          if (valid) ring[(tail + __popc(m & ((1u << lane) - 1u))) & (kRing - 1)] = v;
          tail += __popc(m);
          rp += 32;
          __syncwarp();
        }
        const int cnt = min(kBT, tail - head);
        if (jb >= pc.lb0) {
          const int s = (int)(n % kStages);
          if (!mbar_wait(bar(KV_EMPTY + s), ((n / kStages) & 1u) ^ 1u, kWaitLimitNs, abort_flag)) {
            if (lane == 0) set_abort(abort_flag, status, peer_abort);
            ok = false;
            break;
          }
          if (lane == 0) mbar_arrive_expect_tx(bar(KV_FULL + s), kStageBytes);
          __syncwarp();
          if (lane < 16) {
            int r[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int row = lane * 4 + q;
              r[q] = row < cnt ? ring[(head + row) & (kRing - 1)] : 0;
            }
            const uint32_t dst = sbase + kOffStage + (uint32_t)s * kStageBytes + (uint32_t)lane * 512u;
#pragma unroll
            for (int k = 0; k < kChunks; ++k)
              tma_gather4(dst + (uint32_t)k * kChunkBytes, &tmap_kv, (chunk0 + k) * 64, r[0], r[1], r[2], r[3],
                          bar(KV_FULL + s));
          }
          __syncwarp();
          ++n;
        }
        head += cnt;
      }
    }
    // every issued gather has landed before the CTA may exit
    const uint32_t first = n > (uint32_t)kStages ? n - kStages : 0u;
    for (uint32_t b = first; b < n; ++b) mbar_wait(bar(KV_FULL + (int)(b % kStages)), (b / kStages) & 1u, kWaitLimitNs, nullptr);
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      PieceIter it;
      it.init(p.cum, p.s_q, pair, p.npairs);
      Piece pc;
      uint32_t n = 0, item = 0;
      bool ok = true;
      const int step0 = rank ? 2 : 0;
      while (ok && it.next(pc)) {
        const int nb = pc.lb1 - pc.lb0;
        if (!mbar_wait(bar(Q_FULL), item & 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
        for (int j = 0; j <= nb && ok; ++j) {
          if (j < nb) {
            const uint32_t b = n + (uint32_t)j;
            const int s = (int)(b % kStages);
            if (!mbar_wait(bar(KV_FULL + s), (b / kStages) & 1u, kWaitLimitNs, abort_flag) ||
                !mbar_wait(bar(S_EMPTY), (b & 1u) ^ 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t stage = sbase + kOffStage + (uint32_t)s * kStageBytes;
#pragma unroll
            for (int ks = 0; ks < kQkSteps; ++ks) {
              const int ls = ks + step0;
              const uint64_t bdesc = smem_desc(stage + (uint32_t)(ls >> 2) * kChunkBytes + (uint32_t)(ls & 3) * 32u, 16, 1024);
              mma_ts(tmem + kTmS, tmem + kTmQ + (uint32_t)ks * 8u, bdesc, kIdescQK, ks > 0 ? 1u : 0u);
            }
            mma_commit(bar(S_FULL));
          }
          if (j >= 1) {
            const uint32_t b = n + (uint32_t)(j - 1);
            const int s = (int)(b % kStages);
            const int pb = (int)(b & 1u);
            if (!mbar_wait(bar(P_FULL + pb), (b >> 1) & 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
            if (j == 1 && !mbar_wait(bar(O_FREE), (item & 1u) ^ 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
            tc_fence_after();
            const uint32_t stage = sbase + kOffStage + (uint32_t)s * kStageBytes;
            const uint32_t pbuf = sbase + kOffP + (uint32_t)pb * kPBytes;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t adesc = smem_desc(pbuf + (uint32_t)kk * 32u, 16, 1024);
              const uint64_t bdesc = smem_desc(stage + (uint32_t)kk * 2048u, kChunkBytes, 1024);
              mma_ss(tmem + kTmO, adesc, bdesc, kIdescPV, (j > 1 || kk > 0) ? 1u : 0u);
            }
            mma_commit(bar(KV_EMPTY + s));
            mma_commit(bar(P_EMPTY + pb));
            if (j == nb) mma_commit(bar(O_FULL));
          }
        }
        n += (uint32_t)nb;
        ++item;
      }
      if (!ok) set_abort(abort_flag, status, peer_abort);
      mma_commit(bar(DRAIN));
      mbar_wait(bar(DRAIN), 0, kWaitLimitNs, nullptr);
    }
    __syncwarp();
  } else if (warp >= 4) {
    // ------------------------------------------------------------------ softmax + epilogue
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // head row = TMEM lane
    const uint32_t trow = tmem + ((uint32_t)(quarter * 32) << 16);
    const uint32_t xbase_local = sbase + kOffX;
    const uint32_t xbase_peer = mapa_shared(xbase_local, peer);
    PieceIter it;
    it.init(p.cum, p.s_q, pair, p.npairs);
    Piece pc;
    uint32_t n = 0, item = 0;
    bool ok = true;
    while (ok && it.next(pc)) {
      const int nb = pc.lb1 - pc.lb0;
      const int nval = p.nvalid[pc.t];
      // ---- Q columns [288*rank, 288*rank + 288) of row r into tensor memory
      {
        const bool live = r < p.h_q;
        const uint4* qrow = (const uint4*)(p.q + ((size_t)pc.t * p.h_q + (live ? r : 0)) * kDQK + 288 * rank);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t v[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 w = live ? __ldg(qrow + c * 8 + u) : make_uint4(0, 0, 0, 0);
            v[4 * u] = w.x; v[4 * u + 1] = w.y; v[4 * u + 2] = w.z; v[4 * u + 3] = w.w;
          }
          tmem_st32(trow + kTmQ + (uint32_t)c * 32u, v);
        }
        {
          uint32_t v[16];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const uint4 w = live ? __ldg(qrow + 32 + u) : make_uint4(0, 0, 0, 0);
            v[4 * u] = w.x; v[4 * u + 1] = w.y; v[4 * u + 2] = w.z; v[4 * u + 3] = w.w;
          }
          tmem_st16(trow + kTmQ + 128u, v);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(Q_FULL));
      }
      float rm = -INFINITY, rmfs = -INFINITY, se = 0.f;
      for (int j = 0; j < nb; ++j) {
        const uint32_t b = n + (uint32_t)j;
        const int xb = (int)(b & 1u);
        float s[kBT];
        if (!mbar_wait(bar(S_FULL), b & 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
        tc_fence_after();
        {
          uint32_t v[32];
          tmem_ld32(trow + kTmS, v);
          tmem_wait_ld();
          reg_fence(v);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(v[i]);
          tmem_ld32(trow + kTmS + 32u, v);
          tmem_wait_ld();
          reg_fence(v);
#pragma unroll
          for (int i = 0; i < 32; ++i) s[32 + i] = __uint_as_float(v[i]);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(S_EMPTY));
        // ---- exchange the partial logits with the peer CTA
        if (!mbar_wait(bar(X_EMPTY + xb), ((b >> 1) & 1u) ^ 1u, kWaitLimitNs, abort_flag, true)) { ok = false; break; }
        {
          const uint32_t dst = xbase_peer + (uint32_t)xb * kXBytes + (uint32_t)r * 16u;
#pragma unroll
          for (int k = 0; k < kBT / 4; ++k)
            st_cluster_v4(dst + (uint32_t)k * 2048u, s[4 * k], s[4 * k + 1], s[4 * k + 2], s[4 * k + 3]);
          mbar_arrive_remote(mapa_shared(bar(X_FULL + xb), peer));
        }
        if (!mbar_wait(bar(X_FULL + xb), (b >> 1) & 1u, kWaitLimitNs, abort_flag, true)) { ok = false; break; }
        {
          const float4* src = (const float4*)(smem + kOffX + xb * kXBytes) + r;
#pragma unroll
          for (int k = 0; k < kBT / 4; ++k) {
            const float4 w = src[k * 128];
            s[4 * k] += w.x; s[4 * k + 1] += w.y; s[4 * k + 2] += w.z; s[4 * k + 3] += w.w;
          }
          mbar_arrive_remote(mapa_shared(bar(X_EMPTY + xb), peer));
        }
        // ---- online softmax with skip-scale (log2 domain)
        const int nv = min(kBT, max(0, nval - kBT * (pc.lb0 + j)));
        float cmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < kBT; ++i) {
          s[i] = (i < nv) ? s[i] * p.scale_log2 : -INFINITY;
          cmax = fmaxf(cmax, s[i]);
        }
        rm = fmaxf(rm, cmax);
        const bool trig = rm > rmfs + kThresLog2;
        float alpha = 1.f;
        if (trig) {
          alpha = ex2_approx(rmfs - rm);
          se *= alpha;
          rmfs = rm;
        }
        if (j > 0 && __any_sync(0xffffffffu, trig)) {
          // O holds earlier blocks of this token: rescale it once the previous PV is done
          const uint32_t bp = b - 1u;
          if (!mbar_wait(bar(P_EMPTY + (int)(bp & 1u)), (bp >> 1) & 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < 8; ++c) {
            uint32_t v[32];
            tmem_ld32(trow + kTmO + (uint32_t)c * 32u, v);
            tmem_wait_ld();
            reg_fence(v);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
            tmem_st32(trow + kTmO + (uint32_t)c * 32u, v);
          }
          tmem_wait_st();
        }
        float psum = 0.f;
        uint32_t pk[kBT / 2];
#pragma unroll
        for (int i = 0; i < kBT; i += 2) {
          const float e0 = (i < nv) ? ex2_approx(s[i] - rmfs) : 0.f;
          const float e1 = (i + 1 < nv) ? ex2_approx(s[i + 1] - rmfs) : 0.f;
          psum += e0 + e1;
          pk[i / 2] = pack_bf16x2(e0, e1);
        }
        se += psum;
        const int pb = (int)(b & 1u);
        if (!mbar_wait(bar(P_EMPTY + pb), ((b >> 1) & 1u) ^ 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
        {
          uint8_t* prow = smem + kOffP + pb * kPBytes;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            *(uint4*)(prow + sw128_off((uint32_t)r, (uint32_t)c)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(P_FULL + pb));
      }
      if (!ok) break;
      // ---- epilogue: normalise this CTA's 256 output columns
      if (!mbar_wait(bar(O_FULL), item & 1u, kWaitLimitNs, abort_flag)) { ok = false; break; }
      tc_fence_after();
      const bool has = se > 0.f;
      const float inv = has ? 1.f / se : 0.f;
      const float lse_val = has ? (rmfs + log2f(se)) * kLn2 : -INFINITY;
      const bool live = r < p.h_q;
#pragma unroll 1
      for (int c = 0; c < 8; ++c) {
        uint32_t v[32];
        tmem_ld32(trow + kTmO + (uint32_t)c * 32u, v);
        tmem_wait_ld();
        reg_fence(v);
        if (live) {
          if (pc.full) {
            uint4* dst = (uint4*)(p.out + ((size_t)pc.t * p.h_q + r) * kDV + 256 * rank + 32 * c);
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
            float4* dst = (float4*)(p.part_o + ((size_t)pc.slot * p.h_q + r) * kDV + 256 * rank + 32 * c);
#pragma unroll
            for (int u = 0; u < 8; ++u)
              dst[u] = make_float4(__uint_as_float(v[4 * u]) * inv, __uint_as_float(v[4 * u + 1]) * inv,
                                   __uint_as_float(v[4 * u + 2]) * inv, __uint_as_float(v[4 * u + 3]) * inv);
          }
        }
      }
      if (live && rank == 0) {
        if (pc.full) p.lse[(size_t)pc.t * p.h_q + r] = lse_val;
        else p.part_lse[(size_t)pc.slot * p.h_q + r] = lse_val;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(O_FREE));
      n += (uint32_t)nb;
      ++item;
    }
    if (!ok && lane == 0) set_abort(abort_flag, status, peer_abort);
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 2) tmem_dealloc(tmem, kTmemCols);
  cluster_sync();  // no remote store or arrive may target an exited CTA
}

// Largest number of 2-CTA clusters of the forward kernel that fit at once.
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
  cfg.blockDim = dim3(256, 1, 1);
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

cudaError_t launch_fwd_bf16(const CUtensorMap& tmap, const FwdParams& p, cudaStream_t stream) {
  cudaError_t e = cudaFuncSetAttribute(dsa_fwd_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, fwd::kSmemAlloc);
  if (e != cudaSuccess) return e;
  dsa_fwd_bf16_kernel<<<2 * p.npairs, 256, fwd::kSmemAlloc, stream>>>(tmap, p);
  return cudaGetLastError();
}

}  // namespace dsa

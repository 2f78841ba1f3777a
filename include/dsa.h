/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek Sparse Attention (MLA) forward.
 *
 * What is computed ("Ascend Sparse Attention Forward 算法与优化技术简析",
 * section "数学建模"): for every query token t, with Q_t[h_q, 576],
 * KV[s_kv, 576], an index list idx_t[topk] and a scalar sm_scale,
 *
 *     gathered = KV.index_select(idx_t)                     [topk, 576]
 *     S        = softmax(sm_scale * Q_t @ gathered^T, -1)   [h_q, topk]
 *     out_t    = S @ gathered[:, :512]                       [h_q, 512]
 *     lse_t    = ln(sum(exp(sm_scale * Q_t @ gathered^T)))   [h_q]
 *
 * computed blockwise over index blocks of 128 with the online softmax of section
 * "计算流程": float32 running max / max-for-softmax / sum-of-exp, a float32
 * output accumulator, a rescale that fires only when the running max has moved
 * more than 6 (natural-log units) above the max used for the exponentials
 * ("skip scale"), and S rounded to bf16 before it multiplies V.
 *
 * Index semantics: a slot whose value lies outside [0, s_kv) (the -1 marker
 * included) is excluded exactly; duplicates count once per occurrence; a token
 * with no valid slot gets out = 0 and lse = -inf.  Slot order does not change
 * the result beyond rounding.
 *
 * Memory: every pointer is a DEVICE pointer owned by the caller, except in
 * dsa_sparse_attn_fwd_host (host buffers in and out).  The library allocates no
 * device memory and keeps no per-call state outside the caller's workspace; the
 * exceptions are stated at dsa_sparse_attn_fwd_host (its own copy streams and
 * events for the length of the call), dsa_sparse_attn_fwd_noalloc (a built-in
 * scratch array) and dsa_out_proj (a cuBLASLt handle and algorithm cache).
 * All calls but dsa_sparse_attn_fwd_host are asynchronous on `stream`; their
 * return value reports host-side validation and launch errors only.  A device-side failure
 * (a bounded wait inside a kernel that gave up) is written to the workspace
 * and read back with dsa_read_device_status().  No call aborts or throws.
 *
 * Layouts (row-major, dense, no padding):
 *   q        bf16  [s_q, h_q, 576]
 *   kv       bf16  [s_kv, 576]                          (dsa_sparse_attn_fwd)
 *            uint8 [s_kv, 656] FP8 rows                 (dsa_sparse_attn_fwd_fp8kv):
 *                  bytes   0..511  e4m3 latent channels 0..511
 *                  bytes 512..527  4 x float32 scale, scale g applies to channels 128g..128g+127
 *                  bytes 528..655  64 x bf16 rope channels 512..575
 *            uint8 [s_kv, 448] FP4 rows                 (dsa_sparse_attn_fwd_fp4kv):
 *                  bytes   0..255  e2m1 latent codes, two per byte: byte i holds channel 2i in its
 *                                  low nibble and channel 2i+1 in its high nibble
 *                  bytes 256..319  16 x float32 scale, scale g applies to channels 32g..32g+31
 *                  bytes 320..447  64 x bf16 rope channels 512..575
 *   indices  int32 [s_q, topk]   global row ids into kv
 *   out      bf16  [s_q, h_q, 512]
 *   lse      fp32  [s_q, h_q]    natural-log log-sum-exp of the scaled logits
 * All pointers must be 16-byte aligned.  Shapes: 0 <= s_q, 1 <= h_q <= 128,
 * 0 <= s_kv < 2^31, 1 <= topk.
 */
#ifndef DSA_GB300_H
#define DSA_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define DSA_API __attribute__((visibility("default")))
#else
#define DSA_API
#endif

#define DSA_D_QK 576
#define DSA_D_V 512
#define DSA_D_ROPE 64
#define DSA_FP8_ROW_BYTES 656
#define DSA_FP4_ROW_BYTES 448
#define DSA_MAX_HEADS 128
#define DSA_B_TOPK 128

typedef enum {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,    /* a null pointer where data is needed, or a shape out of range */
  DSA_ERR_UNSUPPORTED = 2,    /* the current device is not sm_103 / lacks the needed resources */
  DSA_ERR_MISALIGNED = 3,     /* a pointer is not 16-byte aligned */
  DSA_ERR_CUDA = 4,           /* a CUDA runtime call or kernel launch failed */
  DSA_ERR_DEVICE_TIMEOUT = 5, /* a bounded wait inside a kernel gave up (read via dsa_read_device_status) */
  DSA_ERR_WORKSPACE = 6       /* workspace null or smaller than dsa_sparse_attn_fwd_workspace_size() */
} dsa_status;

typedef enum { DSA_KV_BF16 = 0, DSA_KV_FP8 = 1, DSA_KV_FP4 = 2 } dsa_kv_format;

/* Bytes of device workspace a forward call with these shapes needs on the
 * current device (scheduler metadata, per-piece partial outputs for tokens
 * whose index blocks are split across CTA pairs, a status word).  Returns 0 for
 * invalid shapes.  The workspace needs no initialisation and may be reused by
 * consecutive calls on one stream; two calls in flight at once need two
 * workspaces. */
DSA_API size_t dsa_sparse_attn_fwd_workspace_size(int s_q, int h_q, int topk, int kv_format);

/* The forward with a bf16 KV cache ("数学建模" / "计算流程" sections cited above).
 * q, kv, indices: inputs (not modified).  out, lse: outputs (fully written for
 * every token and head < h_q).  sm_scale: multiplier of the logits.
 * workspace/workspace_bytes: caller-owned scratch of at least
 * dsa_sparse_attn_fwd_workspace_size(s_q, h_q, topk, DSA_KV_BF16) bytes.
 * Launches, in order on `stream`: a memset of the workspace's control block,
 * a counting/scheduling kernel, the attention kernel, and a kernel that merges
 * the pieces of split tokens. */
DSA_API dsa_status dsa_sparse_attn_fwd(const void* q, const void* kv, const int32_t* indices, int s_q, int h_q, int s_kv,
                               int topk, float sm_scale, void* out, float* lse, void* workspace,
                               size_t workspace_bytes, cudaStream_t stream);

/* The forward with an FP8-e4m3 KV cache of 656-byte rows (layout above; the
 * per-token data and scales sit together as the page's "Decoding KV Cache
 * Layout 优化" section asks).  The latent channels are dequantised as
 * e4m3 * scale and rounded to bf16 before they enter the tensor cores, as the
 * page's "能不能用 1C1V" section describes for decoding.  Arguments as for
 * dsa_sparse_attn_fwd, with kv = uint8 [s_kv, 656]. */
DSA_API dsa_status dsa_sparse_attn_fwd_fp8kv(const void* q, const void* kv_fp8, const int32_t* indices, int s_q, int h_q,
                                     int s_kv, int topk, float sm_scale, void* out, float* lse, void* workspace,
                                     size_t workspace_bytes, cudaStream_t stream);

/* Allocation-free variant of dsa_sparse_attn_fwd, for callers that cannot
 * allocate device memory themselves (code that runs where cudaMalloc is not
 * available or not allowed, such as inside a custom allocator, or a plugin
 * that is handed only its input and output buffers).  The pages have no
 * counterpart; this is a convenience of this library.  Arguments as for
 * dsa_sparse_attn_fwd, without the workspace: the call uses one scratch
 * array compiled into the library instead (about 43 MiB per device, held by
 * every GPU that loads the library until the process exits).
 * Limits: s_q <= 8192, h_q <= 128, and at most 80 resident SM pairs on the
 * device; larger calls return DSA_ERR_WORKSPACE and launch nothing.
 * The first call on a device looks up the array's device address
 * (cudaGetSymbolAddress) with that device current; make that first call
 * before any stream capture.  Every call shares the one array and leaves its
 * contents behind (the call clears what must start at zero itself), so calls
 * whose work overlaps on the GPU (concurrent streams, several host threads)
 * race: serialise them.  Device-side timeouts are recorded in the array, not
 * readable through dsa_read_device_status.  No allocation of any kind is made. */
DSA_API dsa_status dsa_sparse_attn_fwd_noalloc(const void* q, const void* kv, const int32_t* indices, int s_q, int h_q,
                                               int s_kv, int topk, float sm_scale, void* out, float* lse,
                                               cudaStream_t stream);

/* The forward over a paged KV cache ("Flash Attention Infer算子性能优化", section
 * "优化Paged Attention路径": a sequence's KV lives in fixed-size pages of a shared
 * pool and is reached through a block table).
 *   kv_format     DSA_KV_BF16 (kv_pool bf16 [n_rows, 576]), DSA_KV_FP8 (uint8 [n_rows, 656]) or
 *                 DSA_KV_FP4 (uint8 [n_rows, 448]);
 *                 the pool holds n_rows / page_size pages of page_size rows, page k at rows
 *                 [k * page_size, (k + 1) * page_size).
 *   indices       int32 [s_q, topk]: logical positions in the token's own sequence.
 *   seq_of_token  int32 [s_q]: the sequence of each query token, in [0, n_seq).
 *   block_table   int32 [n_seq, max_pages]: physical page of each logical page; < 0 = unmapped.
 * Position v of a token of sequence s reads pool row
 *   block_table[s][v / page_size] * page_size + v % page_size;
 * it is excluded exactly (like -1 in the flat layout) when v < 0, v / page_size >= max_pages,
 * the table entry is negative, s is outside [0, n_seq) or the row is outside [0, n_rows).
 * Everything else (q, out, lse, sm_scale, workspace size and use, stream, errors) is as for
 * dsa_sparse_attn_fwd / dsa_sparse_attn_fwd_fp8kv with s_kv = n_rows; seq_of_token and
 * block_table need 4-byte alignment, page_size, max_pages, n_seq >= 1 and
 * n_seq * max_pages < 2^31 (else DSA_ERR_INVALID_ARG). */
DSA_API dsa_status dsa_sparse_attn_fwd_paged(int kv_format, const void* q, const void* kv_pool, const int32_t* indices,
                                             const int32_t* seq_of_token, const int32_t* block_table, int s_q,
                                             int h_q, int n_rows, int topk, int n_seq, int max_pages, int page_size,
                                             float sm_scale, void* out, float* lse, void* workspace,
                                             size_t workspace_bytes, cudaStream_t stream);

/* The forward with an FP4 (e2m1) KV cache of 448-byte rows (layout above).  The
 * page's "能不能用 1C1V" section names FP4 beside FP8 as a decoding KV format but
 * gives no layout: the row is this library's reading (the FP8 row's pattern with
 * 4-bit codes and one scale per 32 channels).  Latent channels are dequantised as
 * e2m1 * scale and rounded to bf16 before the tensor cores, as for FP8.  Arguments
 * as for dsa_sparse_attn_fwd, with kv = uint8 [s_kv, 448]; the workspace size is
 * dsa_sparse_attn_fwd_workspace_size(..., DSA_KV_FP4). */
DSA_API dsa_status dsa_sparse_attn_fwd_fp4kv(const void* q, const void* kv_fp4, const int32_t* indices, int s_q, int h_q,
                                             int s_kv, int topk, float sm_scale, void* out, float* lse,
                                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The forward from HOST buffers, the query tokens pipelined through the GPU in
 * chunks of chunk_tokens.  The upload of a chunk's inputs, the forward of the
 * chunk before it and the download of the chunk before that run at once, on
 * two copy streams the call creates beside `stream`.  This is a convenience of
 * this library: the method itself works on device memory only.
 *   kv_format      DSA_KV_BF16, DSA_KV_FP8 or DSA_KV_FP4 (picks the row size of kv_host).
 *   q_host, kv_host, indices_host, out_host, lse_host
 *                  host memory with the layouts of dsa_sparse_attn_fwd (kv rows of
 *                  1152, 656 or 448 bytes).  Page-locked memory (cudaHostAlloc)
 *                  lets the copies overlap the compute; pageable memory works
 *                  but serialises them.
 *   device_buffer  >= dsa_sparse_attn_fwd_host_device_bytes(kv_format, s_q, h_q,
 *                  s_kv, topk, chunk_tokens) bytes of device memory, 16-byte
 *                  aligned, owned by the caller; it holds the whole KV, two sets of
 *                  chunk buffers and a workspace, and its contents are scratch.
 *   chunk_tokens   tokens per chunk, >= 1 (s_q or more: one chunk, no overlap); when there are
 *                  several, the first and the last hold half as many, which shortens the upload
 *                  before the first forward and the download after the last one.
 * The work is queued after what `stream` already holds and the call returns
 * when out_host and lse_host hold the result (it synchronises).  Returns
 * DSA_ERR_INVALID_ARG / DSA_ERR_WORKSPACE / DSA_ERR_UNSUPPORTED before any
 * copy for bad arguments, any error of the per-chunk forward, DSA_ERR_CUDA
 * if a copy or synchronisation failed, or DSA_ERR_DEVICE_TIMEOUT if a bounded
 * wait inside any chunk's kernels gave up (the outputs are then not valid). */
DSA_API size_t dsa_sparse_attn_fwd_host_device_bytes(int kv_format, int s_q, int h_q, int s_kv, int topk,
                                                     int chunk_tokens);
DSA_API dsa_status dsa_sparse_attn_fwd_host(int kv_format, const void* q_host, const void* kv_host,
                                            const int32_t* indices_host, int s_q, int h_q, int s_kv, int topk,
                                            float sm_scale, void* out_host, float* lse_host, void* device_buffer,
                                            size_t device_bytes, int chunk_tokens, cudaStream_t stream);

/* Output projection with residual after the attention
 * ("FlashMLA算子Ascend 950移植：从tiling到访存优化全解读", section 3.4, 输出投影与残差合并):
 *   y[t, :] = O[t, :] . W_o + x[t, :]
 * where O[t, :] is the head-major concatenation of the attention output, i.e. the bf16 `out`
 * [s_q, h_q, 512] of a forward read as [s_q, h_q * 512].
 *   o          bf16 [s_q, h_q * 512] (the forward's `out`)
 *   w_o        bf16 [h_q * 512, d_model], row-major
 *   x          bf16 [s_q, d_model] residual, or NULL for none; may equal y (in place)
 *   y          bf16 [s_q, d_model] output (fp32 accumulation, rounded to nearest even)
 *   workspace  >= dsa_out_proj_workspace_size() bytes of device memory, 16-byte aligned
 * d_model must be a multiple of 8 (>= 8) and 1 <= h_q <= 128; all pointers 16-byte aligned.  Runs as
 * one cuBLASLt GEMM on `stream` (asynchronous).  The library keeps one cuBLASLt handle per device and
 * a cache of the chosen algorithm per shape for the life of the process.  Returns DSA_ERR_INVALID_ARG,
 * DSA_ERR_MISALIGNED or DSA_ERR_WORKSPACE before any work for bad arguments, DSA_ERR_UNSUPPORTED if no
 * GEMM algorithm fits, DSA_ERR_CUDA if the GEMM launch failed. */
DSA_API size_t dsa_out_proj_workspace_size(void);
DSA_API dsa_status dsa_out_proj(const void* o, const void* w_o, const void* x, int s_q, int h_q, int d_model,
                                void* y, void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* The forward followed by the output projection on the same stream: out and lse as for the
 * kv_format's forward entry point, then y = out . W_o + x as dsa_out_proj.  The workspace holds the
 * forward's workspace (first, so dsa_read_device_status reads it) and the GEMM's:
 * dsa_sparse_attn_fwd_oproj_workspace_size(s_q, h_q, topk, kv_format) bytes. */
DSA_API size_t dsa_sparse_attn_fwd_oproj_workspace_size(int s_q, int h_q, int topk, int kv_format);
DSA_API dsa_status dsa_sparse_attn_fwd_oproj(int kv_format, const void* q, const void* kv, const int32_t* indices,
                                             int s_q, int h_q, int s_kv, int topk, float sm_scale, const void* w_o,
                                             const void* x, int d_model, void* out, float* lse, void* y,
                                             void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* Synchronises `stream` and returns the device-side status a previous forward
 * call left in `workspace` (DSA_OK or DSA_ERR_DEVICE_TIMEOUT), or DSA_ERR_CUDA
 * if the synchronisation itself failed. */
DSA_API dsa_status dsa_read_device_status(const void* workspace, cudaStream_t stream);

/* A static, human-readable name for a status code. */
DSA_API const char* dsa_status_string(dsa_status status);

/* Number of kernels one forward call launches (the memset excluded). */
DSA_API int dsa_kernels_per_call(void);

/* Profiling hook.  When both events are non-null, every later forward call
 * records `before` on its stream just before the attention kernel and `after`
 * just after it, so a caller can time that kernel alone with
 * cudaEventElapsedTime.  Pass two nulls to switch it off.  The events are
 * created and owned by the caller; the setting is process-wide and not
 * thread-safe (meant for benchmarks). */
DSA_API void dsa_set_timing_events(cudaEvent_t before, cudaEvent_t after);

#ifdef __cplusplus
}
#endif

#endif /* DSA_GB300_H */

/*
 * layer_range_stage (GB300) -- kernel-level entry points.
 *
 * The two dominant steps of a stage forward, callable on their own with caller-owned
 * device buffers: the dequant-fused int8 block-32 GEMV and split-K grouped-query decode
 * attention.  These run the same kernels stage_decode launches.  Return codes are the
 * STAGE_* codes of stage.h (no C++ exception crosses this boundary: stage_op_q8_pack's host
 * staging buffer that cannot be allocated gives STAGE_E_HOST); messages are read with
 * stage_op_last_error().  All device pointers must be 16-byte aligned.
 */
#ifndef LAYER_RANGE_STAGE_OPS_H
#define LAYER_RANGE_STAGE_OPS_H

#include "stage.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Device bytes of a packed [rows x cols] int8 block-32 matrix: the weight bytes (biased,
 * rows padded to a multiple of 256 weights) and the fp16 scale bytes.  STAGE_E_INVALID for
 * rows < 1, cols outside [1, 2^30] or null pointers. */
STAGE_API int stage_op_q8_device_bytes(int64_t rows, int64_t cols, size_t* q_bytes, size_t* s_bytes);

/* Pack a host matrix (layout of stage_q8) into caller device buffers of the sizes above.
 * Synchronous.  Errors: STAGE_E_INVALID (null pointers, a shape stage_op_q8_device_bytes
 * rejects), STAGE_E_HOST (the host staging buffer), STAGE_E_CUDA (the copies). */
STAGE_API int stage_op_q8_pack(const stage_q8* host, void* q_dev, void* s_dev);

/* Embedding rows: out[t][c] = scale(tok[t], c / 32) * q[tok[t]][c] for t < n_tok, c < cols --
 * the dequantised row of each token, as the first stage embeds its tokens ("RFC: pipeline
 * placement across multiple GPUs for models larger than one device", section "What I found":
 * the first stage embeds).  W is a packed [rows x cols] matrix (stage_op_q8_pack); tok_dev:
 * device int32 [n_tok], every entry in [0, rows) (not checked on the device); out_dev: f32
 * [n_tok][cols], 16-byte aligned, cols a multiple of 4.  Runs on `stream`.  Errors:
 * STAGE_E_INVALID (null or unaligned pointers, rows outside [1, 2^30], cols outside
 * [1, 2^24] or not a multiple of 4, n_tok outside [1, 65535]), STAGE_E_CUDA (the launch). */
STAGE_API int stage_op_embed(const void* q_dev, const void* s_dev, int64_t rows, int64_t cols, const int32_t* tok_dev,
                             int n_tok, float* out_dev, void* stream);

/* y[t][r] = sum_k W[r][k] * h[t][k] for t < n_tok, r < rows, where h = x, or
 * h = x / sqrt(mean(x^2) + eps) * gamma when gamma_dev is not NULL (the RMSNorm that
 * precedes every projection of a block: "41. Many GPUs: tensor, pipeline, expert and
 * data parallelism", section "Pipeline parallelism").  W is a packed matrix
 * (stage_op_q8_pack).  x_dev: f32 [n_tok][cols]; y_dev: f32 [n_tok][rows].  Every |h| must
 * be below 2^64 (the dot product takes its inputs scaled by 2^64 in float32); float32
 * rounding error, relative to sum_k (q + 128) |h_k| + 128 |sum_k h_k| per 16-input chunk.
 * Runs on `stream` (a cudaStream_t); no allocation, no synchronisation.  Errors:
 * STAGE_E_INVALID (null or unaligned pointers, rows outside [1, 2^30], cols outside [1, 2^24]
 * or not a multiple of 4, n_tok < 1), STAGE_E_CUDA (the launch). */
STAGE_API int stage_op_gemv(const void* q_dev, const void* s_dev, int64_t rows, int64_t cols, const float* x_dev,
                            int n_tok, const float* gamma_dev, float eps, float* y_dev, void* stream);

/* Tensor-core GEMM of the prefill: y[m][r] = sum_k A[m][k] * W[r][k] for m < M, r < rows,
 * with A bf16 (bit patterns) [M][lda] on the device, lda >= the packed row length
 * (cols rounded up to 256) and multiple of 8, zero beyond cols; W a packed matrix whose
 * weights are rounded to bf16 (bf16(f32(scale) * q)); f32 accumulation (tcgen05, TMEM).
 * y_dev: f32 [M][rows].  Runs on `stream`.  Errors: STAGE_E_INVALID (null or unaligned
 * pointers, M < 1, rows outside [1, 2^30], cols outside [1, 2^24], lda too small or not a
 * multiple of 8), STAGE_E_CUDA (tensor maps or the launch). */
STAGE_API int stage_op_gemm_bf16(const uint16_t* a_dev, int lda, int M, const void* q_dev, const void* s_dev,
                                 int64_t rows, int64_t cols, float* y_dev, void* stream);

/* Scratch bytes stage_op_attention_decode needs for these sizes (0 for a non-positive
 * size). */
STAGE_API size_t stage_op_attention_workspace_bytes(int n_tok, int n_q_heads, int n_kv_heads, int head_dim,
                                                    int n_chunks);

/* Split-K grouped-query decode attention over an fp16 KV cache ("41. Many GPUs: ...",
 * section "Ring attention for very long contexts": partial attention with log-sum-exp
 * and the merge o = sum_s e^(l_s - l) o_s; section "Tensor parallelism": query head j
 * reads KV head j / (n_q_heads / n_kv_heads)).
 *   q_dev: f32 [n_tok][n_q_heads][head_dim] (already rotated);
 *   k_cache_dev, v_cache_dev: fp16 bits [seqs][n_kv_heads][max_len][head_dim];
 *   seq_dev, pos_dev: device int32 [n_tok]: token t attends to positions 0..pos[t] of
 *     sequence seq[t] (the caller guarantees pos[t] < max_len and seq[t] < seqs);
 *   out_dev: f32 [n_tok][n_q_heads][head_dim], softmax(q k^T / sqrt(head_dim)) v;
 *   n_chunks in [1, 64]: the positions of each token are split in n_chunks chunks;
 *   workspace_dev: stage_op_attention_workspace_bytes(...) bytes of device scratch whose
 *     contents must be zero before the first call (each call leaves it ready for the next).
 * head_dim 64 or 128; n_q_heads / n_kv_heads in {1, 2, 4, 8}.  Runs on `stream`.  Errors:
 * STAGE_E_INVALID (null or unaligned pointers, a non-positive size, an unsupported head_dim
 * or group, n_chunks outside [1, 64], n_tok above 65535, a workspace unaligned or smaller
 * than needed), STAGE_E_CUDA (the launch). */
STAGE_API int stage_op_attention_decode(const float* q_dev, const uint16_t* k_cache_dev, const uint16_t* v_cache_dev,
                                        const int32_t* seq_dev, const int32_t* pos_dev, int n_tok, int n_q_heads,
                                        int n_kv_heads, int head_dim, int max_len, int n_chunks, float* out_dev,
                                        void* workspace_dev, size_t workspace_bytes, void* stream);

/* Decode attention that allocates nothing: the same computation and arguments as
 * stage_op_attention_decode, without the workspace.  The pages have no counterpart; this
 * is for callers that cannot allocate device memory at the point they run attention --
 * a host process that owns all device memory through its own allocator and forbids
 * untracked allocations, or a latency-critical loop that must not call cudaMalloc (which
 * can synchronise the device and take unbounded time).
 *   - Scratch is one fixed array inside this library, STAGE_OP_STATIC_SCRATCH_BYTES bytes,
 *     resident on every GPU that loads the library until the process exits.  A request
 *     needing more (stage_op_attention_workspace_bytes) fails with STAGE_E_INVALID.
 *   - The first call on a device looks up that device's address of the array (with the
 *     device current); make that first call before any stream capture.  The address is kept
 *     for the device's primary context (the one the CUDA runtime uses): it does not follow
 *     a cudaDeviceReset, after which the library's device code is loaded again, nor a
 *     driver context other than the primary one made current by the caller -- after either,
 *     reload the library before calling this entry point again.
 *   - Every call reuses the same array and clears its counters on `stream` before the
 *     kernel.  Calls whose kernels overlap on the GPU (on different streams, or different
 *     host threads) race on the array and give wrong results: serialise them.
 *   - No cudaMalloc, cudaFree or allocating library call is made.
 *   - Errors: those of stage_op_attention_decode other than the workspace's, STAGE_E_INVALID
 *     for scratch beyond the array or a device ordinal of 64 or more, STAGE_E_CUDA when the
 *     array's device address cannot be looked up. */
#define STAGE_OP_STATIC_SCRATCH_BYTES (4u << 20)
STAGE_API int stage_op_attention_decode_static(const float* q_dev, const uint16_t* k_cache_dev,
                                               const uint16_t* v_cache_dev, const int32_t* seq_dev,
                                               const int32_t* pos_dev, int n_tok, int n_q_heads, int n_kv_heads,
                                               int head_dim, int max_len, int n_chunks, float* out_dev, void* stream);

/* Message of the last failed stage_op_* call on the calling thread ("" if none). */
STAGE_API const char* stage_op_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* LAYER_RANGE_STAGE_OPS_H */

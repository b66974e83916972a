/*
 * layer_range_stage (GB300) -- C ABI of one pipeline stage.
 *
 * A stage owns a contiguous range [begin, end) of decoder blocks, the resident
 * weights of exactly those blocks, their fp16 KV cache and its workspace.  It
 * takes an F32 hidden activation in and hands an F32 hidden activation out; the
 * first stage (begin == 0) embeds tokens instead of taking a hidden activation,
 * the last stage (end == n_layers) applies the final RMSNorm and owns the
 * readout.
 *   - "RFC: pipeline placement across multiple GPUs for models larger than one
 *     device", section "What I found": each stage owns its resident weights,
 *     model state / KV, heap, workspace and prepared kernels; only the hidden
 *     activation crosses the boundary; a logical step is accepted only after
 *     every stage completes.
 *   - "Multi-node layer splitting and tensor parallelism", section "Supported
 *     stage executors": the dense pipeline transfers F32 hidden activations; each
 *     node loads only its layer weights and KV state; the first stage embeds and
 *     the last computes logits.  Section "Launch a layer pipeline" onwards: the
 *     stage executors accept serialized forward / refill / reset / truncate
 *     controls and keep cache ownership across them.
 *   - "41. Many GPUs: tensor, pipeline, expert and data parallelism", section
 *     "Pipeline parallelism": PipelineStage.forward -- embed on the first stage,
 *     the per-block add_norm / attention / add_norm / MLP loop, one residual
 *     tensor across each boundary, final norm at the end.
 *
 * Conventions for every function below:
 *   - Return 0 (STAGE_OK) on success, a negative STAGE_E_* code on failure.  No
 *     C++ exception crosses this boundary: a host allocation that fails inside a call
 *     returns STAGE_E_HOST.  stage_last_error() gives a message.
 *   - After any error no committed sequence length changes; KV rows written by a
 *     failed or uncommitted call are simply overwritten by the retry.
 *   - Arrays named *_host are read on the host before the call returns; device
 *     buffers (hidden activations, logits) are used asynchronously on the
 *     stage's CUDA stream and must stay alive until that stream reaches the work.
 *   - One call at a time per stage.  A call that finds another call of the same
 *     stage in progress returns STAGE_E_BUSY without side effects.
 *   - Every stage of a pipeline runs on one GPU and one stream; the handoff is a
 *     device buffer, no copy through the host.
 */
#ifndef LAYER_RANGE_STAGE_H
#define LAYER_RANGE_STAGE_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define STAGE_API __attribute__((visibility("default")))
#else
#define STAGE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum {
  STAGE_OK = 0,
  STAGE_E_INVALID = -1,      /* bad config, range, shape, null where required, value out of range */
  STAGE_E_DOES_NOT_FIT = -2, /* stage_required_bytes exceeds the budget or the device's free memory */
  STAGE_E_HANDOFF = -3,      /* tokens given to a non-first stage, hidden given to the first, wrong n/width */
  STAGE_E_POSITION = -4,     /* positions not committed_len + i, or >= max_seq_len */
  STAGE_E_BUSY = -5,         /* another call of this stage is in progress */
  STAGE_E_NOT_LAST = -6,     /* readout requested from a stage that does not own it */
  STAGE_E_CUDA = -7,         /* a CUDA runtime error; the message is in stage_last_error */
  STAGE_E_STATE = -8,        /* weights not loaded, or commit beyond what was written */
  STAGE_E_INJECTED = -9,     /* host-side fault injection (stage_debug_inject) */
  STAGE_E_HOST = -10         /* a host allocation failed (a weight staging buffer, a table): no C++
                                exception leaves the library; the message is in the last-error string */
};

typedef struct stage* stage_t;

/* Model shape.  Dense models set n_experts = top_k = expert_ffn = 0.  ffn and
 * expert_ffn need not be multiples of 32 (the last weight block of a row is then
 * partial).  shared_ffn (MoE only, 0 = none): width of a shared expert added to every
 * token's expert mix with weight sigmoid(shared_score . h) ("41. Many GPUs: tensor,
 * pipeline, expert and data parallelism", the MoE layer listings:
 * out + sigmoid(shared_gate(x)) * shared(x)); stages with one decode on the GEMV path.
 * n_layers is at most 65536.  max_seqs / max_seq_len size the KV cache (at most 65536
 * and 2^24); max_tokens (at most 2^20) bounds the tokens of one prefill or decode call.  gemm_bf16_min_tokens: on dense models, calls
 * with at least this many tokens run their projections on the tensor cores (tcgen05)
 * with bf16 operands -- activations rounded to bf16, weights as bf16(f32(scale) * q) --
 * and f32 accumulation; smaller calls, and every call of a MoE model, use the float32
 * dequant-fused GEMV (0 = never use bf16). */
typedef struct {
  int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
  int n_experts, top_k, expert_ffn;
  float rms_eps, rope_theta;
  int max_seqs, max_seq_len, max_tokens;
  int gemm_bf16_min_tokens;
  int shared_ffn;
} stage_model_cfg;

/* Global block range [begin, end): begin == 0 => the stage embeds; end == n_layers
 * => the stage applies the final norm and owns the readout. */
typedef struct {
  int begin, end;
} stage_layer_range;

/* Host int8 block-32 matrix, row-major [rows x cols]: q[rows][cols] int8 and
 * scale[rows][ceil(cols/32)] IEEE fp16 bit patterns; weight (r, c) is
 * scale[r][c/32] * q[r][c].  Blocks run along the input dimension (cols). */
typedef struct {
  const int8_t* q;
  const uint16_t* scale;
  int64_t rows, cols;
} stage_q8;

/* Host weights of one block.  Shapes: norms [hidden] f32; wq [Hq*D x hidden];
 * wk, wv [Hkv*D x hidden]; wo [hidden x Hq*D]; dense: w_gate, w_up [ffn x hidden],
 * w_down [hidden x ffn]; MoE: router [n_experts x hidden] and arrays of n_experts
 * matrices e_gate, e_up [expert_ffn x hidden], e_down [hidden x expert_ffn]; with a
 * shared expert also shared_score [1 x hidden] (the page's shared_gate, a scalar gate),
 * shared_gate, shared_up [shared_ffn x hidden] and shared_down [hidden x shared_ffn]. */
typedef struct {
  const float *attn_norm, *ffn_norm;
  stage_q8 wq, wk, wv, wo;
  stage_q8 w_gate, w_up, w_down;
  stage_q8 router;
  const stage_q8 *e_gate, *e_up, *e_down;
  stage_q8 shared_score, shared_gate, shared_up, shared_down;
} stage_layer_w;

/* Host weights of a stage: embed [vocab x hidden] only if begin == 0; final_norm
 * [hidden] and lm_head [vocab x hidden] only if end == n_layers; layers has
 * end - begin entries, the owned blocks in order.  Nothing outside the range is
 * read ("each stage loads its owned weights"). */
typedef struct {
  stage_q8 embed;
  const float* final_norm;
  stage_q8 lm_head;
  const stage_layer_w* layers;
} stage_weights;

/* A device float32 activation, row-major [rows x cols] (one row per token).  The
 * stage checks rows == n_tokens and cols == hidden: the checked handoff. */
typedef struct {
  float* data;
  int rows, cols;
} stage_act;

/* Bytes stage_create allocates on the device for this range: owned weights (in the
 * device layout), KV cache, RoPE table and workspace.  0 if cfg/range are invalid. */
STAGE_API size_t stage_required_bytes(const stage_model_cfg* cfg, stage_layer_range range);

/* Placement of the model's blocks over n_devices stages (stage k on device k, in order),
 * from the device budgets alone: contiguous ranges, at least one block per stage, and a
 * placement is legal only if every stage's stage_required_bytes fits its own device's
 * budget -- never the summed memory (RFC page, "Heterogeneous GPUs"; TensorSharp page,
 * "Layer split": balance estimated resident bytes, contiguous layers, at least one layer
 * per selected GPU).  Among the legal placements it returns one that minimises the largest
 * required / budget ratio over the stages (for equal budgets: the most balanced resident
 * bytes), the earliest cut on ties.  Pure host code, no device access.
 * device_budgets: host [n_devices] usable bytes per device.  bounds_out: host int32
 * [n_devices + 1], 0 = b[0] < b[1] < ... < b[n] = n_layers; stage k owns [b[k], b[k+1]).
 * required_out: host [n_devices] or NULL, each stage's stage_required_bytes.
 * Returns STAGE_OK, STAGE_E_INVALID (bad cfg or pointers, n_devices outside [1, n_layers],
 * n_layers above 4096: the tables grow as n_layers^2), or STAGE_E_DOES_NOT_FIT (no legal
 * placement). */
STAGE_API int stage_plan_placement(const stage_model_cfg* cfg, int n_devices, const size_t* device_budgets,
                                   int32_t* bounds_out, size_t* required_out);

/* Create a stage on the current CUDA device.  Fails with STAGE_E_DOES_NOT_FIT --
 * before allocating anything -- when stage_required_bytes exceeds
 * device_budget_bytes or the device's free memory (the per-device fit rule of the
 * RFC page, section "Heterogeneous GPUs": required(stage_i) <= budget(device_i)).
 * weights may be NULL: then load blocks with stage_load_layer and the endpoints
 * with stage_load_endpoints before the first forward.  Host weights are copied;
 * the caller may free them after return.  cuda_stream: a cudaStream_t (NULL = the
 * legacy default stream); every kernel of this stage runs on it. */
STAGE_API int stage_create(const stage_model_cfg* cfg, stage_layer_range range, const stage_weights* weights,
                 size_t device_budget_bytes, void* cuda_stream, stage_t* out);

/* Import the weights of one owned block (global index in [begin, end)), copied from the
 * host (the caller may free them after return; synchronous).  Errors: STAGE_E_INVALID (block
 * not owned, a null or mis-shaped matrix), STAGE_E_BUSY, STAGE_E_HOST (the host staging
 * buffer of a matrix), STAGE_E_CUDA.  A failed import leaves the block unloaded, so a
 * forward returns STAGE_E_STATE until it is imported again. */
STAGE_API int stage_load_layer(stage_t st, int global_layer, const stage_layer_w* w);

/* Import the embedding (first stage) and/or final norm + readout (last stage), with the
 * errors of stage_load_layer (STAGE_E_INVALID for a missing endpoint the stage owns). */
STAGE_API int stage_load_endpoints(stage_t st, const stage_weights* w);

/* Prefill / refill: n_tokens tokens, possibly of several sequences.  For each
 * sequence its tokens appear in order with positions committed_len, committed_len
 * + 1, ...  (seq_ids_host, positions_host, tokens_host: host int32 [n_tokens]).
 * First stage: tokens_host set, hidden_in NULL.  Other stages: tokens_host NULL,
 * hidden_in [n_tokens x hidden].  hidden_out [n_tokens x hidden] receives the
 * residual stream (last stage: the final features rmsnorm(x) * gamma_f); it may be
 * the same buffer as hidden_in.  K/V of every token are written to the cache;
 * attention is causal within each sequence.  Nothing is published: stage_commit does that.
 * Errors, all before any launch unless noted: STAGE_E_STATE (weights not all loaded),
 * STAGE_E_INVALID (n_tokens outside [1, max_tokens], a seq_id outside [0, max_seqs), a
 * token outside [0, vocab)), STAGE_E_HANDOFF (tokens on a later stage or a hidden on the
 * first, a missing input, hidden shapes other than [n_tokens x hidden]), STAGE_E_POSITION
 * (positions not committed_len + i per sequence, or reaching max_seq_len), STAGE_E_BUSY,
 * STAGE_E_INJECTED, STAGE_E_CUDA (a launch failed, or a persistent launch's bounded wait ran
 * out; the retry overwrites the uncommitted rows). */
STAGE_API int stage_prefill(stage_t st, int n_tokens, const int32_t* seq_ids_host, const int32_t* positions_host,
                  const int32_t* tokens_host, const stage_act* hidden_in, const stage_act* hidden_out);

/* Decode: one token for each of `batch` distinct sequences, at position
 * committed_len[seq].  Same conventions and errors as stage_prefill, and STAGE_E_INVALID
 * when batch exceeds max_seqs. */
STAGE_API int stage_decode(stage_t st, int batch, const int32_t* seq_ids_host, const int32_t* positions_host,
                 const int32_t* tokens_host, const stage_act* hidden_in, const stage_act* hidden_out);

/* Readout of the last stage for rows row_index_host[0..n_rows) of its last forward:
 * logits = W_head * features.  logits_out: device f32 [n_rows x vocab] or NULL;
 * argmax_out: device int32 [n_rows] or NULL (greedy token, lowest index on ties).
 * Errors: STAGE_E_NOT_LAST (a stage without the readout), STAGE_E_INVALID (n_rows outside
 * [1, max_tokens], a row outside the last forward's tokens), STAGE_E_BUSY, STAGE_E_CUDA. */
STAGE_API int stage_logits(stage_t st, int n_rows, const int32_t* row_index_host, float* logits_out, int32_t* argmax_out);

/* Publish the written rows: committed_len[seq_ids[i]] = new_len[i].  new_len must
 * lie between the committed length and the highest position written since.  All or
 * nothing: STAGE_E_INVALID (null arrays, a seq_id outside [0, max_seqs)) or STAGE_E_STATE
 * (a length outside that window) changes no length; STAGE_E_BUSY. */
STAGE_API int stage_commit(stage_t st, int n, const int32_t* seq_ids_host, const int32_t* new_len_host);

/* Truncate one sequence to len <= committed_len (later rows are overwritten).  Errors:
 * STAGE_E_INVALID (seq_id), STAGE_E_POSITION (len outside [0, committed_len]), STAGE_E_BUSY. */
STAGE_API int stage_truncate(stage_t st, int seq_id, int len);

/* Forget every sequence (committed lengths to 0).  Errors: STAGE_E_BUSY. */
STAGE_API int stage_reset(stage_t st);

/* The committed length of one sequence into *len_out.  STAGE_E_INVALID for a null stage or
 * pointer, or a seq_id outside [0, max_seqs). */
STAGE_API int stage_committed_len(stage_t st, int seq_id, int* len_out);

/* Copy the cached K and V of one owned block and sequence to the host: positions
 * [0, n_pos) of every KV head, fp16 bit patterns, each [n_kv_heads x n_pos x head_dim].
 * Synchronises the stage's stream.  For inspection and equivalence checks.  Errors:
 * STAGE_E_INVALID (block not owned, seq_id, n_pos outside [0, max_seq_len], null buffers),
 * STAGE_E_BUSY, STAGE_E_CUDA (including an error word left by an earlier launch). */
STAGE_API int stage_read_kv(stage_t st, int global_layer, int seq_id, int n_pos, uint16_t* k_host, uint16_t* v_host);

/* Copy K and V rows from the host into the cache of one owned block and sequence:
 * positions [pos0, pos0 + n_pos) of every KV head, fp16 bit patterns, each
 * [n_kv_heads x n_pos x head_dim] (the layout stage_read_kv returns).  For restoring a cache
 * saved with stage_read_kv, or for starting from a given cache.  pos0 may not leave a gap
 * after the positions already written (STAGE_E_POSITION); the rows count as written, so a
 * following stage_commit of the sequence up to pos0 + n_pos publishes them, jointly with
 * the other stages.  Synchronises the stage's stream.  Errors: STAGE_E_INVALID (block not
 * owned, seq_id, negative pos0 or n_pos, null buffers), STAGE_E_POSITION (past max_seq_len,
 * or a gap), STAGE_E_BUSY, STAGE_E_CUDA. */
STAGE_API int stage_write_kv(stage_t st, int global_layer, int seq_id, int pos0, int n_pos, const uint16_t* k_host,
                             const uint16_t* v_host);

/* Which path a call with n_tokens tokens takes: 0 = float32 dequant-fused GEMV kernels,
 * 1 = bf16 tensor-core GEMMs (dense stages; calls of at most 64 tokens stream each weight
 * once against all their tokens), 2 = float32 persistent decode (a single-token call: every
 * block of the stage in one cooperative launch, on MoE stages with the router and top-k
 * computed inside it; the staged input held as three signed bytes per value with one
 * exponent per 16 values, each dot exact in integers before its float32 scaling, so it
 * agrees with 0 to float32 rounding; its own fixed summation order).  The environment variable LRS_PERSISTENT=0, read at
 * stage_create, turns mode 2 off.  LRS_PDL=0, also read at stage_create, launches the
 * per-kernel paths (modes 0 and 1) without programmatic dependent launch: each kernel then
 * starts only after its predecessor on the stream has finished, instead of overlapping its
 * weight-only prologue with the predecessor's tail (process-wide; for measurement).
 * STAGE_E_INVALID for a null stage or pointer. */
STAGE_API int stage_gemm_mode(stage_t st, int n_tokens, int* mode_out);

/* Message of the stage's last failed call ("" if none; "null stage" for NULL).  Owned by the
 * stage, valid until its next call. */
STAGE_API const char* stage_last_error(stage_t st);

/* Message of the last failed stage_create on the calling thread ("" if none). */
STAGE_API const char* stage_create_error(void);

/* Wait for the stage's stream, then free its device memory, pinned staging and events.
 * NULL is accepted.  Buffers the caller owns (hidden activations, logits) are untouched. */
STAGE_API void stage_destroy(stage_t st);

/* Host-side fault injection for tests (no GPU fault is ever caused):
 *   what = 1: mark the stage busy (value 1) or idle (value 0) as if a call were in progress;
 *   what = 2: the next prefill/decode returns STAGE_E_INJECTED before launching anything;
 *   what = 3 (value 1): the next single-token decode that runs on the persistent kernel (outside
 *     stream capture) waits, in its attention step, for a tag that no step of the launch
 *     writes.  Every such wait runs out after its time limit (0.2 s); the kernel then sets the
 *     stage's error word, waits (bounded) for its own copies in flight and leaves, so the call
 *     reports STAGE_E_CUDA when its error word is read and the next call runs normally.  This
 *     tests the device-side timeout path without faulting or hanging the GPU. */
STAGE_API int stage_debug_inject(stage_t st, int what, int value);

/* ------------------------------------------------------------------------- pipeline
 * Stages chained in order on one GPU and one stream.  Stage k's hidden_out buffer
 * is stage k+1's hidden_in (a pointer handoff).  A step is published jointly:
 * every stage's committed lengths advance only if every stage succeeded (RFC page,
 * "What I propose upstreaming", PR 1: checked activation handoff, joint
 * completion / state publication). */
typedef struct stage_pipeline* stage_pipeline_t;

/* stages: n_stages created stages whose ranges tile [0, n_layers) in order, on one
 * device and stream.  The pipeline does not own them.  Errors: STAGE_E_INVALID (ranges that
 * do not tile the model, differing configs, streams or devices, null pointers), STAGE_E_CUDA
 * (its buffers), STAGE_E_HOST. */
STAGE_API int stage_pipeline_create(stage_t* stages, int n_stages, stage_pipeline_t* out);

/* One step of all stages: prefill (is_prefill = 1) or decode, then the readout of
 * rows row_index_host[0..n_rows) on the last stage.  logits_out (device, may be
 * NULL), next_tokens_host (host int32 [n_rows], may be NULL: the greedy tokens,
 * read back after the step, with every stage's error word).  Every stage's call is
 * validated and its inputs copied in before the first launch, so a call that fails
 * validation runs no stage.  Commits every stage to the new lengths on success.  Errors:
 * any stage's stage_prefill / stage_decode errors (nothing is committed on any stage),
 * STAGE_E_INVALID (a readout row outside the step's tokens), STAGE_E_BUSY (a stage busy). */
STAGE_API int stage_pipeline_step(stage_pipeline_t p, int is_prefill, int n_tokens, const int32_t* seq_ids_host,
                        const int32_t* positions_host, const int32_t* tokens_host, int n_rows,
                        const int32_t* row_index_host, float* logits_out, int32_t* next_tokens_host);

/* n_steps greedy decode steps for `batch` sequences, feeding each greedy token back
 * on the device.  first_tokens_host: the token to feed at each sequence's committed
 * length.  tokens_out_host: host int32 [n_steps x batch], the greedy token of each
 * step.  use_graph = 1 replays one captured CUDA graph per step.  Commits n_steps
 * positions on every stage at the end.  Errors: STAGE_E_INVALID (batch, seq_ids, tokens),
 * STAGE_E_POSITION (a sequence would pass max_seq_len), STAGE_E_BUSY, STAGE_E_CUDA (graph
 * capture or launch, or a kernel's error word); nothing is committed on failure. */
STAGE_API int stage_pipeline_generate(stage_pipeline_t p, int batch, const int32_t* seq_ids_host,
                            const int32_t* first_tokens_host, int n_steps, int use_graph,
                            int32_t* tokens_out_host);

/* Kernel timing for measurement: with enable = 1 every following step (generate or
 * stage_pipeline_step) records a CUDA event pair around the FFN gate/up launch of every
 * block -- the gate/up (or expert gate/up) GEMV, or the gate/up tensor-core GEMM of a call
 * that runs on the tensor cores.  stage_pipeline_kernel_time returns the mean duration
 * (microseconds) of those launches in the last step and their count.  Events sit between kernels, so a timed launch
 * does not overlap its predecessor; leave timing off for the headline measurement. */
STAGE_API int stage_pipeline_kernel_timing(stage_pipeline_t p, int enable);
/* Count 0 while timing is off; STAGE_E_STATE when timing is on but no timed step has run;
 * STAGE_E_INVALID for null pointers. */
STAGE_API int stage_pipeline_kernel_time(stage_pipeline_t p, float* mean_us, int* count);

/* Bytes handed across boundary k (0-based) so far, and the number of handoffs.
 * STAGE_E_INVALID for a boundary outside [0, n_stages - 1) or null pointers. */
STAGE_API int stage_pipeline_handoff_stats(stage_pipeline_t p, int boundary, int64_t* calls, int64_t* bytes);

/* Message of the pipeline's last failed call ("" if none), owned by the pipeline. */
STAGE_API const char* stage_pipeline_last_error(stage_pipeline_t p);
/* Free the pipeline's own buffers and graphs (not the stages).  NULL is accepted. */
STAGE_API void stage_pipeline_destroy(stage_pipeline_t p);

#ifdef __cplusplus
}
#endif
#endif /* LAYER_RANGE_STAGE_H */

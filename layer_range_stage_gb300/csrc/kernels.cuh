// Launch interface of the stage kernels (host side).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace lrs {

enum GemvEpi { EPI_STORE = 0, EPI_RESID = 1, EPI_SWIGLU = 2, EPI_QKV = 3, EPI_MOE_SWIGLU = 4, EPI_SWIGLU_BF16 = 5 };

// Device int8 block-32 matrix: q [N][Kp] stored biased (byte = q + 128), s [N][Kp/32] fp16 bits,
// Kp = K rounded up to 256 (the padding columns face zero inputs).  Row order is the device
// order chosen at import.
// Rows of a device matrix are padded to a multiple of this many weights (every row of bytes
// and of fp16 scales then starts on a 16-byte boundary).
constexpr int kRowPad = 256;
inline int row_pad(int k) { return (k + kRowPad - 1) / kRowPad * kRowPad; }

struct DevQ8 {
  uint8_t* q = nullptr;
  uint16_t* s = nullptr;
  int N = 0, K = 0, Kp = 0;
};

// y[t][n] = sum_k W[n][k] * h[t][k], h = x (or rmsnorm(x) * gamma when gamma != nullptr),
// followed by the epilogue `epi`:
//   EPI_STORE : out[t][n] = y
//   EPI_RESID : out[t][n] = resid[t][n] + y            (the residual add; may run in place)
//   EPI_SWIGLU: device rows (2j, 2j+1) are (gate_j, up_j); out[t][j] = silu(g) * u
//   EPI_QKV   : device rows (2i, 2i+1) of each head are its dims (i, i + D/2); q heads, then
//               k heads, then v heads.  q, k are rotated (rotate-half RoPE at pos[t]); q goes
//               to qout[t][head][D] (f32), k and v to the fp16 cache at (seq[t], kv head, pos[t]).
struct GemvArgs {
  DevQ8 w;
  const float* x = nullptr;
  int ldx = 0;
  const int* x_rows = nullptr;  // optional: token t reads input row x_rows[t]
  int ntok = 0;
  const float* gamma = nullptr;
  float eps = 0.f;
  int epi = EPI_STORE;
  float* out = nullptr;
  int ldo = 0;
  const float* resid = nullptr;
  int ldr = 0;
  // EPI_QKV
  float* qout = nullptr;
  __half* kc = nullptr;
  __half* vc = nullptr;
  const int* seq = nullptr;
  const int* pos = nullptr;
  const float2* rope = nullptr;  // [max_len][D/2] (cos, sin)
  int n_q_heads = 0, n_kv_heads = 0, head_dim = 0, max_len = 0;
  int* err = nullptr;  // device error word: set (never cleared by kernels) when a bounded wait times out
  // Expert gather (routed MoE).  Row gather: device row r of the launch is row r % rows_per_slot
  // of expert ids[r / rows_per_slot].  K gather: 16-weight chunk c of a row is chunk
  // c % seg_chunks of row `row` of expert ids[c / seg_chunks] (expert matrices of seg_rows
  // rows, rows seg_chunks * 16 weights long).
  const int* ids = nullptr;
  const float* slot_w = nullptr;  // EPI_MOE_SWIGLU: out[slot * ldo_slot + i] = silu(g) * u * slot_w[slot]
  int rows_per_slot = 0, seg_chunks = 0, seg_rows = 0, ldo_slot = 0;
};

// Split-K grouped-query decode attention over the fp16 cache with a deterministic merge of
// the chunk partials by the last CTA of each (token, kv head).
struct AttnArgs {
  const float* q = nullptr;      // [ntok][Hq][D]
  const __half* kc = nullptr;    // [max_seqs][Hkv][max_len][D] (this layer)
  const __half* vc = nullptr;
  const int* seq = nullptr;      // [ntok]
  const int* pos = nullptr;      // [ntok]; token t attends to positions 0..pos[t]
  float* out = nullptr;          // [ntok][Hq][D]
  float* part_o = nullptr;       // scratch [ntok][Hkv][n_chunks][Hq/Hkv][D]
  float2* part_ml = nullptr;     // scratch [ntok][Hq][n_chunks] (running max, sum)
  int* counters = nullptr;       // scratch [ntok][Hkv], zero between launches (the kernel re-zeroes)
  int ntok = 0, Hq = 0, Hkv = 0, D = 0, max_len = 0, n_chunks = 1;
  float scale = 1.f;
};

// Tensor-core GEMM of the prefill: C[m][n] = sum_k A[m][k] * W[n][k] with A bf16 activations
// [M][lda] (zero beyond K up to Kp) and W the int8 block-32 matrix dequantised to bf16 in
// shared memory; f32 accumulation in TMEM; epilogues as for the GEMV (EPI_STORE, EPI_RESID,
// EPI_QKV with token t = row m, EPI_SWIGLU_BF16 writing bf16 [M][ldo_bf16]).
struct GemmArgs {
  const __nv_bfloat16* a = nullptr;
  int lda = 0;
  DevQ8 w;
  int M = 0;
  int epi = EPI_STORE;
  float* out = nullptr;
  int ldo = 0;
  const float* resid = nullptr;
  int ldr = 0;
  __nv_bfloat16* out_bf16 = nullptr;
  int ldo_bf16 = 0;
  float* qout = nullptr;
  __half* kc = nullptr;
  __half* vc = nullptr;
  const int* seq = nullptr;
  const int* pos = nullptr;
  const float2* rope = nullptr;
  int n_q_heads = 0, n_kv_heads = 0, head_dim = 0, max_len = 0;
  int* err = nullptr;
  // Calls of at most kGemmSmallTokens tokens (gemm_small_splits): the K-split partials
  // [splits][kGemmSmallTokens][N] f32 and one arrival counter per 128-row weight tile (zero
  // between launches: the last CTA of a tile re-zeroes its counter).  Without them the K range
  // is not split.
  float* ws = nullptr;
  unsigned* tile_cnt = nullptr;
};
cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st);
// The weight-streaming GEMM of small calls: at most this many tokens, weight tiles of 128 rows.
constexpr int kGemmSmallTokens = 64;
constexpr int kGemmSmallRows = 128;
// K splits of a small call's GEMM of an N x Kp matrix (1 when the weight tiles alone fill the
// SMs), and the workspace its split needs (0 without a split).
int gemm_small_splits(int N, int Kp);
size_t gemm_small_ws_bytes(int N, int Kp);
cudaError_t prepare_gemm_tc();
// RMSNorm (gamma != nullptr) or plain copy of f32 rows [ntok][ld_in] to bf16 rows [ntok][ld_out],
// zero-filled from K to ld_out; with `rows`, output row t is input row rows[t].
cudaError_t launch_rows_to_bf16(const float* x, int ld_in, int K, const float* gamma, float eps, int ntok,
                                __nv_bfloat16* out, int ld_out, cudaStream_t st, const int* rows = nullptr);

// Persistent decode of a stage: every block of the stage for one token in one cooperative
// launch (one CTA per SM).  Per block: QKV GEMV (RMSNorm; RoPE + fp16 KV append epilogue),
// split-K attention with the last-arriving chunk merging, O GEMV + residual, (MoE) router and
// ranking, gate/up GEMV (RMSNorm, SwiGLU epilogue), down GEMV + residual; the steps hand their
// vectors over as tagged entries (no grid barrier).  Weight rows stream through a per-warp ring
// of tensor copies that runs ahead across steps and blocks.
struct MegaLayer {
  DevQ8 wqkv, wo, wgu, wdown;  // dense FFN (wgu, wdown) ...
  DevQ8 router, egu, edown;    // ... or routed experts (stacked as in the stage's layout)
  const float* attn_norm = nullptr;
  const float* ffn_norm = nullptr;
  __half* kc = nullptr;  // [max_seqs][Hkv][max_len][D] of this block
  __half* vc = nullptr;
  // Per projection step (QKV, O, router, gate/up, down): the tensor maps of its weight bytes and
  // of its scales, each a box of two rows (a pair) by one ring slot of columns (mega_tensor_maps).
  CUtensorMap tmap[2 * 5];
};
// Fills ml.tmap from the matrices of ml (MoE stages: n_experts > 0).  False if a matrix cannot
// be described (unaligned base).
bool mega_tensor_maps(MegaLayer& ml, bool moe);
// A two-dimensional tiled tensor map (no interleave, L2 promotion of 256 bytes, zero fill).
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw);
struct MegaArgs {
  const MegaLayer* layers = nullptr;  // device [nl]
  int nl = 0;
  const float* hin = nullptr;  // [H] block input of the first block (may equal hout)
  float* hout = nullptr;       // [H] residual stream after the last block
  unsigned long long* tags = nullptr;  // the tagged vectors between steps (mega_tag_entries entries)
  float* qbuf = nullptr;       // [Hq * D] rotated q
  float* obuf = nullptr;       // [Hq * D] attention output
  float* abuf = nullptr;       // [F] SwiGLU output
  float* part_o = nullptr;     // attention split-K partials (layout of AttnArgs, token 0)
  float2* part_ml = nullptr;
  const int* seq = nullptr;    // device [1]
  const int* pos = nullptr;    // device [1]
  const float2* rope = nullptr;
  int H = 0, Hq = 0, Hkv = 0, D = 0, F = 0, max_len = 0, n_chunks = 1;
  int n_experts = 0, top_k = 0, EF = 0;  // MoE stages: experts, selected per token, expert FFN width
  float* logits = nullptr;                // MoE stages: [n_experts] router logits of the current block
  float eps = 1e-5f, scale = 1.f;
  unsigned* bar = nullptr;  // [64]: [0] CTAs done with the SwiGLU step, [1] exit counter, [2 + h]
                            // attention counter of KV head h (zero between launches: the last CTA
                            // out re-zeroes), [63] launch sequence
  int* err = nullptr;
  unsigned bar_extra = 0;  // tests: added to the tag the attention waits for (0 in use)
};
// Whether the persistent decode covers this shape (and the shared memory it needs fits).  MoE:
// n_experts > 0, F = top_k * expert FFN width (the gathered down input).
bool mega_supported(int H, int q_dim, int F, int head_dim, int group, int n_experts = 0, int top_k = 0);
// Entries of MegaArgs::tags for a stage of these shapes.
size_t mega_tag_entries(int H, int q_dim, int kv_dim, int n_experts);
// Attention chunks per KV head used by the persistent decode (about one item per SM).
int mega_chunks(int n_kv_heads);
cudaError_t launch_mega_decode(const MegaArgs& a, cudaStream_t st);
cudaError_t prepare_mega();

int sm_count();
// Sets kernel attributes and records launch limits; call once per process before any
// launch, outside stream capture.
cudaError_t prepare_kernels();
// Programmatic dependent launch of the stage kernels (on by default).
void set_pdl(bool on);
bool pdl_enabled();

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t st);
cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t st);
// Causal attention of a prefill call (same arguments; n_chunks, part_o, part_ml, counters
// unused): tiles of 64 positions shared by 64 query rows of one KV head.
cudaError_t launch_attn_prefill(const AttnArgs& a, cudaStream_t st);
cudaError_t prepare_attn_prefill();
constexpr int kAttnMaxChunks = 64;
bool attn_decode_supported(int head_dim, int group);
cudaError_t launch_embed(const DevQ8& table, const int* tok, int ntok, float* out, int ldo, cudaStream_t st);
cudaError_t launch_final_norm(const float* x, int ldx, const float* gamma, float eps, int H, int ntok,
                              float* feat, float* out, int ldo, cudaStream_t st);
cudaError_t launch_argmax(const float* logits, int V, int n_rows, int* out, cudaStream_t st);
cudaError_t launch_advance(int* pos, const int* tok, int* hist, int* step, int batch, cudaStream_t st);
// Top-k routing of each token over n_experts router logits [ntok][n_experts]: the k largest
// (ties to the lower expert id) in descending order, weights softmax over the selected k.
// Top-k routing of ntok tokens: logits [ntok][ld] (entries 0..n_experts-1 ranked), ids and
// weights [ntok][kw]; kw == k + 1: weight slot k is sigmoid(logits[t][n_experts]) (a shared
// expert's gate).
cudaError_t launch_topk(const float* logits, int ld, int n_experts, int k, int ntok, int kw, int* ids, float* wts,
                        cudaStream_t st);

}  // namespace lrs

// Stage runtime: the C ABI of include/stage.h.
//
// A stage owns one device arena holding its weights (device layout), fp16 KV cache,
// RoPE table and workspace; the same plan sizes stage_required_bytes and the arena, so
// the fit check and the allocation cannot disagree ("RFC: pipeline placement across
// multiple GPUs for models larger than one device", sections "What I found" and
// "Heterogeneous GPUs").  Host-side bookkeeping (committed lengths, validation, joint
// commit) lives here; every number of the forward is computed by the kernels.

#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <limits>
#include <memory>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include <cuda_bf16.h>

#include "../../include/stage.h"
#include "kernels.cuh"

using lrs::DevQ8;

namespace {

constexpr int kMaxChunks = lrs::kAttnMaxChunks;
constexpr size_t kAlign = 256;
constexpr int kMaxLayers = 1 << 16;    // blocks of a model: keeps every layer-count product in range
constexpr int kMaxPlanLayers = 4096;   // the placement planner's tables grow as n_layers^2

inline size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
inline int kpad(int k) { return lrs::row_pad(k); }

struct LayerDev {
  float* attn_norm = nullptr;
  float* ffn_norm = nullptr;
  DevQ8 wqkv, wo, wgu, wdown;  // dense (wgu interleaves gate/up rows)
  DevQ8 router, egu, edown;    // MoE: experts stacked, egu [E][2*EF][Kp(H)], edown [E][H][Kp(EF)];
                               // router [E (+1: the shared expert's scalar gate)][Kp(H)]
  DevQ8 sgu, sdown;            // shared expert: gate/up interleaved [2*SF][Kp(H)], down [H][Kp(SF)]
  bool loaded = false;
};

// Visit every device allocation of a stage in a fixed order.  f(bytes, void** slot).
template <class F>
void walk_plan(const stage_model_cfg& c, int begin, int end, std::vector<LayerDev>* layers, DevQ8* embed,
               DevQ8* head, float** final_norm, __half** kc, __half** vc, float2** rope, float** qbuf,
               float** obuf, float** abuf, float** feat, float** logits, int** argmax, float** part_o,
               float2** part_ml, int** counters, int** d_seq, int** d_pos, int** d_tok, int** d_rows, int** err_word,
               float** moe_logits, int** moe_ids, float** moe_wts, __nv_bfloat16** act_bf16,
               __nv_bfloat16** ffn_bf16, lrs::MegaLayer** mlayers, unsigned long long** mega_tags, unsigned** mega_bar,
               int** shared_id0, float** gemm_ws, unsigned** gemm_cnt, F&& f) {
  auto q8 = [&](DevQ8* m, int N, int K) {
    if (m) {
      m->N = N;
      m->K = K;
      m->Kp = kpad(K);
    }
    f((size_t)N * kpad(K), m ? (void**)&m->q : nullptr);
    f((size_t)N * (kpad(K) / 32) * 2, m ? (void**)&m->s : nullptr);
  };
  const int H = c.hidden, D = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  const bool moe = c.n_experts > 0;
  const int sh = c.shared_ffn > 0 ? 1 : 0;  // a shared expert: one more router row and weight slot
  for (int l = begin; l < end; ++l) {
    LayerDev* L = layers ? &(*layers)[l - begin] : nullptr;
    f((size_t)H * 4, L ? (void**)&L->attn_norm : nullptr);
    f((size_t)H * 4, L ? (void**)&L->ffn_norm : nullptr);
    q8(L ? &L->wqkv : nullptr, (Hq + 2 * Hkv) * D, H);
    q8(L ? &L->wo : nullptr, H, Hq * D);
    if (moe) {
      q8(L ? &L->router : nullptr, c.n_experts + sh, H);
      q8(L ? &L->egu : nullptr, c.n_experts * 2 * c.expert_ffn, H);
      q8(L ? &L->edown : nullptr, c.n_experts * H, c.expert_ffn);
      if (sh) {
        q8(L ? &L->sgu : nullptr, 2 * c.shared_ffn, H);
        q8(L ? &L->sdown : nullptr, H, c.shared_ffn);
      }
    } else {
      q8(L ? &L->wgu : nullptr, 2 * c.ffn, H);
      q8(L ? &L->wdown : nullptr, H, c.ffn);
    }
  }
  if (begin == 0) q8(embed, c.vocab, H);
  if (end == c.n_layers) {
    f((size_t)H * 4, (void**)final_norm);
    q8(head, c.vocab, H);
  }
  const size_t kv = (size_t)(end - begin) * c.max_seqs * Hkv * (size_t)c.max_seq_len * D * 2;
  f(kv, (void**)kc);
  f(kv, (void**)vc);
  f((size_t)c.max_seq_len * (D / 2) * 8, (void**)rope);
  const size_t T = (size_t)c.max_tokens;
  const int ffn_w = moe ? c.top_k * kpad(c.expert_ffn) + (sh ? kpad(c.shared_ffn) : 0) : c.ffn;
  f(T * Hq * D * 4, (void**)qbuf);
  f(T * Hq * D * 4, (void**)obuf);
  f(T * (size_t)std::max(ffn_w, H) * 4, (void**)abuf);
  f(T * H * 4, (void**)feat);
  if (end == c.n_layers) {
    f(T * (size_t)c.vocab * 4, (void**)logits);
    f(T * 4, (void**)argmax);
  }
  const size_t pairs = std::max((size_t)c.max_seqs * kMaxChunks, T * 4);
  f(pairs * Hq * D * 4, (void**)part_o);
  f(pairs * Hq * 8, (void**)part_ml);
  f(T * Hkv * 4, (void**)counters);
  f(T * 4, (void**)d_seq);
  f(T * 4, (void**)d_pos);
  f(T * 4, (void**)d_tok);
  f(T * 4, (void**)d_rows);
  f(4, (void**)err_word);
  // persistent decode: block descriptors, the tagged vectors between its steps, counters
  f((size_t)(end - begin) * sizeof(lrs::MegaLayer), (void**)mlayers);
  f(lrs::mega_tag_entries(H, Hq * D, Hkv * D, c.n_experts) * 8, (void**)mega_tags);
  f(256, (void**)mega_bar);
  if (!moe && c.gemm_bf16_min_tokens > 0) {  // bf16 operands of the tensor-core GEMMs
    f(T * (size_t)std::max(kpad(H), kpad(Hq * D)) * 2, (void**)act_bf16);
    f(T * (size_t)kpad(c.ffn) * 2, (void**)ffn_bf16);
    if (c.gemm_bf16_min_tokens <= lrs::kGemmSmallTokens) {
      // calls of at most kGemmSmallTokens tokens: K-split partials of the weight-streaming GEMM
      // (the largest of the stage's projections and readout) and the tiles' arrival counters
      const int mats[][2] = {{(Hq + 2 * Hkv) * D, H}, {H, Hq * D}, {2 * c.ffn, H}, {H, c.ffn},
                             {end == c.n_layers ? c.vocab : 0, H}};
      size_t ws = 0;
      int tiles = 1;
      for (const auto& m : mats)
        if (m[0] > 0) {
          ws = std::max(ws, lrs::gemm_small_ws_bytes(m[0], kpad(m[1])));
          tiles = std::max(tiles, (m[0] + lrs::kGemmSmallRows - 1) / lrs::kGemmSmallRows);
        }
      f(ws, (void**)gemm_ws);
      f((size_t)tiles * 4, (void**)gemm_cnt);
    }
  }
  if (moe) {
    f(T * (c.n_experts + sh) * 4, (void**)moe_logits);
    f(T * (c.top_k + sh) * 4, (void**)moe_ids);
    f(T * (c.top_k + sh) * 4, (void**)moe_wts);
    if (sh) f(4, (void**)shared_id0);  // expert id 0 of the shared expert's one-slot gate/up launch
  }
}

thread_local std::string g_create_error;

size_t plan_bytes(const stage_model_cfg& c, int begin, int end) {
  size_t total = 0;
  walk_plan(c, begin, end, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
            nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
            nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr,
            [&](size_t b, void**) { total += round_up(b, kAlign); });
  return total;
}

bool cfg_valid(const stage_model_cfg* c, stage_layer_range r, std::string* why) {
  auto bad = [&](const char* m) {
    if (why) *why = m;
    return false;
  };
  if (!c) return bad("null config");
  if (c->n_layers <= 0 || c->hidden <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->head_dim <= 0 ||
      c->vocab <= 0)
    return bad("non-positive model dimension");
  if (c->n_layers > kMaxLayers) return bad("n_layers too large (at most 65536)");
  if (c->n_q_heads % c->n_kv_heads) return bad("n_q_heads must be a multiple of n_kv_heads");
  // every GEMV input row is staged with 16-byte copies
  if (c->hidden % 4 || c->ffn % 4 || c->expert_ffn % 4) return bad("hidden, ffn and expert_ffn must be multiples of 4");
  if (!lrs::attn_decode_supported(c->head_dim, c->n_q_heads / c->n_kv_heads))
    return bad("unsupported head_dim / GQA group (head_dim 64 or 128; group 1, 2, 4 or 8)");
  const bool moe = c->n_experts > 0;
  if (moe && (c->top_k <= 0 || c->top_k > c->n_experts || c->expert_ffn <= 0 || c->top_k > 32))
    return bad("bad MoE shape");
  if (!moe && (c->ffn <= 0 || c->top_k != 0 || c->expert_ffn != 0)) return bad("bad dense FFN shape");
  if (c->shared_ffn < 0 || (c->shared_ffn > 0 && (!moe || c->shared_ffn % 4)))
    return bad("shared_ffn: MoE models only, a multiple of 4");
  if (c->max_seqs <= 0 || c->max_seq_len <= 0 || c->max_tokens <= 0) return bad("non-positive capacity");
  if (c->max_seq_len > (1 << 24) || c->max_tokens > (1 << 20) || c->max_seqs > (1 << 16)) return bad("capacity too large");
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 0.f)) return bad("rms_eps and rope_theta must be positive");
  if (r.begin < 0 || r.end > c->n_layers || r.begin >= r.end) return bad("layer range must satisfy 0 <= begin < end <= n_layers");
  return true;
}

// A C++ exception inside an entry point -- in practice a host allocation that failed (a weight
// staging buffer, a table) -- ends the call with STAGE_E_HOST instead of crossing the C ABI.
// Recording the message may itself fail; that is ignored.
int host_failure(std::string* msg, const char* what) noexcept {
  try {
    if (msg) *msg = std::string("host: ") + what;
  } catch (...) {
  }
  return STAGE_E_HOST;
}

}  // namespace

// ------------------------------------------------------------------------------------------ stage

struct stage {
  stage_model_cfg cfg{};
  int begin = 0, end = 0;
  bool first = false, last = false;
  cudaStream_t stream = nullptr;
  int device = 0;
  char* arena = nullptr;
  size_t arena_bytes = 0;
  std::vector<LayerDev> layers;
  DevQ8 embed, head;
  float* final_norm = nullptr;
  bool endpoints_loaded = false;
  __half *kc = nullptr, *vc = nullptr;
  size_t layer_kv = 0;  // elements per layer
  float2* rope = nullptr;
  float *qbuf = nullptr, *obuf = nullptr, *abuf = nullptr, *feat = nullptr, *logits = nullptr;
  int* argmax = nullptr;
  float* part_o = nullptr;
  float2* part_ml = nullptr;
  int* counters = nullptr;
  int *d_seq = nullptr, *d_pos = nullptr, *d_tok = nullptr, *d_rows = nullptr;
  int* err_word = nullptr;     // device: set by a kernel whose bounded wait timed out
  int* shared_id0 = nullptr;   // device: a zero expert id (the shared expert's gate/up launch)
  float* gemm_ws = nullptr;     // K-split partials of the small calls' GEMMs (lrs::GemmArgs::ws)
  unsigned* gemm_cnt = nullptr;  // their weight tiles' arrival counters
  float* moe_logits = nullptr;  // [max_tokens][n_experts] router logits
  int* moe_ids = nullptr;       // [max_tokens][top_k] selected experts
  float* moe_wts = nullptr;     // [max_tokens][top_k] routing weights
  __nv_bfloat16* act_bf16 = nullptr;  // [max_tokens][Kp] bf16 GEMM operand (normed x, attention out)
  __nv_bfloat16* ffn_bf16 = nullptr;  // [max_tokens][Kp(ffn)] bf16 SwiGLU output
  lrs::MegaLayer* mlayers = nullptr;  // device block descriptors of the persistent decode
  unsigned long long* mega_tags = nullptr;  // its tagged vectors between steps
  unsigned* mega_bar = nullptr;       // its counters (exit, attention, launch sequence)
  bool mega = false;                  // single-token decode calls use the persistent kernel
  bool call_prefill = false;          // the current forward is a prefill call (causal attention kernel)
  std::vector<cudaEvent_t> tev;  // measurement: event pair around each FFN up-projection launch
  bool timing = false;
  int timed_pairs = 0;           // event pairs recorded by the last forward
  int32_t* h_stage = nullptr;  // pinned host staging [4][max_tokens] (seq, pos, tok, rows), then
                               // [max_tokens] read-back tokens and the read-back error word
  cudaEvent_t staged = nullptr;  // recorded after the last copy out of h_stage
  std::vector<int> committed, pending;
  int last_n = 0;
  std::atomic<int> busy{0};
  int fail_next = 0;
  int stall_barrier = 0;  // tests: the next persistent launch's attention waits for a tag never written
  std::string err;
};

namespace {

int set_err(stage* st, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  if (st) st->err = buf;
  return code;
}

int cuda_err(stage* st, cudaError_t e, const char* where) {
  return set_err(st, STAGE_E_CUDA, "%s: %s", where, cudaGetErrorString(e));
}

struct BusyGuard {
  stage* st;
  bool ok;
  explicit BusyGuard(stage* s) : st(s), ok(s->busy.exchange(1) == 0) {}
  ~BusyGuard() {
    if (ok) st->busy.store(0);
  }
};

// Device weights are stored biased: byte = q + 128 (two's complement int8 xor 0x80).
void bias_bytes(std::vector<uint8_t>& q) {
  for (auto& b : q) b ^= 0x80u;
}

// Copy rows of a host q8 matrix into device row order: dst row i <- src row perm(i).
template <class Perm>
int upload_q8(stage* st, const stage_q8& src, const DevQ8& dst, int64_t src_rows, Perm perm, const char* name) {
  if (!src.q || !src.scale) return set_err(st, STAGE_E_INVALID, "%s: null data", name);
  if (src.rows != src_rows || src.cols != dst.K)
    return set_err(st, STAGE_E_INVALID, "%s: shape [%lld x %lld], expected [%lld x %d]", name, (long long)src.rows,
                   (long long)src.cols, (long long)src_rows, dst.K);
  const int nb_src = (dst.K + 31) / 32, nb = dst.Kp / 32;
  std::vector<uint8_t> q((size_t)dst.N * dst.Kp, 0);
  std::vector<uint16_t> s((size_t)dst.N * nb, 0);
  for (int i = 0; i < dst.N; ++i) {
    const int64_t r = perm(i);
    std::memcpy(&q[(size_t)i * dst.Kp], src.q + r * src.cols, (size_t)dst.K);
    std::memcpy(&s[(size_t)i * nb], src.scale + r * nb_src, (size_t)nb_src * 2);
  }
  bias_bytes(q);
  cudaError_t e = cudaMemcpy(dst.q, q.data(), q.size(), cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(dst.s, s.data(), s.size() * 2, cudaMemcpyHostToDevice);
  if (e != cudaSuccess) return cuda_err(st, e, name);
  return STAGE_OK;
}

int upload_plain(stage* st, const stage_q8& src, const DevQ8& dst, const char* name) {
  return upload_q8(st, src, dst, dst.N, [](int i) { return (int64_t)i; }, name);
}

int upload_f32(stage* st, const float* src, float* dst, size_t n, const char* name) {
  if (!src) return set_err(st, STAGE_E_INVALID, "%s: null data", name);
  cudaError_t e = cudaMemcpy(dst, src, n * 4, cudaMemcpyHostToDevice);
  return e == cudaSuccess ? STAGE_OK : cuda_err(st, e, name);
}

// Upload several host matrices stacked in one device matrix (row offset per part).
int upload_stack(stage* st, const stage_q8& src, const DevQ8& whole, int row0, int rows, const char* name) {
  DevQ8 part = whole;
  part.N = rows;
  part.q = whole.q + (size_t)row0 * whole.Kp;
  part.s = whole.s + (size_t)row0 * (whole.Kp / 32);
  return upload_q8(st, src, part, rows, [](int i) { return (int64_t)i; }, name);
}

// Gate and up matrices [F x K] interleaved into device rows (2j, 2j+1) = (gate_j, up_j) of dst.
int upload_gate_up(stage* st, const stage_q8& gate, const stage_q8& up, const DevQ8& dst, int F, const char* name) {
  const int K = dst.K, nb_src = (K + 31) / 32, nb = dst.Kp / 32;
  std::vector<uint8_t> q((size_t)2 * F * dst.Kp, 0);
  std::vector<uint16_t> s((size_t)2 * F * nb, 0);
  const stage_q8* srcs[2] = {&gate, &up};
  for (int which = 0; which < 2; ++which) {
    const stage_q8& m = *srcs[which];
    if (!m.q || !m.scale || m.rows != F || m.cols != K)
      return set_err(st, STAGE_E_INVALID, "%s (%s): bad shape or null", name, which ? "up" : "gate");
    for (int j = 0; j < F; ++j) {
      std::memcpy(&q[(size_t)(2 * j + which) * dst.Kp], m.q + (int64_t)j * K, K);
      std::memcpy(&s[(size_t)(2 * j + which) * nb], m.scale + (int64_t)j * nb_src, (size_t)nb_src * 2);
    }
  }
  bias_bytes(q);
  cudaError_t ce = cudaMemcpy(dst.q, q.data(), q.size(), cudaMemcpyHostToDevice);
  if (ce == cudaSuccess) ce = cudaMemcpy(dst.s, s.data(), s.size() * 2, cudaMemcpyHostToDevice);
  return ce == cudaSuccess ? STAGE_OK : cuda_err(st, ce, name);
}

// The persistent decode's descriptor of block gl: its device weights, norms and KV cache.
int upload_descriptor(stage* st, int gl, const LayerDev& L) {
  lrs::MegaLayer ml;
  ml.wqkv = L.wqkv;
  ml.wo = L.wo;
  ml.wgu = L.wgu;
  ml.wdown = L.wdown;
  ml.router = L.router;
  ml.egu = L.egu;
  ml.edown = L.edown;
  ml.attn_norm = L.attn_norm;
  ml.ffn_norm = L.ffn_norm;
  ml.kc = st->kc + (size_t)(gl - st->begin) * st->layer_kv;
  ml.vc = st->vc + (size_t)(gl - st->begin) * st->layer_kv;
  if (!lrs::mega_tensor_maps(ml, st->cfg.n_experts > 0))
    return set_err(st, STAGE_E_CUDA, "block %d: tensor maps of the persistent decode", gl);
  const cudaError_t ce = cudaMemcpy(st->mlayers + (gl - st->begin), &ml, sizeof ml, cudaMemcpyHostToDevice);
  return ce == cudaSuccess ? STAGE_OK : cuda_err(st, ce, "block descriptor");
}

int load_layer(stage* st, int gl, const stage_layer_w* w) {
  const stage_model_cfg& c = st->cfg;
  if (gl < st->begin || gl >= st->end) return set_err(st, STAGE_E_INVALID, "layer %d outside the owned range [%d, %d)", gl, st->begin, st->end);
  if (!w) return set_err(st, STAGE_E_INVALID, "null layer weights");
  LayerDev& L = st->layers[gl - st->begin];
  L.loaded = false;
  const int H = c.hidden, D = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads, hd = D / 2;
  int rc;
  if ((rc = upload_f32(st, w->attn_norm, L.attn_norm, H, "attn_norm"))) return rc;
  if ((rc = upload_f32(st, w->ffn_norm, L.ffn_norm, H, "ffn_norm"))) return rc;
  // Fused QKV: q heads, k heads, v heads; inside a head device rows (2i, 2i+1) = dims (i, i + D/2).
  struct Part {
    const stage_q8* m;
    int heads, first_head;
    const char* name;
  } parts[3] = {{&w->wq, Hq, 0, "wq"}, {&w->wk, Hkv, Hq, "wk"}, {&w->wv, Hkv, Hq + Hkv, "wv"}};
  for (const Part& p : parts) {
    DevQ8 sub = L.wqkv;
    sub.N = p.heads * D;
    sub.q = L.wqkv.q + (size_t)p.first_head * D * L.wqkv.Kp;
    sub.s = L.wqkv.s + (size_t)p.first_head * D * (L.wqkv.Kp / 32);
    rc = upload_q8(st, *p.m, sub, (int64_t)p.heads * D, [=](int i) {
      const int head = i / D, r = i % D;
      return (int64_t)head * D + ((r & 1) ? (r >> 1) + hd : (r >> 1));
    }, p.name);
    if (rc) return rc;
  }
  if ((rc = upload_plain(st, w->wo, L.wo, "wo"))) return rc;
  if (c.n_experts > 0) {
    if ((rc = upload_stack(st, w->router, L.router, 0, c.n_experts, "router"))) return rc;
    if (c.shared_ffn > 0) {  // the shared expert: its scalar gate as the router's last row
      if ((rc = upload_stack(st, w->shared_score, L.router, c.n_experts, 1, "shared_score"))) return rc;
      if ((rc = upload_gate_up(st, w->shared_gate, w->shared_up, L.sgu, c.shared_ffn, "shared gate/up"))) return rc;
      if ((rc = upload_plain(st, w->shared_down, L.sdown, "shared_down"))) return rc;
    }
    if (!w->e_gate || !w->e_up || !w->e_down) return set_err(st, STAGE_E_INVALID, "null expert arrays");
    const int EF = c.expert_ffn;
    for (int e = 0; e < c.n_experts; ++e) {
      // gate/up of expert e interleaved: device rows (2j, 2j+1) = (gate_j, up_j)
      DevQ8 gu = L.egu;
      gu.N = 2 * EF;
      gu.q = L.egu.q + (size_t)e * 2 * EF * L.egu.Kp;
      gu.s = L.egu.s + (size_t)e * 2 * EF * (L.egu.Kp / 32);
      // even rows from gate, odd rows from up
      std::vector<uint8_t> q((size_t)2 * EF * gu.Kp, 0);
      std::vector<uint16_t> s((size_t)2 * EF * (gu.Kp / 32), 0);
      const stage_q8* srcs[2] = {&w->e_gate[e], &w->e_up[e]};
      for (int which = 0; which < 2; ++which) {
        const stage_q8& m = *srcs[which];
        if (!m.q || !m.scale || m.rows != EF || m.cols != H)
          return set_err(st, STAGE_E_INVALID, "expert %d %s: bad shape or null", e, which ? "up" : "gate");
        const int nb_src = (H + 31) / 32, nb = gu.Kp / 32;
        for (int j = 0; j < EF; ++j) {
          std::memcpy(&q[(size_t)(2 * j + which) * gu.Kp], m.q + (int64_t)j * H, H);
          std::memcpy(&s[(size_t)(2 * j + which) * nb], m.scale + (int64_t)j * nb_src, (size_t)nb_src * 2);
        }
      }
      bias_bytes(q);
      cudaError_t ce = cudaMemcpy(gu.q, q.data(), q.size(), cudaMemcpyHostToDevice);
      if (ce == cudaSuccess) ce = cudaMemcpy(gu.s, s.data(), s.size() * 2, cudaMemcpyHostToDevice);
      if (ce != cudaSuccess) return cuda_err(st, ce, "expert gate/up");
      if ((rc = upload_stack(st, w->e_down[e], L.edown, e * H, H, "expert down"))) return rc;
    }
    if ((rc = upload_descriptor(st, gl, L))) return rc;
  } else {
    const int F = c.ffn;
    std::vector<uint8_t> q((size_t)2 * F * L.wgu.Kp, 0);
    std::vector<uint16_t> s((size_t)2 * F * (L.wgu.Kp / 32), 0);
    const stage_q8* srcs[2] = {&w->w_gate, &w->w_up};
    const int nb_src = (H + 31) / 32, nb = L.wgu.Kp / 32;
    for (int which = 0; which < 2; ++which) {
      const stage_q8& m = *srcs[which];
      if (!m.q || !m.scale || m.rows != F || m.cols != H)
        return set_err(st, STAGE_E_INVALID, "%s: bad shape or null", which ? "w_up" : "w_gate");
      for (int j = 0; j < F; ++j) {
        std::memcpy(&q[(size_t)(2 * j + which) * L.wgu.Kp], m.q + (int64_t)j * H, H);
        std::memcpy(&s[(size_t)(2 * j + which) * nb], m.scale + (int64_t)j * nb_src, (size_t)nb_src * 2);
      }
    }
    bias_bytes(q);
    cudaError_t ce = cudaMemcpy(L.wgu.q, q.data(), q.size(), cudaMemcpyHostToDevice);
    if (ce == cudaSuccess) ce = cudaMemcpy(L.wgu.s, s.data(), s.size() * 2, cudaMemcpyHostToDevice);
    if (ce != cudaSuccess) return cuda_err(st, ce, "gate/up");
    if ((rc = upload_plain(st, w->w_down, L.wdown, "w_down"))) return rc;
    if ((rc = upload_descriptor(st, gl, L))) return rc;
  }
  L.loaded = true;
  return STAGE_OK;
}

int load_endpoints(stage* st, const stage_weights* w) {
  if (!w) return set_err(st, STAGE_E_INVALID, "null weights");
  int rc;
  if (st->first && (rc = upload_plain(st, w->embed, st->embed, "embed"))) return rc;
  if (st->last) {
    if ((rc = upload_f32(st, w->final_norm, st->final_norm, st->cfg.hidden, "final_norm"))) return rc;
    if ((rc = upload_plain(st, w->lm_head, st->head, "lm_head"))) return rc;
  }
  st->endpoints_loaded = true;
  return STAGE_OK;
}

// Weight uploads stage each matrix in a host buffer (up to the size of the readout); a failed
// allocation there ends the upload with STAGE_E_HOST and leaves the stage usable.
template <class F>
int guarded_upload(stage* st, F&& f) {
  try {
    return f();
  } catch (const std::exception& ex) {
    return host_failure(&st->err, ex.what());
  }
}

bool weights_ready(stage* st) {
  if ((st->first || st->last) && !st->endpoints_loaded) return false;
  for (auto& L : st->layers)
    if (!L.loaded) return false;
  return true;
}

// Split-K factor of decode attention: at least about one CTA per SM, and chunks of at most
// ~512 positions for the longest sequence of the call (a batch of ragged contexts is as slow
// as its longest chunk), chunks of >= 32 positions, bounded by the partial-result scratch.
int attn_chunks(const stage* st, int ntok, int max_len_in_call) {
  const size_t pairs = std::max((size_t)st->cfg.max_seqs * kMaxChunks, (size_t)st->cfg.max_tokens * 4);
  int n = (max_len_in_call + 31) / 32;
  const int work = std::max(1, ntok * st->cfg.n_kv_heads);
  const int fill = std::max(1, (lrs::sm_count() + work - 1) / work);  // about one wave
  n = std::min(n, std::max(fill, (max_len_in_call + 511) / 512));
  n = std::min<int>(n, (int)std::min<size_t>(kMaxChunks, pairs / (size_t)ntok));
  return std::max(1, n);
}

// A kernel-timing event: an external event node when the stream is being captured (a plain
// record there would become an internal graph dependency), a plain record otherwise.
void timing_mark(cudaEvent_t ev, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaStreamIsCapturing(s, &cs);
  if (cs == cudaStreamCaptureStatusActive)
    cudaEventRecordWithFlags(ev, s, cudaEventRecordExternal);
  else
    cudaEventRecord(ev, s);
}

// Arithmetic of a call with n tokens: the bf16 tensor-core GEMMs for dense stages once n
// reaches gemm_bf16_min_tokens (when set), the float32 dequant-fused GEMV otherwise.
bool use_tc(const stage* st, int n) {
  return st->cfg.n_experts == 0 && st->cfg.gemm_bf16_min_tokens > 0 && n >= st->cfg.gemm_bf16_min_tokens;
}

// One block on the tensor cores (bf16 operands, f32 accumulation and residual).
int block_tc(stage* st, int li, LayerDev& L, int n, const int* d_seq, const int* d_pos, const float* xin, float* hout,
             __half* kc, __half* vc, int n_chunks, cudaStream_t s) {
  const stage_model_cfg& c = st->cfg;
  const int H = c.hidden, D = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  const int ldh = kpad(H), ldq = kpad(Hq * D), ldf = kpad(c.ffn);
  cudaError_t e;
  if ((e = lrs::launch_rows_to_bf16(xin, H, H, L.attn_norm, c.rms_eps, n, st->act_bf16, ldh, s)) != cudaSuccess)
    return cuda_err(st, e, "norm 1");
  lrs::GemmArgs g;
  g.a = st->act_bf16;
  g.lda = ldh;
  g.w = L.wqkv;
  g.M = n;
  g.epi = lrs::EPI_QKV;
  g.qout = st->qbuf;
  g.kc = kc;
  g.vc = vc;
  g.seq = d_seq;
  g.pos = d_pos;
  g.rope = st->rope;
  g.n_q_heads = Hq;
  g.n_kv_heads = Hkv;
  g.head_dim = D;
  g.max_len = c.max_seq_len;
  g.err = st->err_word;
  g.ws = st->gemm_ws;
  g.tile_cnt = st->gemm_cnt;
  if ((e = lrs::launch_gemm_tc(g, s)) != cudaSuccess) return cuda_err(st, e, "qkv gemm");
  lrs::AttnArgs at;
  at.q = st->qbuf;
  at.kc = kc;
  at.vc = vc;
  at.seq = d_seq;
  at.pos = d_pos;
  at.out = st->obuf;
  at.part_o = st->part_o;
  at.part_ml = st->part_ml;
  at.counters = st->counters;
  at.ntok = n;
  at.Hq = Hq;
  at.Hkv = Hkv;
  at.D = D;
  at.max_len = c.max_seq_len;
  at.n_chunks = n_chunks;
  at.scale = (float)(1.0 / std::sqrt((double)D));
  if ((e = (st->call_prefill ? lrs::launch_attn_prefill(at, s) : lrs::launch_attn_decode(at, s))) != cudaSuccess)
    return cuda_err(st, e, "attention");
  if ((e = lrs::launch_rows_to_bf16(st->obuf, Hq * D, Hq * D, nullptr, 0.f, n, st->act_bf16, ldq, s)) != cudaSuccess)
    return cuda_err(st, e, "attention out");
  lrs::GemmArgs o;
  o.a = st->act_bf16;
  o.lda = ldq;
  o.w = L.wo;
  o.M = n;
  o.epi = lrs::EPI_RESID;
  o.resid = xin;
  o.ldr = H;
  o.out = hout;
  o.ldo = H;
  o.err = st->err_word;
  o.ws = st->gemm_ws;
  o.tile_cnt = st->gemm_cnt;
  if ((e = lrs::launch_gemm_tc(o, s)) != cudaSuccess) return cuda_err(st, e, "o gemm");
  if ((e = lrs::launch_rows_to_bf16(hout, H, H, L.ffn_norm, c.rms_eps, n, st->act_bf16, ldh, s)) != cudaSuccess)
    return cuda_err(st, e, "norm 2");
  lrs::GemmArgs gu;
  gu.a = st->act_bf16;
  gu.lda = ldh;
  gu.w = L.wgu;
  gu.M = n;
  gu.epi = lrs::EPI_SWIGLU_BF16;
  gu.out_bf16 = st->ffn_bf16;
  gu.ldo_bf16 = ldf;
  gu.err = st->err_word;
  gu.ws = st->gemm_ws;
  gu.tile_cnt = st->gemm_cnt;
  if (st->timing) timing_mark(st->tev[2 * li], s);
  if ((e = lrs::launch_gemm_tc(gu, s)) != cudaSuccess) return cuda_err(st, e, "gate_up gemm");
  if (st->timing) timing_mark(st->tev[2 * li + 1], s);
  lrs::GemmArgs dn;
  dn.a = st->ffn_bf16;
  dn.lda = ldf;
  dn.w = L.wdown;
  dn.M = n;
  dn.epi = lrs::EPI_RESID;
  dn.resid = hout;
  dn.ldr = H;
  dn.out = hout;
  dn.ldo = H;
  dn.err = st->err_word;
  dn.ws = st->gemm_ws;
  dn.tile_cnt = st->gemm_cnt;
  if ((e = lrs::launch_gemm_tc(dn, s)) != cudaSuccess) return cuda_err(st, e, "down gemm");
  return STAGE_OK;
}

// The per-stage launch chain.  Inputs are device arrays; hout receives the residual stream
// (the final features on the last stage).
int forward_dev(stage* st, int n, const int* d_seq, const int* d_pos, const int* d_tok, const float* hin, float* hout,
                int n_chunks, cudaStream_t s) {
  const stage_model_cfg& c = st->cfg;
  const int H = c.hidden, D = c.head_dim, Hq = c.n_q_heads, Hkv = c.n_kv_heads;
  cudaError_t e;
  if (st->first && (e = lrs::launch_embed(st->embed, d_tok, n, hout, H, s)) != cudaSuccess) return cuda_err(st, e, "embed");
  const bool tc = use_tc(st, n);
  st->timed_pairs = st->end - st->begin;
  if (n == 1 && st->mega) {  // single-token decode: every block in one persistent launch
    lrs::MegaArgs m;
    m.layers = st->mlayers;
    m.nl = st->end - st->begin;
    m.hin = st->first ? hout : hin;
    m.hout = hout;
    m.tags = st->mega_tags;
    m.qbuf = st->qbuf;
    m.obuf = st->obuf;
    m.abuf = st->abuf;
    m.part_o = st->part_o;
    m.part_ml = st->part_ml;
    m.seq = d_seq;
    m.pos = d_pos;
    m.rope = st->rope;
    m.H = H;
    m.Hq = Hq;
    m.Hkv = Hkv;
    m.D = D;
    const bool moe = c.n_experts > 0;
    m.F = moe ? c.top_k * kpad(c.expert_ffn) : c.ffn;
    m.n_experts = c.n_experts;
    m.top_k = c.top_k;
    m.EF = c.expert_ffn;
    m.logits = st->moe_logits;
    m.max_len = c.max_seq_len;
    m.n_chunks = lrs::mega_chunks(Hkv);
    m.eps = c.rms_eps;
    m.scale = (float)(1.0 / std::sqrt((double)D));
    m.bar = st->mega_bar;
    m.err = st->err_word;
    if (st->stall_barrier) {  // never baked into a captured graph
      cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
      if (cudaStreamIsCapturing(s, &cs) == cudaSuccess && cs == cudaStreamCaptureStatusNone) {
        m.bar_extra = 1;
        st->stall_barrier = 0;
      }
    }
    if (st->timing) timing_mark(st->tev[0], s);
    if ((e = lrs::launch_mega_decode(m, s)) != cudaSuccess) return cuda_err(st, e, "persistent decode");
    if (st->timing) timing_mark(st->tev[1], s);
    st->timed_pairs = 1;
  } else
  for (int li = 0; li < st->end - st->begin; ++li) {
    LayerDev& L = st->layers[li];
    const float* xin = (li == 0 && !st->first) ? hin : hout;
    __half* kc = st->kc + (size_t)li * st->layer_kv;
    __half* vc = st->vc + (size_t)li * st->layer_kv;
    if (tc) {
      const int rc = block_tc(st, li, L, n, d_seq, d_pos, xin, hout, kc, vc, n_chunks, s);
      if (rc) return rc;
      continue;
    }
    lrs::GemvArgs g;
    g.w = L.wqkv;
    g.x = xin;
    g.ldx = H;
    g.ntok = n;
    g.gamma = L.attn_norm;
    g.eps = c.rms_eps;
    g.epi = lrs::EPI_QKV;
    g.qout = st->qbuf;
    g.kc = kc;
    g.vc = vc;
    g.seq = d_seq;
    g.pos = d_pos;
    g.rope = st->rope;
    g.n_q_heads = Hq;
    g.n_kv_heads = Hkv;
    g.head_dim = D;
    g.max_len = c.max_seq_len;
    g.err = st->err_word;
    if ((e = lrs::launch_gemv(g, s)) != cudaSuccess) return cuda_err(st, e, "qkv");

    lrs::AttnArgs a;
    a.q = st->qbuf;
    a.kc = kc;
    a.vc = vc;
    a.seq = d_seq;
    a.pos = d_pos;
    a.out = st->obuf;
    a.part_o = st->part_o;
    a.part_ml = st->part_ml;
    a.counters = st->counters;
    a.ntok = n;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.D = D;
    a.max_len = c.max_seq_len;
    a.n_chunks = n_chunks;
    a.scale = (float)(1.0 / std::sqrt((double)D));
    if ((e = ((st->call_prefill && n > 1) ? lrs::launch_attn_prefill(a, s) : lrs::launch_attn_decode(a, s))) !=
        cudaSuccess)
      return cuda_err(st, e, "attention");

    lrs::GemvArgs o;
    o.w = L.wo;
    o.x = st->obuf;
    o.ldx = Hq * D;
    o.ntok = n;
    o.epi = lrs::EPI_RESID;
    o.resid = xin;
    o.ldr = H;
    o.out = hout;
    o.ldo = H;
    o.err = st->err_word;
    if ((e = lrs::launch_gemv(o, s)) != cudaSuccess) return cuda_err(st, e, "o_proj");

    if (c.n_experts > 0) {
      // routed experts: router GEMV (RMSNorm prologue) -> top-k -> per token the selected
      // experts' gate/up (row gather, SwiGLU scaled by the routing weight) and down
      // (K gather over the k slots, residual add)
      const int E = c.n_experts, kk = c.top_k, EF = c.expert_ffn, KpE = kpad(EF);
      const int SF = c.shared_ffn, sh = SF > 0 ? 1 : 0, kw = kk + sh;  // ids / weights per token
      const int ffn_w = kk * KpE + (sh ? kpad(SF) : 0);                  // abuf per token
      lrs::GemvArgs r;
      r.w = L.router;
      r.x = hout;
      r.ldx = H;
      r.ntok = n;
      r.gamma = L.ffn_norm;
      r.eps = c.rms_eps;
      r.epi = lrs::EPI_STORE;
      r.out = st->moe_logits;
      r.ldo = E + sh;
      r.err = st->err_word;
      if ((e = lrs::launch_gemv(r, s)) != cudaSuccess) return cuda_err(st, e, "router");
      if ((e = lrs::launch_topk(st->moe_logits, E + sh, E, kk, n, kw, st->moe_ids, st->moe_wts, s)) != cudaSuccess)
        return cuda_err(st, e, "top-k");
      for (int t = 0; t < n; ++t) {
        lrs::GemvArgs gu;
        gu.w = L.egu;
        gu.w.N = kk * 2 * EF;
        gu.x = hout + (size_t)t * H;
        gu.ldx = H;
        gu.ntok = 1;
        gu.gamma = L.ffn_norm;
        gu.eps = c.rms_eps;
        gu.epi = lrs::EPI_MOE_SWIGLU;
        gu.out = st->abuf + (size_t)t * ffn_w;
        gu.ids = st->moe_ids + (size_t)t * kw;
        gu.slot_w = st->moe_wts + (size_t)t * kw;
        gu.rows_per_slot = 2 * EF;
        gu.ldo_slot = KpE;
        gu.err = st->err_word;
        if (st->timing && t == 0) timing_mark(st->tev[2 * li], s);
        if ((e = lrs::launch_gemv(gu, s)) != cudaSuccess) return cuda_err(st, e, "expert gate_up");
        if (st->timing && t == 0) timing_mark(st->tev[2 * li + 1], s);
        if (sh) {  // the shared expert's SwiGLU, scaled by sigmoid of its gate (weight slot kk)
          lrs::GemvArgs sg = gu;
          sg.w = L.sgu;
          sg.out = st->abuf + (size_t)t * ffn_w + (size_t)kk * KpE;
          sg.ids = st->shared_id0;
          sg.slot_w = st->moe_wts + (size_t)t * kw + kk;
          sg.rows_per_slot = 2 * SF;
          sg.ldo_slot = kpad(SF);
          if ((e = lrs::launch_gemv(sg, s)) != cudaSuccess) return cuda_err(st, e, "shared gate_up");
        }
        lrs::GemvArgs dn;
        dn.w = L.edown;
        dn.w.N = H;
        dn.w.K = kk * KpE;
        dn.w.Kp = kk * KpE;
        dn.x = st->abuf + (size_t)t * ffn_w;
        dn.ldx = kk * KpE;
        dn.ntok = 1;
        dn.epi = lrs::EPI_RESID;
        dn.resid = hout + (size_t)t * H;
        dn.ldr = H;
        dn.out = hout + (size_t)t * H;
        dn.ldo = H;
        dn.ids = st->moe_ids + (size_t)t * kw;
        dn.seg_chunks = KpE / 16;
        dn.seg_rows = H;
        dn.err = st->err_word;
        if ((e = lrs::launch_gemv(dn, s)) != cudaSuccess) return cuda_err(st, e, "expert down");
        if (sh) {  // + the shared expert's down projection
          lrs::GemvArgs sd;
          sd.w = L.sdown;
          sd.x = st->abuf + (size_t)t * ffn_w + (size_t)kk * KpE;
          sd.ldx = kpad(SF);
          sd.ntok = 1;
          sd.epi = lrs::EPI_RESID;
          sd.resid = hout + (size_t)t * H;
          sd.ldr = H;
          sd.out = hout + (size_t)t * H;
          sd.ldo = H;
          sd.err = st->err_word;
          if ((e = lrs::launch_gemv(sd, s)) != cudaSuccess) return cuda_err(st, e, "shared down");
        }
      }
      continue;
    }
    lrs::GemvArgs gu;
    gu.w = L.wgu;
    gu.x = hout;
    gu.ldx = H;
    gu.ntok = n;
    gu.gamma = L.ffn_norm;
    gu.eps = c.rms_eps;
    gu.epi = lrs::EPI_SWIGLU;
    gu.out = st->abuf;
    gu.ldo = c.ffn;
    gu.err = st->err_word;
    if (st->timing) timing_mark(st->tev[2 * li], s);
    if ((e = lrs::launch_gemv(gu, s)) != cudaSuccess) return cuda_err(st, e, "gate_up");
    if (st->timing) timing_mark(st->tev[2 * li + 1], s);

    lrs::GemvArgs dn;
    dn.w = L.wdown;
    dn.x = st->abuf;
    dn.ldx = c.ffn;
    dn.ntok = n;
    dn.epi = lrs::EPI_RESID;
    dn.resid = hout;
    dn.ldr = H;
    dn.out = hout;
    dn.ldo = H;
    dn.err = st->err_word;
    if ((e = lrs::launch_gemv(dn, s)) != cudaSuccess) return cuda_err(st, e, "down");
  }
  if (st->last &&
      (e = lrs::launch_final_norm(hout, H, st->final_norm, c.rms_eps, H, n, st->feat, hout, H, s)) != cudaSuccess)
    return cuda_err(st, e, "final_norm");
  st->last_n = n;
  return STAGE_OK;
}

// After a synchronisation: report (and clear) a device-side wait timeout of this stage.
int check_device_error(stage* st) {
  int v = 0;
  cudaError_t e = cudaMemcpy(&v, st->err_word, 4, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_err(st, e, "error word");
  if (v) {
    cudaMemset(st->err_word, 0, 4);
    return set_err(st, STAGE_E_CUDA, "a kernel's bounded wait timed out; its outputs are invalid");
  }
  return STAGE_OK;
}

// Host validation of one forward call against the committed lengths (no device access).
int validate_call(stage* st, bool decode, int n, const int32_t* seq, const int32_t* pos, const int32_t* tok,
                  const stage_act* hin, const stage_act* hout, int* max_len_out) {
  const stage_model_cfg& c = st->cfg;
  if (n <= 0 || n > c.max_tokens) return set_err(st, STAGE_E_INVALID, "n_tokens %d outside [1, %d]", n, c.max_tokens);
  if (decode && n > c.max_seqs) return set_err(st, STAGE_E_INVALID, "decode batch %d exceeds max_seqs %d", n, c.max_seqs);
  if (!seq || !pos) return set_err(st, STAGE_E_INVALID, "null seq_ids or positions");
  if (st->first) {
    if (!tok) return set_err(st, STAGE_E_HANDOFF, "the first stage embeds tokens: tokens required");
    if (hin && hin->data) return set_err(st, STAGE_E_HANDOFF, "the first stage takes tokens, not a hidden activation");
  } else {
    if (tok) return set_err(st, STAGE_E_HANDOFF, "stage [%d, %d) takes a hidden activation, not tokens", st->begin, st->end);
    if (!hin || !hin->data) return set_err(st, STAGE_E_HANDOFF, "hidden_in required");
    if (hin->rows != n || hin->cols != c.hidden)
      return set_err(st, STAGE_E_HANDOFF, "hidden_in is [%d x %d], expected [%d x %d]", hin->rows, hin->cols, n, c.hidden);
  }
  if (!hout || !hout->data) return set_err(st, STAGE_E_HANDOFF, "hidden_out required");
  if (((uintptr_t)hout->data & 15) || (hin && hin->data && ((uintptr_t)hin->data & 15)))
    return set_err(st, STAGE_E_HANDOFF, "hidden buffers must be 16-byte aligned");
  if (hout->rows != n || hout->cols != c.hidden)
    return set_err(st, STAGE_E_HANDOFF, "hidden_out is [%d x %d], expected [%d x %d]", hout->rows, hout->cols, n, c.hidden);
  std::vector<int> seen(c.max_seqs, 0);
  int max_len = 0;
  for (int i = 0; i < n; ++i) {
    const int s = seq[i];
    if (s < 0 || s >= c.max_seqs) return set_err(st, STAGE_E_INVALID, "seq_id %d outside [0, %d)", s, c.max_seqs);
    if (decode && seen[s]) return set_err(st, STAGE_E_INVALID, "decode batch repeats seq_id %d", s);
    const int expect = st->committed[s] + seen[s];
    if (pos[i] != expect) return set_err(st, STAGE_E_POSITION, "token %d of seq %d at position %d, expected %d", i, s, pos[i], expect);
    if (pos[i] >= c.max_seq_len) return set_err(st, STAGE_E_POSITION, "position %d >= max_seq_len %d", pos[i], c.max_seq_len);
    if (tok && (tok[i] < 0 || tok[i] >= c.vocab)) return set_err(st, STAGE_E_INVALID, "token id %d outside [0, %d)", tok[i], c.vocab);
    seen[s]++;
    max_len = std::max(max_len, pos[i] + 1);
  }
  *max_len_out = max_len;
  return STAGE_OK;
}

// Validate a forward call and copy its arrays in (through pinned memory into fixed device
// buffers, on the stage's stream); *max_len receives the longest context of the call.
int stage_call_inputs(stage* st, bool decode, int n, const int32_t* seq, const int32_t* pos, const int32_t* tok,
                      const stage_act* hin, const stage_act* hout, int* max_len) {
  if (!weights_ready(st)) return set_err(st, STAGE_E_STATE, "weights not loaded");
  int rc;
  if ((rc = validate_call(st, decode, n, seq, pos, tok, hin, hout, max_len))) return rc;
  if (st->fail_next) {
    const int code = st->fail_next;
    st->fail_next = 0;
    return set_err(st, code, "injected failure");
  }
  // the previous copies out of the staging area must have finished before it is overwritten
  const int T = st->cfg.max_tokens;
  cudaError_t e = cudaEventSynchronize(st->staged);
  if (e != cudaSuccess) return cuda_err(st, e, "staging");
  std::memcpy(st->h_stage, seq, n * 4);
  std::memcpy(st->h_stage + T, pos, n * 4);
  if (tok) std::memcpy(st->h_stage + 2 * T, tok, n * 4);
  e = cudaMemcpyAsync(st->d_seq, st->h_stage, n * 4, cudaMemcpyHostToDevice, st->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(st->d_pos, st->h_stage + T, n * 4, cudaMemcpyHostToDevice, st->stream);
  if (e == cudaSuccess && tok) e = cudaMemcpyAsync(st->d_tok, st->h_stage + 2 * T, n * 4, cudaMemcpyHostToDevice, st->stream);
  if (e == cudaSuccess) e = cudaEventRecord(st->staged, st->stream);
  if (e != cudaSuccess) return cuda_err(st, e, "stage inputs");
  return STAGE_OK;
}

// The launches of a forward call whose inputs are in (stage_call_inputs).
int stage_call_launch(stage* st, bool decode, int n, const int32_t* seq, const int32_t* pos, const stage_act* hin,
                      const stage_act* hout, int max_len) {
  st->call_prefill = !decode;
  const int rc = forward_dev(st, n, st->d_seq, st->d_pos, st->d_tok, hin ? hin->data : nullptr, hout->data,
                             attn_chunks(st, n, max_len), st->stream);
  if (rc) return rc;
  for (int i = 0; i < n; ++i) st->pending[seq[i]] = std::max(st->pending[seq[i]], pos[i] + 1);
  return STAGE_OK;
}

int run_forward(stage* st, bool decode, int n, const int32_t* seq, const int32_t* pos, const int32_t* tok,
                const stage_act* hin, const stage_act* hout) {
  int max_len = 0;
  const int rc = stage_call_inputs(st, decode, n, seq, pos, tok, hin, hout, &max_len);
  return rc ? rc : stage_call_launch(st, decode, n, seq, pos, hin, hout, max_len);
}

}  // namespace

// ------------------------------------------------------------------------------------------ C ABI

extern "C" {

size_t stage_required_bytes(const stage_model_cfg* cfg, stage_layer_range range) try {
  if (!cfg_valid(cfg, range, nullptr)) return 0;
  return plan_bytes(*cfg, range.begin, range.end);
} catch (const std::exception& ex) {
  return 0;  // as for an invalid request
} catch (...) {
  return 0;
}

int stage_plan_placement(const stage_model_cfg* cfg, int n_devices, const size_t* device_budgets,
                         int32_t* bounds_out, size_t* required_out) try {
  if (!cfg || !device_budgets || !bounds_out) return STAGE_E_INVALID;
  const int n = cfg->n_layers, S = n_devices;
  if (S < 1 || S > n || n > kMaxPlanLayers || !cfg_valid(cfg, stage_layer_range{0, n}, nullptr)) return STAGE_E_INVALID;
  // req[a][b]: bytes of a stage owning [a, b) (endpoints, KV and workspace included)
  std::vector<size_t> req((size_t)(n + 1) * (n + 1), 0);
  for (int a = 0; a < n; ++a)
    for (int b = a + 1; b <= n; ++b) req[(size_t)a * (n + 1) + b] = plan_bytes(*cfg, a, b);
  // best[k][b]: the smallest achievable max ratio for stages 0..k-1 covering [0, b); cut[k][b]
  // the start of stage k-1 there.  Ratios compare exactly as required * (1 / budget) in double.
  const double inf = std::numeric_limits<double>::infinity();
  std::vector<double> best((size_t)(S + 1) * (n + 1), inf);
  std::vector<int> cut((size_t)(S + 1) * (n + 1), -1);
  best[0] = 0.0;
  for (int k = 1; k <= S; ++k) {
    const size_t budget = device_budgets[k - 1];
    for (int b = k; b <= n - (S - k); ++b) {
      for (int a = k - 1; a < b; ++a) {
        const double prev = best[(size_t)(k - 1) * (n + 1) + a];
        const size_t r = req[(size_t)a * (n + 1) + b];
        if (prev == inf || r > budget) continue;
        const double cost = std::max(prev, (double)r / (double)std::max<size_t>(budget, 1));
        if (cost < best[(size_t)k * (n + 1) + b]) {
          best[(size_t)k * (n + 1) + b] = cost;
          cut[(size_t)k * (n + 1) + b] = a;
        }
      }
    }
  }
  if (best[(size_t)S * (n + 1) + n] == inf) return STAGE_E_DOES_NOT_FIT;
  bounds_out[S] = n;
  for (int k = S, b = n; k >= 1; --k) {
    const int a = cut[(size_t)k * (n + 1) + b];
    bounds_out[k - 1] = a;
    if (required_out) required_out[k - 1] = req[(size_t)a * (n + 1) + b];
    b = a;
  }
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(nullptr, ex.what());
} catch (...) {
  return host_failure(nullptr, "unknown exception");
}

int stage_create(const stage_model_cfg* cfg, stage_layer_range range, const stage_weights* weights,
                 size_t device_budget_bytes, void* cuda_stream, stage_t* out) try {
  if (!out) return STAGE_E_INVALID;
  *out = nullptr;
  std::string why;
  g_create_error.clear();
  if (!cfg_valid(cfg, range, &why)) {
    g_create_error = why;
    return STAGE_E_INVALID;
  }
  const size_t need = plan_bytes(*cfg, range.begin, range.end);
  char msg[256];
  if (need <= device_budget_bytes) {
    const char* pdl = getenv("LRS_PDL");
    if (pdl && pdl[0] == '0') lrs::set_pdl(false);
    const cudaError_t pe = lrs::prepare_kernels();  // outside any stream capture
    if (pe != cudaSuccess) {
      g_create_error = std::string("kernel setup: ") + cudaGetErrorString(pe);
      return STAGE_E_CUDA;
    }
  }
  if (need > device_budget_bytes) {
    snprintf(msg, sizeof msg, "DoesNotFit: stage needs %zu bytes, device budget is %zu", need, device_budget_bytes);
    g_create_error = msg;
    return STAGE_E_DOES_NOT_FIT;
  }
  size_t free_b = 0, total_b = 0;
  cudaError_t ce = cudaMemGetInfo(&free_b, &total_b);
  if (ce != cudaSuccess) {
    g_create_error = std::string("cudaMemGetInfo: ") + cudaGetErrorString(ce);
    return STAGE_E_CUDA;
  }
  if (need > free_b) {
    snprintf(msg, sizeof msg, "DoesNotFit: stage needs %zu bytes, device has %zu free", need, free_b);
    g_create_error = msg;
    return STAGE_E_DOES_NOT_FIT;
  }

  stage* st = new (std::nothrow) stage();
  if (!st) return STAGE_E_INVALID;
  st->cfg = *cfg;
  st->begin = range.begin;
  st->end = range.end;
  st->first = range.begin == 0;
  st->last = range.end == cfg->n_layers;
  st->stream = (cudaStream_t)cuda_stream;
  cudaGetDevice(&st->device);
  try {
    st->layers.resize(range.end - range.begin);
    st->committed.assign(cfg->max_seqs, 0);
    st->pending.assign(cfg->max_seqs, 0);
  } catch (const std::exception& ex) {
    delete st;
    return host_failure(&g_create_error, ex.what());
  }
  cudaError_t e = cudaMalloc(&st->arena, need);
  if (e != cudaSuccess) {
    g_create_error = std::string("cudaMalloc: ") + cudaGetErrorString(e);
    delete st;
    return e == cudaErrorMemoryAllocation ? STAGE_E_DOES_NOT_FIT : STAGE_E_CUDA;
  }
  st->arena_bytes = need;
  size_t off = 0;
  walk_plan(*cfg, range.begin, range.end, &st->layers, &st->embed, &st->head, &st->final_norm, &st->kc, &st->vc,
            &st->rope, &st->qbuf, &st->obuf, &st->abuf, &st->feat, &st->logits, &st->argmax, &st->part_o,
            &st->part_ml, &st->counters, &st->d_seq, &st->d_pos, &st->d_tok, &st->d_rows, &st->err_word,
            &st->moe_logits, &st->moe_ids, &st->moe_wts, &st->act_bf16, &st->ffn_bf16, &st->mlayers, &st->mega_tags,
            &st->mega_bar, &st->shared_id0, &st->gemm_ws, &st->gemm_cnt, [&](size_t b, void** slot) {
              if (slot) *slot = st->arena + off;
              off += round_up(b, kAlign);
            });
  st->layer_kv = (size_t)cfg->max_seqs * cfg->n_kv_heads * (size_t)cfg->max_seq_len * cfg->head_dim;
  // zero everything once (KV rows never written read as zero; attention counters start at 0)
  e = cudaMemset(st->arena, 0, need);
  // RoPE table: cos/sin of pos * theta^(-2i/D), computed in double on the host
  if (e == cudaSuccess) {
    const int hd = cfg->head_dim / 2;
    const size_t n_tab = (size_t)cfg->max_seq_len * hd;
    std::unique_ptr<float2[]> tab(new (std::nothrow) float2[n_tab]);
    if (!tab) {
      stage_destroy(st);
      return host_failure(&g_create_error, "RoPE table allocation failed");
    }
    for (int p = 0; p < cfg->max_seq_len; ++p)
      for (int i = 0; i < hd; ++i) {
        const double inv = std::pow((double)cfg->rope_theta, -2.0 * i / cfg->head_dim);
        const double ang = (double)p * inv;
        tab[(size_t)p * hd + i] = make_float2((float)std::cos(ang), (float)std::sin(ang));
      }
    e = cudaMemcpy(st->rope, tab.get(), n_tab * sizeof(float2), cudaMemcpyHostToDevice);
  }
  {
    const char* mg = getenv("LRS_PERSISTENT");
    const bool moe = cfg->n_experts > 0;
    st->mega = !(mg && mg[0] == '0') && cfg->shared_ffn == 0 && (!moe || cfg->expert_ffn % 2 == 0) &&
               lrs::mega_supported(cfg->hidden, cfg->n_q_heads * cfg->head_dim,
                                   moe ? cfg->top_k * kpad(cfg->expert_ffn) : cfg->ffn, cfg->head_dim,
                                   cfg->n_q_heads / cfg->n_kv_heads, cfg->n_experts, cfg->top_k);
  }
  if (e == cudaSuccess) e = cudaMallocHost(&st->h_stage, ((size_t)5 * cfg->max_tokens + 16) * 4);
  if (e == cudaSuccess) e = cudaEventCreateWithFlags(&st->staged, cudaEventDisableTiming);
  if (e != cudaSuccess) {
    g_create_error = std::string("stage setup: ") + cudaGetErrorString(e);
    stage_destroy(st);
    return STAGE_E_CUDA;
  }
  if (weights) {
    int rc = guarded_upload(st, [&] { return load_endpoints(st, weights); });
    for (int l = range.begin; !rc && l < range.end; ++l) {
      if (!weights->layers) rc = set_err(st, STAGE_E_INVALID, "null layers");
      else rc = guarded_upload(st, [&] { return load_layer(st, l, &weights->layers[l - range.begin]); });
    }
    if (rc) {
      g_create_error = st->err;
      stage_destroy(st);
      return rc;
    }
  }
  *out = st;
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(&g_create_error, ex.what());
} catch (...) {
  return host_failure(&g_create_error, "unknown exception");
}

int stage_load_layer(stage_t st, int global_layer, const stage_layer_w* w) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  return load_layer(st, global_layer, w);
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_load_endpoints(stage_t st, const stage_weights* w) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  return load_endpoints(st, w);
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_prefill(stage_t st, int n_tokens, const int32_t* seq_ids_host, const int32_t* positions_host,
                  const int32_t* tokens_host, const stage_act* hidden_in, const stage_act* hidden_out) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  return run_forward(st, false, n_tokens, seq_ids_host, positions_host, tokens_host, hidden_in, hidden_out);
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_decode(stage_t st, int batch, const int32_t* seq_ids_host, const int32_t* positions_host,
                 const int32_t* tokens_host, const stage_act* hidden_in, const stage_act* hidden_out) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  return run_forward(st, true, batch, seq_ids_host, positions_host, tokens_host, hidden_in, hidden_out);
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

static int logits_dev(stage* st, int n_rows, const int* d_rows, float* logits_out, int32_t* argmax_out,
                      cudaStream_t s) {
  const stage_model_cfg& c = st->cfg;
  float* lg = logits_out ? logits_out : st->logits;
  cudaError_t e;
  if (use_tc(st, n_rows) && n_rows <= lrs::kGemmSmallTokens) {
    // the rows' features in bf16, then the weight-streaming GEMM: the head is read once
    const int ldh = kpad(c.hidden);
    if ((e = lrs::launch_rows_to_bf16(st->feat, c.hidden, c.hidden, nullptr, 0.f, n_rows, st->act_bf16, ldh, s,
                                      d_rows)) != cudaSuccess)
      return cuda_err(st, e, "readout operand");
    lrs::GemmArgs g;
    g.a = st->act_bf16;
    g.lda = ldh;
    g.w = st->head;
    g.M = n_rows;
    g.epi = lrs::EPI_STORE;
    g.out = lg;
    g.ldo = c.vocab;
    g.err = st->err_word;
    g.ws = st->gemm_ws;
    g.tile_cnt = st->gemm_cnt;
    if ((e = lrs::launch_gemm_tc(g, s)) != cudaSuccess) return cuda_err(st, e, "lm_head");
  } else {
    lrs::GemvArgs h;
    h.w = st->head;
    h.x = st->feat;
    h.ldx = c.hidden;
    h.x_rows = d_rows;
    h.ntok = n_rows;
    h.epi = lrs::EPI_STORE;
    h.out = lg;
    h.ldo = c.vocab;
    h.err = st->err_word;
    if ((e = lrs::launch_gemv(h, s)) != cudaSuccess) return cuda_err(st, e, "lm_head");
  }
  e = lrs::launch_argmax(lg, c.vocab, n_rows, argmax_out ? argmax_out : st->argmax, s);
  if (e != cudaSuccess) return cuda_err(st, e, "argmax");
  return STAGE_OK;
}

int stage_logits(stage_t st, int n_rows, const int32_t* row_index_host, float* logits_out, int32_t* argmax_out) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  if (!st->last) return set_err(st, STAGE_E_NOT_LAST, "stage [%d, %d) does not own the readout", st->begin, st->end);
  if (n_rows <= 0 || n_rows > st->cfg.max_tokens || !row_index_host) return set_err(st, STAGE_E_INVALID, "bad rows");
  for (int i = 0; i < n_rows; ++i)
    if (row_index_host[i] < 0 || row_index_host[i] >= st->last_n)
      return set_err(st, STAGE_E_INVALID, "row %d outside the last forward's %d tokens", row_index_host[i], st->last_n);
  cudaError_t e = cudaEventSynchronize(st->staged);
  if (e != cudaSuccess) return cuda_err(st, e, "staging");
  std::memcpy(st->h_stage + 3 * st->cfg.max_tokens, row_index_host, n_rows * 4);
  e = cudaMemcpyAsync(st->d_rows, st->h_stage + 3 * st->cfg.max_tokens, n_rows * 4, cudaMemcpyHostToDevice, st->stream);
  if (e == cudaSuccess) e = cudaEventRecord(st->staged, st->stream);
  if (e != cudaSuccess) return cuda_err(st, e, "rows");
  return logits_dev(st, n_rows, st->d_rows, logits_out, argmax_out, st->stream);
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_commit(stage_t st, int n, const int32_t* seq_ids_host, const int32_t* new_len_host) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  if (n < 0 || (n > 0 && (!seq_ids_host || !new_len_host))) return set_err(st, STAGE_E_INVALID, "bad commit arrays");
  for (int i = 0; i < n; ++i) {
    const int s = seq_ids_host[i];
    if (s < 0 || s >= st->cfg.max_seqs) return set_err(st, STAGE_E_INVALID, "seq_id %d", s);
    if (new_len_host[i] < st->committed[s] || new_len_host[i] > st->pending[s])
      return set_err(st, STAGE_E_STATE, "seq %d: commit %d outside [committed %d, written %d]", s, new_len_host[i],
                     st->committed[s], st->pending[s]);
  }
  for (int i = 0; i < n; ++i) st->committed[seq_ids_host[i]] = new_len_host[i];
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_truncate(stage_t st, int seq_id, int len) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  if (seq_id < 0 || seq_id >= st->cfg.max_seqs) return set_err(st, STAGE_E_INVALID, "seq_id %d", seq_id);
  if (len < 0 || len > st->committed[seq_id]) return set_err(st, STAGE_E_POSITION, "truncate to %d outside [0, %d]", len, st->committed[seq_id]);
  st->committed[seq_id] = len;
  st->pending[seq_id] = len;
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_reset(stage_t st) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  std::fill(st->committed.begin(), st->committed.end(), 0);
  std::fill(st->pending.begin(), st->pending.end(), 0);
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_committed_len(stage_t st, int seq_id, int* len_out) try {
  if (!st || !len_out || seq_id < 0 || seq_id >= st->cfg.max_seqs) return STAGE_E_INVALID;
  *len_out = st->committed[seq_id];
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_read_kv(stage_t st, int global_layer, int seq_id, int n_pos, uint16_t* k_host, uint16_t* v_host) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  const stage_model_cfg& c = st->cfg;
  if (global_layer < st->begin || global_layer >= st->end || seq_id < 0 || seq_id >= c.max_seqs || n_pos < 0 ||
      n_pos > c.max_seq_len || !k_host || !v_host)
    return set_err(st, STAGE_E_INVALID, "bad KV read arguments");
  cudaError_t e = cudaStreamSynchronize(st->stream);
  const size_t row = (size_t)c.head_dim;
  for (int h = 0; e == cudaSuccess && h < c.n_kv_heads; ++h) {
    const size_t off = (size_t)(global_layer - st->begin) * st->layer_kv +
                       (((size_t)seq_id * c.n_kv_heads + h) * c.max_seq_len) * row;
    e = cudaMemcpy(k_host + (size_t)h * n_pos * row, st->kc + off, (size_t)n_pos * row * 2, cudaMemcpyDeviceToHost);
    if (e == cudaSuccess)
      e = cudaMemcpy(v_host + (size_t)h * n_pos * row, st->vc + off, (size_t)n_pos * row * 2, cudaMemcpyDeviceToHost);
  }
  return e == cudaSuccess ? check_device_error(st) : cuda_err(st, e, "read kv");
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_write_kv(stage_t st, int global_layer, int seq_id, int pos0, int n_pos, const uint16_t* k_host,
                   const uint16_t* v_host) try {
  if (!st) return STAGE_E_INVALID;
  BusyGuard g(st);
  if (!g.ok) return set_err(st, STAGE_E_BUSY, "another call is in progress");
  const stage_model_cfg& c = st->cfg;
  if (global_layer < st->begin || global_layer >= st->end || seq_id < 0 || seq_id >= c.max_seqs || pos0 < 0 ||
      n_pos < 0 || !k_host || !v_host)
    return set_err(st, STAGE_E_INVALID, "bad KV write arguments");
  if ((long long)pos0 + n_pos > c.max_seq_len)
    return set_err(st, STAGE_E_POSITION, "positions [%d, %d) pass max_seq_len %d", pos0, pos0 + n_pos, c.max_seq_len);
  if (pos0 > st->pending[seq_id])
    return set_err(st, STAGE_E_POSITION, "write at %d leaves a gap after position %d", pos0, st->pending[seq_id]);
  cudaError_t e = cudaStreamSynchronize(st->stream);
  const size_t row = (size_t)c.head_dim;
  for (int h = 0; e == cudaSuccess && h < c.n_kv_heads; ++h) {
    const size_t off = (size_t)(global_layer - st->begin) * st->layer_kv +
                       (((size_t)seq_id * c.n_kv_heads + h) * c.max_seq_len + pos0) * row;
    e = cudaMemcpy(st->kc + off, k_host + (size_t)h * n_pos * row, (size_t)n_pos * row * 2, cudaMemcpyHostToDevice);
    if (e == cudaSuccess)
      e = cudaMemcpy(st->vc + off, v_host + (size_t)h * n_pos * row, (size_t)n_pos * row * 2, cudaMemcpyHostToDevice);
  }
  if (e != cudaSuccess) return cuda_err(st, e, "write kv");
  st->pending[seq_id] = std::max(st->pending[seq_id], pos0 + n_pos);
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

int stage_gemm_mode(stage_t st, int n_tokens, int* mode_out) try {
  if (!st || !mode_out) return STAGE_E_INVALID;
  *mode_out = use_tc(st, n_tokens) ? 1 : (n_tokens == 1 && st->mega) ? 2 : 0;
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

const char* stage_last_error(stage_t st) { return st ? st->err.c_str() : "null stage"; }

const char* stage_create_error(void) { return g_create_error.c_str(); }

void stage_destroy(stage_t st) {
  if (!st) return;
  if (st->stream) cudaStreamSynchronize(st->stream);
  if (st->arena) cudaFree(st->arena);
  if (st->h_stage) cudaFreeHost(st->h_stage);
  if (st->staged) cudaEventDestroy(st->staged);
  for (cudaEvent_t ev : st->tev) cudaEventDestroy(ev);
  delete st;
}

int stage_debug_inject(stage_t st, int what, int value) try {
  if (!st) return STAGE_E_INVALID;
  if (what == 1) {
    st->busy.store(value ? 1 : 0);
    return STAGE_OK;
  }
  if (what == 2) {
    st->fail_next = value ? value : STAGE_E_INJECTED;
    return STAGE_OK;
  }
  if (what == 3) {
    st->stall_barrier = value ? 1 : 0;
    return STAGE_OK;
  }
  return STAGE_E_INVALID;
} catch (const std::exception& ex) {
  return host_failure(st ? &st->err : nullptr, ex.what());
} catch (...) {
  return host_failure(st ? &st->err : nullptr, "unknown exception");
}

}  // extern "C"

// ------------------------------------------------------------------------------------------ pipeline

struct stage_pipeline {
  std::vector<stage*> stages;
  float* hbuf = nullptr;  // [max_tokens x hidden] handoff buffer shared by every boundary
  int max_tokens = 0;
  std::vector<int64_t> calls, bytes;
  // device-side greedy generation
  int* d_seq = nullptr;
  int* d_pos = nullptr;
  int* d_tok = nullptr;
  int* d_step = nullptr;
  int* d_hist = nullptr;
  int hist_cap = 0;
  int32_t* h_pin = nullptr;
  cudaStream_t cap = nullptr;  // capture stream of the step graph
  cudaGraphExec_t graph = nullptr;
  std::vector<int> graph_seqs;
  int graph_chunks = 0;
  std::string err;
};

namespace {

int pset(stage_pipeline* p, int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  p->err = buf;
  return code;
}

struct AllBusy {
  std::vector<stage*> held;
  bool ok = true;
  explicit AllBusy(const std::vector<stage*>& v) {
    for (stage* s : v) {
      if (s->busy.exchange(1) != 0) {
        ok = false;
        break;
      }
      held.push_back(s);
    }
  }
  ~AllBusy() {
    for (stage* s : held) s->busy.store(0);
  }
};

}  // namespace

extern "C" {

int stage_pipeline_create(stage_t* stages, int n_stages, stage_pipeline_t* out) try {
  if (!out || !stages || n_stages <= 0) return STAGE_E_INVALID;
  *out = nullptr;
  for (int i = 0; i < n_stages; ++i)
    if (!stages[i]) return STAGE_E_INVALID;
  const stage_model_cfg& c0 = stages[0]->cfg;
  if (stages[0]->begin != 0 || !stages[n_stages - 1]->last) return STAGE_E_INVALID;
  for (int i = 0; i < n_stages; ++i) {
    const stage_model_cfg& c = stages[i]->cfg;
    if (std::memcmp(&c, &c0, sizeof(c)) != 0) return STAGE_E_INVALID;  // same model and settings everywhere
    if (i > 0 && stages[i]->begin != stages[i - 1]->end) return STAGE_E_INVALID;
    if (stages[i]->stream != stages[0]->stream || stages[i]->device != stages[0]->device) return STAGE_E_INVALID;
  }
  stage_pipeline* p = new (std::nothrow) stage_pipeline();
  if (!p) return STAGE_E_INVALID;
  p->stages.assign(stages, stages + n_stages);
  p->max_tokens = c0.max_tokens;
  p->calls.assign(n_stages, 0);
  p->bytes.assign(n_stages, 0);
  cudaError_t e = cudaMalloc(&p->hbuf, (size_t)c0.max_tokens * c0.hidden * 4);
  if (e == cudaSuccess) e = cudaMalloc(&p->d_seq, (size_t)c0.max_seqs * 4 * 4);
  if (e == cudaSuccess) e = cudaMallocHost(&p->h_pin, (size_t)c0.max_seqs * 4 * 4);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->cap, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    stage_pipeline_destroy(p);
    return STAGE_E_CUDA;
  }
  p->d_pos = p->d_seq + c0.max_seqs;
  p->d_tok = p->d_seq + 2 * c0.max_seqs;
  p->d_step = p->d_seq + 3 * c0.max_seqs;
  *out = p;
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(nullptr, ex.what());
} catch (...) {
  return host_failure(nullptr, "unknown exception");
}

int stage_pipeline_step(stage_pipeline_t p, int is_prefill, int n_tokens, const int32_t* seq_ids_host,
                        const int32_t* positions_host, const int32_t* tokens_host, int n_rows,
                        const int32_t* row_index_host, float* logits_out, int32_t* next_tokens_host) try {
  if (!p) return STAGE_E_INVALID;
  AllBusy busy(p->stages);
  if (!busy.ok) return pset(p, STAGE_E_BUSY, "a stage of the pipeline is busy");
  const int H = p->stages[0]->cfg.hidden;
  if (n_tokens <= 0 || n_tokens > p->max_tokens) return pset(p, STAGE_E_INVALID, "n_tokens %d", n_tokens);
  stage_act act{p->hbuf, n_tokens, H};
  // every stage's inputs are validated and copied in before the first launch (no copy sits
  // between two stages' kernels on the stream); nothing is committed unless all succeed
  const size_t ns = p->stages.size();
  std::vector<int> max_len(ns, 0);
  for (size_t i = 0; i < ns; ++i) {
    stage* st = p->stages[i];
    const int rc = stage_call_inputs(st, !is_prefill, n_tokens, seq_ids_host, positions_host,
                                     i == 0 ? tokens_host : nullptr, i == 0 ? nullptr : &act, &act, &max_len[i]);
    if (rc) return pset(p, rc, "stage %zu [%d, %d): %s", i, st->begin, st->end, st->err.c_str());
  }
  for (size_t i = 0; i < ns; ++i) {
    stage* st = p->stages[i];
    const int rc = stage_call_launch(st, !is_prefill, n_tokens, seq_ids_host, positions_host, i == 0 ? nullptr : &act,
                                     &act, max_len[i]);
    if (rc) {
      for (stage* s : p->stages) std::copy(s->committed.begin(), s->committed.end(), s->pending.begin());
      return pset(p, rc, "stage %zu [%d, %d): %s", i, st->begin, st->end, st->err.c_str());
    }
    if (i + 1 < ns) {
      p->calls[i] += 1;
      p->bytes[i] += (int64_t)n_tokens * H * 4;
    }
  }
  stage* last = p->stages.back();
  if (n_rows > 0) {
    for (int i = 0; i < n_rows; ++i)
      if (!row_index_host || row_index_host[i] < 0 || row_index_host[i] >= n_tokens)
        return pset(p, STAGE_E_INVALID, "bad readout row");
    cudaError_t e = cudaEventSynchronize(last->staged);
    if (e == cudaSuccess) {
      std::memcpy(last->h_stage + 3 * last->cfg.max_tokens, row_index_host, n_rows * 4);
      e = cudaMemcpyAsync(last->d_rows, last->h_stage + 3 * last->cfg.max_tokens, n_rows * 4, cudaMemcpyHostToDevice,
                          last->stream);
    }
    if (e == cudaSuccess) e = cudaEventRecord(last->staged, last->stream);
    if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "rows: %s", cudaGetErrorString(e));
    int rc = logits_dev(last, n_rows, last->d_rows, logits_out, nullptr, last->stream);
    if (rc) return pset(p, rc, "%s", last->err.c_str());
    if (next_tokens_host) {
      // the tokens and every stage's error word come back through pinned memory, then one wait
      const int T = last->cfg.max_tokens;
      int32_t* h_tok = last->h_stage + 4 * T;
      e = cudaMemcpyAsync(h_tok, last->argmax, n_rows * 4, cudaMemcpyDeviceToHost, last->stream);
      for (stage* s2 : p->stages)
        if (e == cudaSuccess)
          e = cudaMemcpyAsync(s2->h_stage + 5 * s2->cfg.max_tokens, s2->err_word, 4, cudaMemcpyDeviceToHost,
                              last->stream);
      if (e == cudaSuccess) e = cudaStreamSynchronize(last->stream);
      if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "tokens: %s", cudaGetErrorString(e));
      for (stage* s2 : p->stages)
        if (s2->h_stage[5 * s2->cfg.max_tokens] != 0) {
          cudaMemset(s2->err_word, 0, 4);
          set_err(s2, STAGE_E_CUDA, "a kernel's bounded wait timed out; its outputs are invalid");
          return pset(p, STAGE_E_CUDA, "%s", s2->err.c_str());
        }
      std::memcpy(next_tokens_host, h_tok, n_rows * 4);
    }
  }
  // joint publication
  for (stage* s : p->stages) {
    for (int i = 0; i < n_tokens; ++i) s->committed[seq_ids_host[i]] = std::max(s->committed[seq_ids_host[i]], positions_host[i] + 1);
    std::copy(s->committed.begin(), s->committed.end(), s->pending.begin());
  }
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(p ? &p->err : nullptr, ex.what());
} catch (...) {
  return host_failure(p ? &p->err : nullptr, "unknown exception");
}

int stage_pipeline_generate(stage_pipeline_t p, int batch, const int32_t* seq_ids_host, const int32_t* first_tokens_host,
                            int n_steps, int use_graph, int32_t* tokens_out_host) try {
  if (!p) return STAGE_E_INVALID;
  AllBusy busy(p->stages);
  if (!busy.ok) return pset(p, STAGE_E_BUSY, "a stage of the pipeline is busy");
  stage* s0 = p->stages[0];
  stage* last = p->stages.back();
  const stage_model_cfg& c = s0->cfg;
  if (batch <= 0 || batch > c.max_seqs || n_steps <= 0 || !seq_ids_host || !first_tokens_host || !tokens_out_host)
    return pset(p, STAGE_E_INVALID, "bad generate arguments");
  std::vector<int> seen(c.max_seqs, 0);
  int max_len = 0;
  for (int i = 0; i < batch; ++i) {
    const int s = seq_ids_host[i];
    if (s < 0 || s >= c.max_seqs || seen[s]++) return pset(p, STAGE_E_INVALID, "bad seq_id %d", s);
    for (stage* st : p->stages)
      if (st->committed[s] != s0->committed[s]) return pset(p, STAGE_E_STATE, "stages disagree on seq %d", s);
    if (s0->committed[s] + n_steps > c.max_seq_len) return pset(p, STAGE_E_POSITION, "seq %d would pass max_seq_len", s);
    if (first_tokens_host[i] < 0 || first_tokens_host[i] >= c.vocab) return pset(p, STAGE_E_INVALID, "token id");
    max_len = std::max(max_len, s0->committed[s] + n_steps);
  }
  for (stage* st : p->stages)
    if (!weights_ready(st)) return pset(p, STAGE_E_STATE, "weights not loaded");
  cudaStream_t stream = s0->stream;
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "%s", cudaGetErrorString(e));
  if (n_steps > p->hist_cap) {
    if (p->graph) cudaGraphExecDestroy(p->graph);  // the captured step writes into the history buffer
    p->graph = nullptr;
    if (p->d_hist) cudaFree(p->d_hist);
    p->d_hist = nullptr;
    e = cudaMalloc(&p->d_hist, (size_t)n_steps * c.max_seqs * 4);
    if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "%s", cudaGetErrorString(e));
    p->hist_cap = n_steps;
  }
  for (int i = 0; i < batch; ++i) {
    p->h_pin[i] = seq_ids_host[i];
    p->h_pin[c.max_seqs + i] = s0->committed[seq_ids_host[i]];
    p->h_pin[2 * c.max_seqs + i] = first_tokens_host[i];
  }
  p->h_pin[3 * c.max_seqs] = 0;
  e = cudaMemcpyAsync(p->d_seq, p->h_pin, (size_t)c.max_seqs * 4 * 4, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "%s", cudaGetErrorString(e));
  const int H = c.hidden;
  const int n_chunks = attn_chunks(s0, batch, max_len);
  auto one_step = [&](cudaStream_t s) -> int {
    for (size_t i = 0; i < p->stages.size(); ++i) {
      stage* st = p->stages[i];
      st->call_prefill = false;
      int rc = forward_dev(st, batch, p->d_seq, p->d_pos, p->d_tok, p->hbuf, p->hbuf, n_chunks, s);
      if (rc) return pset(p, rc, "stage %zu: %s", i, st->err.c_str());
    }
    int rc = logits_dev(last, batch, nullptr, nullptr, p->d_tok, s);
    if (rc) return pset(p, rc, "%s", last->err.c_str());
    cudaError_t e2 = lrs::launch_advance(p->d_pos, p->d_tok, p->d_hist, p->d_step, batch, s);
    if (e2 != cudaSuccess) return pset(p, STAGE_E_CUDA, "advance: %s", cudaGetErrorString(e2));
    return STAGE_OK;
  };
  std::vector<int> seqs(seq_ids_host, seq_ids_host + batch);
  if (use_graph) {
    if (!p->graph || p->graph_seqs != seqs || p->graph_chunks != n_chunks) {
      if (p->graph) cudaGraphExecDestroy(p->graph);
      p->graph = nullptr;
      // capture on the pipeline's own non-blocking stream (the stages' stream may be the
      // legacy default stream, which cannot be captured); replay on the stages' stream
      cudaGraph_t g = nullptr;
      e = cudaStreamSynchronize(stream);
      if (e == cudaSuccess) e = cudaStreamBeginCapture(p->cap, cudaStreamCaptureModeThreadLocal);
      if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "capture: %s", cudaGetErrorString(e));
      int rc = one_step(p->cap);
      e = cudaStreamEndCapture(p->cap, &g);
      if (rc) {
        if (g) cudaGraphDestroy(g);
        return rc;
      }
      if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "capture: %s", cudaGetErrorString(e));
      e = cudaGraphInstantiate(&p->graph, g, 0);
      cudaGraphDestroy(g);
      if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "instantiate: %s", cudaGetErrorString(e));
      p->graph_seqs = seqs;
      p->graph_chunks = n_chunks;
    }
    for (int t = 0; t < n_steps; ++t) {
      e = cudaGraphLaunch(p->graph, stream);
      if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "graph launch: %s", cudaGetErrorString(e));
    }
  } else {
    for (int t = 0; t < n_steps; ++t) {
      int rc = one_step(stream);
      if (rc) return rc;
    }
  }
  for (int i = 0; i + 1 < (int)p->stages.size(); ++i) {
    p->calls[i] += n_steps;
    p->bytes[i] += (int64_t)n_steps * batch * H * 4;
  }
  std::vector<int32_t> hist((size_t)n_steps * batch);
  e = cudaMemcpyAsync(hist.data(), p->d_hist, hist.size() * 4, cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return pset(p, STAGE_E_CUDA, "%s", cudaGetErrorString(e));
  for (stage* s2 : p->stages)
    if (check_device_error(s2)) return pset(p, STAGE_E_CUDA, "%s", s2->err.c_str());
  std::memcpy(tokens_out_host, hist.data(), hist.size() * 4);
  for (stage* st : p->stages)
    for (int i = 0; i < batch; ++i) {
      st->committed[seq_ids_host[i]] += n_steps;
      st->pending[seq_ids_host[i]] = st->committed[seq_ids_host[i]];
    }
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(p ? &p->err : nullptr, ex.what());
} catch (...) {
  return host_failure(p ? &p->err : nullptr, "unknown exception");
}

int stage_pipeline_kernel_timing(stage_pipeline_t p, int enable) try {
  if (!p) return STAGE_E_INVALID;
  for (stage* st : p->stages) {
    if (enable && st->tev.empty()) {
      st->tev.resize(2 * (st->end - st->begin));
      for (auto& ev : st->tev)
        if (cudaEventCreate(&ev) != cudaSuccess) return pset(p, STAGE_E_CUDA, "event create");
    }
    st->timing = enable != 0;
  }
  if (p->graph) cudaGraphExecDestroy(p->graph);  // recapture with (or without) the event nodes
  p->graph = nullptr;
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(p ? &p->err : nullptr, ex.what());
} catch (...) {
  return host_failure(p ? &p->err : nullptr, "unknown exception");
}

int stage_pipeline_kernel_time(stage_pipeline_t p, float* mean_us, int* count) try {
  if (!p || !mean_us || !count) return STAGE_E_INVALID;
  double sum = 0;
  int n = 0;
  for (stage* st : p->stages) {
    if (!st->timing) continue;
    for (size_t i = 0; i + 1 < st->tev.size() && (int)i < 2 * st->timed_pairs; i += 2) {
      float ms = 0;
      if (cudaEventElapsedTime(&ms, st->tev[i], st->tev[i + 1]) != cudaSuccess) return pset(p, STAGE_E_STATE, "no timed step");
      sum += ms;
      ++n;
    }
  }
  *count = n;
  *mean_us = n ? (float)(sum * 1000.0 / n) : 0.f;
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(p ? &p->err : nullptr, ex.what());
} catch (...) {
  return host_failure(p ? &p->err : nullptr, "unknown exception");
}

int stage_pipeline_handoff_stats(stage_pipeline_t p, int boundary, int64_t* calls, int64_t* bytes) try {
  if (!p || boundary < 0 || boundary + 1 >= (int)p->stages.size() || !calls || !bytes) return STAGE_E_INVALID;
  *calls = p->calls[boundary];
  *bytes = p->bytes[boundary];
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(p ? &p->err : nullptr, ex.what());
} catch (...) {
  return host_failure(p ? &p->err : nullptr, "unknown exception");
}

const char* stage_pipeline_last_error(stage_pipeline_t p) { return p ? p->err.c_str() : "null pipeline"; }

void stage_pipeline_destroy(stage_pipeline_t p) {
  if (!p) return;
  if (!p->stages.empty() && p->stages[0]->stream) cudaStreamSynchronize(p->stages[0]->stream);
  if (p->graph) cudaGraphExecDestroy(p->graph);
  if (p->hbuf) cudaFree(p->hbuf);
  if (p->d_seq) cudaFree(p->d_seq);
  if (p->d_hist) cudaFree(p->d_hist);
  if (p->h_pin) cudaFreeHost(p->h_pin);
  if (p->cap) cudaStreamDestroy(p->cap);
  delete p;
}

}  // extern "C"

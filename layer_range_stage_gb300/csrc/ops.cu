// Kernel-level entry points of include/stage_ops.h: the GEMV and decode-attention kernels
// of the stage, on caller-owned device buffers.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/stage_ops.h"
#include "kernels.cuh"

// Scratch of stage_op_attention_decode_static: one array per device for the life of the
// process.  In host code this name is only a handle: its device address comes from
// cudaGetSymbolAddress, looked up once per device with that device current.
static __device__ __align__(256) unsigned char g_attn_static_scratch[STAGE_OP_STATIC_SCRATCH_BYTES];

namespace {

thread_local std::string g_op_error;

int op_err(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_op_error = buf;
  return code;
}

int op_cuda(cudaError_t e, const char* where) { return op_err(STAGE_E_CUDA, "%s: %s", where, cudaGetErrorString(e)); }

// A C++ exception inside an entry point (a host staging buffer that could not be allocated)
// ends the call with STAGE_E_HOST instead of crossing the C ABI; recording the message may
// itself fail, which is ignored.
int host_failure(const char* what) noexcept {
  try {
    g_op_error = std::string("host: ") + what;
  } catch (...) {
  }
  return STAGE_E_HOST;
}

bool aligned16(const void* p) { return ((uintptr_t)p & 15) == 0; }

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void* g_static_addr[kMaxDevices] = {};

int static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return op_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return op_err(STAGE_E_INVALID, "device %d beyond the supported %d", dev, kMaxDevices);
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (!g_static_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attn_static_scratch);
    if (e != cudaSuccess || !p) return op_cuda(e == cudaSuccess ? cudaErrorInvalidSymbol : e, "cudaGetSymbolAddress");
    g_static_addr[dev] = p;
  }
  *out = g_static_addr[dev];
  return STAGE_OK;
}

int check_attention(const float* q, const uint16_t* kc, const uint16_t* vc, const int32_t* seq, const int32_t* pos,
                    int n_tok, int hq, int hkv, int d, int max_len, int n_chunks, const float* out) {
  if (!q || !kc || !vc || !seq || !pos || !out) return op_err(STAGE_E_INVALID, "null pointer");
  if (!aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(out))
    return op_err(STAGE_E_INVALID, "q, caches and out must be 16-byte aligned");
  if (n_tok <= 0 || hq <= 0 || hkv <= 0 || max_len <= 0) return op_err(STAGE_E_INVALID, "non-positive size");
  if (hq % hkv || !lrs::attn_decode_supported(d, hq / hkv))
    return op_err(STAGE_E_INVALID, "head_dim must be 64 or 128 and n_q_heads / n_kv_heads in {1, 2, 4, 8}");
  if (n_chunks < 1 || n_chunks > lrs::kAttnMaxChunks) return op_err(STAGE_E_INVALID, "n_chunks outside [1, 64]");
  if (n_tok > 65535) return op_err(STAGE_E_INVALID, "n_tok too large");
  return STAGE_OK;
}

}  // namespace

extern "C" {

const char* stage_op_last_error(void) { return g_op_error.c_str(); }

int stage_op_q8_device_bytes(int64_t rows, int64_t cols, size_t* q_bytes, size_t* s_bytes) try {
  if (rows <= 0 || cols <= 0 || cols > (1 << 30) || !q_bytes || !s_bytes) return op_err(STAGE_E_INVALID, "bad shape");
  const int64_t kp = lrs::row_pad((int)cols);
  *q_bytes = (size_t)(rows * kp);
  *s_bytes = (size_t)(rows * (kp / 32) * 2);
  return STAGE_OK;
} catch (const std::exception& ex) {
  return host_failure(ex.what());
} catch (...) {
  return host_failure("unknown exception");
}

int stage_op_q8_pack(const stage_q8* host, void* q_dev, void* s_dev) try {
  if (!host || !host->q || !host->scale || !q_dev || !s_dev) return op_err(STAGE_E_INVALID, "null pointer");
  size_t qb = 0, sb = 0;
  if (int rc = stage_op_q8_device_bytes(host->rows, host->cols, &qb, &sb)) return rc;
  const int64_t rows = host->rows, cols = host->cols, kp = lrs::row_pad((int)cols);
  const int64_t nb_src = (cols + 31) / 32, nb = kp / 32;
  std::vector<uint8_t> q(qb, 0x80u);  // biased zero in the padding
  std::vector<uint16_t> s(sb / 2, 0);
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c = 0; c < cols; ++c) q[r * kp + c] = (uint8_t)host->q[r * cols + c] ^ 0x80u;
    std::memcpy(&s[r * nb], host->scale + r * nb_src, (size_t)nb_src * 2);
  }
  cudaError_t e = cudaMemcpy(q_dev, q.data(), qb, cudaMemcpyHostToDevice);
  if (e == cudaSuccess) e = cudaMemcpy(s_dev, s.data(), sb, cudaMemcpyHostToDevice);
  return e == cudaSuccess ? STAGE_OK : op_cuda(e, "pack");
} catch (const std::exception& ex) {
  return host_failure(ex.what());
} catch (...) {
  return host_failure("unknown exception");
}

int stage_op_embed(const void* q_dev, const void* s_dev, int64_t rows, int64_t cols, const int32_t* tok_dev,
                   int n_tok, float* out_dev, void* stream) try {
  if (!q_dev || !s_dev || !tok_dev || !out_dev) return op_err(STAGE_E_INVALID, "null pointer");
  if (rows <= 0 || cols <= 0 || rows > (1 << 30) || cols > (1 << 24) || n_tok <= 0 || n_tok > 65535)
    return op_err(STAGE_E_INVALID, "bad shape");
  if (cols % 4) return op_err(STAGE_E_INVALID, "cols must be a multiple of 4");
  if (!aligned16(q_dev) || !aligned16(s_dev) || !aligned16(out_dev)) return op_err(STAGE_E_INVALID, "unaligned pointer");
  cudaError_t e = lrs::prepare_kernels();
  if (e != cudaSuccess) return op_cuda(e, "kernel setup");
  lrs::DevQ8 w;
  w.q = (uint8_t*)q_dev;
  w.s = (uint16_t*)s_dev;
  w.N = (int)rows;
  w.K = (int)cols;
  w.Kp = lrs::row_pad((int)cols);
  e = lrs::launch_embed(w, tok_dev, n_tok, out_dev, (int)cols, (cudaStream_t)stream);
  return e == cudaSuccess ? STAGE_OK : op_cuda(e, "embed");
} catch (const std::exception& ex) {
  return host_failure(ex.what());
} catch (...) {
  return host_failure("unknown exception");
}

int stage_op_gemv(const void* q_dev, const void* s_dev, int64_t rows, int64_t cols, const float* x_dev, int n_tok,
                  const float* gamma_dev, float eps, float* y_dev, void* stream) try {
  if (!q_dev || !s_dev || !x_dev || !y_dev) return op_err(STAGE_E_INVALID, "null pointer");
  if (rows <= 0 || cols <= 0 || rows > (1 << 30) || cols > (1 << 24) || n_tok <= 0)
    return op_err(STAGE_E_INVALID, "bad shape");
  if (cols % 4) return op_err(STAGE_E_INVALID, "cols must be a multiple of 4");
  if (!aligned16(q_dev) || !aligned16(s_dev) || !aligned16(x_dev)) return op_err(STAGE_E_INVALID, "unaligned pointer");
  cudaError_t e = lrs::prepare_kernels();
  if (e != cudaSuccess) return op_cuda(e, "kernel setup");
  lrs::GemvArgs g;
  g.w.q = (uint8_t*)q_dev;
  g.w.s = (uint16_t*)s_dev;
  g.w.N = (int)rows;
  g.w.K = (int)cols;
  g.w.Kp = lrs::row_pad((int)cols);
  g.x = x_dev;
  g.ldx = (int)cols;
  g.ntok = n_tok;
  g.gamma = gamma_dev;
  g.eps = eps;
  g.epi = lrs::EPI_STORE;
  g.out = y_dev;
  g.ldo = (int)rows;
  e = lrs::launch_gemv(g, (cudaStream_t)stream);
  return e == cudaSuccess ? STAGE_OK : op_cuda(e, "gemv");
} catch (const std::exception& ex) {
  return host_failure(ex.what());
} catch (...) {
  return host_failure("unknown exception");
}

int stage_op_gemm_bf16(const uint16_t* a_dev, int lda, int M, const void* q_dev, const void* s_dev, int64_t rows,
                       int64_t cols, float* y_dev, void* stream) try {
  if (!a_dev || !q_dev || !s_dev || !y_dev) return op_err(STAGE_E_INVALID, "null pointer");
  if (M <= 0 || rows <= 0 || cols <= 0 || rows > (1 << 30) || cols > (1 << 24)) return op_err(STAGE_E_INVALID, "bad shape");
  const int kp = lrs::row_pad((int)cols);
  if (lda < kp || lda % 8) return op_err(STAGE_E_INVALID, "lda must be >= %d and a multiple of 8", kp);
  if (!aligned16(a_dev) || !aligned16(q_dev) || !aligned16(s_dev)) return op_err(STAGE_E_INVALID, "unaligned pointer");
  cudaError_t e = lrs::prepare_kernels();
  if (e != cudaSuccess) return op_cuda(e, "kernel setup");
  lrs::GemmArgs g;
  g.a = (const __nv_bfloat16*)a_dev;
  g.lda = lda;
  g.w.q = (uint8_t*)q_dev;
  g.w.s = (uint16_t*)s_dev;
  g.w.N = (int)rows;
  g.w.K = (int)cols;
  g.w.Kp = kp;
  g.M = M;
  g.epi = lrs::EPI_STORE;
  g.out = y_dev;
  g.ldo = (int)rows;
  e = lrs::launch_gemm_tc(g, (cudaStream_t)stream);
  return e == cudaSuccess ? STAGE_OK : op_cuda(e, "gemm");
} catch (const std::exception& ex) {
  return host_failure(ex.what());
} catch (...) {
  return host_failure("unknown exception");
}

size_t stage_op_attention_workspace_bytes(int n_tok, int n_q_heads, int n_kv_heads, int head_dim, int n_chunks) {
  if (n_tok <= 0 || n_q_heads <= 0 || n_kv_heads <= 0 || head_dim <= 0 || n_chunks <= 0) return 0;
  const size_t part_o = (size_t)n_tok * n_q_heads * n_chunks * head_dim * 4;
  const size_t part_ml = (size_t)n_tok * n_q_heads * n_chunks * 8;
  const size_t counters = (size_t)n_tok * n_kv_heads * 4;
  return (part_o + 255) / 256 * 256 + (part_ml + 255) / 256 * 256 + counters;
}

int stage_op_attention_decode(const float* q_dev, const uint16_t* k_cache_dev, const uint16_t* v_cache_dev,
                              const int32_t* seq_dev, const int32_t* pos_dev, int n_tok, int n_q_heads, int n_kv_heads,
                              int head_dim, int max_len, int n_chunks, float* out_dev, void* workspace_dev,
                              size_t workspace_bytes, void* stream) try {
  if (int rc = check_attention(q_dev, k_cache_dev, v_cache_dev, seq_dev, pos_dev, n_tok, n_q_heads, n_kv_heads, head_dim,
                               max_len, n_chunks, out_dev))
    return rc;
  const size_t need = stage_op_attention_workspace_bytes(n_tok, n_q_heads, n_kv_heads, head_dim, n_chunks);
  if (!workspace_dev || workspace_bytes < need || !aligned16(workspace_dev))
    return op_err(STAGE_E_INVALID, "workspace must be 16-byte aligned and hold %zu bytes", need);
  cudaError_t e = lrs::prepare_kernels();
  if (e != cudaSuccess) return op_cuda(e, "kernel setup");
  char* ws = (char*)workspace_dev;
  const size_t part_o = (size_t)n_tok * n_q_heads * n_chunks * head_dim * 4;
  const size_t part_ml = (size_t)n_tok * n_q_heads * n_chunks * 8;
  lrs::AttnArgs a;
  a.q = q_dev;
  a.kc = (const __half*)k_cache_dev;
  a.vc = (const __half*)v_cache_dev;
  a.seq = seq_dev;
  a.pos = pos_dev;
  a.out = out_dev;
  a.part_o = (float*)ws;
  a.part_ml = (float2*)(ws + (part_o + 255) / 256 * 256);
  a.counters = (int*)(ws + (part_o + 255) / 256 * 256 + (part_ml + 255) / 256 * 256);
  a.ntok = n_tok;
  a.Hq = n_q_heads;
  a.Hkv = n_kv_heads;
  a.D = head_dim;
  a.max_len = max_len;
  a.n_chunks = n_chunks;
  a.scale = (float)(1.0 / std::sqrt((double)head_dim));
  e = lrs::launch_attn_decode(a, (cudaStream_t)stream);
  return e == cudaSuccess ? STAGE_OK : op_cuda(e, "attention");
} catch (const std::exception& ex) {
  return host_failure(ex.what());
} catch (...) {
  return host_failure("unknown exception");
}

int stage_op_attention_decode_static(const float* q_dev, const uint16_t* k_cache_dev, const uint16_t* v_cache_dev,
                                     const int32_t* seq_dev, const int32_t* pos_dev, int n_tok, int n_q_heads,
                                     int n_kv_heads, int head_dim, int max_len, int n_chunks, float* out_dev,
                                     void* stream) try {
  if (int rc = check_attention(q_dev, k_cache_dev, v_cache_dev, seq_dev, pos_dev, n_tok, n_q_heads, n_kv_heads, head_dim,
                               max_len, n_chunks, out_dev))
    return rc;
  const size_t need = stage_op_attention_workspace_bytes(n_tok, n_q_heads, n_kv_heads, head_dim, n_chunks);
  if (need > STAGE_OP_STATIC_SCRATCH_BYTES)
    return op_err(STAGE_E_INVALID, "needs %zu bytes of scratch; the library's static scratch holds %u", need,
                  (unsigned)STAGE_OP_STATIC_SCRATCH_BYTES);
  void* scratch = nullptr;
  if (int rc = static_scratch_address(&scratch)) return rc;
  // the chunk counters must start at zero whatever an earlier call left behind
  const size_t part_o = (size_t)n_tok * n_q_heads * n_chunks * head_dim * 4;
  const size_t part_ml = (size_t)n_tok * n_q_heads * n_chunks * 8;
  const size_t counters_off = (part_o + 255) / 256 * 256 + (part_ml + 255) / 256 * 256;
  cudaError_t e = cudaMemsetAsync((char*)scratch + counters_off, 0, (size_t)n_tok * n_kv_heads * 4, (cudaStream_t)stream);
  if (e != cudaSuccess) return op_cuda(e, "clear scratch counters");
  return stage_op_attention_decode(q_dev, k_cache_dev, v_cache_dev, seq_dev, pos_dev, n_tok, n_q_heads, n_kv_heads,
                                   head_dim, max_len, n_chunks, out_dev, scratch, STAGE_OP_STATIC_SCRATCH_BYTES, stream);
} catch (const std::exception& ex) {
  return host_failure(ex.what());
} catch (...) {
  return host_failure("unknown exception");
}

}  // extern "C"

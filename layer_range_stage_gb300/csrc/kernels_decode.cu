// Decode-path kernels of the stage forward (sm_103a).
//
// What they compute follows "41. Many GPUs: tensor, pipeline, expert and data
// parallelism", section "Pipeline parallelism" (per block: add_norm, attention,
// add_norm, MLP; the residual stream carried across blocks and stages) and section
// "Ring attention for very long contexts" (partial attention with log-sum-exp and the
// split-KV merge o = sum_s e^(l_s - l) o_s).  The weights are int8 blocks of 32 along
// the input dimension with one fp16 scale per block.
//
// Determinism: no float atomics anywhere.  Every reduction runs in an order fixed by the
// shapes alone, so a stage boundary (or its absence) cannot change a single bit.

#include <algorithm>
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.cuh"

namespace lrs {

// ------------------------------------------------------------------------------------------
// Dequant-fused GEMV.  A CTA of 256 threads owns a group of R consecutive device rows at a
// time (grid-stride over groups).  Every thread streams 16 weight bytes per row per chunk
// (one 128-bit load; 256 threads cover 4096 weights of a row per pass) and multiplies them
// with 16 activations kept in shared memory; the fp16 block scale multiplies each 16-term
// partial sum.  Warp shuffles, then a fixed-order sum over the 8 warps, give each row.
// The input is read into shared memory once per pass of BT tokens, normalised on the way
// when the RMSNorm prologue is on.  Shared memory holds the activations with an XOR swizzle
// of the four float4 of every 16-float chunk, which makes the per-thread 64-byte reads
// bank-conflict free.

constexpr int kGemvThreads = 256;

__device__ __forceinline__ int swz(int k) {
  const int c = k >> 4, j = (k >> 2) & 3;
  return (c << 4) | ((j ^ ((c >> 1) & 3)) << 2) | (k & 3);
}

template <int R, int BT>
__global__ void __launch_bounds__(kGemvThreads) gemv_q8_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) float smem[];
  const int Kp = a.w.Kp, K = a.w.K, N = a.w.N;
  float* xs = smem;                  // [BT][Kp], swizzled
  float* red = xs + BT * Kp;         // [8][R*BT]
  float* yv = red + 8 * R * BT;      // [R*BT]
  float* nrm = yv + R * BT;          // [8]
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nchunk = Kp >> 4, nblk = Kp >> 5;
  const int ngroups = (N + R - 1) / R;

  for (int t0 = 0; t0 < a.ntok; t0 += BT) {
    const int nt = min(BT, a.ntok - t0);
    __syncthreads();
    for (int b = 0; b < BT; ++b) {
      const float* xr = nullptr;
      if (b < nt) xr = a.x + (size_t)(a.x_rows ? a.x_rows[t0 + b] : (t0 + b)) * a.ldx;
      float rinv = 1.0f;
      if (a.gamma && xr) {
        float ss = 0.f;
        for (int k = tid; k < K; k += kGemvThreads) {
          const float v = xr[k];
          ss = fmaf(v, v, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) nrm[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) tot += nrm[w];
        rinv = 1.0f / sqrtf(tot / (float)K + a.eps);
        __syncthreads();
      }
      for (int k = tid; k < Kp; k += kGemvThreads) {
        float v = 0.f;
        if (xr && k < K) v = a.gamma ? xr[k] * rinv * a.gamma[k] : xr[k];
        xs[b * Kp + swz(k)] = v;
      }
    }
    __syncthreads();

    for (int g = blockIdx.x; g < ngroups; g += gridDim.x) {
      const int row0 = g * R;
      float acc[R][BT];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[r][b] = 0.f;

      for (int c = tid; c < nchunk; c += kGemvThreads) {
        uint4 w[R];
        float sc[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int row = row0 + r;
          if (row < N) {
            w[r] = ld_stream_u4(a.w.q + (size_t)row * Kp + (size_t)c * 16);
            sc[r] = h2f_bits(ld_stream_u16(a.w.s + (size_t)row * nblk + (c >> 1)));
          } else {
            w[r] = make_uint4(0u, 0u, 0u, 0u);
            sc[r] = 0.f;
          }
        }
        const int sw = (c >> 1) & 3;
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          const float4* xp = reinterpret_cast<const float4*>(xs + b * Kp + c * 16);
          const float4 x0 = xp[0 ^ sw], x1 = xp[1 ^ sw], x2 = xp[2 ^ sw], x3 = xp[3 ^ sw];
#pragma unroll
          for (int r = 0; r < R; ++r) acc[r][b] = fmaf(sc[r], dot16_i8(w[r], x0, x1, x2, x3), acc[r][b]);
        }
      }

#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) {
          const float v = warp_sum(acc[r][b]);
          if (lane == 0) red[warp * (R * BT) + r * BT + b] = v;
        }
      __syncthreads();
      if (tid < R * BT) {
        float y = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) y += red[w * (R * BT) + tid];
        yv[tid] = y;
      }
      __syncthreads();

      if (a.epi == EPI_STORE || a.epi == EPI_RESID) {
        if (tid < R * BT) {
          const int r = tid / BT, b = tid % BT, row = row0 + r;
          if (row < N && b < nt) {
            const size_t t = (size_t)(t0 + b);
            float y = yv[tid];
            if (a.epi == EPI_RESID) y = __fadd_rn(a.resid[t * a.ldr + row], y);
            a.out[t * a.ldo + row] = y;
          }
        }
      } else if (tid < (R / 2) * BT) {
        const int j = tid / BT, b = tid % BT, row = row0 + 2 * j;
        if (row < N && b < nt) {
          const size_t t = (size_t)(t0 + b);
          const float y0 = yv[(2 * j) * BT + b], y1 = yv[(2 * j + 1) * BT + b];
          if (a.epi == EPI_SWIGLU) {
            a.out[t * a.ldo + (row >> 1)] = silu(y0) * y1;
          } else {  // EPI_QKV
            const int hd = a.head_dim >> 1, P = row >> 1, head = P / hd, i = P - head * hd;
            const int p = a.pos[t];
            if (head < a.n_q_heads) {
              const float2 cs = a.rope[(size_t)p * hd + i];
              float* qo = a.qout + (t * a.n_q_heads + head) * a.head_dim;
              qo[i] = y0 * cs.x - y1 * cs.y;
              qo[i + hd] = y1 * cs.x + y0 * cs.y;
            } else {
              const bool is_k = head < a.n_q_heads + a.n_kv_heads;
              const int kvh = head - a.n_q_heads - (is_k ? 0 : a.n_kv_heads);
              const size_t base = (((size_t)a.seq[t] * a.n_kv_heads + kvh) * a.max_len + p) * a.head_dim;
              if (is_k) {
                const float2 cs = a.rope[(size_t)p * hd + i];
                a.kc[base + i] = __float2half_rn(y0 * cs.x - y1 * cs.y);
                a.kc[base + i + hd] = __float2half_rn(y1 * cs.x + y0 * cs.y);
              } else {
                a.vc[base + i] = __float2half_rn(y0);
                a.vc[base + i + hd] = __float2half_rn(y1);
              }
            }
          }
        }
      }
      __syncthreads();
    }
  }
}

template <int R, int BT>
static size_t gemv_smem(int Kp) {
  return sizeof(float) * ((size_t)BT * Kp + 8 * R * BT + R * BT + 8);
}

template <int R, int BT>
static cudaError_t launch_gemv_t(const GemvArgs& a, cudaStream_t st) {
  // occupancy per shared-memory size, computed once per size (host-side only)
  static size_t cached_smem[16];
  static int cached_occ[16];
  static int n_cached = 0;
  static bool attr_set = false;
  const size_t smem = gemv_smem<R, BT>(a.w.Kp);
  cudaError_t e = cudaSuccess;
  if (!attr_set) {
    e = cudaFuncSetAttribute(gemv_q8_kernel<R, BT>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024 + 1024);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  int occ = -1;
  for (int i = 0; i < n_cached; ++i)
    if (cached_smem[i] == smem) occ = cached_occ[i];
  if (occ < 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, gemv_q8_kernel<R, BT>, kGemvThreads, smem);
    if (e != cudaSuccess) return e;
    if (n_cached < 16) {
      cached_smem[n_cached] = smem;
      cached_occ[n_cached] = occ;
      ++n_cached;
    }
  }
  if (occ < 1) return cudaErrorInvalidConfiguration;
  const int ngroups = (a.w.N + R - 1) / R;
  const int grid = std::max(1, std::min(ngroups, sm_count() * occ));
  gemv_q8_kernel<R, BT><<<grid, kGemvThreads, smem, st>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t st) {
  if (a.ntok <= 0 || a.w.N <= 0) return cudaSuccess;
  const size_t budget = 200 * 1024;
  if (a.ntok >= 4 && gemv_smem<4, 4>(a.w.Kp) <= budget) return launch_gemv_t<4, 4>(a, st);
  if (a.ntok >= 2 && gemv_smem<4, 2>(a.w.Kp) <= budget) return launch_gemv_t<4, 2>(a, st);
  return launch_gemv_t<4, 1>(a, st);
}

// ------------------------------------------------------------------------------------------
// Split-K GQA decode attention.  Grid (n_chunks, Hkv, ntok), 128 threads.  The CTA takes the
// G = Hq / Hkv query heads that share KV head blockIdx.y and the positions of its chunk of
// 0..pos[t]; it walks the chunk in tiles of 128 positions (one per thread for the scores)
// with a running max / sum, then writes its partial (unnormalised output, max, sum).  The
// last CTA of a (token, kv head) to finish -- found with one integer atomic, no waiting --
// merges the chunks in chunk order.

template <int D, int G>
__global__ void __launch_bounds__(128) attn_decode_kernel(const AttnArgs a) {
  constexpr int NT = 128;
  constexpr int TPR = D / 4;       // threads per V row (4 dims each)
  constexpr int NPG = NT / TPR;    // position groups in the PV product
  __shared__ __align__(16) float qs[G][D];
  __shared__ float ps[G][NT];
  __shared__ float red[4][G];
  __shared__ __align__(16) float ored[NPG][G][D];
  __shared__ int is_last;

  const int chunk = blockIdx.x, kvh = blockIdx.y, t = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = a.pos[t] + 1, sid = a.seq[t];
  const int clen = (L + a.n_chunks - 1) / a.n_chunks;
  const int c0 = min(L, chunk * clen), c1 = min(L, c0 + clen);
  const size_t head0 = (size_t)t * a.Hq + (size_t)kvh * G;

  for (int i = tid; i < G * D; i += NT) qs[i / D][i % D] = a.q[head0 * D + i];
  __syncthreads();

  const __half* kb = a.kc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;
  const __half* vb = a.vc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;

  float m[G], l[G], o[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g) {
    m[g] = -INFINITY;
    l[g] = 0.f;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[g][e] = 0.f;
  }
  const int d0 = (tid % TPR) * 4, pg = tid / TPR;

  for (int p0 = c0; p0 < c1; p0 += NT) {
    const int np = min(NT, c1 - p0);
    float sc[G];
#pragma unroll
    for (int g = 0; g < G; ++g) sc[g] = -INFINITY;
    if (tid < np) {
#pragma unroll
      for (int g = 0; g < G; ++g) sc[g] = 0.f;
      const uint4* kr = reinterpret_cast<const uint4*>(kb + (size_t)(p0 + tid) * D);
#pragma unroll 4
      for (int i = 0; i < D / 8; ++i) {
        const uint4 kk = kr[i];
        const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kk.x));
        const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kk.y));
        const float2 k45 = __half22float2(*reinterpret_cast<const __half2*>(&kk.z));
        const float2 k67 = __half22float2(*reinterpret_cast<const __half2*>(&kk.w));
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4*>(&qs[g][8 * i]);
          const float4 qb = *reinterpret_cast<const float4*>(&qs[g][8 * i + 4]);
          float s = sc[g];
          s = fmaf(qa.x, k01.x, s);
          s = fmaf(qa.y, k01.y, s);
          s = fmaf(qa.z, k23.x, s);
          s = fmaf(qa.w, k23.y, s);
          s = fmaf(qb.x, k45.x, s);
          s = fmaf(qb.y, k45.y, s);
          s = fmaf(qb.z, k67.x, s);
          s = fmaf(qb.w, k67.y, s);
          sc[g] = s;
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) sc[g] *= a.scale;
    }
    // tile max per head
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float v = warp_max(sc[g]);
      if (lane == 0) red[warp][g] = v;
    }
    __syncthreads();
    float mnew[G], alpha[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float mt = fmaxf(fmaxf(red[0][g], red[1][g]), fmaxf(red[2][g], red[3][g]));
      mnew[g] = fmaxf(m[g], mt);
      alpha[g] = (m[g] == -INFINITY) ? 0.f : expf(m[g] - mnew[g]);
      const float e = (tid < np) ? expf(sc[g] - mnew[g]) : 0.f;
      ps[g][tid] = e;
      sc[g] = e;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float v = warp_sum(sc[g]);
      if (lane == 0) red[warp][g] = v;
    }
    __syncthreads();
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float lt = (red[0][g] + red[1][g]) + (red[2][g] + red[3][g]);
      l[g] = l[g] * alpha[g] + lt;
      m[g] = mnew[g];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[g][e] *= alpha[g];
    }
    for (int p = pg; p < np; p += NPG) {
      const uint2 vv = *reinterpret_cast<const uint2*>(vb + (size_t)(p0 + p) * D + d0);
      const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
      const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float w = ps[g][p];
        o[g][0] = fmaf(w, v01.x, o[g][0]);
        o[g][1] = fmaf(w, v01.y, o[g][1]);
        o[g][2] = fmaf(w, v23.x, o[g][2]);
        o[g][3] = fmaf(w, v23.y, o[g][3]);
      }
    }
    __syncthreads();
  }

#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) ored[pg][g][d0 + e] = o[g][e];
  __syncthreads();
  for (int i = tid; i < G * D; i += NT) {
    const int g = i / D, d = i % D;
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < NPG; ++q) s += ored[q][g][d];
    a.part_o[((head0 + g) * a.n_chunks + chunk) * D + d] = s;
  }
#pragma unroll
  for (int g = 0; g < G; ++g)
    if (tid == g) a.part_ml[(head0 + g) * a.n_chunks + chunk] = make_float2(m[g], l[g]);

  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int prev = atomicAdd(&a.counters[(size_t)t * a.Hkv + kvh], 1);
    is_last = (prev == a.n_chunks - 1);
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  for (int i = tid; i < G * D; i += NT) {
    const int g = i / D, d = i % D;
    const float2* ml = a.part_ml + (head0 + g) * a.n_chunks;
    const float* po = a.part_o + (head0 + g) * a.n_chunks * D + d;
    float M = -INFINITY;
    for (int c = 0; c < a.n_chunks; ++c) M = fmaxf(M, __ldcg(ml + c).x);
    float Ls = 0.f, acc = 0.f;
    for (int c = 0; c < a.n_chunks; ++c) {
      const float2 mc = __ldcg(ml + c);
      if (mc.y > 0.f) {
        const float w = expf(mc.x - M);
        Ls = fmaf(mc.y, w, Ls);
        acc = fmaf(w, __ldcg(po + (size_t)c * D), acc);
      }
    }
    a.out[(head0 + g) * D + d] = acc / Ls;
  }
  if (tid == 0) a.counters[(size_t)t * a.Hkv + kvh] = 0;
}

bool attn_decode_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4 || group == 8);
}

template <int D>
static cudaError_t launch_attn_d(const AttnArgs& a, cudaStream_t st) {
  const dim3 grid(a.n_chunks, a.Hkv, a.ntok);
  switch (a.Hq / a.Hkv) {
    case 1: attn_decode_kernel<D, 1><<<grid, 128, 0, st>>>(a); break;
    case 2: attn_decode_kernel<D, 2><<<grid, 128, 0, st>>>(a); break;
    case 4: attn_decode_kernel<D, 4><<<grid, 128, 0, st>>>(a); break;
    case 8: attn_decode_kernel<D, 8><<<grid, 128, 0, st>>>(a); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t st) {
  if (a.ntok <= 0) return cudaSuccess;
  if (!attn_decode_supported(a.D, a.Hq / a.Hkv) || a.Hq % a.Hkv) return cudaErrorInvalidValue;
  if (a.n_chunks < 1 || a.n_chunks > 65535) return cudaErrorInvalidValue;
  return a.D == 64 ? launch_attn_d<64>(a, st) : launch_attn_d<128>(a, st);
}

// ------------------------------------------------------------------------------------------
// Embedding row gather: x[t][k] = scale[tok][k/32] * q[tok][k] (exact in float32).

__global__ void embed_kernel(const DevQ8 tab, const int* tok, float* out, int ldo) {
  const int t = blockIdx.x, row = tok[t];
  const int8_t* q = tab.q + (size_t)row * tab.Kp;
  const uint16_t* s = tab.s + (size_t)row * (tab.Kp >> 5);
  for (int k = threadIdx.x; k < tab.K; k += blockDim.x) out[(size_t)t * ldo + k] = h2f_bits(s[k >> 5]) * (float)q[k];
}

cudaError_t launch_embed(const DevQ8& table, const int* tok, int ntok, float* out, int ldo, cudaStream_t st) {
  if (ntok <= 0) return cudaSuccess;
  embed_kernel<<<ntok, 256, 0, st>>>(table, tok, out, ldo);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Final RMSNorm of the last stage: f = x / sqrt(mean(x^2) + eps) * gamma, written to
// the stage's feature buffer and to the caller's hidden_out.  Same reduction order as the
// GEMV prologue.

__global__ void final_norm_kernel(const float* x, int ldx, const float* gamma, float eps, int H, float* feat,
                                  float* out, int ldo) {
  __shared__ float nrm[8];
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* xr = x + (size_t)t * ldx;
  float ss = 0.f;
  for (int k = tid; k < H; k += 256) {
    const float v = xr[k];
    ss = fmaf(v, v, ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) nrm[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < 8; ++w) tot += nrm[w];
  const float rinv = 1.0f / sqrtf(tot / (float)H + eps);
  for (int k = tid; k < H; k += 256) {
    const float f = xr[k] * rinv * gamma[k];
    feat[(size_t)t * H + k] = f;
    out[(size_t)t * ldo + k] = f;
  }
}

cudaError_t launch_final_norm(const float* x, int ldx, const float* gamma, float eps, int H, int ntok, float* feat,
                              float* out, int ldo, cudaStream_t st) {
  if (ntok <= 0) return cudaSuccess;
  final_norm_kernel<<<ntok, 256, 0, st>>>(x, ldx, gamma, eps, H, feat, out, ldo);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Greedy token: argmax over a logits row, the lowest index among equal maxima.

__device__ __forceinline__ void better(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

__global__ void argmax_kernel(const float* logits, int V, int* out) {
  __shared__ float sv[32];
  __shared__ int si[32];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* lg = logits + (size_t)r * V;
  float v = -INFINITY;
  int idx = INT_MAX;
  for (int k = tid; k < V; k += blockDim.x) better(v, idx, lg[k], k);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, o);
    better(v, idx, v2, i2);
  }
  if (lane == 0) {
    sv[warp] = v;
    si[warp] = idx;
  }
  __syncthreads();
  if (tid == 0) {
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) better(v, idx, sv[w], si[w]);
    out[r] = (idx == INT_MAX) ? 0 : idx;
  }
}

cudaError_t launch_argmax(const float* logits, int V, int n_rows, int* out, cudaStream_t st) {
  if (n_rows <= 0) return cudaSuccess;
  argmax_kernel<<<n_rows, 1024, 0, st>>>(logits, V, out);
  return cudaGetLastError();
}

// ------------------------------------------------------------------------------------------
// Device-side greedy feedback of a replayed decode step: every sequence moves one position
// on, and the step's greedy tokens are appended to the history.

__global__ void advance_kernel(int* pos, const int* tok, int* hist, int* step, int batch) {
  const int i = threadIdx.x;
  const int s = *step;
  if (i < batch) {
    hist[(size_t)s * batch + i] = tok[i];
    pos[i] += 1;
  }
  __syncthreads();
  if (i == 0) *step = s + 1;
}

cudaError_t launch_advance(int* pos, const int* tok, int* hist, int* step, int batch, cudaStream_t st) {
  advance_kernel<<<1, std::max(32, ((batch + 31) / 32) * 32), 0, st>>>(pos, tok, hist, step, batch);
  return cudaGetLastError();
}

int sm_count() {
  static int n = 0;
  if (n == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 1;
  }
  return n;
}

}  // namespace lrs

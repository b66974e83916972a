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
#include <utility>

#include "common.cuh"
#include "kernels.cuh"
#include "q8dot.cuh"

namespace lrs {

static bool g_pdl = true;
void set_pdl(bool on) { g_pdl = on; }
bool pdl_enabled() { return g_pdl; }

// Every kernel of the stage chain is launched with programmatic stream serialization, so
// it can start (and, for the GEMVs, begin streaming its weights) while its predecessor
// drains; each kernel orders its reads of predecessor outputs after pdl_wait().
template <typename... KArgs, typename... Args>
static cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// ------------------------------------------------------------------------------------------
// Dequant-fused GEMV (the per-chunk arithmetic is in q8dot.cuh: one byte extract + one
// FFMA per weight byte).
//
// Work split: KS warps of a CTA own R consecutive rows at a time (grid-stride over row
// groups), each warp a 1/KS slice of K; its lanes stream 16 bytes per row per chunk with U
// chunks in flight per row, so KS is chosen to let every warp issue all of its loads at
// once.  Warps reduce with shuffles; the KS partial sums of a row meet in shared memory in
// slice order behind a named barrier of those KS warps only.  The first batch of weights
// is requested before waiting for the predecessor kernel.  The
// CTA's shared memory holds the (normalised, scaled) input once per pass of BT tokens,
// copied in with cp.async, and its chunk sums; an XOR swizzle of the four float4 of each
// 16-float chunk keeps the lanes' 64-byte reads bank-conflict free.

constexpr int kGemvThreads = 256;
constexpr size_t kGemvSmemBudget = 200 * 1024;

// GATHER: 0 plain rows, 1 row gather (expert gate/up), 2 K gather (expert down).
template <int R, int U, int BT, int KS, int GATHER = 0>
__global__ void __launch_bounds__(kGemvThreads, BT == 1 ? 3 : 2) gemv_q8_kernel(const GemvArgs a) {
  extern __shared__ __align__(16) float smem[];
  constexpr int NW = kGemvThreads / 32, RG = NW / KS;  // warps, row groups per CTA
  const int Kp = a.w.Kp, K = a.w.K, N = a.w.N;
  const int nchunk = Kp >> 4, nblk = Kp >> 5;
  float* xs = smem;                  // [BT][Kp] inputs * 2^64, swizzled
  float* xc = xs + BT * Kp;          // [BT][nchunk] chunk sums of the inputs
  float* nrm = xc + BT * nchunk;     // [8]
  float* red = nrm + 8;              // [RG][KS][R*BT] slice partial sums
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int kslice = warp % KS, rgrp = warp / KS;
  const int ngroups = (N + R - 1) / R;
  const int gwarp = blockIdx.x * RG + rgrp, nwarps = gridDim.x * RG;

  uint4 w[U][R];
  float sc[U][R];
  auto load_batch = [&](int row0, int cb) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int c = cb + 32 * u + lane;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const int row = row0 + r;
        if (c < nchunk && row < N) {
          size_t qoff, soff;
          if (GATHER == 1) {  // row gather: the row belongs to the expert of its slot
            const size_t wrow = (size_t)a.ids[row / a.rows_per_slot] * a.rows_per_slot + row % a.rows_per_slot;
            qoff = wrow * Kp + (size_t)c * 16;
            soff = wrow * nblk + (c >> 1);
          } else if (GATHER == 2) {  // K gather: chunk c lies in the row of the expert of its segment
            const int j = c / a.seg_chunks, cl = c - j * a.seg_chunks;
            const size_t wrow = (size_t)a.ids[j] * a.seg_rows + row;
            qoff = wrow * ((size_t)a.seg_chunks * 16) + (size_t)cl * 16;
            soff = wrow * (size_t)(a.seg_chunks >> 1) + (cl >> 1);
          } else {
            qoff = (size_t)row * Kp + (size_t)c * 16;
            soff = (size_t)row * nblk + (c >> 1);
          }
          w[u][r] = ld_stream_u4(a.w.q + qoff);
          sc[u][r] = h2f_bits(ld_stream_u16(a.w.s + soff));
        } else {
          w[u][r] = make_uint4(0u, 0u, 0u, 0u);
          sc[u][r] = 0.f;
        }
      }
    }
  };
  // The weights do not depend on the predecessor kernel: fetch this warp's first batch
  // before waiting for it (single-pass launches only).
  pdl_trigger();
  bool prefetched = false;
  // (gathered weights depend on the router's output: no prefetch before the wait then)
  if (GATHER == 0 && a.ntok <= BT && gwarp < ngroups) {
    load_batch(gwarp * R, kslice * 32 * U);
    prefetched = true;
  }
  pdl_wait();

  for (int t0 = 0; t0 < a.ntok; t0 += BT) {
    const int nt = min(BT, a.ntok - t0);
    __syncthreads();
    // 1. raw inputs -> shared memory, every copy in flight at once
    const int k4 = K >> 2;
    for (int b = 0; b < nt; ++b) {
      const float* xr = a.x + (size_t)(a.x_rows ? a.x_rows[t0 + b] : (t0 + b)) * a.ldx;
      for (int i = tid; i < k4; i += kGemvThreads) cp_async16(xs + b * Kp + 4 * i, xr + 4 * i);
      for (int k = 4 * k4 + tid; k < K; k += kGemvThreads) xs[b * Kp + k] = xr[k];
    }
    cp_async_wait_all();
    for (int b = 0; b < BT; ++b)
      for (int k = (b < nt ? K : 0) + tid; k < Kp; k += kGemvThreads) xs[b * Kp + k] = 0.f;
    __syncthreads();
    // 2. RMSNorm scale per token (fixed reduction order)
    float rinv[BT];
#pragma unroll
    for (int b = 0; b < BT; ++b) {
      rinv[b] = 1.0f;
      if (a.gamma && b < nt) {
        float ss = 0.f;
        for (int k = tid; k < K; k += kGemvThreads) {
          const float v = xs[b * Kp + k];
          ss = fmaf(v, v, ss);
        }
        ss = warp_sum(ss);
        if (lane == 0) nrm[warp] = ss;
        __syncthreads();
        float tot = 0.f;
#pragma unroll
        for (int w8 = 0; w8 < 8; ++w8) tot += nrm[w8];
        rinv[b] = 1.0f / sqrtf(tot / (float)K + a.eps);
        __syncthreads();
      }
    }
    // 3. in place, one thread per 16-input chunk: normalise, scale by 2^64, swizzle, chunk sum
    for (int i = tid; i < BT * nchunk; i += kGemvThreads) {
      const int b = i / nchunk, c = i - b * nchunk;
      float* xp = xs + b * Kp + c * 16;
      float v[16];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float4 t4 = reinterpret_cast<const float4*>(xp)[j];
        v[4 * j] = t4.x;
        v[4 * j + 1] = t4.y;
        v[4 * j + 2] = t4.z;
        v[4 * j + 3] = t4.w;
      }
      float sum = 0.f;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int k = c * 16 + j;
        float h = v[j];
        if (a.gamma) h = (k < K) ? h * rinv[b] * a.gamma[k] : 0.f;
        v[j] = h;
        sum += h;
      }
      const int sw = (c >> 1) & 3;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        reinterpret_cast<float4*>(xp)[j ^ sw] =
            make_float4(v[4 * j] * kXScale, v[4 * j + 1] * kXScale, v[4 * j + 2] * kXScale, v[4 * j + 3] * kXScale);
      xc[i] = sum;
    }
    __syncthreads();

    for (int g = gwarp; g < ngroups; g += nwarps) {
      const int row0 = g * R;
      float acc[R][BT];
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[r][b] = 0.f;

      for (int cb = kslice * 32 * U; cb < nchunk; cb += KS * 32 * U) {
        if (prefetched) {
          prefetched = false;  // the first batch of the first task is already in registers
        } else {
          load_batch(row0, cb);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = cb + 32 * u + lane;
          if (c < nchunk) {
            const int sw = (c >> 1) & 3;
#pragma unroll
            for (int b = 0; b < BT; ++b) {
              const float4* xp = reinterpret_cast<const float4*>(xs + b * Kp + c * 16);
              const float4 x0 = xp[0 ^ sw], x1 = xp[1 ^ sw], x2 = xp[2 ^ sw], x3 = xp[3 ^ sw];
              const float corr = -128.0f * xc[b * nchunk + c];
#pragma unroll
              for (int r = 0; r < R; ++r) {
                const float t = fmaf(dot16_u8(w[u][r], x0, x1, x2, x3), kPScale, corr);
                acc[r][b] = fmaf(sc[u][r], t, acc[r][b]);
              }
            }
          }
        }
      }
#pragma unroll
      for (int r = 0; r < R; ++r)
#pragma unroll
        for (int b = 0; b < BT; ++b) acc[r][b] = warp_sum(acc[r][b]);
      if (KS > 1) {
        // the KS slices of this row group meet in shared memory, summed in slice order
        float* rg = red + rgrp * KS * R * BT;
        if (lane == 0) {
#pragma unroll
          for (int r = 0; r < R; ++r)
#pragma unroll
            for (int b = 0; b < BT; ++b) rg[kslice * R * BT + r * BT + b] = acc[r][b];
        }
        named_bar(1 + rgrp, KS * 32);
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < KS; ++k) sum += rg[k * R * BT + r * BT + b];
            acc[r][b] = sum;
          }
        named_bar(1 + rgrp, KS * 32);
        if (kslice != 0) continue;
      }

      // epilogue: lane i takes value i (rows) or pair i (row pairs)
      if (a.epi == EPI_STORE || a.epi == EPI_RESID) {
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            const int row = row0 + r;
            if (lane == r * BT + b && row < N && b < nt) {
              const size_t t = (size_t)(t0 + b);
              float y = acc[r][b];
              if (a.epi == EPI_RESID) y = __fadd_rn(a.resid[t * a.ldr + row], y);
              a.out[t * a.ldo + row] = y;
            }
          }
      } else {
#pragma unroll
        for (int j = 0; j < R / 2; ++j)
#pragma unroll
          for (int b = 0; b < BT; ++b) {
            const int row = row0 + 2 * j;
            if (lane != j * BT + b || row >= N || b >= nt) continue;
            const size_t t = (size_t)(t0 + b);
            const float y0 = acc[2 * j][b], y1 = acc[2 * j + 1][b];
            if (a.epi == EPI_SWIGLU) {
              a.out[t * a.ldo + (row >> 1)] = silu(y0) * y1;
            } else if (a.epi == EPI_MOE_SWIGLU) {
              const int slot = row / a.rows_per_slot, i = (row % a.rows_per_slot) >> 1;
              a.out[t * a.ldo + (size_t)slot * a.ldo_slot + i] = silu(y0) * y1 * a.slot_w[slot];
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
    }
  }
}

// xs [BT][Kp] + xc [BT][Kp/16] + nrm [8] + red [warps][R*BT]
template <int R, int BT>
static size_t gemv_smem(int Kp) {
  return sizeof(float) * ((size_t)BT * Kp + (size_t)BT * (Kp / 16) + 8 + (size_t)(kGemvThreads / 32) * R * BT);
}

// Launch attributes are fixed once, outside any stream capture (prepare_kernels); the
// launch itself only computes the grid from the recorded register count.
template <int R, int U, int BT, int KS, int GATHER>
struct GemvInfo {
  static int regs;
};
template <int R, int U, int BT, int KS, int GATHER>
int GemvInfo<R, U, BT, KS, GATHER>::regs = 0;

template <int R, int U, int BT, int KS, int GATHER = 0>
static cudaError_t prepare_gemv() {
  cudaError_t e = cudaFuncSetAttribute(gemv_q8_kernel<R, U, BT, KS, GATHER>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGemvSmemBudget + 4096);
  if (e != cudaSuccess) return e;
  cudaFuncAttributes fa;
  e = cudaFuncGetAttributes(&fa, gemv_q8_kernel<R, U, BT, KS, GATHER>);
  if (e != cudaSuccess) return e;
  GemvInfo<R, U, BT, KS, GATHER>::regs = fa.numRegs;
  return cudaSuccess;
}

// Resident CTAs per SM from the per-SM limits (threads, registers, shared memory).
static int occupancy(int regs, int threads, size_t smem) {
  const int by_threads = 2048 / threads;
  const int regs_rounded = (regs + 7) / 8 * 8;
  const int by_regs = std::max(1, 65536 / (regs_rounded * threads));
  const int by_smem = std::max(1, (int)((228 * 1024) / (smem + 1024)));
  return std::max(1, std::min(by_threads, std::min(by_regs, by_smem)));
}

template <int R, int U, int BT, int KS, int GATHER = 0>
static cudaError_t launch_gemv_t(const GemvArgs& a, cudaStream_t st) {
  if (GemvInfo<R, U, BT, KS, GATHER>::regs == 0) return cudaErrorNotReady;  // prepare_kernels() was not called
  const size_t smem = gemv_smem<R, BT>(a.w.Kp);
  const int occ = occupancy(GemvInfo<R, U, BT, KS, GATHER>::regs, kGemvThreads, smem);
  const int ngroups = (a.w.N + R - 1) / R;
  const int groups_per_cta = (kGemvThreads / 32) / KS;
  const int grid = std::max(1, std::min((ngroups + groups_per_cta - 1) / groups_per_cta, sm_count() * occ));
  return launch_k(gemv_q8_kernel<R, U, BT, KS, GATHER>, dim3(grid), dim3(kGemvThreads), smem, st, a);
}

cudaError_t launch_gemv(const GemvArgs& a, cudaStream_t st) {
  if (a.ntok <= 0 || a.w.N <= 0) return cudaSuccess;
  const size_t budget = kGemvSmemBudget;
  if (a.ntok >= 4 && gemv_smem<2, 4>(a.w.Kp) <= budget) return launch_gemv_t<2, 2, 4, 1>(a, st);
  if (a.ntok >= 2 && gemv_smem<2, 2>(a.w.Kp) <= budget) return launch_gemv_t<2, 4, 2, 1>(a, st);
  // one load round per warp: K split over KS warps so that KS * 32 lanes * U chunks cover K
  const int nchunk = a.w.Kp / 16;
  if (a.rows_per_slot || a.seg_chunks) {
    if (a.ntok != 1) return cudaErrorInvalidValue;  // expert launches are per token
    if (a.rows_per_slot) {
      if (nchunk > 2 * 32 * 4) return launch_gemv_t<2, 4, 1, 4, 1>(a, st);
      if (nchunk > 32 * 4) return launch_gemv_t<2, 4, 1, 2, 1>(a, st);
      return launch_gemv_t<2, 4, 1, 1, 1>(a, st);
    }
    if (nchunk > 2 * 32 * 4) return launch_gemv_t<2, 4, 1, 4, 2>(a, st);
    if (nchunk > 32 * 4) return launch_gemv_t<2, 4, 1, 2, 2>(a, st);
    return launch_gemv_t<2, 4, 1, 1, 2>(a, st);
  }
  if (nchunk > 4 * 32 * 4) return launch_gemv_t<2, 4, 1, 8>(a, st);
  if (nchunk > 2 * 32 * 4) return launch_gemv_t<2, 4, 1, 4>(a, st);
  if (nchunk > 32 * 4) return launch_gemv_t<2, 4, 1, 2>(a, st);
  return launch_gemv_t<2, 4, 1, 1>(a, st);
}

// ------------------------------------------------------------------------------------------
// Split-K GQA decode attention.  Grid (n_chunks, Hkv, ntok), 128 threads, about one wave of
// CTAs.  The CTA takes the G = Hq / Hkv query heads that share KV head blockIdx.y and the
// positions of its chunk of 0..pos[t].  It walks the chunk in tiles of 64 positions: all
// threads first copy the K and V rows of the tile into shared memory with cp.async (every
// copy of the tile in flight at once), then threads 2p and 2p + 1 score position p for every
// head (half of the dims each), a running max / sum per head is kept, and the
// probability-weighted V rows accumulate.  Shared memory is kept to ~43 KB (the PV sums of the
// position groups reuse the tile area at the end) so that five CTAs share an SM and one CTA's
// copies overlap the others' arithmetic.  The
// chunk's partial (unnormalised output, max, sum) goes to scratch; the last CTA of a
// (token, kv head) to finish -- found with one integer atomic, no waiting -- merges the
// chunks in chunk order after copying every partial into shared memory in one round trip.

constexpr int kAttnThreads = 128;
constexpr int kAttnTile = 64;

template <int D, int G>
struct AttnSmem {
  static constexpr int KROW = D + 8;  // halves per K/V row in shared memory (16-byte pad)
  static constexpr int TPR = D / 4;   // threads per V row in the PV product (4 dims each)
  static constexpr int NPG = kAttnThreads / TPR;
  static constexpr size_t kv = (size_t)kAttnTile * KROW * 2;  // bytes of one K or V tile
  static constexpr size_t q = (size_t)G * D * 4;
  static constexpr size_t p = (size_t)G * kAttnTile * 4;
  static constexpr size_t o = (size_t)NPG * G * D * 4;
  static constexpr size_t w = (size_t)kAttnMaxChunks * G * 4;
  static constexpr size_t stats = (size_t)4 * G * 4;
  static constexpr size_t total = 2 * kv + q + p + w + stats;  // o reuses the K/V tile area
  static_assert(o <= 2 * kv, "PV sums of the position groups over the K/V tiles");
  static_assert((size_t)G * kAttnMaxChunks * 8 <= q + p, "merge (max, sum) pairs over q and the scores");
  // chunks whose partials fit in the K/V tile area for the one-shot merge
  static constexpr int merge_chunks = (int)((2 * kv) / ((size_t)G * D * 4));
};

template <int D, int G>
__global__ void __launch_bounds__(kAttnThreads) attn_decode_kernel(const AttnArgs a) {
  using S = AttnSmem<D, G>;
  constexpr int NT = kAttnThreads, TP = kAttnTile, KROW = S::KROW, TPR = S::TPR, NPG = S::NPG;
  extern __shared__ __align__(16) unsigned char sm_raw[];
  __half* ks = reinterpret_cast<__half*>(sm_raw);
  __half* vs = ks + TP * KROW;
  float* qs = reinterpret_cast<float*>(sm_raw + 2 * S::kv);
  float* ps = qs + G * D;                   // [G][TP]
  float* ored = reinterpret_cast<float*>(sm_raw);  // [NPG][G][D] after the last tile
  float* wts = ps + G * TP;                 // [n_chunks][G]
  float* st_m = wts + kAttnMaxChunks * G;   // [G] running max
  float* st_l = st_m + G;                   // [G] running sum
  float* st_a = st_l + G;                   // [G] rescale of this tile
  float* st_L = st_a + G;                   // [G] merged sum (merge phase)
  __shared__ int is_last;

  const int chunk = blockIdx.x, kvh = blockIdx.y, t = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_trigger();
  pdl_wait();
  const int L = a.pos[t] + 1, sid = a.seq[t];
  const int clen = (L + a.n_chunks - 1) / a.n_chunks;
  const int c0 = min(L, chunk * clen), c1 = min(L, c0 + clen);
  const size_t head0 = (size_t)t * a.Hq + (size_t)kvh * G;

  for (int i = tid; i < G * D / 4; i += NT)
    reinterpret_cast<float4*>(qs)[i] = reinterpret_cast<const float4*>(a.q + head0 * D)[i];
  if (tid < G) {
    st_m[tid] = -INFINITY;
    st_l[tid] = 0.f;
  }
  const __half* kb = a.kc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;
  const __half* vb = a.vc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;

  float o[G][4];
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[g][e] = 0.f;
  const int d0 = (tid % TPR) * 4, pg = tid / TPR;

  for (int p0 = c0; p0 < c1; p0 += TP) {
    const int np = min(TP, c1 - p0);
    __syncthreads();  // previous tile fully consumed (and q / stats initialised)
    constexpr int PIECES = D / 8;  // 16-byte pieces per row
    for (int i = tid; i < np * PIECES; i += NT) {
      const int r = i / PIECES, c = i - r * PIECES;
      cp_async16(ks + r * KROW + c * 8, kb + (size_t)(p0 + r) * D + c * 8);
      cp_async16(vs + r * KROW + c * 8, vb + (size_t)(p0 + r) * D + c * 8);
    }
    cp_async_wait_all();
    __syncthreads();
    // scores: threads 2p and 2p + 1 -> position p, half of the dims each, every head
    {
      const int pp = tid >> 1, hf = tid & 1;
      float sc[G];
#pragma unroll
      for (int g = 0; g < G; ++g) sc[g] = 0.f;
      const __half* kr = ks + pp * KROW + hf * (D / 2);
#pragma unroll 4
      for (int i = 0; i < (pp < np ? D / 16 : 0); ++i) {
        const uint4 kk = *reinterpret_cast<const uint4*>(kr + 8 * i);
        const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kk.x));
        const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kk.y));
        const float2 k45 = __half22float2(*reinterpret_cast<const __half2*>(&kk.z));
        const float2 k67 = __half22float2(*reinterpret_cast<const __half2*>(&kk.w));
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float4 qa = *reinterpret_cast<const float4*>(qs + g * D + hf * (D / 2) + 8 * i);
          const float4 qb = *reinterpret_cast<const float4*>(qs + g * D + hf * (D / 2) + 8 * i + 4);
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
      for (int g = 0; g < G; ++g) sc[g] += __shfl_xor_sync(0xffffffffu, sc[g], 1);
      if (pp < np && hf == 0)
#pragma unroll
        for (int g = 0; g < G; ++g) ps[g * TP + pp] = sc[g] * a.scale;
    }
    __syncthreads();
    // per head: tile max, probabilities, running (max, sum); warp w handles heads w, w + 4, ...
    for (int g = warp; g < G; g += NT / 32) {
      float sv[TP / 32];
      float mt = -INFINITY;
#pragma unroll
      for (int k2 = 0; k2 < TP / 32; ++k2) {
        const int p = lane + 32 * k2;
        sv[k2] = p < np ? ps[g * TP + p] : -INFINITY;
        mt = fmaxf(mt, sv[k2]);
      }
      mt = warp_max(mt);
      const float mold = st_m[g];
      const float mnew = fmaxf(mold, mt);
      float lsum = 0.f;
#pragma unroll
      for (int k2 = 0; k2 < TP / 32; ++k2) {
        const int p = lane + 32 * k2;
        const float e = p < np ? expf(sv[k2] - mnew) : 0.f;
        ps[g * TP + p] = e;
        lsum += e;
      }
      const float lt = warp_sum(lsum);
      if (lane == 0) {
        const float alpha = (mold == -INFINITY) ? 0.f : expf(mold - mnew);
        st_a[g] = alpha;
        st_l[g] = st_l[g] * alpha + lt;
        st_m[g] = mnew;
      }
    }
    __syncthreads();
    // PV: thread -> 4 dims of V, positions pg, pg + NPG, ...
#pragma unroll
    for (int g = 0; g < G; ++g) {
      const float al = st_a[g];
#pragma unroll
      for (int e = 0; e < 4; ++e) o[g][e] *= al;
    }
    for (int pp = pg; pp < np; pp += NPG) {
      const uint2 vv = *reinterpret_cast<const uint2*>(vs + pp * KROW + d0);
      const float2 v01 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
      const float2 v23 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float w = ps[g * TP + pp];
        o[g][0] = fmaf(w, v01.x, o[g][0]);
        o[g][1] = fmaf(w, v01.y, o[g][1]);
        o[g][2] = fmaf(w, v23.x, o[g][2]);
        o[g][3] = fmaf(w, v23.y, o[g][3]);
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int g = 0; g < G; ++g)
#pragma unroll
    for (int e = 0; e < 4; ++e) ored[(pg * G + g) * D + d0 + e] = o[g][e];
  __syncthreads();
  // partial of this chunk: [t][kvh][chunk][G][D] and (max, sum) per head
  float* po = a.part_o + (((size_t)t * a.Hkv + kvh) * a.n_chunks + chunk) * (G * D);
  for (int i = tid; i < G * D; i += NT) {
    float s = 0.f;
#pragma unroll
    for (int q2 = 0; q2 < NPG; ++q2) s += ored[q2 * G * D + i];
    po[i] = s;
  }
  if (tid < G) a.part_ml[(head0 + tid) * a.n_chunks + chunk] = make_float2(st_m[tid], st_l[tid]);

  __syncthreads();  // every partial write, then one acquire-release arrival (no separate fence)
  if (tid == 0) {
    const int prev = (int)atom_add_acq_rel(reinterpret_cast<unsigned*>(&a.counters[(size_t)t * a.Hkv + kvh]), 1u);
    is_last = (prev == a.n_chunks - 1);
  }
  __syncthreads();
  if (!is_last) return;
  // merge: chunk weights e^(m_c - M) per head, then the weighted sums in chunk order
  const int nch = a.n_chunks;
  const float* pbase = a.part_o + ((size_t)t * a.Hkv + kvh) * nch * (G * D);
  const bool staged = nch <= S::merge_chunks;
  float* pst = reinterpret_cast<float*>(sm_raw);  // [nch][G*D] partials, over the K/V tiles
  if (staged)
    for (int i = tid; i < nch * G * D / 4; i += NT) cp_async16(pst + 4 * i, pbase + 4 * i);
  float2* mls = reinterpret_cast<float2*>(qs);  // [G][nch] (max, sum), over q and the scores (read by now)
  for (int i = tid; i < G * nch; i += NT) mls[i] = __ldcg(a.part_ml + head0 * nch + i);
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int c = 0; c < nch; ++c) M = fmaxf(M, mls[tid * nch + c].x);
    float Ls = 0.f;
    for (int c = 0; c < nch; ++c) {
      const float2 mc = mls[tid * nch + c];
      const float w = mc.y > 0.f ? expf(mc.x - M) : 0.f;
      wts[c * G + tid] = w;
      Ls = fmaf(mc.y, w, Ls);
    }
    st_L[tid] = Ls;
  }
  cp_async_wait_all();
  __syncthreads();
  for (int i = tid; i < G * D; i += NT) {
    const int g = i / D;
    float acc = 0.f;
    if (staged) {
      for (int c = 0; c < nch; ++c) acc = fmaf(wts[c * G + g], pst[(size_t)c * (G * D) + i], acc);
    } else {
      int c = 0;
      for (; c + 8 <= nch; c += 8) {
        float v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] = __ldcg(pbase + (size_t)(c + j) * (G * D) + i);
#pragma unroll
        for (int j = 0; j < 8; ++j) acc = fmaf(wts[(c + j) * G + g], v[j], acc);
      }
      for (; c < nch; ++c) acc = fmaf(wts[c * G + g], __ldcg(pbase + (size_t)c * (G * D) + i), acc);
    }
    a.out[head0 * D + i] = acc / st_L[g];
  }
  if (tid == 0) a.counters[(size_t)t * a.Hkv + kvh] = 0;
}

bool attn_decode_supported(int head_dim, int group) {
  return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4 || group == 8);
}

template <int D, int G>
static cudaError_t prepare_attn() {
  return cudaFuncSetAttribute(attn_decode_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)AttnSmem<D, G>::total);
}

template <int D, int G>
static cudaError_t launch_attn_dg(const AttnArgs& a, cudaStream_t st) {
  const dim3 grid(a.n_chunks, a.Hkv, a.ntok);
  return launch_k(attn_decode_kernel<D, G>, grid, dim3(kAttnThreads), AttnSmem<D, G>::total, st, a);
}

template <int D>
static cudaError_t launch_attn_d(const AttnArgs& a, cudaStream_t st) {
  switch (a.Hq / a.Hkv) {
    case 1: return launch_attn_dg<D, 1>(a, st);
    case 2: return launch_attn_dg<D, 2>(a, st);
    case 4: return launch_attn_dg<D, 4>(a, st);
    case 8: return launch_attn_dg<D, 8>(a, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_decode(const AttnArgs& a, cudaStream_t st) {
  if (a.ntok <= 0) return cudaSuccess;
  if (!attn_decode_supported(a.D, a.Hq / a.Hkv) || a.Hq % a.Hkv) return cudaErrorInvalidValue;
  if (a.n_chunks < 1 || a.n_chunks > kAttnMaxChunks) return cudaErrorInvalidValue;
  return a.D == 64 ? launch_attn_d<64>(a, st) : launch_attn_d<128>(a, st);
}

// ------------------------------------------------------------------------------------------
// Embedding row gather: x[t][k] = scale[tok][k/32] * q[tok][k] (exact in float32).  The
// table is stored biased like every weight matrix (byte = q + 128).

// One token per CTA; a thread dequantises 16 consecutive weights from one 16-byte load.
__global__ void embed_kernel(const DevQ8 tab, const int* tok, float* out, int ldo) {
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, row = tok[t];
  const uint8_t* q = tab.q + (size_t)row * tab.Kp;
  const uint16_t* s = tab.s + (size_t)row * (tab.Kp >> 5);
  float* o = out + (size_t)t * ldo;
  for (int k0 = threadIdx.x * 16; k0 < tab.K; k0 += blockDim.x * 16) {
    const uint4 w = __ldg(reinterpret_cast<const uint4*>(q + k0));
    const float sc = h2f_bits(s[k0 >> 5]);
    const uint32_t words[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int k = k0 + j;
      if (k < tab.K) o[k] = sc * (float)((int)((words[j >> 2] >> (8 * (j & 3))) & 0xFFu) - 128);
    }
  }
}

cudaError_t launch_embed(const DevQ8& table, const int* tok, int ntok, float* out, int ldo, cudaStream_t st) {
  if (ntok <= 0) return cudaSuccess;
  return launch_k(embed_kernel, dim3(ntok), dim3(256), 0, st, table, tok, out, ldo);
}

// ------------------------------------------------------------------------------------------
// Final RMSNorm of the last stage: f = x / sqrt(mean(x^2) + eps) * gamma, written to the
// stage's feature buffer and to the caller's hidden_out.  Same reduction order as the GEMV
// prologue.

// One token per CTA of kFinalNormThreads; float4 accesses (H, ldx and ldo are multiples of 4).
constexpr int kFinalNormThreads = 1024;
__global__ void __launch_bounds__(kFinalNormThreads) final_norm_kernel(const float* x, int ldx, const float* gamma,
                                                                      float eps, int H, float* feat, float* out,
                                                                      int ldo) {
  __shared__ float nrm[kFinalNormThreads / 32];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, H4 = H >> 2;
  const float4* xr = reinterpret_cast<const float4*>(x + (size_t)t * ldx);
  float ss = 0.f;
  for (int k = tid; k < H4; k += kFinalNormThreads) {
    const float4 v = xr[k];
    ss = fmaf(v.x, v.x, ss);
    ss = fmaf(v.y, v.y, ss);
    ss = fmaf(v.z, v.z, ss);
    ss = fmaf(v.w, v.w, ss);
  }
  ss = warp_sum(ss);
  if (lane == 0) nrm[warp] = ss;
  __syncthreads();
  float tot = 0.f;
#pragma unroll
  for (int w = 0; w < kFinalNormThreads / 32; ++w) tot += nrm[w];
  const float rinv = 1.0f / sqrtf(tot / (float)H + eps);
  const float4* g4 = reinterpret_cast<const float4*>(gamma);
  for (int k = tid; k < H4; k += kFinalNormThreads) {
    const float4 v = xr[k], g = g4[k];
    const float4 f = make_float4(v.x * rinv * g.x, v.y * rinv * g.y, v.z * rinv * g.z, v.w * rinv * g.w);
    reinterpret_cast<float4*>(feat + (size_t)t * H)[k] = f;
    reinterpret_cast<float4*>(out + (size_t)t * ldo)[k] = f;
  }
}

cudaError_t launch_final_norm(const float* x, int ldx, const float* gamma, float eps, int H, int ntok, float* feat,
                              float* out, int ldo, cudaStream_t st) {
  if (ntok <= 0) return cudaSuccess;
  if ((H | ldx | ldo) & 3) return cudaErrorInvalidValue;
  return launch_k(final_norm_kernel, dim3(ntok), dim3(kFinalNormThreads), 0, st, x, ldx, gamma, eps, H, feat, out,
                  ldo);
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
  pdl_trigger();
  pdl_wait();
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* lg = logits + (size_t)r * V;
  float v = -INFINITY;
  int idx = INT_MAX;
  // float4 loads, several in flight per thread (rows are 16-byte aligned when V % 4 == 0); the
  // comparison keeps the largest value and the lowest index on ties whatever the visit order
  const int V4 = (V & 3) ? 0 : V >> 2;
  const float4* lg4 = reinterpret_cast<const float4*>(lg);
#pragma unroll 8
  for (int k = tid; k < V4; k += blockDim.x) {
    const float4 q = __ldcg(lg4 + k);
    better(v, idx, q.x, 4 * k);
    better(v, idx, q.y, 4 * k + 1);
    better(v, idx, q.z, 4 * k + 2);
    better(v, idx, q.w, 4 * k + 3);
  }
  for (int k = 4 * V4 + tid; k < V; k += blockDim.x) better(v, idx, lg[k], k);
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
  return launch_k(argmax_kernel, dim3(n_rows), dim3(1024), 0, st, logits, V, out);
}

// ------------------------------------------------------------------------------------------
// Device-side greedy feedback of a replayed decode step: every sequence moves one position
// on, and the step's greedy tokens are appended to the history.

__global__ void advance_kernel(int* pos, const int* tok, int* hist, int* step, int batch) {
  pdl_trigger();
  pdl_wait();
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
  return launch_k(advance_kernel, dim3(1), dim3(std::max(32, ((batch + 31) / 32) * 32)), 0, st, pos, tok, hist,
                  step, batch);
}

// ------------------------------------------------------------------------------------------
// Top-k routing ("41. Many GPUs: ...", section "MoE layers under tensor parallelism": the
// gate returns per-token routing weights and expert ids).  One CTA per token, one thread
// per expert: an expert's rank is the number of experts with a larger logit, or an equal
// one and a lower id; the k lowest ranks are selected, in rank order.  Softmax over all
// experts followed by renormalisation over the selected k equals a softmax over the
// selected logits, which is what is computed.  Logit rows have stride ld; ids and weights
// rows have stride kw.  kw > k: the model has a shared expert whose scalar gate logit is
// row entry E, and weight slot k receives sigmoid of it (section "Expert parallelism with
// all-to-all": the shared expert is added with sigmoid(shared_gate(x))).

__global__ void topk_kernel(const float* logits, int ld, int E, int k, int kw, int* ids, float* wts) {
  extern __shared__ float lg[];
  __shared__ float sel[32];
  __shared__ int sel_id[32];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x;
  for (int e = threadIdx.x; e < E; e += blockDim.x) lg[e] = logits[(size_t)t * ld + e];
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const float v = lg[e];
    int rank = 0;
    for (int f = 0; f < E; ++f) {
      const float u = lg[f];
      rank += (u > v) || (u == v && f < e);
    }
    if (rank < k) {
      sel[rank] = v;
      sel_id[rank] = e;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const float m = sel[0];
    float z = 0.f;
    for (int j = 0; j < k; ++j) z += expf(sel[j] - m);
    for (int j = 0; j < k; ++j) {
      ids[(size_t)t * kw + j] = sel_id[j];
      wts[(size_t)t * kw + j] = expf(sel[j] - m) / z;
    }
    if (kw > k) wts[(size_t)t * kw + k] = 1.0f / (1.0f + expf(-logits[(size_t)t * ld + E]));
  }
}

cudaError_t launch_topk(const float* logits, int ld, int n_experts, int k, int ntok, int kw, int* ids, float* wts,
                        cudaStream_t st) {
  if (ntok <= 0) return cudaSuccess;
  if (k < 1 || k > 32 || k > n_experts || ld < n_experts || kw < k || kw > k + 1 || (kw > k && ld <= n_experts))
    return cudaErrorInvalidValue;
  const int threads = std::min(1024, ((n_experts + 31) / 32) * 32);
  return launch_k(topk_kernel, dim3(ntok), dim3(threads), (size_t)n_experts * 4, st, logits, ld, n_experts, k, kw,
                  ids, wts);
}

cudaError_t prepare_kernels() {
  static cudaError_t done = cudaErrorNotReady;
  if (done == cudaSuccess) return done;
  sm_count();
  cudaError_t e = prepare_gemv<2, 4, 1, 1>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 1, 2>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 1, 4>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 1, 8>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 2, 1>();
  if (e == cudaSuccess) e = prepare_gemv<2, 2, 4, 1>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 1, 1, 1>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 1, 2, 1>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 1, 4, 1>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 1, 1, 2>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 1, 2, 2>();
  if (e == cudaSuccess) e = prepare_gemv<2, 4, 1, 4, 2>();

  if (e == cudaSuccess) e = prepare_gemm_tc();
  if (e == cudaSuccess) e = prepare_attn<64, 1>();
  if (e == cudaSuccess) e = prepare_attn<64, 2>();
  if (e == cudaSuccess) e = prepare_attn<64, 4>();
  if (e == cudaSuccess) e = prepare_attn<64, 8>();
  if (e == cudaSuccess) e = prepare_attn<128, 1>();
  if (e == cudaSuccess) e = prepare_attn<128, 2>();
  if (e == cudaSuccess) e = prepare_attn<128, 4>();
  if (e == cudaSuccess) e = prepare_attn<128, 8>();
  if (e == cudaSuccess) e = prepare_mega();
  if (e == cudaSuccess) e = prepare_attn_prefill();
  done = e;
  return e;
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

// Prefill-path kernels (sm_103a): the tcgen05 tensor-core GEMM with int8 -> bf16 weight
// dequantisation in shared memory, and the bf16 conversion of activations.
//
// "41. Many GPUs: tensor, pipeline, expert and data parallelism", section "Pipeline
// parallelism": a prefill step is the same block loop as decode over all prompt tokens;
// here the projections of those tokens are dense GEMMs on the tensor cores.  Operands are
// bf16 (activations rounded once, weights as bf16(f32(scale) * q)), accumulation is f32.

#include <algorithm>
#include <cfloat>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace lrs {

// CTA tile: 256 tokens (two M = 128 MMAs) x 256 weight rows (N = 256) x 64 of K per step.
constexpr int kGBM = 256, kGBN = 256, kGBK = 64, kGStages = 3, kGThreads = 256;
constexpr uint32_t kGTileA = kGBM * kGBK * 2;        // 32 KB bf16, 128B-swizzled K-major
constexpr uint32_t kGTileB = kGBN * kGBK * 2;        // 32 KB bf16, 128B-swizzled K-major
constexpr uint32_t kGRawB = kGBN * kGBK;             // 16 KB int8 (biased)
constexpr uint32_t kGRawS = kGBN * 4;                // 2 fp16 scales per row
constexpr uint32_t kGOffA = 0;
constexpr uint32_t kGOffB = kGOffA + kGStages * kGTileA;     // 2 dequantised B buffers
constexpr uint32_t kGOffRB = kGOffB + 2 * kGTileB;
constexpr uint32_t kGOffRS = kGOffRB + kGStages * kGRawB;
constexpr uint32_t kGOffBar = kGOffRS + kGStages * kGRawS;
constexpr uint32_t kGSmem = kGOffBar + 64 + 1024;          // + barriers, tmem slot, alignment slack
constexpr uint32_t kGTmemCols = 512;                        // two 128 x 256 f32 accumulators
constexpr uint64_t kGWaitNs = 2000000000ull;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__global__ void __launch_bounds__(kGThreads, 1) gemm_tc_kernel(const GemmArgs a) {
  extern __shared__ unsigned char g_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)g_raw + 1023) & ~(uintptr_t)1023);
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + kGOffBar);  // [2] MMA completion
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kGOffBar + 16);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kGOffBar + 32);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // M tiles vary fastest across the grid: the CTAs that share a weight tile run together
  // and read it from DRAM once (the activations, a few MB, stay in L2 for every N tile)
  const int m0 = blockIdx.x * kGBM, n0 = blockIdx.y * kGBN;
  const int N = a.w.N, Kp = a.w.Kp, M = a.M;
  const int nk = Kp / kGBK;

  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    *abort_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kGTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();
  pdl_wait();

  auto issue_loads = [&](int kt) {
    if (kt < nk) {
      const int s = kt % kGStages;
      unsigned char* as = sm + kGOffA + s * kGTileA;
      unsigned char* rb = sm + kGOffRB + s * kGRawB;
      unsigned char* rs = sm + kGOffRS + s * kGRawS;
#pragma unroll
      for (int i = 0; i < (kGBM * 8) / kGThreads; ++i) {  // activations: 256 rows x 8 chunks of 16 B
        const int idx = tid + i * kGThreads, r = idx >> 3, c = idx & 7;
        const int gm = m0 + r;
        const __nv_bfloat16* src = gm < M ? a.a + (size_t)gm * a.lda + kt * kGBK + c * 8 : a.a;
        cp_async16_zfill(as + r * 128 + ((c ^ (r & 7)) << 4), src, gm < M ? 16u : 0u);
      }
#pragma unroll
      for (int i = 0; i < (kGBN * 4) / kGThreads; ++i) {  // weights: 256 rows x 4 chunks of 16 int8
        const int idx = tid + i * kGThreads, n = idx >> 2, j = idx & 3;
        const int gn = n0 + n;
        const uint8_t* src = gn < N ? a.w.q + (size_t)gn * Kp + kt * kGBK + j * 16 : a.w.q;
        cp_async16_zfill(rb + n * 64 + j * 16, src, gn < N ? 16u : 0u);
      }
      {  // the 2 block scales of row tid for this K step
        const int gn = n0 + tid;
        if (gn < N)
          cp_async4(rs + tid * 4, a.w.s + (size_t)gn * (Kp / 32) + kt * 2);
        else
          *reinterpret_cast<uint32_t*>(rs + tid * 4) = 0u;
      }
    }
    cp_async_commit();
  };

  auto wait_mma = [&](int kt) {  // MMAs of K step kt (and all before) complete
    if (!*abort_flag && !mbar_wait(&bar[kt & 1], (uint32_t)(kt >> 1) & 1u, kGWaitNs)) {
      if (a.err) atomicExch(a.err, 1);
      *abort_flag = 1;
    }
  };

  constexpr uint32_t idesc = idesc_bf16_f32(128, kGBN);
  issue_loads(0);
  issue_loads(1);
  for (int kt = 0; kt < nk; ++kt) {
    const int s = kt % kGStages, buf = kt & 1;
    cp_async_wait_group<1>();
    __syncthreads();
    if (kt >= 2) wait_mma(kt - 2);  // the B buffer about to be written was read by step kt - 2
    {  // dequantise weight row `tid` of this step into the swizzled bf16 tile
      const unsigned char* rb = sm + kGOffRB + s * kGRawB + tid * 64;
      const uint32_t sraw = *reinterpret_cast<const uint32_t*>(sm + kGOffRS + s * kGRawS + tid * 4);
      const float s0 = __half2float(__ushort_as_half((uint16_t)(sraw & 0xFFFFu)));
      const float s1 = __half2float(__ushort_as_half((uint16_t)(sraw >> 16)));
      unsigned char* bt = sm + kGOffB + buf * kGTileB;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 w = *reinterpret_cast<const uint4*>(rb + j * 16);
        const float sc = j < 2 ? s0 : s1;
        const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t x = wd[q];
          const float f0 = sc * (float)((int)(x & 0xFFu) - 128);
          const float f1 = sc * (float)((int)((x >> 8) & 0xFFu) - 128);
          const float f2 = sc * (float)((int)((x >> 16) & 0xFFu) - 128);
          const float f3 = sc * (float)((int)(x >> 24) - 128);
          o[2 * q] = pack_bf16x2(f0, f1);
          o[2 * q + 1] = pack_bf16x2(f2, f3);
        }
        *reinterpret_cast<uint4*>(bt + sw128_offset(tid, 16 * j)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(bt + sw128_offset(tid, 16 * j + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
    }
    fence_async_smem();
    __syncthreads();
    if (tid == 0 && !*abort_flag) {
      tc_fence_after();
      const uint32_t a_base = smem_u32(sm + kGOffA + s * kGTileA);
      const uint32_t b_base = smem_u32(sm + kGOffB + buf * kGTileB);
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int kk = 0; kk < kGBK / 16; ++kk)
          umma_bf16(tmem + h * kGBN, desc_sw128(a_base + h * (128 * 128) + kk * 32), desc_sw128(b_base + kk * 32),
                    idesc, (kt > 0 || kk > 0) ? 1u : 0u);
      umma_commit(&bar[buf]);
    }
    if (kt >= 1) wait_mma(kt - 1);  // the stage about to be refilled was read by step kt - 1
    issue_loads(kt + 2);
  }
  wait_mma(nk - 1);
  cp_async_wait_group<0>();
  tc_fence_after();

  // ---- epilogue: warp w reads TMEM lanes 32 (w % 4) .. +31, columns of its half ----
  const int p = warp & 3, chalf = warp >> 2;
#pragma unroll 1
  for (int h = 0; h < 2; ++h) {
    const int gm = m0 + h * 128 + 32 * p + lane;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      const int c0 = chalf * 128 + cc * 32;
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(32 * p) << 16) + (uint32_t)(h * kGBN + c0), r);
      tmem_wait_ld();
      if (*abort_flag || gm >= M) continue;
      const int gn0 = n0 + c0;
      if (a.epi == EPI_STORE || a.epi == EPI_RESID) {
        float* orow = a.out + (size_t)gm * a.ldo;
        const float* rrow = a.epi == EPI_RESID ? a.resid + (size_t)gm * a.ldr : nullptr;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int gn = gn0 + i;
          if (gn < N) {
            float v = __uint_as_float(r[i]);
            if (rrow) v = __fadd_rn(rrow[gn], v);
            orow[gn] = v;
          }
        }
      } else if (a.epi == EPI_SWIGLU_BF16) {
        __nv_bfloat16* orow = a.out_bf16 + (size_t)gm * a.ldo_bf16;
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int gn = gn0 + i;
          if (gn < N) orow[gn >> 1] = __float2bfloat16_rn(silu(__uint_as_float(r[i])) * __uint_as_float(r[i + 1]));
        }
      } else {  // EPI_QKV: column pairs (2i, 2i+1) of a head are its dims (i, i + D/2)
        const int hd = a.head_dim >> 1, pp = a.pos[gm];
#pragma unroll
        for (int i = 0; i < 32; i += 2) {
          const int gn = gn0 + i;
          if (gn >= N) continue;
          const float y0 = __uint_as_float(r[i]), y1 = __uint_as_float(r[i + 1]);
          const int P = gn >> 1, head = P / hd, ii = P - head * hd;
          if (head < a.n_q_heads) {
            const float2 cs = a.rope[(size_t)pp * hd + ii];
            float* qo = a.qout + ((size_t)gm * a.n_q_heads + head) * a.head_dim;
            qo[ii] = y0 * cs.x - y1 * cs.y;
            qo[ii + hd] = y1 * cs.x + y0 * cs.y;
          } else {
            const bool is_k = head < a.n_q_heads + a.n_kv_heads;
            const int kvh = head - a.n_q_heads - (is_k ? 0 : a.n_kv_heads);
            const size_t base = (((size_t)a.seq[gm] * a.n_kv_heads + kvh) * a.max_len + pp) * a.head_dim;
            if (is_k) {
              const float2 cs = a.rope[(size_t)pp * hd + ii];
              a.kc[base + ii] = __float2half_rn(y0 * cs.x - y1 * cs.y);
              a.kc[base + ii + hd] = __float2half_rn(y1 * cs.x + y0 * cs.y);
            } else {
              a.vc[base + ii] = __float2half_rn(y0);
              a.vc[base + ii + hd] = __float2half_rn(y1);
            }
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kGTmemCols);
}

cudaError_t prepare_gemm_tc() {
  return cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
}

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st) {
  if (a.M <= 0 || a.w.N <= 0) return cudaSuccess;
  if (a.w.Kp % kGBK || a.lda < a.w.Kp || a.lda % 8) return cudaErrorInvalidValue;
  const dim3 grid((a.M + kGBM - 1) / kGBM, (a.w.N + kGBN - 1) / kGBN);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = kGSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, a);
}

// ------------------------------------------------------------------------------------------
// f32 rows -> bf16 rows (the GEMM operand), with the RMSNorm when gamma is given; the
// reduction order matches the GEMV prologue.

__global__ void rows_to_bf16_kernel(const float* x, int ld_in, int K, const float* gamma, float eps,
                                    __nv_bfloat16* out, int ld_out) {
  __shared__ float nrm[8];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* xr = x + (size_t)t * ld_in;
  float rinv = 1.0f;
  if (gamma) {
    float ss = 0.f;
    for (int k = tid; k < K; k += 256) {
      const float v = xr[k];
      ss = fmaf(v, v, ss);
    }
    ss = warp_sum(ss);
    if (lane == 0) nrm[warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < 8; ++w) tot += nrm[w];
    rinv = 1.0f / sqrtf(tot / (float)K + eps);
  }
  __nv_bfloat16* orow = out + (size_t)t * ld_out;
  for (int k = tid; k < ld_out; k += 256) {
    float v = 0.f;
    if (k < K) v = gamma ? xr[k] * rinv * gamma[k] : xr[k];
    orow[k] = __float2bfloat16_rn(v);
  }
}

cudaError_t launch_rows_to_bf16(const float* x, int ld_in, int K, const float* gamma, float eps, int ntok,
                                __nv_bfloat16* out, int ld_out, cudaStream_t st) {
  if (ntok <= 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ntok);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, rows_to_bf16_kernel, x, ld_in, K, gamma, eps, out, ld_out);
}

// ------------------------------------------------------------------------------------------
// Causal attention of a prefill call, tiled (CUDA cores, f32 math over the fp16 cache).
//
// "41. Many GPUs: tensor, pipeline, expert and data parallelism", section "Ring attention for
// very long contexts": softmax(q k^T / sqrt(D)) v with a running max and sum over tiles of
// positions (the same log-sum-exp recurrence its merge uses), here over the tiles of one
// sequence in order.  A CTA takes 64 query rows -- the G query heads of one KV head for 64 / G
// consecutive tokens of the call -- and every K/V tile of 64 positions it loads serves all of
// them.  Token t attends to positions 0..pos[t] of sequence seq[t]; a block that spans two
// sequences walks each sequence's tiles in turn with the other rows masked.  The tokens' own
// K/V rows are already in the cache (written by the QKV projection).

constexpr int kPR = 64;       // query rows per CTA
constexpr int kPT = 64;       // positions per K/V tile
constexpr int kPThreads = 256;

template <int D>
struct PrefillSmem {
  static constexpr int QROW = D + 4;   // floats per q row (bank offset between rows)
  static constexpr int KROW = D + 8;   // halves per K/V row (16-byte pad)
  static constexpr int SROW = kPT + 4; // floats per probability row
  static constexpr size_t q = (size_t)kPR * QROW * 4;
  static constexpr size_t kv = (size_t)kPT * KROW * 2;
  static constexpr size_t p = (size_t)kPR * SROW * 4;
  static constexpr size_t total = q + 2 * kv + p + 4 * kPR * 4;
};

template <int D, int G>
__global__ void __launch_bounds__(kPThreads, 2) attn_prefill_kernel(const AttnArgs a) {
  using S = PrefillSmem<D>;
  constexpr int QB = kPR / G;  // tokens per CTA
  extern __shared__ __align__(16) unsigned char ps_raw[];
  float* qs = reinterpret_cast<float*>(ps_raw);
  __half* ks = reinterpret_cast<__half*>(ps_raw + S::q);
  __half* vs = ks + kPT * S::KROW;
  float* pr = reinterpret_cast<float*>(ps_raw + S::q + 2 * S::kv);
  int* rseq = reinterpret_cast<int*>(pr + kPR * S::SROW);  // [kPR] sequence of the row's token (-1: none)
  int* rpos = rseq + kPR;                                   // [kPR] its position
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, tr = tid >> 3, tc = tid & 7;
  const int kvh = blockIdx.y, t0 = blockIdx.x * QB;
  // rows r = i * G + g: token t0 + i, query head kvh * G + g
  for (int i = tid; i < kPR * (D / 4); i += kPThreads) {
    const int r = i / (D / 4), c4 = i - r * (D / 4);
    const int t = t0 + r / G, g = r % G;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < a.ntok) v = reinterpret_cast<const float4*>(a.q + ((size_t)t * a.Hq + (size_t)kvh * G + g) * D)[c4];
    *reinterpret_cast<float4*>(qs + r * S::QROW + 4 * c4) = v;
  }
  for (int r = tid; r < kPR; r += kPThreads) {
    const int t = t0 + r / G;
    rseq[r] = t < a.ntok ? a.seq[t] : -1;
    rpos[r] = t < a.ntok ? a.pos[t] : -1;
  }
  __syncthreads();
  // this thread: rows tr and tr + 32; positions tc + 8 j of a tile; output dims tc + 8 k
  const int r0 = tr, r1 = tr + 32;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float o0[D / 8], o1[D / 8];
#pragma unroll
  for (int k = 0; k < D / 8; ++k) o0[k] = o1[k] = 0.f;
  const int sq0 = rseq[r0], sq1 = rseq[r1], pp0 = rpos[r0], pp1 = rpos[r1];

  // walk the distinct sequences of the block in order of first appearance (rows of one
  // sequence need not be adjacent); every thread reads the same row table, so the walk is
  // uniform across the CTA
  for (int rs = 0; rs < kPR; ++rs) {
    const int sid = rseq[rs];
    if (sid < 0) continue;
    bool seen = false;
    for (int q = 0; q < rs; ++q) seen |= rseq[q] == sid;
    if (seen) continue;
    int maxpos = -1;
    for (int r = rs; r < kPR; ++r)
      if (rseq[r] == sid) maxpos = max(maxpos, rpos[r]);
    const __half* kb = a.kc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;
    const __half* vb = a.vc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;
    const bool own0 = sq0 == sid, own1 = sq1 == sid;
    for (int p0 = 0; p0 <= maxpos; p0 += kPT) {
      const int np = min(kPT, maxpos + 1 - p0);
      __syncthreads();  // the previous tile is consumed
      for (int i = tid; i < np * (D / 8); i += kPThreads) {
        const int r = i / (D / 8), c = i - r * (D / 8);
        cp_async16(ks + r * S::KROW + c * 8, kb + (size_t)(p0 + r) * D + c * 8);
        cp_async16(vs + r * S::KROW + c * 8, vb + (size_t)(p0 + r) * D + c * 8);
      }
      cp_async_wait_all();
      __syncthreads();
      // scores of rows r0, r1 at positions tc + 8 j
      float s0[8], s1[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) s0[j] = s1[j] = 0.f;
      const float* q0 = qs + r0 * S::QROW;
      const float* q1 = qs + r1 * S::QROW;
#pragma unroll 2
      for (int d = 0; d < D; d += 8) {
        const float4 qa0 = *reinterpret_cast<const float4*>(q0 + d), qb0 = *reinterpret_cast<const float4*>(q0 + d + 4);
        const float4 qa1 = *reinterpret_cast<const float4*>(q1 + d), qb1 = *reinterpret_cast<const float4*>(q1 + d + 4);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint4 kk = *reinterpret_cast<const uint4*>(ks + (tc + 8 * j) * S::KROW + d);
          const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kk.x));
          const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kk.y));
          const float2 k45 = __half22float2(*reinterpret_cast<const __half2*>(&kk.z));
          const float2 k67 = __half22float2(*reinterpret_cast<const __half2*>(&kk.w));
          float x = s0[j];
          x = fmaf(qa0.x, k01.x, x);
          x = fmaf(qa0.y, k01.y, x);
          x = fmaf(qa0.z, k23.x, x);
          x = fmaf(qa0.w, k23.y, x);
          x = fmaf(qb0.x, k45.x, x);
          x = fmaf(qb0.y, k45.y, x);
          x = fmaf(qb0.z, k67.x, x);
          x = fmaf(qb0.w, k67.y, x);
          s0[j] = x;
          float y = s1[j];
          y = fmaf(qa1.x, k01.x, y);
          y = fmaf(qa1.y, k01.y, y);
          y = fmaf(qa1.z, k23.x, y);
          y = fmaf(qa1.w, k23.y, y);
          y = fmaf(qb1.x, k45.x, y);
          y = fmaf(qb1.y, k45.y, y);
          y = fmaf(qb1.z, k67.x, y);
          y = fmaf(qb1.w, k67.y, y);
          s1[j] = y;
        }
      }
      // causal mask, running max and sum per row (the 8 lanes of a row agree via shuffles)
      float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const int p = p0 + tc + 8 * j;
        s0[j] = (own0 && tc + 8 * j < np && p <= pp0) ? s0[j] * a.scale : -INFINITY;
        s1[j] = (own1 && tc + 8 * j < np && p <= pp1) ? s1[j] * a.scale : -INFINITY;
        mt0 = fmaxf(mt0, s0[j]);
        mt1 = fmaxf(mt1, s1[j]);
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        mt0 = fmaxf(mt0, __shfl_xor_sync(0xffffffffu, mt0, o));
        mt1 = fmaxf(mt1, __shfl_xor_sync(0xffffffffu, mt1, o));
      }
      const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
      const float al0 = (mn0 == -INFINITY || m0 == -INFINITY) ? (m0 == -INFINITY ? 0.f : 1.f) : expf(m0 - mn0);
      const float al1 = (mn1 == -INFINITY || m1 == -INFINITY) ? (m1 == -INFINITY ? 0.f : 1.f) : expf(m1 - mn1);
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float e0 = s0[j] == -INFINITY ? 0.f : expf(s0[j] - mn0);
        const float e1 = s1[j] == -INFINITY ? 0.f : expf(s1[j] - mn1);
        pr[r0 * S::SROW + tc + 8 * j] = e0;
        pr[r1 * S::SROW + tc + 8 * j] = e1;
        ls0 += e0;
        ls1 += e1;
      }
#pragma unroll
      for (int o = 1; o < 8; o <<= 1) {
        ls0 += __shfl_xor_sync(0xffffffffu, ls0, o);
        ls1 += __shfl_xor_sync(0xffffffffu, ls1, o);
      }
      l0 = l0 * al0 + ls0;
      l1 = l1 * al1 + ls1;
      m0 = mn0;
      m1 = mn1;
      __syncwarp();  // the row's 8 lanes are in this warp: their probabilities are written
      // o += P V for dims tc + 8 k
#pragma unroll
      for (int k = 0; k < D / 8; ++k) {
        o0[k] *= al0;
        o1[k] *= al1;
      }
      for (int p = 0; p < np; ++p) {
        const float w0 = pr[r0 * S::SROW + p], w1 = pr[r1 * S::SROW + p];
        const __half* vr = vs + p * S::KROW;
#pragma unroll
        for (int k = 0; k < D / 8; ++k) {
          const float v = __half2float(vr[tc + 8 * k]);
          o0[k] = fmaf(w0, v, o0[k]);
          o1[k] = fmaf(w1, v, o1[k]);
        }
      }
    }
  }
  // normalise and store
  const int ta = t0 + r0 / G, tb = t0 + r1 / G;
  if (sq0 >= 0 && ta < a.ntok) {
    float* out = a.out + ((size_t)ta * a.Hq + (size_t)kvh * G + r0 % G) * D;
    const float inv = 1.0f / l0;
#pragma unroll
    for (int k = 0; k < D / 8; ++k) out[tc + 8 * k] = o0[k] * inv;
  }
  if (sq1 >= 0 && tb < a.ntok) {
    float* out = a.out + ((size_t)tb * a.Hq + (size_t)kvh * G + r1 % G) * D;
    const float inv = 1.0f / l1;
#pragma unroll
    for (int k = 0; k < D / 8; ++k) out[tc + 8 * k] = o1[k] * inv;
  }
}

template <int D, int G>
static cudaError_t prepare_attn_prefill_dg() {
  return cudaFuncSetAttribute(attn_prefill_kernel<D, G>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)PrefillSmem<D>::total);
}

cudaError_t prepare_attn_prefill() {
  const cudaError_t r[] = {prepare_attn_prefill_dg<64, 1>(),  prepare_attn_prefill_dg<64, 2>(),
                           prepare_attn_prefill_dg<64, 4>(),  prepare_attn_prefill_dg<64, 8>(),
                           prepare_attn_prefill_dg<128, 1>(), prepare_attn_prefill_dg<128, 2>(),
                           prepare_attn_prefill_dg<128, 4>(), prepare_attn_prefill_dg<128, 8>()};
  for (cudaError_t x : r)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

template <int D, int G>
static cudaError_t launch_attn_prefill_dg(const AttnArgs& a, cudaStream_t st) {
  constexpr int QB = kPR / G;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.ntok + QB - 1) / QB, a.Hkv);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = PrefillSmem<D>::total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_prefill_kernel<D, G>, a);
}

cudaError_t launch_attn_prefill(const AttnArgs& a, cudaStream_t st) {
  if (a.ntok <= 0) return cudaSuccess;
  const int G = a.Hq / a.Hkv;
  if (a.D == 64) {
    switch (G) {
      case 1: return launch_attn_prefill_dg<64, 1>(a, st);
      case 2: return launch_attn_prefill_dg<64, 2>(a, st);
      case 4: return launch_attn_prefill_dg<64, 4>(a, st);
      case 8: return launch_attn_prefill_dg<64, 8>(a, st);
    }
  } else if (a.D == 128) {
    switch (G) {
      case 1: return launch_attn_prefill_dg<128, 1>(a, st);
      case 2: return launch_attn_prefill_dg<128, 2>(a, st);
      case 4: return launch_attn_prefill_dg<128, 4>(a, st);
      case 8: return launch_attn_prefill_dg<128, 8>(a, st);
    }
  }
  return cudaErrorInvalidValue;
}

}  // namespace lrs

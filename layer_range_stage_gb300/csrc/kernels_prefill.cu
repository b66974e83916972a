// Prefill-path kernels (sm_103a): the tcgen05 tensor-core GEMM with int8 -> bf16 weight
// dequantisation in shared memory, its variant for calls of at most 64 tokens (batched
// decode: the weights as the 128-row MMA operand, each read once, K split over CTAs where the
// weight tiles are few), the bf16 conversion of activations, and the causal attention of a
// prefill call on the tensor cores.
//
// "41. Many GPUs: tensor, pipeline, expert and data parallelism", section "Pipeline
// parallelism": a prefill step is the same block loop as decode over all prompt tokens;
// here the projections of those tokens are dense GEMMs on the tensor cores.  Operands are
// bf16 (activations rounded once, weights as bf16(f32(scale) * q)), accumulation is f32.

#include <algorithm>
#include <cfloat>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"
#include "kernels.cuh"
#include "tc.cuh"

namespace lrs {

// CTA tile: 256 tokens (two M = 128 MMAs) x 256 weight rows (N = 256) x 64 of K per step.
// Warp roles during the main loop, coupled only by mbarriers:
//   warps 0-7: dequantise each int8 weight tile into a 128B-swizzled bf16 tile,
//     bf16(f32(scale) * q), one row per thread;
//   warp 8 (one thread): TMA loads of the activations through a 128B-swizzled tensor map
//     (they land in the tensor core's K-major layout), after the programmatic-launch wait;
//   warp 10 (one thread): TMA loads of the raw int8 weight tiles and fp16 scale groups through
//     plain tensor maps; the weights do not depend on the previous kernel and start at once;
//   warp 9 (one thread): issues the tcgen05 MMAs of a K step once its activation stage and
//     bf16 weight tile are full, and commits their completion to the stages' "empty" barriers;
// then warps 0-7 run the epilogue from TMEM.  Every wait is bounded (and gives up at once
// when another role has given up); a CTA that gives up sets the error word, waits (bounded)
// for the copies and MMAs it started, releases TMEM and leaves.
constexpr int kGBM = 256, kGBN = 256, kGBK = 64, kGThreads = 352;
constexpr int kGDeq = 256;  // dequantising threads (warps 0-7), one weight row each
constexpr int kGSA = 3;  // activation stages
constexpr int kGSR = 3;  // raw weight stages
constexpr uint32_t kGTileA = kGBM * kGBK * 2;        // 32 KB bf16, 128B-swizzled K-major
constexpr uint32_t kGTileB = kGBN * kGBK * 2;        // 32 KB bf16, 128B-swizzled K-major
constexpr uint32_t kGRawB = kGBN * kGBK;             // 16 KB int8 (biased), row-major
constexpr uint32_t kGRawS = kGBN * 16;               // 8 fp16 scales per row = 4 K steps
constexpr uint32_t kGOffA = 0;
constexpr uint32_t kGOffB = kGOffA + kGSA * kGTileA;     // 2 dequantised B buffers
constexpr uint32_t kGOffRB = kGOffB + 2 * kGTileB;       // raw weight stages
constexpr uint32_t kGOffRS = kGOffRB + kGSR * kGRawB;    // 2 scale stages
constexpr uint32_t kGOffBar = kGOffRS + 2 * kGRawS;
constexpr uint32_t kGSmem = kGOffBar + 256 + 1024;       // + barriers, tmem slot, alignment slack
constexpr uint32_t kGTmemCols = 512;                     // two 128 x 256 f32 accumulators
constexpr uint64_t kGWaitNs = 500000000ull;              // 0.5 s
constexpr uint64_t kGDrainNs = 100000000ull;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}


// Bounded wait that also gives up as soon as another role of the CTA has given up.
__device__ __forceinline__ bool gwait(uint64_t* bar, uint32_t parity, volatile int* abort_flag, int* err) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (global_ns() - t0 > kGWaitNs) {
      *abort_flag = 1;
      if (err) atomicExch(err, 1);
      return false;
    }
  }
  return true;
}

struct GBars {  // mbarriers of the main loop
  uint64_t a_full[kGSA], a_empty[kGSA], r_full[kGSR], r_empty[kGSR];
  uint64_t s_full[2], s_empty[2], b_full[2], b_empty[2], acc_full, mma_drain;
};

__global__ void __launch_bounds__(kGThreads, 1)
    gemm_tc_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tB,
                   const __grid_constant__ CUtensorMap tS) {
  extern __shared__ unsigned char g_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)g_raw + 1023) & ~(uintptr_t)1023);
  GBars* B = reinterpret_cast<GBars*>(sm + kGOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kGOffBar + sizeof(GBars));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kGOffBar + sizeof(GBars) + 8);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // M tiles vary fastest across the grid: the CTAs that share a weight tile run together
  // and read it from DRAM once (the activations, a few MB, stay in L2 for every N tile)
  const int m0 = blockIdx.x * kGBM, n0 = blockIdx.y * kGBN;
  const int N = a.w.N, M = a.M;
  const int nk = a.w.Kp / kGBK;

  if (tid == 0) {
    for (int i = 0; i < kGSA; ++i) {
      mbar_init(&B->a_full[i], 1);
      mbar_init(&B->a_empty[i], 1);
    }
    for (int i = 0; i < kGSR; ++i) {
      mbar_init(&B->r_full[i], 1);
      mbar_init(&B->r_empty[i], kGDeq);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B->s_full[i], 1);
      mbar_init(&B->s_empty[i], kGDeq);
      mbar_init(&B->b_full[i], kGDeq);
      mbar_init(&B->b_empty[i], 1);
    }
    mbar_init(&B->acc_full, 1);
    mbar_init(&B->mma_drain, 1);
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

  if (warp == 8) {
    // ---------------- activation loads ----------------
    if (lane == 0) {
      int ia = 0;
      pdl_wait();  // the activations are the previous kernel's output
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % kGSA;
        if (kt >= kGSA && !gwait(&B->a_empty[s], (uint32_t)((kt / kGSA) + 1) & 1u, abort_flag, a.err)) break;
        mbar_arrive_expect_tx(&B->a_full[s], kGTileA);
        tma_load_2d(sm + kGOffA + s * kGTileA, &tA, kt * kGBK, m0, &B->a_full[s]);
        ++ia;
      }
      if (*abort_flag)  // nothing may still be landing in shared memory when the CTA leaves
        for (int k = max(0, ia - kGSA); k < ia; ++k)
          mbar_wait(&B->a_full[k % kGSA], (uint32_t)(k / kGSA) & 1u, kGDrainNs);
    }
  } else if (warp == 10) {
    // ---------------- weight loads: raw tiles, and a scale group every 4 K steps ----------------
    if (lane == 0) {
      int ir = 0, is = 0;
      for (int kt = 0; kt < nk; ++kt) {
        const int r = kt % kGSR;
        if (kt >= kGSR && !gwait(&B->r_empty[r], (uint32_t)((kt / kGSR) + 1) & 1u, abort_flag, a.err)) break;
        if ((kt & 3) == 0) {
          const int g = kt >> 2, gs = g & 1;
          if (g >= 2 && !gwait(&B->s_empty[gs], (uint32_t)((g / 2) + 1) & 1u, abort_flag, a.err)) break;
          mbar_arrive_expect_tx(&B->s_full[gs], kGRawS);
          tma_load_2d(sm + kGOffRS + gs * kGRawS, &tS, g * 8, n0, &B->s_full[gs]);
          ++is;
        }
        mbar_arrive_expect_tx(&B->r_full[r], kGRawB);
        tma_load_2d(sm + kGOffRB + r * kGRawB, &tB, kt * kGBK, n0, &B->r_full[r]);
        ++ir;
      }
      if (*abort_flag) {
        for (int k = max(0, ir - kGSR); k < ir; ++k)
          mbar_wait(&B->r_full[k % kGSR], (uint32_t)(k / kGSR) & 1u, kGDrainNs);
        for (int k = max(0, is - 2); k < is; ++k) mbar_wait(&B->s_full[k & 1], (uint32_t)(k / 2) & 1u, kGDrainNs);
      }
    }
  } else if (warp < 8) {
    // ---------------- dequantise: row `tid` of every weight tile ----------------
    // A byte b moved into the low mantissa bits of 2^23 is the float 2^23 + b; subtracting
    // 2^23 + 128 gives q = b - 128 exactly, and f32(scale) * q is exact (11 + 8 bits).
    const int row = tid;
    for (int kt = 0; kt < nk; ++kt) {
      const int r = kt % kGSR, bb = kt & 1, g = kt >> 2;
      if (!gwait(&B->r_full[r], (uint32_t)(kt / kGSR) & 1u, abort_flag, a.err)) break;
      if ((kt & 3) == 0 && !gwait(&B->s_full[g & 1], (uint32_t)(g / 2) & 1u, abort_flag, a.err)) break;
      if (kt >= 2 && !gwait(&B->b_empty[bb], (uint32_t)((kt / 2) + 1) & 1u, abort_flag, a.err)) break;
      const unsigned char* rb = sm + kGOffRB + r * kGRawB;
      const unsigned char* rs = sm + kGOffRS + (g & 1) * kGRawS;
      unsigned char* bt = sm + kGOffB + bb * kGTileB;
      const uint32_t sraw = *reinterpret_cast<const uint32_t*>(rs + row * 16 + (kt & 3) * 4);
      const float s0 = __half2float(__ushort_as_half((uint16_t)(sraw & 0xFFFFu)));
      const float s1 = __half2float(__ushort_as_half((uint16_t)(sraw >> 16)));
      constexpr float kBias = 8388736.0f;  // 2^23 + 128
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int j = (jj + row) & 3;  // rotated: neighbouring rows read different banks
        const uint4 w = *reinterpret_cast<const uint4*>(rb + row * 64 + j * 16);
        const float sc = j < 2 ? s0 : s1;
        const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
        uint32_t o[8];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint32_t x = wd[q];
          const float f0 = sc * (__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440)) - kBias);
          const float f1 = sc * (__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7441)) - kBias);
          const float f2 = sc * (__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7442)) - kBias);
          const float f3 = sc * (__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7443)) - kBias);
          o[2 * q] = pack_bf16x2(f0, f1);
          o[2 * q + 1] = pack_bf16x2(f2, f3);
        }
        *reinterpret_cast<uint4*>(bt + sw128_offset(row, 16 * j)) = make_uint4(o[0], o[1], o[2], o[3]);
        *reinterpret_cast<uint4*>(bt + sw128_offset(row, 16 * j + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
      }
      fence_async_smem();  // the bf16 tile is read next by the tensor core (async proxy)
      mbar_arrive(&B->b_full[bb]);
      mbar_arrive(&B->r_empty[r]);
      if ((kt & 3) == 3) mbar_arrive(&B->s_empty[g & 1]);
    }
  } else if (warp == 9) {
    // ---------------- MMA issue ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(128, kGBN);
      int issued = 0;
      for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % kGSA, bb = kt & 1;
        if (!gwait(&B->a_full[s], (uint32_t)(kt / kGSA) & 1u, abort_flag, a.err)) break;
        if (!gwait(&B->b_full[bb], (uint32_t)(kt / 2) & 1u, abort_flag, a.err)) break;
        tc_fence_after();
        const uint32_t a_base = smem_u32(sm + kGOffA + s * kGTileA);
        const uint32_t b_base = smem_u32(sm + kGOffB + bb * kGTileB);
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int kk = 0; kk < kGBK / 16; ++kk)
            umma_bf16(tmem + h * kGBN, desc_sw128(a_base + h * (128 * 128) + kk * 32), desc_sw128(b_base + kk * 32),
                      idesc, (kt > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&B->a_empty[s]);
        umma_commit(&B->b_empty[bb]);
        ++issued;
      }
      if (issued == nk) {
        umma_commit(&B->acc_full);
      } else if (issued > 0) {  // given up: let the MMAs already issued finish before TMEM is released
        umma_commit(&B->mma_drain);
        mbar_wait(&B->mma_drain, 0u, kGDrainNs);
      }
    }
  }
  __syncthreads();
  if (tid == 0 && !*abort_flag) gwait(&B->acc_full, 0u, abort_flag, a.err);
  __syncthreads();
  const bool ok = !*abort_flag;
  tc_fence_after();
  pdl_wait();  // the epilogue reads the residual / writes outputs the previous kernel may touch

  // ---- epilogue (warps 0-7): warp w reads TMEM lanes 32 (w % 4) .. +31, columns of its half ----
  // Each 32 x 32 block goes through shared memory (the activation stages are idle now) so
  // that a warp writes whole row segments: lane = column for the stores.
  const int p = warp & 3, chalf = (warp >> 2) & 1;
  float* stg = reinterpret_cast<float*>(sm + kGOffA) + warp * (32 * 33);  // [32][33] per warp
#pragma unroll 1
  for (int h = 0; h < 2 && ok && warp < 8; ++h) {
    const int rbase = m0 + h * 128 + 32 * p;
    // the rows' positions and sequences (QKV), one load per lane, shared by shuffles below
    const int prow = rbase + lane;
    const int pos_l = (a.epi == EPI_QKV && prow < M) ? a.pos[prow] : 0;
    const int seq_l = (a.epi == EPI_QKV && prow < M) ? a.seq[prow] : 0;
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      const int c0 = chalf * 128 + cc * 32;
      const int gn0 = n0 + c0;
      const int gn = gn0 + lane;
      // the global inputs of the epilogue are requested before the accumulators are read, all
      // at once (every load of the block in flight together, not one per row)
      float rv[32];
      if (a.epi == EPI_RESID) {
#pragma unroll
        for (int j = 0; j < 32; ++j)
          rv[j] = (rbase + j < M && gn < N) ? a.resid[(size_t)(rbase + j) * a.ldr + gn] : 0.f;
      }
      const int qi = lane & 15, qhalf = lane >> 4;  // QKV: column pair qi, rows 2 jj + qhalf
      const int hd = a.head_dim >> 1, qP = (gn0 >> 1) + qi, qhead = hd ? qP / hd : 0, qii = qP - qhead * hd;
      float2 cs[16];
      if (a.epi == EPI_QKV) {
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int jr = 2 * jj + qhalf;
          const int pp = __shfl_sync(0xffffffffu, pos_l, jr);
          cs[jj] = (qhead < a.n_q_heads + a.n_kv_heads && rbase + jr < M) ? a.rope[(size_t)pp * hd + qii]
                                                                          : make_float2(1.f, 0.f);
        }
      }
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(32 * p) << 16) + (uint32_t)(h * kGBN + c0), r);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 32; ++i) stg[lane * 33 + i] = __uint_as_float(r[i]);
      __syncwarp();
      if (a.epi == EPI_QKV) {  // column pairs (2i, 2i+1) of a head are its dims (i, i + D/2)
        const int i = qi, half = qhalf, head = qhead, ii = qii;  // two rows per pass, 16 pairs each
#pragma unroll
        for (int jj = 0; jj < 16; ++jj) {
          const int jr = 2 * jj + half, gm = rbase + jr;
          const int pp = __shfl_sync(0xffffffffu, pos_l, jr), sq = __shfl_sync(0xffffffffu, seq_l, jr);
          if (gm >= M || gn0 + 2 * i >= N) continue;
          const float y0 = stg[jr * 33 + 2 * i], y1 = stg[jr * 33 + 2 * i + 1];
          if (head < a.n_q_heads) {
            float* qo = a.qout + ((size_t)gm * a.n_q_heads + head) * a.head_dim;
            qo[ii] = y0 * cs[jj].x - y1 * cs[jj].y;
            qo[ii + hd] = y1 * cs[jj].x + y0 * cs[jj].y;
          } else {
            const bool is_k = head < a.n_q_heads + a.n_kv_heads;
            const int kvh = head - a.n_q_heads - (is_k ? 0 : a.n_kv_heads);
            const size_t base = (((size_t)sq * a.n_kv_heads + kvh) * a.max_len + pp) * a.head_dim;
            if (is_k) {
              a.kc[base + ii] = __float2half_rn(y0 * cs[jj].x - y1 * cs[jj].y);
              a.kc[base + ii + hd] = __float2half_rn(y1 * cs[jj].x + y0 * cs[jj].y);
            } else {
              a.vc[base + ii] = __float2half_rn(y0);
              a.vc[base + ii + hd] = __float2half_rn(y1);
            }
          }
        }
      } else if (a.epi == EPI_SWIGLU_BF16) {  // columns (2i, 2i+1) are (gate_i, up_i): 16 outputs per row
        const int i = lane & 15, half = lane >> 4;    // two rows per pass, 16 lanes each
        const int go = (gn0 >> 1) + i;
#pragma unroll 4
        for (int j = 0; j < 32; j += 2) {
          const int jr = j + half, gm = rbase + jr;
          const float g = stg[jr * 33 + 2 * i], u = stg[jr * 33 + 2 * i + 1];
          if (gm < M && gn0 + 2 * i < N) a.out_bf16[(size_t)gm * a.ldo_bf16 + go] = __float2bfloat16_rn(silu(g) * u);
        }
      } else {  // EPI_STORE / EPI_RESID
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int gm = rbase + j;
          if (gm >= M || gn >= N) continue;
          float v = stg[j * 33 + lane];
          if (a.epi == EPI_RESID) v = __fadd_rn(rv[j], v);
          a.out[(size_t)gm * a.ldo + gn] = v;
        }
      }
      __syncwarp();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kGTmemCols);
}

// ------------------------------------------------------------------------------------------
// The GEMM of a call of at most kGemmSmallTokens tokens (batched decode, and the readout of
// such a call).  Every weight is read once, so the operands are swapped: A = 128 dequantised
// weight rows (the MMA's M), B = the tokens' activations (N = 64, zero beyond M); D[row][token]
// sits in 64 TMEM columns.  The K range of a weight tile may be split over `splits` CTAs (the
// grid's y), so that projections with few weight tiles still cover the SMs: each writes its
// f32 partial to the workspace, and the last CTA of the tile to arrive adds the partials in
// split order and runs the epilogue (one summation order whatever the arrival order).  Roles
// as in gemm_tc_kernel, with two dequantising threads per weight row (32 of K each).
constexpr int kSN = kGemmSmallRows, kST = kGemmSmallTokens, kSK = 64;
constexpr int kSSA = 4;  // activation stages
constexpr int kSSR = 4;  // raw weight stages of 256 columns (one scale group): 256-byte row runs
constexpr int kSSB = 3;  // dequantised weight buffers of one K step
constexpr uint32_t kSTileW = kSN * kSK * 2;  // 16 KB bf16 weights, 128B-swizzled K-major
constexpr uint32_t kSTileA = kST * kSK * 2;  // 8 KB bf16 activations, 128B-swizzled K-major
constexpr uint32_t kSRawBox = kSN * 128;     // 16 KB int8: 128 columns of the tile's rows, 128B-swizzled
constexpr uint32_t kSRawW = 2 * kSRawBox;    // a raw stage: 256 columns
constexpr uint32_t kSRawS = kSN * 16;        // its 8 fp16 scales per row
constexpr uint32_t kSOffW = 0;                             // dequantised weight buffers
constexpr uint32_t kSOffA = kSOffW + kSSB * kSTileW;       // activation stages
constexpr uint32_t kSOffRW = kSOffA + kSSA * kSTileA;      // raw weight stages
constexpr uint32_t kSOffRS = kSOffRW + kSSR * kSRawW;      // the raw stages' scales
constexpr uint32_t kSOffBar = kSOffRS + kSSR * kSRawS;
constexpr uint32_t kSSmem = kSOffBar + 512 + 1024;         // + barriers, tmem slot, flags, alignment slack
constexpr uint32_t kSTmemCols = 64;

struct SBars {
  uint64_t a_full[kSSA], a_empty[kSSA], r_full[kSSR], r_empty[kSSR];
  uint64_t b_full[kSSB], b_empty[kSSB], acc_full, mma_drain;
};

__global__ void __launch_bounds__(kGThreads, 1)
    gemm_small_kernel(const GemmArgs a, const __grid_constant__ CUtensorMap tA, const __grid_constant__ CUtensorMap tW,
                      const __grid_constant__ CUtensorMap tS, int splits) {
  extern __shared__ unsigned char g_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)g_raw + 1023) & ~(uintptr_t)1023);
  SBars* B = reinterpret_cast<SBars*>(sm + kSOffBar);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(sm + kSOffBar + sizeof(SBars));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + kSOffBar + sizeof(SBars) + 8);
  volatile int* last_flag = abort_flag + 1;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int n0 = blockIdx.x * kSN, split = blockIdx.y;
  const int N = a.w.N, M = a.M;
  // this CTA's K steps: whole scale groups (4 steps of 64) of its split
  const int ng = a.w.Kp / 256;
  const int kt0 = 4 * (int)((long long)split * ng / splits), kt1 = 4 * (int)((long long)(split + 1) * ng / splits);
  const int nk = kt1 - kt0;

  if (tid == 0) {
    for (int i = 0; i < kSSA; ++i) {
      mbar_init(&B->a_full[i], 1);
      mbar_init(&B->a_empty[i], 1);
    }
    for (int i = 0; i < kSSR; ++i) {
      mbar_init(&B->r_full[i], 1);
      mbar_init(&B->r_empty[i], kGDeq);
    }
    for (int i = 0; i < kSSB; ++i) {
      mbar_init(&B->b_full[i], kGDeq);
      mbar_init(&B->b_empty[i], 1);
    }
    mbar_init(&B->acc_full, 1);
    mbar_init(&B->mma_drain, 1);
    *abort_flag = 0;
    *last_flag = 0;
    mbar_fence_init();
  }
  if (warp == 0) {
    tmem_alloc(tmem_slot, kSTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_trigger();

  if (warp == 8) {
    // ---------------- activation loads (the call's tokens, zero beyond M) ----------------
    if (lane == 0) {
      int ia = 0;
      pdl_wait();  // the activations are the previous kernel's output
      for (int i = 0; i < nk; ++i) {
        const int s = i % kSSA;
        if (i >= kSSA && !gwait(&B->a_empty[s], (uint32_t)((i / kSSA) + 1) & 1u, abort_flag, a.err)) break;
        mbar_arrive_expect_tx(&B->a_full[s], kSTileA);
        tma_load_2d(sm + kSOffA + s * kSTileA, &tA, (kt0 + i) * kSK, 0, &B->a_full[s]);
        ++ia;
      }
      if (*abort_flag)  // nothing may still be landing in shared memory when the CTA leaves
        for (int k = max(0, ia - kSSA); k < ia; ++k)
          mbar_wait(&B->a_full[k % kSSA], (uint32_t)(k / kSSA) & 1u, kGDrainNs);
    }
  } else if (warp == 10) {
    // ---------------- weight loads: a raw stage is 256 columns (two swizzled boxes) and their scales ----------------
    if (lane == 0) {
      int ir = 0;
      for (int g = 0; g < nk / 4; ++g) {
        const int r = g % kSSR, kc = (kt0 >> 2) + g;  // the scale group
        if (g >= kSSR && !gwait(&B->r_empty[r], (uint32_t)((g / kSSR) + 1) & 1u, abort_flag, a.err)) break;
        mbar_arrive_expect_tx(&B->r_full[r], kSRawW + kSRawS);
        unsigned char* rw = sm + kSOffRW + r * kSRawW;
        tma_load_2d(rw, &tW, kc * 256, n0, &B->r_full[r]);
        tma_load_2d(rw + kSRawBox, &tW, kc * 256 + 128, n0, &B->r_full[r]);
        tma_load_2d(sm + kSOffRS + r * kSRawS, &tS, kc * 8, n0, &B->r_full[r]);
        ++ir;
      }
      if (*abort_flag)
        for (int k = max(0, ir - kSSR); k < ir; ++k)
          mbar_wait(&B->r_full[k % kSSR], (uint32_t)(k / kSSR) & 1u, kGDrainNs);
    }
  } else if (warp < 8) {
    // ---------------- dequantise: half `hf` (32 of K) of weight row `row` of every tile ----------------
    const int row = tid >> 1, hf = tid & 1;
    constexpr float kBias = 8388736.0f;  // 2^23 + 128 (see gemm_tc_kernel)
    bool go = true;
    for (int g = 0; g < nk / 4 && go; ++g) {
      const int r = g % kSSR;
      if (!gwait(&B->r_full[r], (uint32_t)(g / kSSR) & 1u, abort_flag, a.err)) break;
      const unsigned char* rw = sm + kSOffRW + r * kSRawW;
      const unsigned char* rs = sm + kSOffRS + r * kSRawS;
      for (int u = 0; u < 4; ++u) {  // the K steps of the stage
        const int i = 4 * g + u, bb = i % kSSB;
        if (i >= kSSB && !gwait(&B->b_empty[bb], (uint32_t)((i / kSSB) + 1) & 1u, abort_flag, a.err)) {
          go = false;
          break;
        }
        unsigned char* wt = sm + kSOffW + bb * kSTileW;
        const float sc =
            __half2float(__ushort_as_half(*reinterpret_cast<const uint16_t*>(rs + row * 16 + (2 * u + hf) * 2)));
        const unsigned char* rb = rw + (u >> 1) * kSRawBox + row * 128;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int c = (u & 1) * 4 + hf * 2 + j;  // the 16-byte chunk of the box row (swizzled by row)
          const uint4 w = *reinterpret_cast<const uint4*>(rb + ((c ^ (row & 7)) << 4));
          const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
          uint32_t o[8];
#pragma unroll
          for (int q = 0; q < 4; ++q) {  // two weights per packed subtract and multiply (exact, as above)
            const uint32_t x = wd[q];
            const float2 lo = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7440)),
                                                               __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7441))),
                                                   make_float2(-kBias, -kBias)),
                                        make_float2(sc, sc));
            const float2 hi = __fmul2_rn(__fadd2_rn(make_float2(__uint_as_float(__byte_perm(x, 0x4B000000u, 0x7442)),
                                                               __uint_as_float(__byte_perm(x, 0x4B000000u, 0x7443))),
                                                   make_float2(-kBias, -kBias)),
                                        make_float2(sc, sc));
            o[2 * q] = pack_bf16x2(lo.x, lo.y);
            o[2 * q + 1] = pack_bf16x2(hi.x, hi.y);
          }
          const int col = hf * 32 + j * 16;
          *reinterpret_cast<uint4*>(wt + sw128_offset(row, col)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(wt + sw128_offset(row, col + 8)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_async_smem();  // the bf16 tile is read next by the tensor core (async proxy)
        mbar_arrive(&B->b_full[bb]);
      }
      if (go) mbar_arrive(&B->r_empty[r]);
    }
  } else if (warp == 9) {
    // ---------------- MMA issue: D[128 rows][64 tokens] += W_tile * A_tile^T ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kSN, kST);
      int issued = 0;
      for (int i = 0; i < nk; ++i) {
        const int s = i % kSSA, bb = i % kSSB;
        if (!gwait(&B->a_full[s], (uint32_t)(i / kSSA) & 1u, abort_flag, a.err)) break;
        if (!gwait(&B->b_full[bb], (uint32_t)(i / kSSB) & 1u, abort_flag, a.err)) break;
        tc_fence_after();
        const uint32_t w_base = smem_u32(sm + kSOffW + bb * kSTileW);
        const uint32_t a_base = smem_u32(sm + kSOffA + s * kSTileA);
#pragma unroll
        for (int kk = 0; kk < kSK / 16; ++kk)
          umma_bf16(tmem, desc_sw128(w_base + kk * 32), desc_sw128(a_base + kk * 32), idesc, (i > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&B->a_empty[s]);
        umma_commit(&B->b_empty[bb]);
        ++issued;
      }
      if (issued == nk) {
        umma_commit(&B->acc_full);
      } else if (issued > 0) {  // given up: let the MMAs already issued finish before TMEM is released
        umma_commit(&B->mma_drain);
        mbar_wait(&B->mma_drain, 0u, kGDrainNs);
      }
    }
  }
  __syncthreads();
  if (tid == 0 && !*abort_flag) gwait(&B->acc_full, 0u, abort_flag, a.err);
  __syncthreads();
  const bool ok = !*abort_flag;
  tc_fence_after();
  pdl_wait();  // the epilogue reads the residual / writes outputs the previous kernel may touch

  // ---- epilogue (warps 0-7): warp w holds weight rows n0 + 32 (w % 4) + lane (TMEM lanes) and
  // tokens t0 .. t0 + 31, t0 = 32 (w / 4) (TMEM columns); a store of one token is 32 rows wide ----
  const int row = n0 + 32 * (warp & 3) + lane, t0 = 32 * ((warp >> 2) & 1);
  float v[32];
  if (warp < 8) {
    uint32_t r[32];
    tmem_ld32(tmem + ((uint32_t)(32 * (warp & 3)) << 16) + (uint32_t)t0, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
  }
  bool run = ok;
  if (splits > 1) {
    if (warp < 8 && row < N)
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (t0 + i < M) a.ws[((size_t)split * kST + t0 + i) * N + row] = v[i];
    __syncthreads();  // every partial write, then one acquire-release arrival (no separate fence)
    if (tid == 0) {
      const bool last = atom_add_acq_rel(a.tile_cnt + blockIdx.x, 1u) == (unsigned)splits - 1;
      if (last) a.tile_cnt[blockIdx.x] = 0u;  // every split of the tile has arrived: ready for the next launch
      *last_flag = last;
    }
    __syncthreads();
    run = ok && *last_flag;
    if (run) {
      if (warp < 8 && row < N) {  // split by split, the 32 tokens' partials in flight together
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.f;
        for (int sp = 0; sp < splits; ++sp)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (t0 + i < M) v[i] += __ldcg(a.ws + ((size_t)sp * kST + t0 + i) * N + row);
      }
    }
  }
  if (run && warp < 8) {
    // the tokens' positions and sequences: one load per lane (token t0 + lane), then shuffles
    const int pos_l = (a.epi == EPI_QKV && t0 + lane < M) ? a.pos[t0 + lane] : 0;
    const int seq_l = (a.epi == EPI_QKV && t0 + lane < M) ? a.seq[t0 + lane] : 0;
    if (a.epi == EPI_QKV) {  // rows (2P, 2P+1) of a head are its dims (i, i + D/2): lane pairs
      const int hd = a.head_dim >> 1, P = row >> 1, head = P / hd, ii = P - head * hd;
      const bool rotated = head < a.n_q_heads + a.n_kv_heads;
#pragma unroll 8
      for (int i0 = 0; i0 < 32; i0 += 8) {
        float2 cs[8];  // the RoPE factors of eight tokens, requested together
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int pp = __shfl_sync(0xffffffffu, pos_l, i0 + k);
          cs[k] = (rotated && !(lane & 1) && t0 + i0 + k < M && row < N) ? a.rope[(size_t)pp * hd + ii]
                                                                         : make_float2(1.f, 0.f);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int i = i0 + k;
          const float y0 = v[i], y1 = __shfl_down_sync(0xffffffffu, v[i], 1);
          const int pp = __shfl_sync(0xffffffffu, pos_l, i), sq = __shfl_sync(0xffffffffu, seq_l, i);
          const int t = t0 + i;
          if ((lane & 1) || t >= M || row >= N) continue;
          if (head < a.n_q_heads) {
            float* qo = a.qout + ((size_t)t * a.n_q_heads + head) * a.head_dim;
            qo[ii] = y0 * cs[k].x - y1 * cs[k].y;
            qo[ii + hd] = y1 * cs[k].x + y0 * cs[k].y;
          } else {
            const bool is_k = head < a.n_q_heads + a.n_kv_heads;
            const int kvh = head - a.n_q_heads - (is_k ? 0 : a.n_kv_heads);
            const size_t base = (((size_t)sq * a.n_kv_heads + kvh) * a.max_len + pp) * a.head_dim;
            if (is_k) {
              a.kc[base + ii] = __float2half_rn(y0 * cs[k].x - y1 * cs[k].y);
              a.kc[base + ii + hd] = __float2half_rn(y1 * cs[k].x + y0 * cs[k].y);
            } else {
              a.vc[base + ii] = __float2half_rn(y0);
              a.vc[base + ii + hd] = __float2half_rn(y1);
            }
          }
        }
      }
    } else if (a.epi == EPI_SWIGLU_BF16) {  // rows (2j, 2j+1) are (gate_j, up_j): lane pairs
#pragma unroll 4
      for (int i = 0; i < 32; ++i) {
        const float g = v[i], u = __shfl_down_sync(0xffffffffu, v[i], 1);
        const int t = t0 + i;
        if (!(lane & 1) && t < M && row < N) a.out_bf16[(size_t)t * a.ldo_bf16 + (row >> 1)] = __float2bfloat16_rn(silu(g) * u);
      }
    } else {  // EPI_STORE / EPI_RESID: the residuals of the 32 tokens requested together
      float rv[32];
#pragma unroll
      for (int i = 0; i < 32; ++i)
        rv[i] = (a.epi == EPI_RESID && t0 + i < M && row < N) ? a.resid[(size_t)(t0 + i) * a.ldr + row] : 0.f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int t = t0 + i;
        if (t >= M || row >= N) continue;
        float y = v[i];
        if (a.epi == EPI_RESID) y = __fadd_rn(rv[i], y);
        a.out[(size_t)t * a.ldo + row] = y;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kSTmemCols);
}

cudaError_t prepare_gemm_tc() {
  static_assert(sizeof(GBars) + 16 <= 256, "barrier block");
  static_assert(sizeof(SBars) + 16 <= 512, "barrier block of the small-call GEMM");
  static_assert(kSSmem <= 227 * 1024, "shared memory of the small-call GEMM");
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(gemm_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSSmem);
  return e;
}

int gemm_small_splits(int N, int Kp) {
  // only when the weight tiles alone leave SMs idle: then the split count with the fewest
  // waves of full-K time, ceil(tiles * S / SMs) / S
  const int tiles = (N + kSN - 1) / kSN, ng = Kp / 256, G = std::max(1, sm_count());
  if (tiles >= G) return 1;
  int best = 1;
  double best_cost = (double)((tiles + G - 1) / G);
  for (int S = 2; S <= std::min(8, ng); ++S) {
    const double cost = (double)((tiles * S + G - 1) / G) / S;
    if (cost < best_cost - 1e-9) {
      best = S;
      best_cost = cost;
    }
  }
  return best;
}

size_t gemm_small_ws_bytes(int N, int Kp) {
  const int S = gemm_small_splits(N, Kp);
  return S > 1 ? (size_t)S * kST * (size_t)N * 4 : 0;
}

namespace {
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

}  // namespace

bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
               uint64_t row_bytes, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle sw) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return enc(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st) {
  if (a.M <= 0 || a.w.N <= 0) return cudaSuccess;
  // Kp a multiple of 256 (scale groups of 4 K steps), 16-byte aligned rows and bases
  if (a.w.Kp % 256 || a.lda < a.w.Kp || a.lda % 8 || ((uintptr_t)a.a & 15) || ((uintptr_t)a.w.q & 15) ||
      ((uintptr_t)a.w.s & 15))
    return cudaErrorInvalidValue;
  CUtensorMap tA, tB, tS;
  if (a.M <= kST) {  // a small call: the weight-streaming kernel
    const int S = (a.ws && a.tile_cnt) ? gemm_small_splits(a.w.N, a.w.Kp) : 1;
    if (!encode_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.a, (uint64_t)a.w.Kp, (uint64_t)a.M, (uint64_t)a.lda * 2,
                   kSK, kST, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w.q, (uint64_t)a.w.Kp, (uint64_t)a.w.N, (uint64_t)a.w.Kp,
                   128, kSN, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !encode_2d(&tS, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.w.s, (uint64_t)(a.w.Kp / 32), (uint64_t)a.w.N,
                   (uint64_t)(a.w.Kp / 16), 8, kSN, CU_TENSOR_MAP_SWIZZLE_NONE))
      return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((a.w.N + kSN - 1) / kSN, S);
    cfg.blockDim = dim3(kGThreads);
    cfg.dynamicSmemBytes = kSSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl_enabled() ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, gemm_small_kernel, a, tA, tB, tS, S);
  }
  if (!encode_2d(&tA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, a.a, (uint64_t)a.w.Kp, (uint64_t)a.M, (uint64_t)a.lda * 2,
                 kGBK, kGBM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode_2d(&tB, CU_TENSOR_MAP_DATA_TYPE_UINT8, a.w.q, (uint64_t)a.w.Kp, (uint64_t)a.w.N, (uint64_t)a.w.Kp,
                 kGBK, kGBN, CU_TENSOR_MAP_SWIZZLE_NONE) ||
      !encode_2d(&tS, CU_TENSOR_MAP_DATA_TYPE_UINT16, a.w.s, (uint64_t)(a.w.Kp / 32), (uint64_t)a.w.N,
                 (uint64_t)(a.w.Kp / 16), 8, kGBN, CU_TENSOR_MAP_SWIZZLE_NONE))
    return cudaErrorInvalidValue;
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
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, a, tA, tB, tS);
}

// ------------------------------------------------------------------------------------------
// f32 rows -> bf16 rows (the GEMM operand), with the RMSNorm when gamma is given; the
// reduction order matches the GEMV prologue.

__global__ void rows_to_bf16_kernel(const float* x, int ld_in, int K, const float* gamma, float eps,
                                    __nv_bfloat16* out, int ld_out, const int* rows) {
  __shared__ float nrm[8];
  pdl_trigger();
  pdl_wait();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* xr = x + (size_t)(rows ? rows[t] : t) * ld_in;
  __nv_bfloat16* orow = out + (size_t)t * ld_out;
  // rows of at most 8192 values in 16-byte pieces: each thread keeps its (at most eight) float4
  // pieces in registers between the sum of squares and the output
  constexpr int NV = 8;
  const bool vec = K <= 256 * 4 * NV && ((K | ld_in | ld_out) & 3) == 0 &&
                   !(((uintptr_t)x | (uintptr_t)(gamma ? gamma : x)) & 15) && !((uintptr_t)out & 7);
  float rinv = 1.0f;
  if (vec) {
    const int n4 = K >> 2;
    float4 v[NV];
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int i = tid + 256 * j;
      v[j] = i < n4 ? reinterpret_cast<const float4*>(xr)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
      ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
    }
    if (gamma) {
      ss = warp_sum(ss);
      if (lane == 0) nrm[warp] = ss;
      __syncthreads();
      float tot = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) tot += nrm[w];
      rinv = 1.0f / sqrtf(tot / (float)K + eps);
    }
#pragma unroll
    for (int j = 0; j < NV; ++j) {
      const int i = tid + 256 * j;
      if (4 * i >= ld_out) break;
      float4 y = v[j];
      if (gamma && i < n4) {
        const float4 g = reinterpret_cast<const float4*>(gamma)[i];
        y = make_float4(y.x * rinv * g.x, y.y * rinv * g.y, y.z * rinv * g.z, y.w * rinv * g.w);
      }
      reinterpret_cast<uint2*>(orow)[i] = make_uint2(pack_bf16x2(y.x, y.y), pack_bf16x2(y.z, y.w));
    }
    for (int i = tid + 256 * NV; 4 * i < ld_out; i += 256)  // zero beyond the kept pieces
      reinterpret_cast<uint2*>(orow)[i] = make_uint2(0u, 0u);
    return;
  }
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
  for (int k = tid; k < ld_out; k += 256) {
    float v = 0.f;
    if (k < K) v = gamma ? xr[k] * rinv * gamma[k] : xr[k];
    orow[k] = __float2bfloat16_rn(v);
  }
}

cudaError_t launch_rows_to_bf16(const float* x, int ld_in, int K, const float* gamma, float eps, int ntok,
                                __nv_bfloat16* out, int ld_out, cudaStream_t st, const int* rows) {
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
  return cudaLaunchKernelEx(&cfg, rows_to_bf16_kernel, x, ld_in, K, gamma, eps, out, ld_out, rows);
}

// ------------------------------------------------------------------------------------------
// Causal attention of a prefill call on the tensor cores (mma m16n8k16: fp16 operands, f32
// accumulation).
//
// "41. Many GPUs: tensor, pipeline, expert and data parallelism", section "Ring attention for
// very long contexts": softmax(q k^T / sqrt(D)) v with a running max and sum over tiles of
// positions (the same log-sum-exp recurrence its merge uses), here over the tiles of one
// sequence in order.  A CTA takes 64 query rows -- the G query heads of one KV head for 64 / G
// consecutive tokens of the call -- in four warps of 16 rows; every K/V tile of 64 positions
// it loads serves all of them.  K and V are the fp16 cache as stored; q is rounded to fp16
// once, the probabilities to fp16 per tile, every sum is f32.  Token t attends to positions
// 0..pos[t] of sequence seq[t]; a block that spans two sequences walks each sequence's tiles
// in turn with the other rows masked.  The tokens' own K/V rows are already in the cache.

constexpr int kPR = 64;        // query rows per CTA (four warps of 16)
constexpr int kPT = 64;        // positions per K/V tile
constexpr int kPThreads = 128;

// The q rows are staged over the first K/V buffer: they are read into registers before the
// barrier that opens every sequence's walk, and the walk's first tile lands after it.  68.5 KB
// per CTA: three CTAs per SM (the registers allow three as well).
template <int D>
struct PrefillSmem {
  static constexpr int HROW = D + 8;                       // halves per row: conflict-free ldmatrix
  static constexpr size_t q = (size_t)kPR * HROW * 2;      // q rows, fp16 (over the K/V buffers)
  static constexpr size_t tile = (size_t)kPT * HROW * 2;   // one K or V tile
  static constexpr size_t kv = 2 * 2 * tile;               // [2 buffers][K, V]
  static constexpr size_t total = kv + 2 * kPR * 4;        // + each row's sequence and position
  static_assert(q <= kv, "q staging over the K/V buffers");
};

__device__ __forceinline__ void ldsm_x4(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(smem_u32(p)));
}
// c (16 x 8, f32) += a (16 x 16, fp16, row-major fragments) * b (16 x 8, fp16, column fragments)
__device__ __forceinline__ void mma_16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
               "{%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

// Lane l of a warp holds rows (l / 4) and (l / 4 + 8) of its 16, positions / dims 2 (l % 4) and
// + 1 of every 8-column tile (the accumulator layout of mma m16n8k16).
template <int D, int G>
__global__ void __launch_bounds__(kPThreads) attn_prefill_kernel(const AttnArgs a) {
  using S = PrefillSmem<D>;
  constexpr int QB = kPR / G;          // tokens per CTA
  constexpr int HROW = S::HROW;
  constexpr int KS = D / 16;           // k steps of q k^T
  constexpr int NT = D / 8;            // 8-dim tiles of the output
  constexpr int PN = kPT / 8;          // 8-position tiles of the scores
  extern __shared__ __align__(16) unsigned char ps_raw[];
  __half* kvs = reinterpret_cast<__half*>(ps_raw);          // [buffer][K, V][kPT][HROW]
  __half* qs = kvs;                                           // q rows until the first walk
  int* rseq = reinterpret_cast<int*>(ps_raw + S::kv);         // [kPR] sequence of the row's token (-1: none)
  int* rpos = rseq + kPR;                                      // [kPR] its position
  pdl_trigger();
  pdl_wait();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // the grid runs the blocks of later tokens first (KV head fastest): within a sequence they
  // walk the most tiles, so the last CTAs to start are the shortest ones
  const int kvh = blockIdx.x, t0 = (gridDim.y - 1 - blockIdx.y) * QB;
  // rows r = i * G + g: token t0 + i, query head kvh * G + g; q to fp16
  for (int i = tid; i < kPR * (D / 4); i += kPThreads) {
    const int r = i / (D / 4), c4 = i - r * (D / 4);
    const int t = t0 + r / G, g = r % G;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (t < a.ntok) v = reinterpret_cast<const float4*>(a.q + ((size_t)t * a.Hq + (size_t)kvh * G + g) * D)[c4];
    __half2* dst = reinterpret_cast<__half2*>(qs + r * HROW + 4 * c4);
    dst[0] = __floats2half2_rn(v.x, v.y);
    dst[1] = __floats2half2_rn(v.z, v.w);
  }
  for (int r = tid; r < kPR; r += kPThreads) {
    const int t = t0 + r / G;
    rseq[r] = t < a.ntok ? a.seq[t] : -1;
    rpos[r] = t < a.ntok ? a.pos[t] : -1;
  }
  __syncthreads();
  const int mi = lane >> 3, mr = lane & 7;  // ldmatrix: the matrix and row this lane addresses
  uint32_t qf[KS][4];                       // this warp's 16 q rows as A fragments
#pragma unroll
  for (int ks = 0; ks < KS; ++ks)
    ldsm_x4(qf[ks][0], qf[ks][1], qf[ks][2], qf[ks][3],
            qs + (warp * 16 + mr + (mi & 1) * 8) * HROW + ks * 16 + (mi >> 1) * 8);
  const int ra = warp * 16 + (lane >> 2), rb = ra + 8;
  const int sqa = rseq[ra], sqb = rseq[rb], ppa = rpos[ra], ppb = rpos[rb];
  float o[NT][4];
#pragma unroll
  for (int n = 0; n < NT; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;

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
    const bool owna = sqa == sid, ownb = sqb == sid;
    auto fetch = [&](int p0, int buf) {  // the tile at p0 into buffer buf; rows past the sequence are zero
      const int np = min(kPT, maxpos + 1 - p0);
      __half* tk = kvs + (size_t)buf * 2 * kPT * HROW;
      __half* tv = tk + kPT * HROW;
      for (int i = tid; i < kPT * (D / 8); i += kPThreads) {
        const int r = i / (D / 8), c = i - r * (D / 8);
        if (r < np) {
          cp_async16(tk + r * HROW + c * 8, kb + (size_t)(p0 + r) * D + c * 8);
          cp_async16(tv + r * HROW + c * 8, vb + (size_t)(p0 + r) * D + c * 8);
        } else {
          *reinterpret_cast<uint4*>(tk + r * HROW + c * 8) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(tv + r * HROW + c * 8) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      cp_async_commit();
    };
    __syncthreads();  // the q staging, or the previous walk, is done with the tile buffers
    fetch(0, 0);
    int buf = 0;
    for (int p0 = 0; p0 <= maxpos; p0 += kPT, buf ^= 1) {
      const int np = min(kPT, maxpos + 1 - p0);
      if (p0 + kPT <= maxpos) {
        fetch(p0 + kPT, buf ^ 1);
        cp_async_wait_group<1>();
      } else {
        cp_async_wait_group<0>();
      }
      __syncthreads();  // tile `buf` landed (and its zero rows are written) for every thread
      const __half* tk = kvs + (size_t)buf * 2 * kPT * HROW;
      const __half* tv = tk + kPT * HROW;
      // scores: s[n] is the 16 x 8 tile of positions p0 + 8 n .. + 7
      float sc[PN][4];
#pragma unroll
      for (int n = 0; n < PN; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
#pragma unroll
      for (int n2 = 0; n2 < PN / 2; ++n2)
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t b0, b1, b2, b3;  // K rows [pos][dim] are the column fragments of k^T
          ldsm_x4(b0, b1, b2, b3, tk + (n2 * 16 + mr + (mi >> 1) * 8) * HROW + ks * 16 + (mi & 1) * 8);
          mma_16816(sc[2 * n2], qf[ks], b0, b1);
          mma_16816(sc[2 * n2 + 1], qf[ks], b2, b3);
        }
      // scale, causal mask (own sequence, position in the tile and <= the row's), running max
      float mta = -INFINITY, mtb = -INFINITY;
#pragma unroll
      for (int n = 0; n < PN; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int c = n * 8 + (lane & 3) * 2 + e, p = p0 + c;
          sc[n][e] = (owna && c < np && p <= ppa) ? sc[n][e] * a.scale : -INFINITY;
          sc[n][2 + e] = (ownb && c < np && p <= ppb) ? sc[n][2 + e] * a.scale : -INFINITY;
          mta = fmaxf(mta, sc[n][e]);
          mtb = fmaxf(mtb, sc[n][2 + e]);
        }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {  // the four lanes of a row
        mta = fmaxf(mta, __shfl_xor_sync(0xffffffffu, mta, off));
        mtb = fmaxf(mtb, __shfl_xor_sync(0xffffffffu, mtb, off));
      }
      const float mna = fmaxf(ma, mta), mnb = fmaxf(mb, mtb);
      const float ala = ma == -INFINITY ? 0.f : expf(ma - mna);
      const float alb = mb == -INFINITY ? 0.f : expf(mb - mnb);
      float lsa = 0.f, lsb = 0.f;
#pragma unroll
      for (int n = 0; n < PN; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          sc[n][e] = sc[n][e] == -INFINITY ? 0.f : expf(sc[n][e] - mna);
          sc[n][2 + e] = sc[n][2 + e] == -INFINITY ? 0.f : expf(sc[n][2 + e] - mnb);
          lsa += sc[n][e];
          lsb += sc[n][2 + e];
        }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        lsa += __shfl_xor_sync(0xffffffffu, lsa, off);
        lsb += __shfl_xor_sync(0xffffffffu, lsb, off);
      }
      la = la * ala + lsa;
      lb = lb * alb + lsb;
      ma = mna;
      mb = mnb;
#pragma unroll
      for (int n = 0; n < NT; ++n) {
        o[n][0] *= ala;
        o[n][1] *= ala;
        o[n][2] *= alb;
        o[n][3] *= alb;
      }
      // o += p v: the probabilities of positions 16 k .. + 15 as an A fragment, V through
      // transposed loads (rows [pos][dim] are the row fragments of v)
#pragma unroll
      for (int k = 0; k < PN / 2; ++k) {
        const uint32_t pf[4] = {half2_bits(sc[2 * k][0], sc[2 * k][1]), half2_bits(sc[2 * k][2], sc[2 * k][3]),
                                half2_bits(sc[2 * k + 1][0], sc[2 * k + 1][1]),
                                half2_bits(sc[2 * k + 1][2], sc[2 * k + 1][3])};
#pragma unroll
        for (int n2 = 0; n2 < NT / 2; ++n2) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(b0, b1, b2, b3, tv + (k * 16 + mr + (mi & 1) * 8) * HROW + n2 * 16 + (mi >> 1) * 8);
          mma_16816(o[2 * n2], pf, b0, b1);
          mma_16816(o[2 * n2 + 1], pf, b2, b3);
        }
      }
      __syncthreads();  // the tile is consumed before the buffer is refilled
    }
  }
  // normalise and store
  const int ta = t0 + ra / G, tb = t0 + rb / G;
  if (sqa >= 0 && ta < a.ntok) {
    float* out = a.out + ((size_t)ta * a.Hq + (size_t)kvh * G + ra % G) * D + (lane & 3) * 2;
    const float inv = 1.0f / la;
#pragma unroll
    for (int n = 0; n < NT; ++n) *reinterpret_cast<float2*>(out + n * 8) = make_float2(o[n][0] * inv, o[n][1] * inv);
  }
  if (sqb >= 0 && tb < a.ntok) {
    float* out = a.out + ((size_t)tb * a.Hq + (size_t)kvh * G + rb % G) * D + (lane & 3) * 2;
    const float inv = 1.0f / lb;
#pragma unroll
    for (int n = 0; n < NT; ++n) *reinterpret_cast<float2*>(out + n * 8) = make_float2(o[n][2] * inv, o[n][3] * inv);
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
  cfg.gridDim = dim3(a.Hkv, (a.ntok + QB - 1) / QB);
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

// Prefill-path kernels (sm_103a): the tcgen05 tensor-core GEMM with int8 -> bf16 weight
// dequantisation in shared memory, and the bf16 conversion of activations.
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

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
          "r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
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
#pragma unroll 1
    for (int cc = 0; cc < 4; ++cc) {
      const int c0 = chalf * 128 + cc * 32;
      uint32_t r[32];
      tmem_ld32(tmem + ((uint32_t)(32 * p) << 16) + (uint32_t)(h * kGBN + c0), r);
      tmem_wait_ld();
      const int gn0 = n0 + c0;
#pragma unroll
      for (int i = 0; i < 32; ++i) stg[lane * 33 + i] = __uint_as_float(r[i]);
      __syncwarp();
      const int gn = gn0 + lane;
      if (a.epi == EPI_QKV) {  // column pairs (2i, 2i+1) of a head are its dims (i, i + D/2)
        const int i = lane & 15, half = lane >> 4;  // two rows per pass, 16 pairs each
        const int hd = a.head_dim >> 1, P = (gn0 >> 1) + i, head = P / hd, ii = P - head * hd;
#pragma unroll 2
        for (int j = 0; j < 32; j += 2) {
          const int jr = j + half, gm = rbase + jr;
          if (gm >= M || gn0 + 2 * i >= N) continue;
          const float y0 = stg[jr * 33 + 2 * i], y1 = stg[jr * 33 + 2 * i + 1];
          const int pp = a.pos[gm];
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
#pragma unroll 4
        for (int j = 0; j < 32; ++j) {
          const int gm = rbase + j;
          if (gm >= M || gn >= N) continue;
          float v = stg[j * 33 + lane];
          if (a.epi == EPI_RESID) v = __fadd_rn(a.resid[(size_t)gm * a.ldr + gn], v);
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

cudaError_t prepare_gemm_tc() {
  static_assert(sizeof(GBars) + 16 <= 256, "barrier block");
  return cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
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
}  // namespace

cudaError_t launch_gemm_tc(const GemmArgs& a, cudaStream_t st) {
  if (a.M <= 0 || a.w.N <= 0) return cudaSuccess;
  // Kp a multiple of 256 (scale groups of 4 K steps), 16-byte aligned rows and bases
  if (a.w.Kp % 256 || a.lda < a.w.Kp || a.lda % 8 || ((uintptr_t)a.a & 15) || ((uintptr_t)a.w.q & 15) ||
      ((uintptr_t)a.w.s & 15))
    return cudaErrorInvalidValue;
  CUtensorMap tA, tB, tS;
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
constexpr int kPT = 32;       // positions per K/V tile
constexpr int kPThreads = 256;

template <int D>
struct PrefillSmem {
  static constexpr int QROW = D + 4;    // floats per q / K / V row (bank offset between rows)
  static constexpr int HROW = D + 8;    // halves per raw K/V row (16-byte pad)
  static constexpr int SROW = kPT + 4;  // floats per probability row
  static constexpr size_t q = (size_t)kPR * QROW * 4;
  static constexpr size_t kf = (size_t)kPT * QROW * 4;      // K tile, f32
  static constexpr size_t raw = (size_t)2 * kPT * HROW * 2;  // one raw K + V tile, fp16
  static constexpr size_t p = (size_t)kPR * SROW * 4;
  static constexpr size_t total = q + 2 * kf + 2 * raw + p + 2 * kPR * 4;
};

// Thread (tr, tc) = (tid / 8, tid % 8): query rows tr and tr + 32; scores at positions
// tc + 8 j of a tile; output dims 4 tc + 32 m + e.  K and V tiles are converted to f32 in
// shared memory once (one copy for all threads); the raw fp16 rows of the next tile stream in
// with cp.async meanwhile.
template <int D, int G>
__global__ void __launch_bounds__(kPThreads, 2) attn_prefill_kernel(const AttnArgs a) {
  using S = PrefillSmem<D>;
  constexpr int QB = kPR / G;    // tokens per CTA
  constexpr int NM = D / 32;     // float4 groups of output dims per thread
  extern __shared__ __align__(16) unsigned char ps_raw[];
  float* qs = reinterpret_cast<float*>(ps_raw);
  float* kf = reinterpret_cast<float*>(ps_raw + S::q);
  float* vf = kf + kPT * S::QROW;
  __half* rawb = reinterpret_cast<__half*>(ps_raw + S::q + 2 * S::kf);  // [2 buffers][K, V][kPT][HROW]
  float* pr = reinterpret_cast<float*>(ps_raw + S::q + 2 * S::kf + 2 * S::raw);
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
  const int r0 = tr, r1 = tr + 32;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float4 o0[NM], o1[NM];
#pragma unroll
  for (int m = 0; m < NM; ++m) o0[m] = o1[m] = make_float4(0.f, 0.f, 0.f, 0.f);
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
    auto fetch = [&](int p0, int buf) {  // raw fp16 rows of the tile at p0 into buffer buf
      const int np = min(kPT, maxpos + 1 - p0);
      __half* rk = rawb + (size_t)buf * 2 * kPT * S::HROW;
      __half* rv = rk + kPT * S::HROW;
      for (int i = tid; i < np * (D / 8); i += kPThreads) {
        const int r = i / (D / 8), c = i - r * (D / 8);
        cp_async16(rk + r * S::HROW + c * 8, kb + (size_t)(p0 + r) * D + c * 8);
        cp_async16(rv + r * S::HROW + c * 8, vb + (size_t)(p0 + r) * D + c * 8);
      }
      cp_async_commit();
    };
    __syncthreads();  // the previous walk is done with the raw buffers
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
      __syncthreads();  // raw tile `buf` landed for every thread; the previous f32 tile is consumed
      {  // convert to f32 (rows beyond np are zero)
        const __half* rk = rawb + (size_t)buf * 2 * kPT * S::HROW;
        const __half* rv = rk + kPT * S::HROW;
        for (int i = tid; i < kPT * (D / 8); i += kPThreads) {
          const int r = i / (D / 8), c = i - r * (D / 8);
          float4 k0 = make_float4(0.f, 0.f, 0.f, 0.f), k1 = k0, v0 = k0, v1 = k0;
          if (r < np) {
            const uint4 kk = *reinterpret_cast<const uint4*>(rk + r * S::HROW + c * 8);
            const uint4 vv = *reinterpret_cast<const uint4*>(rv + r * S::HROW + c * 8);
            const float2 a0 = __half22float2(*reinterpret_cast<const __half2*>(&kk.x));
            const float2 a1 = __half22float2(*reinterpret_cast<const __half2*>(&kk.y));
            const float2 a2 = __half22float2(*reinterpret_cast<const __half2*>(&kk.z));
            const float2 a3 = __half22float2(*reinterpret_cast<const __half2*>(&kk.w));
            const float2 b0 = __half22float2(*reinterpret_cast<const __half2*>(&vv.x));
            const float2 b1 = __half22float2(*reinterpret_cast<const __half2*>(&vv.y));
            const float2 b2 = __half22float2(*reinterpret_cast<const __half2*>(&vv.z));
            const float2 b3 = __half22float2(*reinterpret_cast<const __half2*>(&vv.w));
            k0 = make_float4(a0.x, a0.y, a1.x, a1.y);
            k1 = make_float4(a2.x, a2.y, a3.x, a3.y);
            v0 = make_float4(b0.x, b0.y, b1.x, b1.y);
            v1 = make_float4(b2.x, b2.y, b3.x, b3.y);
          }
          *reinterpret_cast<float4*>(kf + r * S::QROW + c * 8) = k0;
          *reinterpret_cast<float4*>(kf + r * S::QROW + c * 8 + 4) = k1;
          *reinterpret_cast<float4*>(vf + r * S::QROW + c * 8) = v0;
          *reinterpret_cast<float4*>(vf + r * S::QROW + c * 8 + 4) = v1;
        }
      }
      __syncthreads();
      // scores of rows r0, r1 at positions tc + 8 j
      float s0[kPT / 8], s1[kPT / 8];
#pragma unroll
      for (int j = 0; j < kPT / 8; ++j) s0[j] = s1[j] = 0.f;
      const float* q0 = qs + r0 * S::QROW;
      const float* q1 = qs + r1 * S::QROW;
#pragma unroll 4
      for (int d = 0; d < D; d += 4) {
        const float4 qa = *reinterpret_cast<const float4*>(q0 + d);
        const float4 qb = *reinterpret_cast<const float4*>(q1 + d);
#pragma unroll
        for (int j = 0; j < kPT / 8; ++j) {
          const float4 kk = *reinterpret_cast<const float4*>(kf + (tc + 8 * j) * S::QROW + d);
          s0[j] = fmaf(qa.x, kk.x, s0[j]);
          s0[j] = fmaf(qa.y, kk.y, s0[j]);
          s0[j] = fmaf(qa.z, kk.z, s0[j]);
          s0[j] = fmaf(qa.w, kk.w, s0[j]);
          s1[j] = fmaf(qb.x, kk.x, s1[j]);
          s1[j] = fmaf(qb.y, kk.y, s1[j]);
          s1[j] = fmaf(qb.z, kk.z, s1[j]);
          s1[j] = fmaf(qb.w, kk.w, s1[j]);
        }
      }
      // causal mask, running max and sum per row (the 8 lanes of a row agree via shuffles)
      float mt0 = -INFINITY, mt1 = -INFINITY;
#pragma unroll
      for (int j = 0; j < kPT / 8; ++j) {
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
      for (int j = 0; j < kPT / 8; ++j) {
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
#pragma unroll
      for (int m = 0; m < NM; ++m) {
        o0[m].x *= al0; o0[m].y *= al0; o0[m].z *= al0; o0[m].w *= al0;
        o1[m].x *= al1; o1[m].y *= al1; o1[m].z *= al1; o1[m].w *= al1;
      }
      for (int p = 0; p < np; ++p) {
        const float w0 = pr[r0 * S::SROW + p], w1 = pr[r1 * S::SROW + p];
        const float* vr = vf + p * S::QROW + 4 * tc;
#pragma unroll
        for (int m = 0; m < NM; ++m) {
          const float4 v = *reinterpret_cast<const float4*>(vr + 32 * m);
          o0[m].x = fmaf(w0, v.x, o0[m].x); o0[m].y = fmaf(w0, v.y, o0[m].y);
          o0[m].z = fmaf(w0, v.z, o0[m].z); o0[m].w = fmaf(w0, v.w, o0[m].w);
          o1[m].x = fmaf(w1, v.x, o1[m].x); o1[m].y = fmaf(w1, v.y, o1[m].y);
          o1[m].z = fmaf(w1, v.z, o1[m].z); o1[m].w = fmaf(w1, v.w, o1[m].w);
        }
      }
    }
  }
  // normalise and store
  const int ta = t0 + r0 / G, tb = t0 + r1 / G;
  if (sq0 >= 0 && ta < a.ntok) {
    float* out = a.out + ((size_t)ta * a.Hq + (size_t)kvh * G + r0 % G) * D + 4 * tc;
    const float inv = 1.0f / l0;
#pragma unroll
    for (int m = 0; m < NM; ++m)
      *reinterpret_cast<float4*>(out + 32 * m) = make_float4(o0[m].x * inv, o0[m].y * inv, o0[m].z * inv, o0[m].w * inv);
  }
  if (sq1 >= 0 && tb < a.ntok) {
    float* out = a.out + ((size_t)tb * a.Hq + (size_t)kvh * G + r1 % G) * D + 4 * tc;
    const float inv = 1.0f / l1;
#pragma unroll
    for (int m = 0; m < NM; ++m)
      *reinterpret_cast<float4*>(out + 32 * m) = make_float4(o1[m].x * inv, o1[m].y * inv, o1[m].z * inv, o1[m].w * inv);
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

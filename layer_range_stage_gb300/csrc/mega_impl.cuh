// Persistent decode of a dense stage (sm_103a): every block of the stage for one token in
// one cooperative launch, one CTA per SM.
//
// What it computes is the decode block loop of "41. Many GPUs: tensor, pipeline, expert
// and data parallelism", section "Pipeline parallelism" (add_norm, attention, add_norm,
// MLP per block, the residual stream carried through), with the split-KV attention merge
// of section "Ring attention for very long contexts".  The arithmetic per weight is the
// dequant-fused dot product of q8dot.cuh.
//
// Why one launch: a batch-1 decode step is a chain of small dependent matrix-vector
// products.  Launched one kernel each, every product pays its own ramp and tail while HBM
// idles, and a successor cannot start streaming until its predecessor's CTAs leave the
// SMs.  Here the weight stream never stops: each warp owns a fixed sequence of weight
// slices (its share of every projection of every block, known before the first
// activation exists) and keeps two of them in flight as bulk copies into shared memory,
// running ahead across phases and blocks; the activations meet the weights at five grid
// barriers per block (six in MoE stages).
//
// Work split of a projection with N rows: a task is a row pair (2t, 2t + 1) -- the pairs the
// RoPE and SwiGLU epilogues need, and for the other projections two rows that share each
// load of the staged input -- cut into P column blocks of at most 2 KB per row; a ring slot
// holds a block's two row pieces side by side.  Task t belongs to warp t mod (warps of the
// grid), so at any moment the grid reads one window of the matrix.  A warp sums its blocks
// in order and reduces with shuffles: every output has one fixed summation order.
//
// MoE stages: the router rows are a phase of the weight stream like the projections (a logit
// per task, written to global memory); after one more grid barrier every CTA ranks all the
// logits itself (top-k with ties to the lower id, softmax over the selected: the same
// arithmetic on the same data, so every CTA picks the same experts), and the gate/up and
// down slices of the selected experts stream in once it is known (the weight stream pauses
// there: those slices depend on the routing).
//
// Grid barrier: a counter that only grows within a launch (release add, acquire polling,
// bounded by time) and is reset by the last CTA to leave.  Every wait is bounded; a CTA
// that runs out of time sets the error word, waits (bounded) for its own copies in flight
// and leaves.

// This header holds the kernel and its device code; kernels_mega.cu instantiates the dense
// kernels and holds the host entry points, kernels_mega_moe.cu the MoE kernels.

#pragma once

#include <algorithm>
#include <cfloat>

#include "common.cuh"
#include "kernels.cuh"
#include "q8dot.cuh"

namespace lrs {
namespace {


constexpr int kMW = 16;                       // warps per CTA
constexpr int kMT = kMW * 32;                 // threads per CTA
constexpr int kDepth = 2;                     // weight slots per warp
constexpr int kSlotQ = 4096;                  // weight bytes per slot
constexpr int kSlotS = kSlotQ / 16;           // scale bytes per slot (one fp16 per 32 weights)
template <int D>
constexpr int attn_tile() { return D == 64 ? 256 : 128; }  // attention positions per tile (64 KB of K + V)
constexpr int kMaxKp = 16384;                 // largest projection input (floats in shared memory)
constexpr uint64_t kWaitNs = 200000000ull;    // bound of every wait: 0.2 s
constexpr size_t kMaxSmem = 227 * 1024;

// shared memory, from a 128-byte aligned base (bulk copies want 16 bytes, float4 16)
constexpr size_t kOffRingQ = 0;
constexpr size_t kOffRingS = kOffRingQ + (size_t)kMW * kDepth * kSlotQ;
constexpr size_t kOffBars = kOffRingS + (size_t)kMW * kDepth * kSlotS;  // kMW*kDepth slot barriers + 1
constexpr size_t kOffRed = kOffBars + 512;                               // 32 floats + flags
constexpr size_t kOffMoe = kOffRed + 512;                                 // routing (MoE stages)
constexpr int kMaxExperts = 256, kMaxTopK = 32;
constexpr size_t kOffLogits = kOffMoe, kOffIds = kOffLogits + kMaxExperts * 4, kOffWts = kOffIds + kMaxTopK * 4,
                 kOffSel = kOffWts + kMaxTopK * 4, kOffSelId = kOffSel + kMaxTopK * 4,
                 kOffReady = kOffSelId + kMaxTopK * 4;
constexpr size_t kOffSplit = kOffMoe + (kMaxExperts + 4 * kMaxTopK + 4) * 4;  // [kPhases] Split
constexpr size_t kOffWptr = kOffSplit + 224;                               // [kMW][2] stream pointers
// the phases of a block's weight stream
constexpr int kPhQKV = 0, kPhO = 1, kPhRouter = 2, kPhGU = 3, kPhDown = 4, kPhases = 5;
constexpr size_t kOffXraw = kOffMoe + 2048;                               // [Kp(H)] floats

__host__ __device__ constexpr int pad256(int k) { return (k + 255) / 256 * 256; }

template <int D, int G>
struct AttnLayout {
  static constexpr int T = attn_tile<D>();
  // PV step: a thread takes one dim pair of HPV heads (head group) over one position group
  static constexpr int HPV = G < 4 ? G : 4, NHG = G / HPV, PG = kMT / (D / 2 * NHG);
  static constexpr size_t ks = 0;                                // K tile [T][D] fp16
  static constexpr size_t vs = ks + (size_t)T * D * 2;           // V tile [T][D] fp16
  static constexpr size_t qs = vs + (size_t)T * D * 2;           // q [G][D] f32 (see q_slot)
  static constexpr size_t sc = qs + (size_t)G * D * 4;           // scores [G][T]
  static constexpr size_t pt = sc + (size_t)G * T * 4;           // probabilities [T][G]
  static constexpr size_t st = pt + (size_t)T * G * 4;           // m, l, alpha, merged sum [4][G]
  static constexpr size_t total = st + (size_t)4 * G * 4;
  // after the tiles of an item: the PV partial sums of the position groups [PG][G][D] over the
  // K/V tiles.  Merge: (m, l) [G][64] and chunk weights [64][G] over q and the scores; this
  // CTA's slice of every chunk partial [n_chunks][ceil(G * D / n_chunks)] over the K/V tiles
  static constexpr size_t mls = qs;
  static constexpr size_t wts = qs + (size_t)G * 64 * 8;
  static_assert(wts + (size_t)64 * G * 4 <= st, "merge scratch");
  static_assert((size_t)(G * D + 64) * 4 <= (size_t)2 * T * D * 2, "merge slice scratch over the K/V tiles");
  static_assert((size_t)PG * G * D * 4 <= (size_t)2 * T * D * 2, "PV partial sums over the K/V tiles");
};

// Where dim d of a head's q sits in shared memory: per 8-dim chunk j the low four dims at
// 4 j, the high four at D / 2 + 4 j, so that 8 lanes reading 8 consecutive chunks touch 8
// consecutive 16-byte words (one shared-memory wavefront).
template <int D>
__device__ __forceinline__ int q_slot(int d) {
  return ((d & 4) ? D / 2 : 0) + ((d >> 3) << 2) + (d & 3);
}

__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// How a projection is dealt over the grid.  Rows go in pairs (2P, 2P + 1): the pairs the RoPE
// and SwiGLU epilogues need, and for the other projections two rows that share each load of
// the staged input.  CTA c owns pairs [p0, p0 + np) with p0 = c * NP / G, so every CTA holds
// the same number of pairs to within one.  Inside a CTA the pairs' K ranges are laid end to end
// (np * Kp columns) and cut into 16 contiguous warp ranges of whole 256-column units, so a
// warp may hold the tail of one pair, some whole pairs and the head of another; each warp sums
// its pieces, and after the phase the CTA adds, per pair, the pieces of the warps that hold
// it in warp order -- one fixed summation order per output.
struct Split {
  int NP;    // pairs of the projection
  int Kp;    // columns of a pair's K range (mode 2: top_k expert pieces of PS columns)
  int seg;   // columns between source discontinuities (Kp, or PS in mode 2)
  int mode;  // 0 plain rows; 1 rows of the selected experts (rps rows each); 2 piece j of a row
             // from selected expert j (K gathered over the experts)
  int rps;
  int p0, np;  // this CTA's pairs: p0 + i * pstride for i < np
  int pstride;
  int upp;     // units (256 columns) of a pair: Kp / 256
  int U;       // this CTA's units: np * upp
};

constexpr int kUnit = 256;             // columns of a unit (warp ranges and segments are whole units)
constexpr int kSlotCols = kSlotQ / 2;  // columns of each row in a ring slot
constexpr int kMaxPieces = 16;         // pairs a warp's range may touch in one projection
constexpr int kMaxCtaPairs = 256;      // pairs a CTA may hold in one projection
// per-projection scratch after the staged input: warp partials, piece counters, the warp
// ranges, the RoPE factors of the CTA's QKV pairs
constexpr size_t kPsPart = 0, kPsCnt = kPsPart + (size_t)kMW * kMaxPieces * 8, kPsWu0 = kPsCnt + kMaxCtaPairs * 4,
                 kPsPf = kPsWu0 + 128, kPsRope = kPsPf + 128, kPsBytes = kPsRope + (size_t)kMaxCtaPairs * 8;

// A position in a warp's range of one projection: CTA-local pair pr, column k of the pair, ks =
// column within its source segment, and the columns of the range still to go.  The issuer and
// the consumer of a warp's ring walk the same sequence of cursors, so a slot's contents never
// have to be written down.
struct Cur {
  int pr, k, ks, left;
};

// The weight stream of one warp: block l, projection ph, the cursor of the next slot, and the
// counts of slots issued and consumed.
struct Stream {
  int l, ph;
  Cur q;
  int issued, consumed;
};

// Everything in shared memory is at a fixed offset from one base (no pointer per region
// kept in registers).
struct Ctx {
  const MegaArgs* a;
  unsigned char* sm;
  unsigned char* ps;  // per-projection scratch after the staged input (see kPs*)
  int lane, warp;
  // [kMW][kMaxPieces] partial sums (rows 2P, 2P + 1) of pairs split between warps
  __device__ float2* part() const { return reinterpret_cast<float2*>(ps + kPsPart); }
  __device__ int* cnt() const { return reinterpret_cast<int*>(ps + kPsCnt); }     // [kMaxCtaPairs] pieces done
  __device__ int* wu0() const { return reinterpret_cast<int*>(ps + kPsWu0); }     // [kMW + 1] first unit of each warp
  __device__ int* pf() const { return reinterpret_cast<int*>(ps + kPsPf); }       // [kMW] first pair of each warp
  __device__ float2* rope_s() const { return reinterpret_cast<float2*>(ps + kPsRope); }  // [kMaxCtaPairs] (QKV)
  __device__ unsigned char* ringq() const { return sm + kOffRingQ; }
  __device__ unsigned char* rings() const { return sm + kOffRingS; }
  __device__ uint64_t* bars() const { return reinterpret_cast<uint64_t*>(sm + kOffBars); }  // [kMW][kDepth], attention
  __device__ float* red() const { return reinterpret_cast<float*>(sm + kOffRed); }          // [32] reduction scratch
  __device__ volatile int* flag() const {  // [0] error seen by this CTA, [1] last-arriver flag
    return reinterpret_cast<volatile int*>(sm + kOffRed + 256);
  }
  __device__ float* logits() const { return reinterpret_cast<float*>(sm + kOffLogits); }  // [n_experts] (MoE)
  __device__ int* moe_ids() const { return reinterpret_cast<int*>(sm + kOffIds); }        // [top_k] selected experts
  __device__ float* moe_wts() const { return reinterpret_cast<float*>(sm + kOffWts); }    // [top_k] their weights
  __device__ float* sel() const { return reinterpret_cast<float*>(sm + kOffSel); }        // [top_k] ranking scratch
  __device__ int* sel_id() const { return reinterpret_cast<int*>(sm + kOffSelId); }
  __device__ volatile int* moe_ready() const {  // last block whose routing is known
    return reinterpret_cast<volatile int*>(sm + kOffReady);
  }
  __device__ const Split* split() const { return reinterpret_cast<const Split*>(sm + kOffSplit); }  // [kPhases]
  // [kMW][2] weights and scales of each warp's stream cursor (l, ph): an issue reads them
  // here, not from the block descriptor
  __device__ const void** wptr() const { return reinterpret_cast<const void**>(sm + kOffWptr); }
};

// The projections of a block: weights of phase ph.
template <bool MOE>
__device__ __forceinline__ const DevQ8& phase_w(const MegaLayer& L, int ph) {
  if (MOE && ph == kPhRouter) return L.router;
  if (MOE && ph >= kPhGU) return ph == kPhGU ? L.egu : L.edown;
  return ph == kPhQKV ? L.wqkv : ph == kPhO ? L.wo : ph == kPhGU ? L.wgu : L.wdown;
}

// ph: kPhQKV, kPhO, kPhRouter (MoE stages: one logit per row, into global memory), kPhGU
// (dense, or the selected experts' rows), kPhDown (dense, or gathered over the experts).
// Computed once per launch (from block 0: every block has the same shapes).
__device__ Split split_of(const MegaArgs& a, int ph, int cta, int G) {
  const MegaLayer& L = a.layers[0];
  const bool moe = a.n_experts > 0;
  Split p;
  p.mode = 0;
  p.rps = 0;
  if (ph == kPhRouter && !moe) {  // dense stages: no router rows
    p.NP = 0;
    p.Kp = p.seg = kUnit;
  } else {
    const DevQ8& w = moe ? phase_w<true>(L, ph) : phase_w<false>(L, ph);
    int N = w.N;
    p.Kp = p.seg = w.Kp;
    if (moe && ph == kPhGU) {
      N = a.top_k * 2 * a.EF;
      p.mode = 1;
      p.rps = 2 * a.EF;
    } else if (moe && ph == kPhDown) {
      N = a.H;
      p.mode = 2;
      p.Kp = a.top_k * w.Kp;
    }
    p.NP = N / 2;
  }
  p.p0 = (int)((long long)cta * p.NP / G);
  p.pstride = 1;
  p.np = (int)((long long)(cta + 1) * p.NP / G) - p.p0;
  p.upp = p.Kp / kUnit;
  p.U = p.np * p.upp;
  return p;
}

// Units [u0, u1) of warp w in a projection.
__device__ __forceinline__ int warp_u0(const Split& p, int w) { return w * p.U / kMW; }

// The cursor at the start of warp w's range in projection p.
__device__ __forceinline__ Cur cur_start(const Split& p, int w) {
  const int u0 = warp_u0(p, w), u1 = warp_u0(p, w + 1);
  Cur q;
  q.pr = u0 / p.upp;
  q.k = (u0 - q.pr * p.upp) * kUnit;
  q.ks = q.k % p.seg;
  q.left = (u1 - u0) * kUnit;
  return q;
}

// Columns of the slot at q: to the end of the range, of the pair or of the source segment, at
// most kSlotCols.
__device__ __forceinline__ int cur_len(const Split& p, const Cur& q) {
  return min(min(q.left, kSlotCols), min(p.Kp - q.k, p.seg - q.ks));
}

__device__ __forceinline__ void cur_advance(const Split& p, Cur& q, int len) {
  q.left -= len;
  q.k += len;
  q.ks += len;
  if (q.ks == p.seg) q.ks = 0;
  if (q.k == p.Kp) {
    q.k = 0;
    q.ks = 0;
    ++q.pr;
  }
}

// Global addresses of rows (2P, 2P + 1) of a projection at column k (P phase-global).
template <bool MOE>
__device__ __forceinline__ void pair_src(const Ctx& c, const Split& p, const uint8_t* wq, const uint16_t* ws, int P,
                                         int k, int kk, const uint8_t*& q, const uint16_t*& sc, size_t& qstride,
                                         size_t& sstride) {
  if (MOE && p.mode == 2) {  // K gathered: columns [j PS, (j + 1) PS) from selected expert j; kk = k % PS
    const int j = (k - kk) / p.seg;
    const size_t r = (size_t)c.moe_ids()[j] * (size_t)(2 * p.NP) + 2 * P;
    q = wq + r * p.seg + kk;
    sc = ws + r * (p.seg / 32) + kk / 32;
    qstride = p.seg;
    sstride = p.seg / 32;
    return;
  }
  size_t r = 2 * (size_t)P;
  if (MOE && p.mode == 1) r = (size_t)c.moe_ids()[2 * P / p.rps] * p.rps + (2 * P) % p.rps;
  q = wq + r * p.Kp + k;
  sc = ws + r * (p.Kp / 32) + k / 32;
  qstride = p.Kp;
  sstride = p.Kp / 32;
}

// Move a cursor to the first non-empty warp range at or after (l, ph).
template <bool MOE>
__device__ __forceinline__ void stream_normalise(const Ctx& c, Stream& s) {
  bool moved = false;
  while (s.l < c.a->nl && s.q.left == 0) {
    if (++s.ph == kPhases) {
      s.ph = 0;
      ++s.l;
    }
    s.q = cur_start(c.split()[s.ph], c.warp);
    moved = true;
  }
  if (moved && s.l < c.a->nl && c.lane == 0) {
    const DevQ8& w = phase_w<MOE>(c.a->layers[s.l], s.ph);
    c.wptr()[2 * c.warp] = w.q;
    c.wptr()[2 * c.warp + 1] = w.s;
  }
  __syncwarp();
}

// Issue the next slot of this warp's stream (if any) into the ring: cur_len columns of one pair
// from the cursor, row 2P's bytes at the start of the slot and row 2P + 1's at kSlotCols.
// Slices of the selected experts wait until the routing of their block is known.
template <bool MOE>
__device__ __forceinline__ void stream_issue(const Ctx& c, Stream& s) {
  if (s.l >= c.a->nl) return;
  if (MOE && s.ph >= kPhGU && s.l > *c.moe_ready()) return;
  const Split& p = c.split()[s.ph];
  const int slot = s.issued % kDepth;
  const int len = cur_len(p, s.q);
  if (c.lane == 0) {
    const uint8_t* q;
    const uint16_t* sc;
    size_t qst, sst;
    pair_src<MOE>(c, p, static_cast<const uint8_t*>(c.wptr()[2 * c.warp]),
                  static_cast<const uint16_t*>(c.wptr()[2 * c.warp + 1]), p.p0 + s.q.pr * p.pstride, s.q.k, s.q.ks,
                  q, sc, qst, sst);
    uint64_t* bar = c.bars() + c.warp * kDepth + slot;
    unsigned char* dq = c.ringq() + (size_t)(c.warp * kDepth + slot) * kSlotQ;
    unsigned char* ds = c.rings() + (size_t)(c.warp * kDepth + slot) * kSlotS;
    fence_async_smem();  // the slot's previous contents were read through the generic proxy
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * (len + len / 16)));
    bulk_g2s(dq, q, (uint32_t)len, bar);
    bulk_g2s(dq + kSlotCols, q + qst, (uint32_t)len, bar);
    bulk_g2s(ds, sc, (uint32_t)(len / 16), bar);
    bulk_g2s(ds + kSlotCols / 16, sc + sst, (uint32_t)(len / 16), bar);
  }
  ++s.issued;
  cur_advance(p, s.q, len);
  if (s.q.left == 0) stream_normalise<MOE>(c, s);
}

// Top the ring up to kDepth slots (after the routing of a block became known).
template <bool MOE>
__device__ __forceinline__ void stream_refill(const Ctx& c, Stream& s) {
  while (s.issued - s.consumed < kDepth && s.l < c.a->nl) {
    const int before = s.issued;
    stream_issue<MOE>(c, s);
    if (s.issued == before) break;
  }
}

// After a failed wait: wait (bounded) for this warp's copies still in flight.
__device__ void stream_drain(const Ctx& c, Stream& s) {
  for (int k = s.consumed; k < s.issued; ++k)
    mbar_wait(c.bars() + c.warp * kDepth + k % kDepth, (unsigned)(k / kDepth) & 1u, kWaitNs);
  s.consumed = s.issued;
}

__device__ __forceinline__ void set_error(const Ctx& c) {
  atomicExch(c.a->err, 1);
  c.flag()[0] = 1;
}

// Grid barrier number `k` (1-based) of this launch; false when the wait ran out.
__device__ bool grid_barrier(const Ctx& c, unsigned k) {
  __syncthreads();
  if (threadIdx.x == 0 && !c.flag()[0]) {
    const unsigned target = k * gridDim.x + c.a->bar_extra;
    red_release_add(c.a->bar, 1u);
    if (ld_acquire_u32(c.a->bar) < target) {
      const uint64_t t0 = global_ns();
      while (ld_acquire_u32(c.a->bar) < target)
        if (global_ns() - t0 > kWaitNs) {
          set_error(c);
          break;
        }
    }
  }
  __syncthreads();
  return !c.flag()[0];
}

// Leaving: the last CTA out resets the barrier counters for the next launch (every CTA has
// stopped polling by the time it counts itself out).
__device__ void grid_leave(const Ctx& c) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(c.a->bar + 1, 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(c.a->bar, 0u);
      for (int h = 0; h < c.a->Hkv; ++h) atomicExch(c.a->bar + 2 + h, 0u);
      atomicExch(c.a->bar + 1, 0u);
    }
  }
}

// A projection input from global memory (written earlier in this launch: read through L2)
// into shared memory: normalised by RMSNorm with gamma when given, scaled by 2^64,
// swizzled per 16-float chunk, with chunk sums.  With gamma the raw values land in xraw
// (kept for the residual adds) and gamma in xs, which is then overwritten in place; without,
// the raw values land in xs.  Every 16-byte piece is an asynchronous copy issued before any
// is waited for (stage_finish), so the staging costs one round trip to L2 and no registers.
__device__ void stage_issue(const float* x, int K, int Kp, const float* gamma, float* xs, float* xraw) {
  const int tid = threadIdx.x;
  float* raw = gamma ? xraw : xs;
  for (int i = tid; i < (Kp >> 2); i += kMT) {  // K is a multiple of 4: a piece lies wholly inside or outside
    if (4 * i < K) {
      cp_async16(raw + 4 * i, x + 4 * i);
      if (gamma) cp_async16(xs + 4 * i, gamma + 4 * i);
    } else {
      reinterpret_cast<float4*>(raw)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (gamma) reinterpret_cast<float4*>(xs)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
}

// The second half of the staging (after stage_issue and any other loads of the phase's setup):
// wait for the copies, then RMSNorm, scaling, swizzle and chunk sums in place.
__device__ void stage_finish(const Ctx& c, int K, int Kp, const float* gamma, float eps, float* xs, float* xc,
                             float* xraw) {
  const int tid = threadIdx.x, nchunk = Kp >> 4;
  const float* raw = gamma ? xraw : xs;
  cp_async_wait_all();
  __syncthreads();
  float rinv = 1.0f;
  if (gamma) {
    float ss = 0.f;
    for (int i = tid; i < (K >> 2); i += kMT) {
      const float4 v = reinterpret_cast<const float4*>(xraw)[i];
      ss = fmaf(v.x, v.x, ss);
      ss = fmaf(v.y, v.y, ss);
      ss = fmaf(v.z, v.z, ss);
      ss = fmaf(v.w, v.w, ss);
    }
    ss = warp_sum(ss);
    if (c.lane == 0) c.red()[c.warp] = ss;
    __syncthreads();
    float tot = 0.f;
#pragma unroll
    for (int w = 0; w < kMW; ++w) tot += c.red()[w];
    rinv = 1.0f / sqrtf(tot / (float)K + eps);
  }
  for (int ch = tid; ch < nchunk; ch += kMT) {
    float h[16];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 v = reinterpret_cast<const float4*>(raw)[ch * 4 + j];
      h[4 * j] = v.x;
      h[4 * j + 1] = v.y;
      h[4 * j + 2] = v.z;
      h[4 * j + 3] = v.w;
      if (gamma) {
        const float4 g = reinterpret_cast<const float4*>(xs)[ch * 4 + j];
        h[4 * j] = h[4 * j] * rinv * g.x;
        h[4 * j + 1] = h[4 * j + 1] * rinv * g.y;
        h[4 * j + 2] = h[4 * j + 2] * rinv * g.z;
        h[4 * j + 3] = h[4 * j + 3] * rinv * g.w;
      }
    }
    float sum = 0.f;
#pragma unroll
    for (int j = 0; j < 16; ++j) sum += h[j];
    const int sw = (ch >> 1) & 3;
    float* xp = xs + ch * 16;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      reinterpret_cast<float4*>(xp)[j ^ sw] =
          make_float4(h[4 * j] * kXScale, h[4 * j + 1] * kXScale, h[4 * j + 2] * kXScale, h[4 * j + 3] * kXScale);
    xc[ch] = sum;
  }
  __syncthreads();
}

// Both rows of a 16-weight chunk against one 16-float chunk of the staged input: the sums
// b_j x'_j 2^-149 of q8dot.cuh, each over two independent pairs of packed products (depth 4).
__device__ __forceinline__ void dot16x2(const uint4 wa, const uint4 wb, const float4 x0, const float4 x1,
                                        const float4 x2, const float4 x3, float& da, float& db) {
  const float2 xa0 = make_float2(x0.x, x0.y), xb0 = make_float2(x0.z, x0.w);
  const float2 xa1 = make_float2(x1.x, x1.y), xb1 = make_float2(x1.z, x1.w);
  const float2 xa2 = make_float2(x2.x, x2.y), xb2 = make_float2(x2.z, x2.w);
  const float2 xa3 = make_float2(x3.x, x3.y), xb3 = make_float2(x3.z, x3.w);
  float2 a0 = __fmul2_rn(make_float2(q8_b0(wa.x), q8_b1(wa.x)), xa0);
  float2 a1 = __fmul2_rn(make_float2(q8_b2(wa.x), q8_b3(wa.x)), xb0);
  float2 b0 = __fmul2_rn(make_float2(q8_b0(wb.x), q8_b1(wb.x)), xa0);
  float2 b1 = __fmul2_rn(make_float2(q8_b2(wb.x), q8_b3(wb.x)), xb0);
  a0 = __ffma2_rn(make_float2(q8_b0(wa.y), q8_b1(wa.y)), xa1, a0);
  a1 = __ffma2_rn(make_float2(q8_b2(wa.y), q8_b3(wa.y)), xb1, a1);
  b0 = __ffma2_rn(make_float2(q8_b0(wb.y), q8_b1(wb.y)), xa1, b0);
  b1 = __ffma2_rn(make_float2(q8_b2(wb.y), q8_b3(wb.y)), xb1, b1);
  a0 = __ffma2_rn(make_float2(q8_b0(wa.z), q8_b1(wa.z)), xa2, a0);
  a1 = __ffma2_rn(make_float2(q8_b2(wa.z), q8_b3(wa.z)), xb2, a1);
  b0 = __ffma2_rn(make_float2(q8_b0(wb.z), q8_b1(wb.z)), xa2, b0);
  b1 = __ffma2_rn(make_float2(q8_b2(wb.z), q8_b3(wb.z)), xb2, b1);
  a0 = __ffma2_rn(make_float2(q8_b0(wa.w), q8_b1(wa.w)), xa3, a0);
  a1 = __ffma2_rn(make_float2(q8_b2(wa.w), q8_b3(wa.w)), xb3, a1);
  b0 = __ffma2_rn(make_float2(q8_b0(wb.w), q8_b1(wb.w)), xa3, b0);
  b1 = __ffma2_rn(make_float2(q8_b2(wb.w), q8_b3(wb.w)), xb3, b1);
  da = (a0.x + a0.y) + (a1.x + a1.y);
  db = (b0.x + b0.y) + (b1.x + b1.y);
}

// The epilogue of pair i (CTA-local) of projection ph of block l, from its row sums.
template <bool MOE>
__device__ __forceinline__ void epilogue_pair(const Ctx& c, int l, int ph, int i, float y0, float y1,
                                              const float* xraw, int pos, int sid) {
  const MegaArgs& a = *c.a;
  const Split& p = c.split()[ph];
  const int t = p.p0 + i * p.pstride;  // the pair, projection-wide
  if (ph == kPhQKV) {  // rows (2t, 2t+1) are dims (j, j + D/2) of one head: RoPE, then q or fp16 K/V
    const int hd = a.D >> 1, head = t / hd, j = t - head * hd;
    if (head < a.Hq) {
      const float2 cs = c.rope_s()[i];
      float* qo = a.qbuf + (size_t)head * a.D;
      qo[j] = y0 * cs.x - y1 * cs.y;
      qo[j + hd] = y1 * cs.x + y0 * cs.y;
    } else {
      const bool is_k = head < a.Hq + a.Hkv;
      const int kvh = head - a.Hq - (is_k ? 0 : a.Hkv);
      const MegaLayer& L = a.layers[l];
      const size_t base = (((size_t)sid * a.Hkv + kvh) * a.max_len + pos) * a.D;
      if (is_k) {
        const float2 cs = c.rope_s()[i];
        L.kc[base + j] = __float2half_rn(y0 * cs.x - y1 * cs.y);
        L.kc[base + j + hd] = __float2half_rn(y1 * cs.x + y0 * cs.y);
      } else {
        L.vc[base + j] = __float2half_rn(y0);
        L.vc[base + j + hd] = __float2half_rn(y1);
      }
    }
  } else if (ph == kPhO) {
    a.x1[2 * t] = __fadd_rn(xraw[2 * t], y0);
    a.x1[2 * t + 1] = __fadd_rn(xraw[2 * t + 1], y1);
  } else if (MOE && ph == kPhRouter) {
    a.logits[2 * t] = y0;
    a.logits[2 * t + 1] = y1;
  } else if (ph == kPhGU) {
    if (MOE) {  // pair t: expert slot t / EF, unit t % EF; scaled by the routing weight
      const int slot = t / a.EF, j = t - slot * a.EF;
      a.abuf[(size_t)slot * pad256(a.EF) + j] = silu(y0) * y1 * c.moe_wts()[slot];
    } else {
      a.abuf[t] = silu(y0) * y1;
    }
  } else {
    a.hout[2 * t] = __fadd_rn(xraw[2 * t], y0);
    a.hout[2 * t + 1] = __fadd_rn(xraw[2 * t + 1], y1);
  }
}

// This warp's piece of pair i (CTA-local) is summed.  A pair held by one warp goes straight to
// its epilogue; a pair split between warps is finished by the warp whose piece completes it
// (a shared-memory counter per pair): it adds the warps' pieces in a fixed order -- a tree over
// the 16 warp slots, absent warps contributing zero -- so every output has one summation order
// whichever warp finishes it.
template <bool MOE>
__device__ __forceinline__ void finish_piece(const Ctx& c, int l, int ph, int i, int pfirst, float acc0, float acc1,
                                             const float* xraw, int pos, int sid) {
  const Split& p = c.split()[ph];
  acc0 = warp_sum(acc0);
  acc1 = warp_sum(acc1);
  const int ua = i * p.upp, ub = ua + p.upp;
  bool holds = false;
  if (c.lane < kMW) {
    const int w0 = c.wu0()[c.lane], w1 = c.wu0()[c.lane + 1];
    holds = w0 < w1 && w0 < ub && w1 > ua;
  }
  const int nw = __popc(__ballot_sync(0xffffffffu, holds));
  float y0 = acc0, y1 = acc1;
  if (nw > 1) {
    int done = 0;
    if (c.lane == 0) {
      c.part()[c.warp * kMaxPieces + i - pfirst] = make_float2(acc0, acc1);
      __threadfence_block();
      done = atomicAdd(c.cnt() + i, 1);
    }
    done = __shfl_sync(0xffffffffu, done, 0);
    if (done != nw - 1) return;  // another warp's piece completes the pair
    __threadfence_block();
    float2 v = make_float2(0.f, 0.f);
    if (holds) v = c.part()[c.lane * kMaxPieces + i - c.pf()[c.lane]];
#pragma unroll
    for (int o = kMW / 2; o > 0; o >>= 1) {
      v.x += __shfl_xor_sync(0xffffffffu, v.x, o);
      v.y += __shfl_xor_sync(0xffffffffu, v.y, o);
    }
    y0 = v.x;
    y1 = v.y;
  }
  if (c.lane == 0) epilogue_pair<MOE>(c, l, ph, i, y0, y1, xraw, pos, sid);
}

// The per-projection scratch of phase ph: piece counters, warp ranges and (QKV) the RoPE factors
// of the CTA's q and k pairs.  A CTA barrier must follow before the projection.
__device__ void phase_setup(const Ctx& c, int ph, int pos) {
  const MegaArgs& a = *c.a;
  const Split& p = c.split()[ph];
  const int tid = threadIdx.x;
  for (int i = tid; i < p.np; i += kMT) c.cnt()[i] = 0;
  if (tid <= kMW) c.wu0()[tid] = tid * p.U / kMW;
  if (tid < kMW) c.pf()[tid] = tid * p.U / kMW / p.upp;
  if (ph == kPhQKV) {
    const int hd = a.D >> 1;
    for (int i = tid; i < p.np; i += kMT) {
      const int t = p.p0 + i * p.pstride, head = t / hd;
      if (head < a.Hq + a.Hkv) c.rope_s()[i] = __ldg(a.rope + (size_t)pos * hd + (t - head * hd));
    }
  }
}

// One projection of block l: consume this warp's range from the ring, refilling behind; each
// finished pair piece goes to finish_piece.  Returns false (for the whole warp) after a
// timed-out wait (error set, copies drained); the caller makes the outcome CTA-uniform.
template <bool MOE>
__device__ bool gemv_phase(const Ctx& c, Stream& s, int l, int ph, const float* xs, const float* xc,
                           const float* xraw, int pos, int sid) {
  const Split& p = c.split()[ph];
  Cur q = cur_start(p, c.warp);
  const int pfirst = q.pr;
  float acc0 = 0.f, acc1 = 0.f;
  int cur = -1;
  while (q.left > 0) {
    const int slot = s.consumed % kDepth;
    const bool landed = mbar_wait(c.bars() + c.warp * kDepth + slot, (unsigned)(s.consumed / kDepth) & 1u, kWaitNs);
    if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform decision
      if (c.lane == 0) set_error(c);
      stream_drain(c, s);
      return false;
    }
    const unsigned char* sq = c.ringq() + (size_t)(c.warp * kDepth + slot) * kSlotQ;
    const unsigned char* ss = c.rings() + (size_t)(c.warp * kDepth + slot) * kSlotS;
    const int len = cur_len(p, q), k = q.k;
    {
      if (q.pr != cur) {
        if (cur >= 0) finish_piece<MOE>(c, l, ph, cur, pfirst, acc0, acc1, xraw, pos, sid);
        acc0 = acc1 = 0.f;
        cur = q.pr;
      }
      const unsigned char* q0 = sq;
      const unsigned char* q1 = q0 + kSlotCols;
      const unsigned char* s0 = ss;
      const unsigned char* s1 = s0 + kSlotCols / 16;
      const int nch = len >> 4, cb = k >> 4;
#pragma unroll 2
      for (int cl = c.lane; cl < nch; cl += 32) {
        const int ch = cb + cl;
        const int sw = (ch >> 1) & 3;
        const float4* xp = reinterpret_cast<const float4*>(xs + ch * 16);
        const float4 x0 = xp[0 ^ sw], x1 = xp[1 ^ sw], x2 = xp[2 ^ sw], x3 = xp[3 ^ sw];
        const float corr = -128.0f * xc[ch];
        const uint4 w0 = *reinterpret_cast<const uint4*>(q0 + cl * 16);
        const uint4 w1 = *reinterpret_cast<const uint4*>(q1 + cl * 16);
        const float f0 = h2f_bits(*reinterpret_cast<const uint16_t*>(s0 + (cl >> 1) * 2));
        const float f1 = h2f_bits(*reinterpret_cast<const uint16_t*>(s1 + (cl >> 1) * 2));
        float d0, d1;
        dot16x2(w0, w1, x0, x1, x2, x3, d0, d1);
        acc0 = fmaf(f0, fmaf(d0, kPScale, corr), acc0);
        acc1 = fmaf(f1, fmaf(d1, kPScale, corr), acc1);
      }
      cur_advance(p, q, len);
    }
    __syncwarp();  // the slot is consumed: refill it
    ++s.consumed;
    stream_issue<MOE>(c, s);
  }
  if (cur >= 0) finish_piece<MOE>(c, l, ph, cur, pfirst, acc0, acc1, xraw, pos, sid);
  return true;
}

// Routing of MoE block l, after the grid barrier that follows the router phase (whose tasks
// wrote the logits to global memory): every CTA reads all logits, takes the top_k by rank
// (ties to the lower id) and their softmax; ids, weights and the ready block into shared
// memory.
__device__ void rank_experts(const Ctx& c, int l) {
  const MegaArgs& a = *c.a;
  float* sel = c.sel();
  int* sel_id = c.sel_id();
  int* ids = c.moe_ids();
  float* wts = c.moe_wts();
  const int E = a.n_experts, k = a.top_k;
  if (threadIdx.x < k) sel_id[threadIdx.x] = threadIdx.x;  // valid ids whatever the logits hold
  for (int e = threadIdx.x; e < E; e += kMT) c.logits()[e] = __ldcg(a.logits + e);
  __syncthreads();
  // rank of expert e: 4 threads, each counting over a quarter of the experts
  const int qlen = (E + 3) >> 2;
  for (int base = c.warp * 32; base < E * 4; base += kMT) {
    const int idx = base + c.lane, e = idx >> 2, qq = idx & 3;
    float v = 0.f;
    int rank = 0;
    if (e < E) {
      v = c.logits()[e];
      const int f1 = min(E, (qq + 1) * qlen);
      for (int f = qq * qlen; f < f1; ++f) {
        const float u = c.logits()[f];
        rank += (u > v) || (u == v && f < e);
      }
    }
    rank += __shfl_xor_sync(0xffffffffu, rank, 1);
    rank += __shfl_xor_sync(0xffffffffu, rank, 2);
    if (e < E && qq == 0 && rank < k) {
      sel[rank] = v;
      sel_id[rank] = e;
    }
  }
  __syncthreads();
  if (c.warp == 0) {  // softmax over the selected logits (sel[0] is the largest)
    const float m = sel[0];
    const float ev = c.lane < k ? expf(sel[c.lane] - m) : 0.f;
    const float z = warp_sum(ev);
    if (c.lane < k) {
      ids[c.lane] = sel_id[c.lane];
      wts[c.lane] = ev / z;
    }
    if (c.lane == 0) *c.moe_ready() = l;
  }
  __syncthreads();
}

// Positions [c0, c1) of attention item `it` (KV head it % Hkv, chunk it / Hkv).
__device__ __forceinline__ void item_range(const MegaArgs& a, int it, int pos, int& kvh, int& chunk, int& c0,
                                           int& c1) {
  kvh = it % a.Hkv;
  chunk = it / a.Hkv;
  const int L = pos + 1, clen = (L + a.n_chunks - 1) / a.n_chunks;
  c0 = min(L, chunk * clen);
  c1 = min(L, c0 + clen);
}

// Thread 0: bulk copies of the K and V rows [p0, p0 + nold) (positions written by earlier
// steps) into the attention tile; completes on the attention barrier.
template <int D, int G>
__device__ __forceinline__ void attn_issue(const Ctx& c, unsigned char* area, const __half* kb, const __half* vb,
                                           int p0, int nold) {
  using AL = AttnLayout<D, G>;
  uint64_t* bar = c.bars() + kMW * kDepth;
  fence_async_smem();
  mbar_arrive_expect_tx(bar, (uint32_t)(2 * nold * D * 2));
  if (nold > 0) {
    bulk_g2s(area + AL::ks, kb + (size_t)p0 * D, (uint32_t)(nold * D * 2), bar);
    bulk_g2s(area + AL::vs, vb + (size_t)p0 * D, (uint32_t)(nold * D * 2), bar);
  }
}

// Split-K attention of block l over this CTA's items; the last chunk of a KV head to finish
// together with the other chunks of its head merges a slice of the head's outputs into
// obuf.  `prefetched`: tile 0 of the first item was issued before the preceding barrier.
template <int D, int G>
__device__ bool attention_phase(const Ctx& c, int l, unsigned char* area, unsigned& aphase, bool prefetched, int pos,
                                int sid) {
  using AL = AttnLayout<D, G>;
  constexpr int T = AL::T, PG = AL::PG, DP = D / 2, HPV = AL::HPV, NHG = AL::NHG;
  const MegaArgs& a = *c.a;
  const MegaLayer& Ly = a.layers[l];
  __half* Ks = reinterpret_cast<__half*>(area + AL::ks);
  __half* Vs = reinterpret_cast<__half*>(area + AL::vs);
  float* qs = reinterpret_cast<float*>(area + AL::qs);
  float* S = reinterpret_cast<float*>(area + AL::sc);
  float* Pt = reinterpret_cast<float*>(area + AL::pt);
  float* st_m = reinterpret_cast<float*>(area + AL::st);
  float* st_l = st_m + G;
  float* st_a = st_l + G;
  float* st_L = st_a + G;
  float* red = reinterpret_cast<float*>(area + AL::ks);  // [PG][G][D] after the last tile
  const int tid = threadIdx.x;
  const int nch = a.n_chunks, items = a.Hkv * nch;
  uint64_t* abar = c.bars() + kMW * kDepth;
  // PV: dims (2 dp, 2 dp + 1) of heads hg HPV .. hg HPV + HPV - 1, positions pg + PG k
  const int dp = tid % DP, hg = (tid / DP) % NHG, pg = tid / (DP * NHG);
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    int kvh, chunk, c0, c1;
    item_range(a, it, pos, kvh, chunk, c0, c1);
    const __half* kb = Ly.kc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;
    const __half* vb = Ly.vc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;
    for (int i = tid; i < G * D; i += kMT) {
      const int g = i / D, d = i - g * D;
      qs[g * D + q_slot<D>(d)] = __ldcg(a.qbuf + (size_t)kvh * G * D + i);
    }
    if (tid < G) {
      st_m[tid] = -INFINITY;
      st_l[tid] = 0.f;
    }
    float2 o[HPV];
#pragma unroll
    for (int h = 0; h < HPV; ++h) o[h] = make_float2(0.f, 0.f);
    for (int p0 = c0; p0 < c1; p0 += T) {
      const int np = min(T, c1 - p0);
      const int nold = max(0, min(np, pos - p0));
      if (!(prefetched && p0 == c0 && it == (int)blockIdx.x) && tid == 0) attn_issue<D, G>(c, area, kb, vb, p0, nold);
      if (nold < np) {  // the current position: written by this launch's QKV phase, read through L2
        const int r = pos - p0;
        for (int i = tid; i < D / 8; i += kMT) {
          reinterpret_cast<uint4*>(Ks + (size_t)r * D)[i] = __ldcg(reinterpret_cast<const uint4*>(kb + (size_t)pos * D) + i);
          reinterpret_cast<uint4*>(Vs + (size_t)r * D)[i] = __ldcg(reinterpret_cast<const uint4*>(vb + (size_t)pos * D) + i);
        }
      }
      const bool landed = mbar_wait(abar, aphase & 1u, kWaitNs);
      if (!__syncthreads_and(landed)) {  // CTA-uniform decision (also orders the row copy above)
        if (tid == 0) set_error(c);
        return false;
      }
      ++aphase;
      // scores: the 16-byte pieces of a K row are walked in a rotated order so that the lanes'
      // rows fall in distinct banks
      for (int idx = tid; idx < G * T; idx += kMT) {
        const int g = idx / T, p = idx - g * T;
        if (p < np) {
          const __half* kr = Ks + (size_t)p * D;
          const float* qg = qs + g * D;
          float sc = 0.f;
#pragma unroll 4
          for (int i = 0; i < D / 8; ++i) {
            const int j = (i + p) & (D / 8 - 1);
            const uint4 kk = *reinterpret_cast<const uint4*>(kr + 8 * j);
            const float4 qa = *reinterpret_cast<const float4*>(qg + 4 * j);
            const float4 qb = *reinterpret_cast<const float4*>(qg + D / 2 + 4 * j);
            const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kk.x));
            const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kk.y));
            const float2 k45 = __half22float2(*reinterpret_cast<const __half2*>(&kk.z));
            const float2 k67 = __half22float2(*reinterpret_cast<const __half2*>(&kk.w));
            sc = fmaf(qa.x, k01.x, sc);
            sc = fmaf(qa.y, k01.y, sc);
            sc = fmaf(qa.z, k23.x, sc);
            sc = fmaf(qa.w, k23.y, sc);
            sc = fmaf(qb.x, k45.x, sc);
            sc = fmaf(qb.y, k45.y, sc);
            sc = fmaf(qb.z, k67.x, sc);
            sc = fmaf(qb.w, k67.y, sc);
          }
          S[g * T + p] = sc * a.scale;
        }
      }
      __syncthreads();
      if (c.warp < G) {  // warp g: tile max, probabilities, running (max, sum) of head g
        const int g = c.warp;
        float sv[T / 32];
        float mt = -INFINITY;
#pragma unroll
        for (int k2 = 0; k2 < T / 32; ++k2) {
          const int p = c.lane + 32 * k2;
          sv[k2] = p < np ? S[g * T + p] : -INFINITY;
          mt = fmaxf(mt, sv[k2]);
        }
        mt = warp_max(mt);
        const float mold = st_m[g];
        const float mnew = fmaxf(mold, mt);
        float lsum = 0.f;
#pragma unroll
        for (int k2 = 0; k2 < T / 32; ++k2) {
          const int p = c.lane + 32 * k2;
          const float e = p < np ? expf(sv[k2] - mnew) : 0.f;
          Pt[p * G + g] = e;
          lsum += e;
        }
        const float lt = warp_sum(lsum);
        if (c.lane == 0) {
          const float alpha = (mold == -INFINITY) ? 0.f : expf(mold - mnew);
          st_a[g] = alpha;
          st_l[g] = st_l[g] * alpha + lt;
          st_m[g] = mnew;
        }
      }
      __syncthreads();
      // PV: this thread's dim pair of its head group over positions pg, pg + PG, ...
#pragma unroll
      for (int h = 0; h < HPV; ++h) {
        const float al = st_a[hg * HPV + h];
        o[h].x *= al;
        o[h].y *= al;
      }
      for (int p = pg; p < np; p += PG) {
        const float2 v = __half22float2(*reinterpret_cast<const __half2*>(Vs + (size_t)p * D + 2 * dp));
        float pr[HPV];
        if constexpr (HPV == 4) {
          const float4 q4 = *reinterpret_cast<const float4*>(Pt + p * G + hg * HPV);
          pr[0] = q4.x;
          pr[1] = q4.y;
          pr[2] = q4.z;
          pr[3] = q4.w;
        } else {
#pragma unroll
          for (int h = 0; h < HPV; ++h) pr[h] = Pt[p * G + hg * HPV + h];
        }
#pragma unroll
        for (int h = 0; h < HPV; ++h) {
          o[h].x = fmaf(pr[h], v.x, o[h].x);
          o[h].y = fmaf(pr[h], v.y, o[h].y);
        }
      }
      __syncthreads();  // the tile is consumed before the next one lands
    }
    // the position groups' sums (over the K/V tiles), then the partial of this chunk (token 0
    // of the AttnArgs layout), then arrive on the head's counter
#pragma unroll
    for (int h = 0; h < HPV; ++h) reinterpret_cast<float2*>(red + ((size_t)pg * G + hg * HPV + h) * D)[dp] = o[h];
    __syncthreads();
    float* po = a.part_o + ((size_t)kvh * nch + chunk) * (G * D);
    for (int i = tid; i < G * D; i += kMT) {
      float v = 0.f;
#pragma unroll
      for (int q = 0; q < PG; ++q) v += red[(size_t)q * G * D + i];
      po[i] = v;
    }
    if (tid < G) a.part_ml[((size_t)kvh * G + tid) * nch + chunk] = make_float2(st_m[tid], st_l[tid]);
    // the CTA barrier orders every thread's partial writes before thread 0's release (cumulative
    // at GPU scope), which the merging CTAs acquire
    __syncthreads();
    if (tid == 0) red_release_add(a.bar + 2 + kvh, 1u);
  }
  // Merge, spread over the chunks: once every chunk of its head has arrived, the CTA of
  // chunk j merges outputs [j SL, (j + 1) SL) of the head -- weights e^(m_c - M) per head,
  // weighted sums in chunk order.  (Every CTA arrives on all of its items before waiting.)
  constexpr int GD = G * D;
  const int SL = (GD + nch - 1) / nch;
  for (int it = blockIdx.x; it < items; it += gridDim.x) {
    int kvh, chunk, c0, c1;
    item_range(a, it, pos, kvh, chunk, c0, c1);
    if (tid == 0) {
      const unsigned target = (unsigned)(l + 1) * (unsigned)nch;
      const unsigned* hc = a.bar + 2 + kvh;
      if (ld_acquire_u32(hc) < target) {
        const uint64_t t0 = global_ns();
        while (ld_acquire_u32(hc) < target)
          if (global_ns() - t0 > kWaitNs) {
            set_error(c);
            break;
          }
      }
    }
    __syncthreads();
    if (c.flag()[0]) return false;
    const int i0 = min(GD, chunk * SL), n = min(GD, i0 + SL) - i0;
    float2* mls = reinterpret_cast<float2*>(area + AL::mls);  // [G][nch]
    float* wts = reinterpret_cast<float*>(area + AL::wts);    // [nch][G]
    float* pst = reinterpret_cast<float*>(area + AL::ks);     // [nch][SL] this slice of every partial
    for (int i = tid; i < G * nch; i += kMT) mls[i] = __ldcg(a.part_ml + (size_t)kvh * G * nch + i);
    for (int i = tid; i < nch * n; i += kMT) {
      const int ck = i / n, k = i - ck * n;
      pst[ck * SL + k] = __ldcg(a.part_o + ((size_t)kvh * nch + ck) * GD + i0 + k);
    }
    __syncthreads();
    if (c.warp < G) {  // warp g: the chunk weights of head g (lanes over the chunks)
      const int g = c.warp;
      float M = -INFINITY;
      for (int ck = c.lane; ck < nch; ck += 32) M = fmaxf(M, mls[g * nch + ck].x);
      M = warp_max(M);
      float Ls = 0.f;
      for (int ck = c.lane; ck < nch; ck += 32) {
        const float2 mc = mls[g * nch + ck];
        const float w = mc.y > 0.f ? expf(mc.x - M) : 0.f;
        wts[ck * G + g] = w;
        Ls = fmaf(mc.y, w, Ls);
      }
      Ls = warp_sum(Ls);
      if (c.lane == 0) st_L[g] = Ls;
    }
    __syncthreads();
    for (int k = c.warp; k < n; k += kMW) {  // a warp per output, lanes over the chunks
      const int g = (i0 + k) / D;
      float acc = 0.f;
      for (int ck = c.lane; ck < nch; ck += 32) acc = fmaf(wts[ck * G + g], pst[ck * SL + k], acc);
      acc = warp_sum(acc);
      if (c.lane == 0) a.obuf[(size_t)kvh * GD + i0 + k] = acc / st_L[g];
    }
    __syncthreads();
  }
  return true;
}

// MOE: the stage's blocks route over experts (a.n_experts > 0); compiled apart so that the
// dense kernel carries none of it.
template <int D, int G, bool MOE>
__global__ void __launch_bounds__(kMT, 1) mega_decode_kernel(const MegaArgs a) {
  extern __shared__ unsigned char mg_raw[];
  unsigned char* sm = reinterpret_cast<unsigned char*>(((uintptr_t)mg_raw + 127) & ~(uintptr_t)127);
  const int KpH = pad256(a.H);
  const size_t off_u = (kOffXraw + (size_t)KpH * 4 + 127) & ~(size_t)127;
  Ctx c;
  c.a = &a;
  c.sm = sm;
  static_assert(kOffReady + 4 <= kOffSplit, "routing scratch");
  static_assert(kOffSplit + kPhases * sizeof(Split) <= kOffWptr, "splits");
  static_assert(kOffWptr % 16 == 0 && kOffWptr + kMW * 2 * sizeof(void*) <= kOffXraw, "stream pointers");
  Split* splits = reinterpret_cast<Split*>(sm + kOffSplit);
  c.lane = threadIdx.x & 31;
  c.warp = threadIdx.x >> 5;
  float* xraw = reinterpret_cast<float*>(sm + kOffXraw);
  unsigned char* area = sm + off_u;  // union: projection input and warp partials, or attention tiles
  const int KpQ = pad256(a.Hq * a.D), KpF = pad256(a.F);
  const int Kx = max(KpH, max(KpQ, KpF));
  float* xs = reinterpret_cast<float*>(area);
  float* xc = xs + Kx;
  c.ps = reinterpret_cast<unsigned char*>(xc + Kx / 16);

  if (threadIdx.x < kMW * kDepth + 1) mbar_init(c.bars() + threadIdx.x, 1);
  if (threadIdx.x == 0) {
    c.flag()[0] = 0;
    c.flag()[1] = 0;
    *c.moe_ready() = -1;
  }
  if (threadIdx.x < kPhases) splits[threadIdx.x] = split_of(a, threadIdx.x, blockIdx.x, gridDim.x);
  mbar_fence_init();
  __syncthreads();
  const int pos = __ldcg(a.pos), sid = __ldcg(a.seq);

  Stream s;
  s.l = 0;
  s.ph = 0;
  s.q = cur_start(splits[0], c.warp);
  s.issued = 0;
  s.consumed = 0;
  if (c.lane == 0 && a.nl > 0) {
    const DevQ8& w0 = phase_w<MOE>(a.layers[0], 0);
    c.wptr()[2 * c.warp] = w0.q;
    c.wptr()[2 * c.warp + 1] = w0.s;
  }
  __syncwarp();
  if (s.q.left == 0) stream_normalise<MOE>(c, s);
  for (int d = 0; d < kDepth; ++d) stream_issue<MOE>(c, s);

  unsigned nbar = 0, aphase = 0;
  bool ok = true;
  constexpr bool moe = MOE;
  // one call site per step (the projection step is the same code for every phase: the kernel
  // stays small enough for the instruction cache)
  for (int l = 0; l < a.nl && ok; ++l) {
    const MegaLayer& L = a.layers[l];
    for (int ph = 0; ph < kPhases && ok; ++ph) {
      if (ph == kPhRouter && !moe) continue;
      if (ph == kPhGU && moe) {
        stream_refill<MOE>(c, s);  // the routing is known: the selected experts' slices stream in
        phase_setup(c, ph, pos);
        __syncthreads();
      } else {
        // the projection's input: QKV and the router (or the dense gate/up) normalise the
        // residual (gamma_1, gamma_2; the raw residual is kept for the residual adds), O and
        // down take the attention output and the SwiGLU output as they are; the experts'
        // gate/up reuses the router's input
        const bool norm2 = ph == kPhRouter || ph == kPhGU;
        const float* in = ph == kPhQKV ? (l == 0 ? a.hin : a.hout) : ph == kPhO ? a.obuf : ph == kPhDown ? a.abuf : a.x1;
        const int K = ph == kPhO ? a.Hq * a.D : ph == kPhDown ? a.F : a.H;
        const int Kp = ph == kPhO ? KpQ : ph == kPhDown ? KpF : KpH;
        const float* gamma = ph == kPhQKV ? L.attn_norm : norm2 ? L.ffn_norm : nullptr;
        // the gamma of the next normalising stage is fetched into L2 one phase ahead (the weight
        // stream evicts it between blocks): one 128-byte line per CTA
        if (threadIdx.x == 0 && (ph == kPhO || ph == kPhDown)) {
          const float* g = ph == kPhO ? L.ffn_norm : (l + 1 < a.nl ? a.layers[l + 1].attn_norm : nullptr);
          for (int i = blockIdx.x * 32; g && i < a.H; i += gridDim.x * 32) prefetch_l2_last(g + i);
        }
        stage_issue(in, K, Kp, gamma, xs, xraw);
        phase_setup(c, ph, pos);
        stage_finish(c, K, Kp, gamma, a.eps, xs, xc, xraw);
      }
      ok = __syncthreads_and(gemv_phase<MOE>(c, s, l, ph, xs, xc, xraw, pos, sid));
      if (ph == kPhQKV) {
        // tile 0 of this CTA's first attention item (positions of earlier steps) streams in
        // while the grid meets
        bool pre = false;
        if (ok && (int)blockIdx.x < a.Hkv * a.n_chunks) {
          int kvh, chunk, c0, c1;
          item_range(a, blockIdx.x, pos, kvh, chunk, c0, c1);
          if (c0 < c1) {
            pre = true;
            if (threadIdx.x == 0) {
              const __half* kb = L.kc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;
              const __half* vb = L.vc + ((size_t)sid * a.Hkv + kvh) * (size_t)a.max_len * D;
              const int np = min(AttnLayout<D, G>::T, c1 - c0);
              attn_issue<D, G>(c, area, kb, vb, c0, max(0, min(np, pos - c0)));
            }
          }
        }
        if (ok) ok = grid_barrier(c, ++nbar);
        if (!ok) {
          if (pre && threadIdx.x == 0) mbar_wait(c.bars() + kMW * kDepth, aphase & 1u, kWaitNs);
          break;
        }
        ok = attention_phase<D, G>(c, l, area, aphase, pre, pos, sid);
      }
      // the residual after the last projection of the last block is the launch's output
      if (ok && (ph < kPhDown || l + 1 < a.nl)) ok = grid_barrier(c, ++nbar);
      if (MOE && ok && ph == kPhRouter) rank_experts(c, l);
    }
  }
  if (!ok) stream_drain(c, s);
  grid_leave(c);
}

size_t mega_smem(int H, int q_dim, int F, int D, int G) {
  const int KpH = pad256(H), Kx = std::max(KpH, std::max(pad256(q_dim), pad256(F)));
  const size_t off_u = (kOffXraw + (size_t)KpH * 4 + 127) & ~(size_t)127;
  size_t attn = 0;
  if (D == 64) attn = G == 1 ? AttnLayout<64, 1>::total : G == 2 ? AttnLayout<64, 2>::total
                    : G == 4 ? AttnLayout<64, 4>::total : AttnLayout<64, 8>::total;
  else attn = G == 1 ? AttnLayout<128, 1>::total : G == 2 ? AttnLayout<128, 2>::total
            : G == 4 ? AttnLayout<128, 4>::total : AttnLayout<128, 8>::total;
  const size_t u = std::max((size_t)Kx * 4 + (size_t)(Kx / 16) * 4 + kPsBytes, attn);
  return off_u + u + 128;  // + alignment of the dynamic base
}

template <int D, int G, bool MOE>
cudaError_t prepare_mega_dg() {
  return cudaFuncSetAttribute(mega_decode_kernel<D, G, MOE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)kMaxSmem);
}

template <int D, int G, bool MOE>
cudaError_t launch_mega_dg(const MegaArgs& a, size_t smem, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(sm_count());
  cfg.blockDim = dim3(kMT);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, mega_decode_kernel<D, G, MOE>, a);
}

// Shared-memory attribute of the eight (head dim, group) kernels of one kind.
template <bool MOE>
cudaError_t prepare_mega_all() {
  const cudaError_t r[] = {prepare_mega_dg<64, 1, MOE>(),  prepare_mega_dg<64, 2, MOE>(),
                           prepare_mega_dg<64, 4, MOE>(),  prepare_mega_dg<64, 8, MOE>(),
                           prepare_mega_dg<128, 1, MOE>(), prepare_mega_dg<128, 2, MOE>(),
                           prepare_mega_dg<128, 4, MOE>(), prepare_mega_dg<128, 8, MOE>()};
  for (cudaError_t x : r)
    if (x != cudaSuccess) return x;
  return cudaSuccess;
}

template <bool MOE>
cudaError_t launch_mega_all(const MegaArgs& a, size_t smem, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  if (a.D == 64) {
    switch (G) {
      case 1: return launch_mega_dg<64, 1, MOE>(a, smem, st);
      case 2: return launch_mega_dg<64, 2, MOE>(a, smem, st);
      case 4: return launch_mega_dg<64, 4, MOE>(a, smem, st);
      default: return launch_mega_dg<64, 8, MOE>(a, smem, st);
    }
  }
  switch (G) {
    case 1: return launch_mega_dg<128, 1, MOE>(a, smem, st);
    case 2: return launch_mega_dg<128, 2, MOE>(a, smem, st);
    case 4: return launch_mega_dg<128, 4, MOE>(a, smem, st);
    default: return launch_mega_dg<128, 8, MOE>(a, smem, st);
  }
}

}  // namespace

// The MoE kernels (kernels_mega_moe.cu).
cudaError_t prepare_mega_moe();
cudaError_t launch_mega_moe(const MegaArgs& a, size_t smem, cudaStream_t st);

}  // namespace lrs

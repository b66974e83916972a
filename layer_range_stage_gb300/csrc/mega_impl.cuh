// Persistent decode of a stage, dense or MoE (sm_103a): every block of the stage for one token
// in one cooperative launch, one CTA per SM.
//
// What it computes is the decode block loop of "41. Many GPUs: tensor, pipeline, expert
// and data parallelism", section "Pipeline parallelism" (add_norm, attention, add_norm,
// MLP per block, the residual stream carried through), with the split-KV attention merge
// of section "Ring attention for very long contexts".  The arithmetic per weight is the
// integer-form dot product of q8dot.cuh: dp4a on the stored weight bytes against three signed
// bytes per staged input, exact before its float32 scaling.
//
// Why one launch: a batch-1 decode step is a chain of small dependent matrix-vector
// products.  Launched one kernel each, every product pays its own ramp and tail while HBM
// idles, and a successor cannot start streaming until its predecessor's CTAs leave the
// SMs.  Here the weight stream never stops: each warp owns a fixed sequence of weight
// slices (its share of every projection of every block, known before the first
// activation exists) and keeps two of them in flight as tensor copies into shared memory,
// running ahead across projections and blocks.
//
// Work split of a projection: CTA c owns a contiguous range of row pairs (2t, 2t + 1) -- the
// pairs the RoPE and SwiGLU epilogues need, and for the other projections two rows that share
// each read of the staged input -- cut into slots of at most 2048 columns; the CTA's slots, in
// memory order, are dealt to its warps in groups (see Split).  Every output has one fixed
// summation order.
//
// Hand-offs without grid barriers: every vector one step passes to the next (q, the current K
// and V rows, the attention output, the post-attention residual, the block output, the router
// logits) is written as tagged 64-bit entries (launch sequence and block in the high word), and
// a consumer waits only for the entries it reads; the SwiGLU output goes by plain stores and a
// counter.  A CTA reads a step's input only if it has work in the step, so every reader of a
// vector contributes to what that vector's next writers wait for.
//
// MoE stages: the router rows are a projection of the weight stream like the others (tagged
// logits); every CTA gathers the logits and ranks them itself (top-k with ties to the lower id,
// softmax over the selected: the same arithmetic on the same data, so every CTA picks the same
// experts), and the gate/up and down slices of the selected experts stream in once it is known
// (the weight stream pauses there: those slices depend on the routing).
//
// Every wait is bounded by time; a CTA that runs out sets the error word, waits (bounded) for
// its own copies in flight and leaves, and the last CTA to leave resets the counters.

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
constexpr size_t kOffWptr = kOffSplit + 272;                               // [kMW][2] stream pointers
// the phases of a block's weight stream
constexpr int kPhQKV = 0, kPhO = 1, kPhRouter = 2, kPhGU = 3, kPhDown = 4, kPhases = 5;
constexpr int kSeqWord = 63;  // word of the counter block holding the launch sequence
constexpr size_t kOffXraw = kOffMoe + 2176;                               // [Kp(H)] floats

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
  static_assert(G * D <= 2 * kMT && (2 * T * D * 2) / (G * D * 4) >= 1, "merge: two outputs per thread, a chunk batch");
};

// Where dim d of a head's q sits in shared memory: per 8-dim chunk j the low four dims at
// 4 j, the high four at D / 2 + 4 j, so that 8 lanes reading 8 consecutive chunks touch 8
// consecutive 16-byte words (one shared-memory wavefront).
template <int D>
__device__ __forceinline__ int q_slot(int d) {
  return ((d & 4) ? D / 2 : 0) + ((d >> 3) << 2) + (d & 3);
}

// The counters: after a CTA barrier, one thread's release (or acquire-release) operation at GPU
// scope publishes every write the CTA made before the barrier (release is cumulative), and an
// acquire by one thread followed by a CTA barrier orders every thread's later reads after the
// writes it observed -- no separate fence on either side.
__device__ __forceinline__ void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Tagged values: the vectors handed from one step of a block to the next are written as 64-bit
// words (tag << 32 | f32 bits), tag = launch sequence * 256 + block + 1, with single 64-bit
// stores, so a reader that sees the tag it expects has the value too.  A reader polls exactly
// the entries it needs -- no grid barrier, one round trip to L2 once the last of them is in.
typedef unsigned long long tagged_t;

__device__ __forceinline__ void st_tag(tagged_t* p, float v, unsigned tag) {
  const tagged_t w = ((tagged_t)tag << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ ulonglong2 ld_tag2(const tagged_t* p) {  // two entries, 16-byte aligned
  ulonglong2 r;
  asm volatile("ld.relaxed.gpu.global.v2.b64 {%0, %1}, [%2];" : "=l"(r.x), "=l"(r.y) : "l"(p) : "memory");
  return r;
}
__device__ __forceinline__ unsigned tag_of(tagged_t w) { return (unsigned)(w >> 32); }
__device__ __forceinline__ float val_of(tagged_t w) { return __uint_as_float((unsigned)w); }

// How a projection is dealt over the grid.  Rows go in pairs (2P, 2P + 1): the pairs the RoPE
// and SwiGLU epilogues need, and for the other projections two rows that share each load of
// the staged input.  CTA c owns pairs [p0, p0 + np) with p0 = c * NP / G, so every CTA holds
// the same number of pairs to within one.  A pair's K range is cut into slots of at most
// kSlotCols columns (one ring slot each: a column block of both rows).  The CTA's slots, in
// memory order, form groups of gs consecutive slots -- a whole pair (gs = slots per pair), or
// one slot when whole pairs would leave the CTA's warps unevenly loaded -- and group g goes to
// warp g mod 16.  At any moment the CTA's warps read one dense window of the matrix (DRAM rows
// are opened once for many requests), and every warp holds the same number of slots to within
// one group.  A pair split between warps is finished by the warp that completes it: the slots'
// partial sums are added in slot order.
struct Split {
  int NP;    // pairs of the projection
  int Kp;    // columns of a pair's K range (mode 2: top_k expert pieces of PS columns)
  int seg;   // columns between source discontinuities (Kp, or PS in mode 2)
  int mode;  // 0 plain rows; 1 rows of the selected experts (rps rows each); 2 piece j of a row
             // from selected expert j (K gathered over the experts)
  int rps;
  int p0, np;  // this CTA's pairs
  int sp;      // slots of a pair
  int sl;      // columns of a slot (the last of a pair may be shorter), a multiple of 256
  int gs;      // slots of a group: sp, or 1
  int ng;      // this CTA's groups: np * sp / gs
  int dq, dr;  // gs == 1: kMW slots further on is dq pairs and dr slots further on
};

constexpr int kSlotCols = kSlotQ / 2;  // columns of each row in a ring slot
constexpr int kMaxCtaPairs = 256;      // pairs (and split-pair slots) a CTA may hold in one projection
// per-projection scratch after the staged input: slot partials, slot counters of split pairs,
// the RoPE factors of the CTA's QKV pairs
constexpr size_t kPsPart = 0, kPsCnt = kPsPart + (size_t)kMaxCtaPairs * 8, kPsRope = kPsCnt + kMaxCtaPairs * 4,
                 kPsBytes = kPsRope + (size_t)kMaxCtaPairs * 8;

// A warp's position in one projection: its group count m (groups w + 16 m are its own), the
// current slot (CTA-local pair pr, slot j of the pair) and r, the slot's place in its group.
// The issuer and the consumer of a warp's ring walk the same sequence of cursors, so a slot's
// contents never have to be written down.
struct Cur {
  int m, pr, j, r;
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
  unsigned seq;  // this launch's sequence number (tags: seq * 256 + block + 1)
  __device__ unsigned tag(int l) const { return seq * 256u + (unsigned)l + 1u; }
  // the tagged vectors (layout of mega_tag_entries): q [Hq * D], the current K and V rows
  // [2][Hkv * D], attention output [Hq * D], x1 [H], block output [H], router logits [n_experts]
  __device__ tagged_t* tq() const { return a->tags; }
  __device__ tagged_t* tkv() const { return a->tags + (size_t)a->Hq * a->D; }
  __device__ tagged_t* to() const { return tkv() + (size_t)2 * a->Hkv * a->D; }
  __device__ tagged_t* tx1() const { return to() + (size_t)a->Hq * a->D; }
  __device__ tagged_t* th() const { return tx1() + a->H; }
  __device__ tagged_t* tlog() const { return th() + a->H; }
  // [np * sp] partial sums (rows 2P, 2P + 1) of the slots of pairs split between warps
  __device__ float2* part() const { return reinterpret_cast<float2*>(ps + kPsPart); }
  __device__ int* cnt() const { return reinterpret_cast<int*>(ps + kPsCnt); }     // [kMaxCtaPairs] pieces done
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
  // [kMW][2] tensor maps (weights, scales) of each warp's stream cursor (l, ph): an issue reads
  // them here, not from the block descriptor
  __device__ const void** wptr() const { return reinterpret_cast<const void**>(sm + kOffWptr); }
};

// The projections of a block: weights of phase ph.
template <bool MOE>
__host__ __device__ __forceinline__ const DevQ8& phase_w(const MegaLayer& L, int ph) {
  if (MOE && ph == kPhRouter) return L.router;
  if (MOE && ph >= kPhGU) return ph == kPhGU ? L.egu : L.edown;
  return ph == kPhQKV ? L.wqkv : ph == kPhO ? L.wo : ph == kPhGU ? L.wgu : L.wdown;
}

// ph: kPhQKV, kPhO, kPhRouter (MoE stages: one logit per row, into global memory), kPhGU
// (dense, or the selected experts' rows), kPhDown (dense, or gathered over the experts).
// Computed once per launch (from block 0: every block has the same shapes).  Host-callable too,
// so that its cover of every pair and slot is checked on the host for every shape.
__host__ __device__ Split split_of(const MegaArgs& a, int ph, int cta, int G) {
  const MegaLayer& L = a.layers[0];
  const bool moe = a.n_experts > 0;
  Split p;
  p.mode = 0;
  p.rps = 0;
  if (ph == kPhRouter && !moe) {  // dense stages: no router rows
    p.NP = 0;
    p.Kp = p.seg = kSlotCols;
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
  p.np = (int)((long long)(cta + 1) * p.NP / G) - p.p0;
  // slots of sl columns: a source piece (mode 2), else kSlotCols
  p.sp = p.mode == 2 ? p.Kp / p.seg : (p.Kp + kSlotCols - 1) / kSlotCols;
  p.sl = p.mode == 2 ? p.seg : min(kSlotCols, p.Kp);  // the last slot of a pair may be shorter
  // whole pairs per warp unless single slots spread the CTA's slots more evenly
  const int by_pair = (p.np + kMW - 1) / kMW * p.sp, by_slot = (p.np * p.sp + kMW - 1) / kMW;
  p.gs = (by_slot < by_pair && p.np * p.sp <= kMaxCtaPairs) ? 1 : p.sp;
  p.ng = p.np * p.sp / p.gs;
  p.dq = kMW / p.sp;
  p.dr = kMW % p.sp;
  return p;
}

// The cursor of warp w's first slot in projection p (valid while w + 16 m < ng).
__host__ __device__ __forceinline__ Cur cur_start(const Split& p, int w) {
  Cur q;
  q.m = 0;
  q.r = 0;
  const int g = w * p.gs;
  q.pr = g / p.sp;
  q.j = g - q.pr * p.sp;
  return q;
}

__host__ __device__ __forceinline__ bool cur_valid(const Split& p, const Cur& q, int w) { return w + kMW * q.m < p.ng; }

// First column and columns of slot j of a pair.
__host__ __device__ __forceinline__ int slot_k(const Split& p, int j) { return j * p.sl; }
__host__ __device__ __forceinline__ int slot_len(const Split& p, int j) { return min(p.sl, p.Kp - j * p.sl); }

__host__ __device__ __forceinline__ void cur_advance(const Split& p, Cur& q) {
  if (++q.r < p.gs) {  // the next slot of a whole-pair group
    ++q.j;
    return;
  }
  q.r = 0;
  ++q.m;
  if (p.gs == p.sp) {  // the warp's next pair
    q.pr += kMW;
    q.j = 0;
  } else {  // single slots: kMW slots further on
    q.pr += p.dq;
    q.j += p.dr;
    if (q.j >= p.sp) {
      q.j -= p.sp;
      ++q.pr;
    }
  }
}

// Global addresses of rows (2P, 2P + 1) of a projection at column k (P phase-global).
// Row (the pair's first) and first column of slot j of pair P in the matrix of projection p
// (MoE: the stacked experts' rows).
template <bool MOE>
__device__ __forceinline__ void pair_rc(const Ctx& c, const Split& p, int P, int j, int& r, int& k) {
  if (MOE && p.mode == 2) {  // K gathered: slot j is the row's piece from selected expert j
    r = c.moe_ids()[j] * (2 * p.NP) + 2 * P;
    k = 0;
    return;
  }
  r = 2 * P;
  if (MOE && p.mode == 1) r = c.moe_ids()[2 * P / p.rps] * p.rps + (2 * P) % p.rps;
  k = slot_k(p, j);
}

// Move a cursor to the first projection at or after (l, ph) in which this warp holds slots.
template <bool MOE>
__device__ __forceinline__ void stream_normalise(const Ctx& c, Stream& s) {
  bool moved = false;
  while (s.l < c.a->nl && !cur_valid(c.split()[s.ph], s.q, c.warp)) {
    if (++s.ph == kPhases) {
      s.ph = 0;
      ++s.l;
    }
    s.q = cur_start(c.split()[s.ph], c.warp);
    moved = true;
  }
  if (moved && s.l < c.a->nl && c.lane == 0) {
    c.wptr()[2 * c.warp] = &c.a->layers[s.l].tmap[2 * s.ph];
    c.wptr()[2 * c.warp + 1] = &c.a->layers[s.l].tmap[2 * s.ph + 1];
  }
  __syncwarp();
}

// Issue the next slot of this warp's stream (if any) into the ring: slot j of pair pr, row 2P's
// bytes at the start of the ring slot and row 2P + 1's sl bytes further on (two tensor-map
// boxes: bytes and scales).  Slices of the selected experts wait until the routing of their
// block is known.
template <bool MOE>
__device__ __forceinline__ void stream_issue(const Ctx& c, Stream& s) {
  if (s.l >= c.a->nl) return;
  if (MOE && s.ph >= kPhGU && s.l > *c.moe_ready()) return;
  const Split& p = c.split()[s.ph];
  const int slot = s.issued % kDepth;
  if (c.lane == 0) {
    int r, k;
    pair_rc<MOE>(c, p, p.p0 + s.q.pr, s.q.j, r, k);
    uint64_t* bar = c.bars() + c.warp * kDepth + slot;
    unsigned char* dq = c.ringq() + (size_t)(c.warp * kDepth + slot) * kSlotQ;
    unsigned char* ds = c.rings() + (size_t)(c.warp * kDepth + slot) * kSlotS;
    fence_async_smem();  // the slot's previous contents were read through the generic proxy
    // one box of the pair's two rows for the bytes and one for the scales (8-byte elements): row
    // 2P + 1 lands sl bytes (sl / 16 scale bytes) after row 2P; columns past Kp read as zero
    mbar_arrive_expect_tx(bar, (uint32_t)(2 * (p.sl + p.sl / 16)));
    tma_load_2d(dq, c.wptr()[2 * c.warp], k >> 3, r, bar);
    tma_load_2d(ds, c.wptr()[2 * c.warp + 1], k >> 7, r, bar);
  }
  ++s.issued;
  cur_advance(p, s.q);
  if (!cur_valid(p, s.q, c.warp)) stream_normalise<MOE>(c, s);
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

// Leaving: the last CTA out resets the SwiGLU and attention counters and advances the launch
// sequence
// (every CTA has stopped polling by the time it counts itself out).
__device__ void grid_leave(const Ctx& c) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned prev = atomicAdd(c.a->bar + 1, 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(c.a->bar, 0u);
      for (int h = 0; h < c.a->Hkv; ++h) atomicExch(c.a->bar + 2 + h, 0u);
      atomicExch(c.a->bar + kSeqWord, c.seq + 1u);
      atomicExch(c.a->bar + 1, 0u);
    }
  }
}

// A projection input from global memory (written earlier in this launch: read through L2)
// into shared memory, for stage_finish to turn into the integer form of every 16-input chunk
// (RMSNorm with gamma first, when given).  With gamma the raw values land in xraw (kept for
// the residual adds) and gamma in xs, which is then overwritten in place; without, the raw
// values land in xs.  Every 16-byte piece is an asynchronous copy issued before any
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

// One pair of entries (16-byte aligned) of a tagged vector, waited for (bounded).
__device__ __forceinline__ bool poll_pair(const Ctx& c, const tagged_t* p, unsigned tag, float2& v) {
  ulonglong2 w = ld_tag2(p);
  uint64_t t0 = 0;
  while (tag_of(w.x) != tag || tag_of(w.y) != tag) {
    const uint64_t now = global_ns();
    if (!t0) {
      t0 = now;
    } else if (now - t0 > kWaitNs) {
      set_error(c);
      return false;
    }
    __nanosleep(64);
    w = ld_tag2(p);
  }
  v = make_float2(val_of(w.x), val_of(w.y));
  return true;
}

// Wait (bounded) until entries [0, n) of a tagged vector carry `tag` and put their values in
// dst; entries whose index within a piece of `piece` entries is `valid` or more are never
// written and read as zero.  n, piece and valid are even.  All entries are fetched at once with
// asynchronous copies into `scratch` (shared memory, n tagged entries); the pairs not yet
// carrying the tag are fetched again, all at once, pass after pass (one L2 round trip per
// pass).  n <= 128 kMT.  Returns false after a timed-out wait
// (error set); the caller makes the outcome CTA-uniform.
__device__ bool gather_tagged(const Ctx& c, const tagged_t* src, int n, int piece, int valid, unsigned tag,
                              tagged_t* scratch, float* dst) {
  const int npair = n >> 1;
  // the pairs of this thread (i = threadIdx.x + kMT k) still to come, one bit per k (n <= 64 kMT)
  unsigned long long pending = 0;
  for (int k = 0, i = threadIdx.x; i < npair; ++k, i += kMT) {
    if ((2 * i) % piece < valid) {
      cp_async16(scratch + 2 * i, src + 2 * i);
      pending |= 1ull << k;
    } else {
      dst[2 * i] = 0.f;
      dst[2 * i + 1] = 0.f;
    }
  }
  uint64_t t0 = 0;
  while (true) {
    cp_async_wait_all();
    unsigned long long left = 0;
    for (unsigned long long m = pending; m; m &= m - 1) {  // the pairs fetched in this pass
      const int k = __ffsll((long long)m) - 1, i = threadIdx.x + kMT * k;
      const tagged_t w0 = scratch[2 * i], w1 = scratch[2 * i + 1];
      if (tag_of(w0) == tag && tag_of(w1) == tag) {
        dst[2 * i] = val_of(w0);
        dst[2 * i + 1] = val_of(w1);
      } else {
        left |= 1ull << k;
      }
    }
    if (!left) return true;
    const uint64_t now = global_ns();
    if (!t0) {
      t0 = now;
    } else if (now - t0 > kWaitNs) {
      set_error(c);
      return false;
    }
    pending = left;  // one more pass: every missing pair fetched again at once
    for (unsigned long long m = pending; m; m &= m - 1) {
      const int i = threadIdx.x + kMT * (__ffsll((long long)m) - 1);
      cp_async16(scratch + 2 * i, src + 2 * i);
    }
  }
}

// The staging of a projection whose input is a tagged vector of this launch: gamma (when given)
// is issued first, then the input is gathered as its entries arrive (into xraw with gamma, else
// into xs), zero beyond K up to Kp.  `scratch`: 2K floats of shared memory that hold nothing
// else during the gather.  Returns false (CTA-uniform) after a timed-out wait.
__device__ bool stage_gather(const Ctx& c, const tagged_t* x, int K, int Kp, int piece, int valid, unsigned tag,
                             const float* gamma, float* xs, float* xraw, tagged_t* scratch) {
  const int tid = threadIdx.x;
  float* raw = gamma ? xraw : xs;
  if (gamma)
    for (int i = tid; i < (Kp >> 2); i += kMT) {
      if (4 * i < K) cp_async16(xs + 4 * i, gamma + 4 * i);
      else reinterpret_cast<float4*>(xs)[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  const bool ok = gather_tagged(c, x, K, piece, valid, tag, scratch, raw);
  for (int i = K + tid; i < Kp; i += kMT) raw[i] = 0.f;
  return __syncthreads_and(ok);
}

// The staging of a projection whose input is written by every CTA before it counts itself done
// on `counter` (the SwiGLU output, too wide to carry tags in shared memory): wait (thread 0,
// bounded) for `target` arrivals, then copy the input in as stage_issue does.  Returns false
// (CTA-uniform) after a timed-out wait.
__device__ bool stage_counted(const Ctx& c, const unsigned* counter, unsigned target, const float* x, int K, int Kp,
                              float* xs, float* xraw) {
  if (threadIdx.x == 0 && ld_acquire_u32(counter) < target) {
    const uint64_t t0 = global_ns();
    while (ld_acquire_u32(counter) < target) {
      if (global_ns() - t0 > kWaitNs) {
        set_error(c);
        break;
      }
      __nanosleep(64);
    }
  }
  __syncthreads();
  if (c.flag()[0]) return false;
  stage_issue(x, K, Kp, nullptr, xs, xraw);
  return true;
}

// The second half of the staging (after stage_issue and any other loads of the phase's setup):
// wait for the copies, then RMSNorm and the integer form of every 16-input chunk (q8dot.cuh) in
// place: 64 bytes per chunk, as many as its floats.
__device__ void stage_finish(const Ctx& c, int K, int Kp, const float* gamma, float eps, float* xs, float* xraw) {
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
  // two lanes per chunk (2 nchunk is a multiple of 32: whole warps); each lane reads its eight
  // inputs before the pair's first shuffle and writes after it, so the in-place form is safe
  for (int t = tid; t < 2 * nchunk; t += kMT) {
    const int ch = t >> 1, half = t & 1;
    float h[8];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const float4 v = reinterpret_cast<const float4*>(raw)[ch * 4 + half * 2 + j];
      h[4 * j] = v.x;
      h[4 * j + 1] = v.y;
      h[4 * j + 2] = v.z;
      h[4 * j + 3] = v.w;
      if (gamma) {
        const float4 g = reinterpret_cast<const float4*>(xs)[ch * 4 + half * 2 + j];
        h[4 * j] = h[4 * j] * rinv * g.x;
        h[4 * j + 1] = h[4 * j + 1] * rinv * g.y;
        h[4 * j + 2] = h[4 * j + 2] * rinv * g.z;
        h[4 * j + 3] = h[4 * j + 3] * rinv * g.w;
      }
    }
    uint2 q[4];
    q8_chunk_encode2(h, half, q[0], q[1], q[2], q[3]);
    const int sw = (ch >> 1) & 3;  // the chunk's four 16-byte pieces, swizzled: lanes reading
    uint2* xp = reinterpret_cast<uint2*>(xs + ch * 16);  // consecutive chunks hit distinct banks
#pragma unroll
    for (int j = 0; j < 4; ++j) xp[2 * (j ^ sw) + half] = q[j];
  }
  __syncthreads();
}

// The epilogue of pair i (CTA-local) of projection ph of block l, from its row sums.
template <bool MOE>
__device__ __forceinline__ void epilogue_pair(const Ctx& c, int l, int ph, int i, float y0, float y1,
                                              const float* xraw, int pos, int sid) {
  const MegaArgs& a = *c.a;
  const Split& p = c.split()[ph];
  const int t = p.p0 + i;  // the pair, projection-wide
  if (ph == kPhQKV) {  // rows (2t, 2t+1) are dims (j, j + D/2) of one head: RoPE, then q or fp16 K/V
    const int hd = a.D >> 1, head = t / hd, j = t - head * hd;
    const unsigned tg = c.tag(l);
    if (head < a.Hq) {
      const float2 cs = c.rope_s()[i];
      tagged_t* qo = c.tq() + (size_t)head * a.D;
      st_tag(qo + j, y0 * cs.x - y1 * cs.y, tg);
      st_tag(qo + j + hd, y1 * cs.x + y0 * cs.y, tg);
    } else {
      // the fp16 cache row, and its values (as rounded) tagged for this launch's attention
      const bool is_k = head < a.Hq + a.Hkv;
      const int kvh = head - a.Hq - (is_k ? 0 : a.Hkv);
      const MegaLayer& L = a.layers[l];
      const size_t base = (((size_t)sid * a.Hkv + kvh) * a.max_len + pos) * a.D;
      __half h0, h1;
      if (is_k) {
        const float2 cs = c.rope_s()[i];
        h0 = __float2half_rn(y0 * cs.x - y1 * cs.y);
        h1 = __float2half_rn(y1 * cs.x + y0 * cs.y);
      } else {
        h0 = __float2half_rn(y0);
        h1 = __float2half_rn(y1);
      }
      __half* cache = is_k ? L.kc : L.vc;
      cache[base + j] = h0;
      cache[base + j + hd] = h1;
      tagged_t* kv = c.tkv() + ((size_t)(is_k ? 0 : a.Hkv) + kvh) * a.D;
      st_tag(kv + j, __half2float(h0), tg);
      st_tag(kv + j + hd, __half2float(h1), tg);
    }
  } else if (ph == kPhO) {
    st_tag(c.tx1() + 2 * t, __fadd_rn(xraw[2 * t], y0), c.tag(l));
    st_tag(c.tx1() + 2 * t + 1, __fadd_rn(xraw[2 * t + 1], y1), c.tag(l));
  } else if (MOE && ph == kPhRouter) {
    st_tag(c.tlog() + 2 * t, y0, c.tag(l));
    st_tag(c.tlog() + 2 * t + 1, y1, c.tag(l));
  } else if (ph == kPhGU) {  // plain stores: the CTA counts itself done after the projection
    if (MOE) {  // pair t: expert slot t / EF, unit t % EF; scaled by the routing weight
      const int slot = t / a.EF, j = t - slot * a.EF;
      a.abuf[(size_t)slot * pad256(a.EF) + j] = silu(y0) * y1 * c.moe_wts()[slot];
    } else {
      a.abuf[t] = silu(y0) * y1;
    }
  } else if (l + 1 < a.nl) {  // the block output: the next block's input
    st_tag(c.th() + 2 * t, __fadd_rn(xraw[2 * t], y0), c.tag(l));
    st_tag(c.th() + 2 * t + 1, __fadd_rn(xraw[2 * t + 1], y1), c.tag(l));
  } else {  // the launch's output
    a.hout[2 * t] = __fadd_rn(xraw[2 * t], y0);
    a.hout[2 * t + 1] = __fadd_rn(xraw[2 * t + 1], y1);
  }
}

// This warp's slot j of pair i (CTA-local) is summed.  A whole-pair group (gs == sp) goes
// straight to the epilogue once its last slot is in; a pair dealt slot by slot is finished by
// the warp whose slot completes it (a shared-memory counter per pair), which adds the slots'
// sums in slot order, so every output has one summation order whichever warp finishes it.
template <bool MOE>
__device__ __forceinline__ void finish_slot(const Ctx& c, int l, int ph, int i, int j, float& acc0, float& acc1,
                                            const float* xraw, int pos, int sid) {
  const Split& p = c.split()[ph];
  if (p.gs == p.sp) {
    if (j != p.sp - 1) return;  // the pair goes on in this warp's next slot
    const float y0 = warp_sum(acc0), y1 = warp_sum(acc1);
    acc0 = acc1 = 0.f;
    if (c.lane == 0) epilogue_pair<MOE>(c, l, ph, i, y0, y1, xraw, pos, sid);
    return;
  }
  const float y0 = warp_sum(acc0), y1 = warp_sum(acc1);
  acc0 = acc1 = 0.f;
  if (c.lane == 0) {
    float2* part = c.part() + i * p.sp;
    part[j] = make_float2(y0, y1);
    __threadfence_block();
    if (atomicAdd(c.cnt() + i, 1) == p.sp - 1) {  // the pair's last slot
      __threadfence_block();
      float2 v = part[0];
      for (int u = 1; u < p.sp; ++u) {
        const float2 w = part[u];
        v.x += w.x;
        v.y += w.y;
      }
      epilogue_pair<MOE>(c, l, ph, i, v.x, v.y, xraw, pos, sid);
    }
  }
}

// The per-projection scratch of phase ph: slot counters of split pairs and (QKV) the RoPE factors
// of the CTA's q and k pairs (asynchronous copies, completed by the staging's wait).  A CTA
// barrier must follow before the projection.
__device__ void phase_setup(const Ctx& c, int ph, int pos) {
  const MegaArgs& a = *c.a;
  const Split& p = c.split()[ph];
  const int tid = threadIdx.x;
  if (p.gs != p.sp)
    for (int i = tid; i < p.np; i += kMT) c.cnt()[i] = 0;
  if (ph == kPhQKV) {
    const int hd = a.D >> 1;
    for (int i = tid; i < p.np; i += kMT) {
      const int t = p.p0 + i, head = t / hd;
      if (head < a.Hq + a.Hkv) cp_async8(c.rope_s() + i, a.rope + (size_t)pos * hd + (t - head * hd));
    }
  }
}

// One projection of block l: consume this warp's range from the ring, refilling behind; each
// finished pair piece goes to finish_piece.  Returns false (for the whole warp) after a
// timed-out wait (error set, copies drained); the caller makes the outcome CTA-uniform.
template <bool MOE>
__device__ bool gemv_phase(const Ctx& c, Stream& s, int l, int ph, const float* xs,
                           const float* xraw, int pos, int sid) {
  const Split& p = c.split()[ph];
  float acc0 = 0.f, acc1 = 0.f;
  for (Cur q = cur_start(p, c.warp); cur_valid(p, q, c.warp); cur_advance(p, q)) {
    const int slot = s.consumed % kDepth;
    const bool landed = mbar_wait(c.bars() + c.warp * kDepth + slot, (unsigned)(s.consumed / kDepth) & 1u, kWaitNs);
    if (!__all_sync(0xffffffffu, landed)) {  // warp-uniform decision
      if (c.lane == 0) set_error(c);
      stream_drain(c, s);
      return false;
    }
    // the slot's bytes go to registers (lane: chunks lane + 32 u of both rows) and the ring slot
    // is refilled at once, so the ring keeps kDepth slots in flight while this one is summed
    const unsigned char* sq = c.ringq() + (size_t)(c.warp * kDepth + slot) * kSlotQ;
    const unsigned char* ss = c.rings() + (size_t)(c.warp * kDepth + slot) * kSlotS;
    const int nch = slot_len(p, q.j) >> 4, cb = slot_k(p, q.j) >> 4;
    constexpr int U = kSlotCols / 16 / 32;  // chunks of a row per lane
    uint4 wa[U], wb[U];
    uint32_t sab[U];  // the two rows' fp16 scales of each chunk
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cl = c.lane + 32 * u;
      if (cl < nch) {
        wa[u] = *reinterpret_cast<const uint4*>(sq + cl * 16);
        wb[u] = *reinterpret_cast<const uint4*>(sq + p.sl + cl * 16);
        sab[u] = (uint32_t)*reinterpret_cast<const uint16_t*>(ss + (cl >> 1) * 2) |
                 ((uint32_t)*reinterpret_cast<const uint16_t*>(ss + p.sl / 16 + (cl >> 1) * 2) << 16);
      }
    }
    __syncwarp();  // the slot is read: refill it
    ++s.consumed;
    stream_issue<MOE>(c, s);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int cl = c.lane + 32 * u;
      if (cl < nch) {
        const int ch = cb + cl;
        const int sw = (ch >> 1) & 3;
        const uint4* xp = reinterpret_cast<const uint4*>(xs + ch * 16);
        const uint4 l0 = xp[0 ^ sw], l1 = xp[1 ^ sw], l2 = xp[2 ^ sw], k = xp[3 ^ sw];
        const float ek = __uint_as_float(k.w);  // the chunk's unit u
        const float f0 = h2f_bits((uint16_t)(sab[u] & 0xFFFFu)) * ek, f1 = h2f_bits((uint16_t)(sab[u] >> 16)) * ek;
        acc0 = fmaf(f0, q8_chunk_dot(wa[u], l0, l1, l2, k), acc0);
        acc1 = fmaf(f1, q8_chunk_dot(wb[u], l0, l1, l2, k), acc1);
      }
    }
    finish_slot<MOE>(c, l, ph, q.pr, q.j, acc0, acc1, xraw, pos, sid);
  }
  return true;
}

// Routing of MoE block l: every CTA gathers all router logits (tagged, as they arrive), takes
// the top_k by rank (ties to the lower id) and their softmax; ids, weights and the ready block
// into shared memory.  False after a timed-out wait (CTA-uniform).
__device__ bool rank_experts(const Ctx& c, int l) {
  const MegaArgs& a = *c.a;
  float* sel = c.sel();
  int* sel_id = c.sel_id();
  int* ids = c.moe_ids();
  float* wts = c.moe_wts();
  const int E = a.n_experts, k = a.top_k;
  if (threadIdx.x < k) sel_id[threadIdx.x] = threadIdx.x;  // valid ids whatever the logits hold
  // the slot partials' region is free between the router projection and the experts' setup
  const bool got = gather_tagged(c, c.tlog(), E, E, E, c.tag(l), reinterpret_cast<tagged_t*>(c.part()), c.logits());
  if (!__syncthreads_and(got)) return false;
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
  return true;
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

// Split-K attention of block l over this CTA's items (KV head, chunk of positions): q of the
// head's group and (for the chunk holding the current position) the current K and V rows are
// gathered from their tagged vectors as they arrive; the chunk's partial (running max and sum,
// unnormalised output) goes to global memory, and the chunk that arrives last on its head's
// counter merges all of the head's chunks (weights e^(m_c - M), sums in chunk order) into the
// tagged attention output.  `prefetched`: tile 0 of the first item was issued earlier.
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
    const unsigned tg = c.tag(l) + a.bar_extra;
    bool got = true;
    for (int i = tid; 2 * i < G * D && got; i += kMT) {  // q of the group, as it arrives
      const int g = 2 * i / D, d = 2 * i - g * D;
      float2 v;
      got = poll_pair(c, c.tq() + (size_t)kvh * G * D + 2 * i, tg, v);
      qs[g * D + q_slot<D>(d)] = v.x;
      qs[g * D + q_slot<D>(d + 1)] = v.y;
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
      if (nold < np) {  // the current position: this launch's K and V rows, from their tagged copies
        const int r = pos - p0;
        for (int i = tid; 2 * i < 2 * D && got; i += kMT) {
          const bool is_v = 2 * i >= D;
          const int d = 2 * i - (is_v ? D : 0);
          float2 v;
          got = poll_pair(c, c.tkv() + ((size_t)(is_v ? a.Hkv : 0) + kvh) * D + d, tg, v);
          *reinterpret_cast<__half2*>((is_v ? Vs : Ks) + (size_t)r * D + d) = __floats2half2_rn(v.x, v.y);
        }
      }
      const bool landed = mbar_wait(abar, aphase & 1u, kWaitNs);
      if (!__syncthreads_and(landed && got)) {  // CTA-uniform decision (also orders the row copy above)
        if (tid == 0) set_error(c);
        return false;
      }
      ++aphase;
      // scores: four lanes per position, a quarter of the dims each, all G heads of the group at
      // once (every K element read once); the 16-byte pieces of a quarter are walked in a
      // rotated order so that the lanes' rows fall in distinct banks; the quarters are added
      // with two shuffles
      constexpr int QD = D / 4, QP = QD / 8;
      for (int idx = tid; idx < 4 * T; idx += kMT) {
        const int p = idx >> 2, qt = idx & 3;
        float acc[G];
#pragma unroll
        for (int g = 0; g < G; ++g) acc[g] = 0.f;
        if (p < np) {
          const __half* kr = Ks + (size_t)p * D + qt * QD;
#pragma unroll 1
          for (int i = 0; i < QP; ++i) {
            const int j = (i + p) & (QP - 1);
            const uint4 kk = *reinterpret_cast<const uint4*>(kr + 8 * j);
            const float2 k01 = __half22float2(*reinterpret_cast<const __half2*>(&kk.x));
            const float2 k23 = __half22float2(*reinterpret_cast<const __half2*>(&kk.y));
            const float2 k45 = __half22float2(*reinterpret_cast<const __half2*>(&kk.z));
            const float2 k67 = __half22float2(*reinterpret_cast<const __half2*>(&kk.w));
            const int m = qt * QP + j;  // the 8-dim piece of the head's D dims
#pragma unroll
            for (int g = 0; g < G; ++g) {
              const float4 qa = *reinterpret_cast<const float4*>(qs + g * D + 4 * m);
              const float4 qb = *reinterpret_cast<const float4*>(qs + g * D + D / 2 + 4 * m);
              float sc = acc[g];
              sc = fmaf(qa.x, k01.x, sc);
              sc = fmaf(qa.y, k01.y, sc);
              sc = fmaf(qa.z, k23.x, sc);
              sc = fmaf(qa.w, k23.y, sc);
              sc = fmaf(qb.x, k45.x, sc);
              sc = fmaf(qb.y, k45.y, sc);
              sc = fmaf(qb.z, k67.x, sc);
              sc = fmaf(qb.w, k67.y, sc);
              acc[g] = sc;
            }
          }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
          acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 1);
          acc[g] += __shfl_xor_sync(0xffffffffu, acc[g], 2);
        }
        if (qt == 0 && p < np)
#pragma unroll
          for (int g = 0; g < G; ++g) S[g * T + p] = acc[g] * a.scale;
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
    // every thread's partial writes, then one arrival on the head's counter (monotonic within a
    // launch); the chunk that completes the head merges it
    __syncthreads();
    if (tid == 0) c.flag()[1] = atom_add_acq_rel(a.bar + 2 + kvh, 1u) == (unsigned)(l + 1) * (unsigned)nch - 1u;
    __syncthreads();
    if (!c.flag()[1]) continue;
    constexpr int GD = G * D;
    constexpr int CB = (2 * T * D * 2) / (GD * 4);  // chunk partials that fit over the K/V tiles
    float2* mls = reinterpret_cast<float2*>(area + AL::mls);  // [G][nch]
    float* wts = reinterpret_cast<float*>(area + AL::wts);    // [nch][G]
    float* pst = reinterpret_cast<float*>(area + AL::ks);     // [CB][GD] chunk partials
    const float* pk = a.part_o + (size_t)kvh * nch * GD;
    // the (max, sum) pairs and the first chunks' partials of the head, each fetched at once
    for (int i = tid; i < G * nch; i += kMT) cp_async8(mls + i, a.part_ml + (size_t)kvh * G * nch + i);
    for (int i = tid; i < min(nch, CB) * GD / 4; i += kMT) cp_async16(pst + 4 * i, pk + 4 * i);
    cp_async_wait_all();
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
    // a thread per output (GD <= 2 kMT), the chunks in order, CB chunks per batch
    float acc0 = 0.f, acc1 = 0.f;
    for (int ck0 = 0; ck0 < nch; ck0 += CB) {
      if (ck0 > 0) {
        __syncthreads();  // the previous batch is read
        for (int i = tid; i < min(CB, nch - ck0) * GD / 4; i += kMT)
          cp_async16(pst + 4 * i, pk + (size_t)ck0 * GD + 4 * i);
        cp_async_wait_all();
        __syncthreads();
      }
      for (int ck = ck0; ck < min(nch, ck0 + CB); ++ck) {
        const float* pc = pst + (size_t)(ck - ck0) * GD;
        acc0 = fmaf(wts[ck * G + tid / D], pc[tid], acc0);
        if (tid + kMT < GD) acc1 = fmaf(wts[ck * G + (tid + kMT) / D], pc[tid + kMT], acc1);
      }
    }
    if (tid < GD) st_tag(c.to() + (size_t)kvh * GD + tid, acc0 / st_L[tid / D], c.tag(l));
    if (tid + kMT < GD) st_tag(c.to() + (size_t)kvh * GD + tid + kMT, acc1 / st_L[(tid + kMT) / D], c.tag(l));
    __syncthreads();  // the merge scratch is read before the next item's tile lands
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
  // the union area: the per-projection scratch, then the staged input (a tagged input is
  // gathered beyond the current projection's Kp), or the attention tiles
  c.ps = area;
  float* xs = reinterpret_cast<float*>(area + kPsBytes);

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
  c.seq = __ldcg(a.bar + kSeqWord);

  Stream s;
  s.l = 0;
  s.ph = 0;
  s.q = cur_start(splits[0], c.warp);
  s.issued = 0;
  s.consumed = 0;
  if (c.lane == 0 && a.nl > 0) {
    c.wptr()[2 * c.warp] = &a.layers[0].tmap[0];
    c.wptr()[2 * c.warp + 1] = &a.layers[0].tmap[1];
  }
  __syncwarp();
  if (!cur_valid(splits[0], s.q, c.warp)) stream_normalise<MOE>(c, s);
  for (int d = 0; d < kDepth; ++d) stream_issue<MOE>(c, s);

  unsigned aphase = 0;
  bool ok = true;
  constexpr bool moe = MOE;
  // One call site per step (the projection step is the same code for every phase: the kernel
  // stays small enough for the instruction cache).  No grid barrier: each step waits for the
  // tagged entries it reads, and a CTA reads a step's input only if it has work in the step --
  // so every reader of a vector produces a share of what the vector's next writers wait for.
  for (int l = 0; l < a.nl && ok; ++l) {
    const MegaLayer& L = a.layers[l];
    for (int ph = 0; ph < kPhases && ok; ++ph) {
      if (ph == kPhRouter && !moe) continue;
      const Split& sp = splits[ph];
      if (ph == kPhGU && moe) {
        stream_refill<MOE>(c, s);  // the routing is known: the selected experts' slices stream in
        phase_setup(c, ph, pos);
        __syncthreads();
      } else if (sp.np > 0 || (MOE && ph == kPhRouter)) {  // MoE: every CTA stages the router input
        // the projection's input: QKV and the router (or the dense gate/up) normalise the
        // residual (gamma_1, gamma_2; the raw residual is kept for the residual adds), O and
        // down take the attention output and the SwiGLU output as they are; the experts'
        // gate/up reuses the router's input
        const bool norm2 = ph == kPhRouter || ph == kPhGU;
        const int K = ph == kPhO ? a.Hq * a.D : ph == kPhDown ? a.F : a.H;
        const int Kp = ph == kPhO ? KpQ : ph == kPhDown ? KpF : KpH;
        const float* gamma = ph == kPhQKV ? L.attn_norm : norm2 ? L.ffn_norm : nullptr;
        // the gamma of the next normalising step is fetched into L2 one step ahead (the weight
        // stream evicts it between blocks): one 128-byte line per CTA
        if (threadIdx.x == 0 && (ph == kPhO || ph == kPhDown)) {
          const float* g = ph == kPhO ? L.ffn_norm : (l + 1 < a.nl ? a.layers[l + 1].attn_norm : nullptr);
          for (int i = blockIdx.x * 32; g && i < a.H; i += gridDim.x * 32) prefetch_l2_last(g + i);
        }
        phase_setup(c, ph, pos);
        if (ph == kPhQKV && l == 0) {  // the launch's input, written before the launch
          stage_issue(a.hin, K, Kp, gamma, xs, xraw);
        } else if (ph == kPhDown) {  // the SwiGLU output of every CTA
          ok = stage_counted(c, a.bar, (unsigned)(l + 1) * gridDim.x, a.abuf, K, Kp, xs, xraw);
        } else {
          const tagged_t* in = ph == kPhQKV ? c.th() : ph == kPhO ? c.to() : c.tx1();
          ok = stage_gather(c, in, K, Kp, K, K, c.tag(ph == kPhQKV ? l - 1 : l), gamma, xs, xraw,
                            reinterpret_cast<tagged_t*>(xs + Kp));
        }
        if (!ok) break;
        stage_finish(c, K, Kp, gamma, a.eps, xs, xraw);
      }
      ok = __syncthreads_and(gemv_phase<MOE>(c, s, l, ph, xs, xraw, pos, sid));
      if (ok && ph == kPhGU && threadIdx.x == 0)  // this CTA's SwiGLU outputs are written (barrier above)
        red_release_add(a.bar, 1u);
      if (ok && ph == kPhQKV) {
        // tile 0 of this CTA's first attention item (positions of earlier steps) streams in
        // while q, k and v arrive
        bool pre = false;
        if ((int)blockIdx.x < a.Hkv * a.n_chunks) {
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
        ok = attention_phase<D, G>(c, l, area, aphase, pre, pos, sid);
        if (!ok && pre && threadIdx.x == 0) mbar_wait(c.bars() + kMW * kDepth, aphase & 1u, kWaitNs);
      }
      if (MOE && ok && ph == kPhRouter) ok = rank_experts(c, l);
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
  // the staged input (the integer form: as many bytes as its floats), or a tagged input (H or
  // q_dim entries of 8 bytes) gathered beyond the projection's Kp floats
  const size_t gather = std::max((size_t)pad256(H) * 4 + (size_t)H * 8, (size_t)pad256(q_dim) * 4 + (size_t)q_dim * 8);
  const size_t u = std::max(kPsBytes + std::max((size_t)Kx * 4, gather), attn);
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

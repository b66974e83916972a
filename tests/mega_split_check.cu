// Host check of the persistent decode's work split: split_of and the warp cursors of
// mega_impl.cuh, compiled for the host and run for every model shape below over several grid
// sizes.  For each projection it checks what the weight stream's tensor copies rely on:
//   - the CTAs' pair ranges partition the projection's row pairs, and every row count is even
//     (a slot box is two rows);
//   - every slot starts inside its row on a 256-column boundary (both boxes of a slot then start
//     on a 16-byte boundary) and is at most a ring slot wide;
//   - the 16 warps' cursors visit every (pair, slot) of the CTA exactly once, and no warp holds
//     more than one group more than another;
//   - a CTA's split-pair scratch (kMaxCtaPairs entries) holds its pairs, for every grid size at
//     which the persistent decode accepts the shape, and the slots of its pairs whenever pairs of
//     several slots are dealt slot by slot.
// Prints one line per failure and a summary; exits 1 if anything failed.
#include <cstdio>
#include <vector>

#include "mega_impl.cuh"

using namespace lrs;

namespace {

struct Shape {
  const char* name;
  int H, Hq, Hkv, D, F;   // F: dense FFN width (0 for MoE)
  int E, top_k, EF;       // MoE: experts, selected per token, expert FFN width
};

int g_fail = 0;
long g_checked = 0;

void fail(const Shape& s, int G, int ph, int cta, const char* what, int a, int b) {
  if (g_fail++ < 40) std::printf("FAIL %s G=%d phase=%d cta=%d: %s (%d, %d)\n", s.name, G, ph, cta, what, a, b);
}

DevQ8 mat(int N, int K) {
  DevQ8 m;
  m.N = N;
  m.K = K;
  m.Kp = pad256(K);
  return m;
}

void check_shape(const Shape& s, int G) {
  const bool moe = s.E > 0;
  MegaLayer L;
  L.wqkv = mat((s.Hq + 2 * s.Hkv) * s.D, s.H);
  L.wo = mat(s.H, s.Hq * s.D);
  if (moe) {
    L.router = mat(s.E, s.H);
    L.egu = mat(s.E * 2 * s.EF, s.H);
    L.edown = mat(s.E * s.H, s.EF);
  } else {
    L.wgu = mat(2 * s.F, s.H);
    L.wdown = mat(s.H, s.F);
  }
  MegaArgs a;
  a.layers = &L;
  a.nl = 1;
  a.H = s.H;
  a.Hq = s.Hq;
  a.Hkv = s.Hkv;
  a.D = s.D;
  a.F = moe ? s.top_k * pad256(s.EF) : s.F;
  a.n_experts = s.E;
  a.top_k = s.top_k;
  a.EF = s.EF;
  // rows of each projection as the stream sees them (MoE gate/up: the selected experts' rows;
  // down: H rows gathered over the experts)
  const int rows[kPhases] = {L.wqkv.N, L.wo.N, moe ? s.E : 0, moe ? s.top_k * 2 * s.EF : 2 * s.F, s.H};
  for (int ph = 0; ph < kPhases; ++ph) {
    if (rows[ph] % 2) fail(s, G, ph, -1, "odd row count", rows[ph], 0);
    // the persistent decode declines a shape whose fullest CTA holds more pairs than this
    const bool accepted = (rows[ph] / 2 + G - 1) / G <= kMaxCtaPairs;
    int next = 0;
    for (int cta = 0; cta < G; ++cta) {
      const Split p = split_of(a, ph, cta, G);
      ++g_checked;
      if (p.p0 != next) fail(s, G, ph, cta, "pair ranges not contiguous", p.p0, next);
      next = p.p0 + p.np;
      if (p.NP * 2 != rows[ph]) fail(s, G, ph, cta, "pairs of the projection", p.NP, rows[ph]);
      if (p.np == 0) continue;
      if (p.sl <= 0 || p.sl % 256 || p.sl > kSlotCols) fail(s, G, ph, cta, "slot width", p.sl, kSlotCols);
      if (p.sp < 1) fail(s, G, ph, cta, "slots per pair", p.sp, 0);
      for (int j = 0; j < p.sp; ++j) {
        const int k = slot_k(p, j), len = slot_len(p, j);
        if (k % 256 || len <= 0 || k + len > p.Kp) fail(s, G, ph, cta, "slot outside its row", k, len);
        if (p.mode == 2 && (k != j * p.seg || len != p.seg)) fail(s, G, ph, cta, "gathered piece", k, len);
      }
      if (p.gs != 1 && p.gs != p.sp) fail(s, G, ph, cta, "group size", p.gs, p.sp);
      if (p.ng * p.gs != p.np * p.sp) fail(s, G, ph, cta, "groups", p.ng, p.np * p.sp);
      if (accepted && p.np > kMaxCtaPairs) fail(s, G, ph, cta, "pairs above the scratch", p.np, kMaxCtaPairs);
      // single-slot groups of pairs with several slots: every slot's partial has an entry
      if (p.gs == 1 && p.sp > 1 && p.np * p.sp > kMaxCtaPairs)
        fail(s, G, ph, cta, "slots above the scratch", p.np * p.sp, 0);
      std::vector<int> seen((size_t)p.np * p.sp, 0);
      int most = 0, least = 1 << 30;
      for (int w = 0; w < kMW; ++w) {
        Cur q = cur_start(p, w);
        int mine = 0;
        while (cur_valid(p, q, w)) {
          if (q.pr < 0 || q.pr >= p.np || q.j < 0 || q.j >= p.sp) {
            fail(s, G, ph, cta, "cursor outside the CTA's slots", q.pr, q.j);
            break;
          }
          ++seen[(size_t)q.pr * p.sp + q.j];
          if (++mine > p.np * p.sp) {
            fail(s, G, ph, cta, "cursor does not end", w, mine);
            break;
          }
          cur_advance(p, q);
        }
        most = mine > most ? mine : most;
        least = mine < least ? mine : least;
      }
      for (size_t i = 0; i < seen.size(); ++i)
        if (seen[i] != 1) {
          fail(s, G, ph, cta, "slot visited other than once", (int)i, seen[i]);
          break;
        }
      if (most - least > p.gs) fail(s, G, ph, cta, "warps unevenly loaded", most, least);
    }
    if (next * 2 != rows[ph]) fail(s, G, ph, G, "pairs covered", next, rows[ph] / 2);
  }
}

}  // namespace

int main() {
  const Shape shapes[] = {
      {"tiny dense", 256, 4, 2, 64, 688, 0, 0, 0},
      {"8B dense", 4096, 32, 8, 128, 14336, 0, 0, 0},
      {"70B dense", 8192, 64, 8, 128, 28672, 0, 0, 0},
      {"dense, hidden not a multiple of 256", 4100, 32, 8, 128, 11008, 0, 0, 0},
      {"A3B MoE", 2048, 32, 4, 128, 0, 128, 8, 768},
      {"small MoE", 256, 4, 2, 64, 0, 8, 2, 64},
      {"MoE, expert width not a multiple of 256", 1024, 16, 4, 64, 0, 16, 4, 96},
  };
  const int grids[] = {152, 148, 132, 160, 304, 76, 7, 2, 1, 3};
  for (const Shape& s : shapes)
    for (int G : grids) check_shape(s, G);
  std::printf("%ld splits checked, %d failures\n", g_checked, g_fail);
  return g_fail ? 1 : 0;
}

// Persistent decode: the dense kernels and the host entry points (the kernel itself is in
// mega_impl.cuh).

#include <cstring>

#include "mega_impl.cuh"

namespace lrs {
namespace {

bool g_mega_ready = false;

}  // namespace

bool mega_supported(int H, int q_dim, int F, int head_dim, int group, int n_experts, int top_k) {
  if (!g_mega_ready) return false;
  if (n_experts > kMaxExperts || top_k > kMaxTopK || (n_experts > 0 && top_k < 1)) return false;
  if (n_experts > 0 && F % top_k) return false;
  if (n_experts & 1) return false;  // router rows go in pairs
  if (head_dim != 64 && head_dim != 128) return false;
  if (group != 1 && group != 2 && group != 4 && group != 8) return false;
  if (q_dim / head_dim / group > 62) return false;  // per-KV-head counters in the 64-word barrier block
  if ((H & 3) || (q_dim & 3) || (F & 3)) return false;
  const int Kx = std::max(pad256(H), std::max(pad256(q_dim), pad256(F)));
  if (Kx > kMaxKp) return false;
  // pairs of the fullest CTA in each projection (rows: QKV, O, router, gate/up or the selected
  // experts' rows, down)
  const int G = sm_count();
  const int rows[] = {q_dim + 2 * (q_dim / group), H, n_experts, 2 * F, H};
  for (int r : rows)
    if ((r / 2 + G - 1) / G > kMaxCtaPairs) return false;
  if (n_experts > 0 && F / top_k > kSlotCols) return false;  // an expert's down piece fits a slot
  return mega_smem(H, q_dim, F, head_dim, group) <= kMaxSmem;
}

bool mega_tensor_maps(MegaLayer& ml, bool moe) {
  std::memset(static_cast<void*>(ml.tmap), 0, sizeof ml.tmap);
  const DevQ8* m[kPhases] = {&ml.wqkv, &ml.wo, moe ? &ml.router : nullptr, moe ? &ml.egu : &ml.wgu,
                             moe ? &ml.edown : &ml.wdown};
  for (int ph = 0; ph < kPhases; ++ph) {
    if (!m[ph] || !m[ph]->q || m[ph]->N <= 0) continue;
    const DevQ8& w = *m[ph];
    // a ring slot of two rows (the last slot of a row may reach past Kp: zero filled); the
    // bytes and the fp16 scales as 8-byte elements
    const int sl = std::min(kSlotCols, w.Kp);
    if (w.Kp % 256 || ((uintptr_t)w.q & 15) || ((uintptr_t)w.s & 15)) return false;
    if (!encode_2d(&ml.tmap[2 * ph], CU_TENSOR_MAP_DATA_TYPE_UINT64, w.q, (uint64_t)w.Kp / 8, (uint64_t)w.N,
                   (uint64_t)w.Kp, (uint32_t)sl / 8, 2, CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !encode_2d(&ml.tmap[2 * ph + 1], CU_TENSOR_MAP_DATA_TYPE_UINT64, w.s, (uint64_t)w.Kp / 128, (uint64_t)w.N,
                   (uint64_t)w.Kp / 16, (uint32_t)sl / 128, 2, CU_TENSOR_MAP_SWIZZLE_NONE))
      return false;
  }
  return true;
}

size_t mega_tag_entries(int H, int q_dim, int kv_dim, int n_experts) {
  return (size_t)2 * q_dim + 2 * (size_t)kv_dim + 2 * (size_t)H + ((n_experts + 1) & ~1);
}

int mega_chunks(int n_kv_heads) { return std::max(1, std::min(kAttnMaxChunks, sm_count() / std::max(1, n_kv_heads))); }

cudaError_t prepare_mega() {
  int dev = 0, coop = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
  if (e != cudaSuccess) return e;
  if (!coop) return cudaSuccess;  // persistent decode unavailable: mega_supported() stays false
  if ((e = prepare_mega_all<false>()) != cudaSuccess || (e = prepare_mega_moe()) != cudaSuccess) return e;
  int nb = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, mega_decode_kernel<128, 4, false>, kMT, kMaxSmem - 128);
  if (e != cudaSuccess) return e;
  g_mega_ready = nb >= 1;
  return cudaSuccess;
}

cudaError_t launch_mega_decode(const MegaArgs& a, cudaStream_t st) {
  const int G = a.Hq / a.Hkv;
  if (!mega_supported(a.H, a.Hq * a.D, a.F, a.D, G, a.n_experts, a.top_k)) return cudaErrorInvalidValue;
  if (a.n_chunks < 1 || a.n_chunks > kAttnMaxChunks || a.nl > 255 || !a.tags) return cudaErrorInvalidValue;
  const size_t smem = mega_smem(a.H, a.Hq * a.D, a.F, a.D, G);
  return a.n_experts > 0 ? launch_mega_moe(a, smem, st) : launch_mega_all<false>(a, smem, st);
}

}  // namespace lrs

// Persistent decode: the MoE kernels (router and top-k inside the launch; the kernel itself is
// in mega_impl.cuh).

#include "mega_impl.cuh"

namespace lrs {

cudaError_t prepare_mega_moe() { return prepare_mega_all<true>(); }

cudaError_t launch_mega_moe(const MegaArgs& a, size_t smem, cudaStream_t st) {
  return launch_mega_all<true>(a, smem, st);
}

}  // namespace lrs

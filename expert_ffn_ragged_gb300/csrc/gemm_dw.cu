// gemm_dw.cu -- the trans_ragged_dot grouped GEMM (per-group weight gradient):
// bf16 output, f32 output, f32 accumulation into the output; single-CTA and
// CTA-pair variants.
#include "gemm_kernel.cuh"

namespace rd {
template <bool PAIR>
static cudaError_t launch_dw(int epi, const CUtensorMap& a, const CUtensorMap& b,
                             const GemmArgs& args, int grid, cudaStream_t s) {
  switch (epi) {
    case kEpiF32: return launch_gemm_impl<kOpDw, kEpiF32, PAIR>(a, b, args, grid, s);
    case kEpiF32Acc: return launch_gemm_impl<kOpDw, kEpiF32Acc, PAIR>(a, b, args, grid, s);
    default: return launch_gemm_impl<kOpDw, kEpiNone, PAIR>(a, b, args, grid, s);
  }
}

cudaError_t launch_gemm_dw(bool pair, int epi, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmArgs& args, int grid, cudaStream_t s) {
  return pair ? launch_dw<true>(epi, a, b, args, grid, s) : launch_dw<false>(epi, a, b, args, grid, s);
}
}  // namespace rd

// gemm_dw.cu -- the trans_ragged_dot grouped GEMM (per-group weight gradient),
// single-CTA and CTA-pair variants.
#include "gemm_kernel.cuh"

namespace rd {
cudaError_t launch_gemm_dw(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmArgs& args, int grid, cudaStream_t s) {
  return pair ? launch_gemm_impl<kOpDw, false, true>(a, b, args, grid, s)
              : launch_gemm_impl<kOpDw, false, false>(a, b, args, grid, s);
}
}  // namespace rd

// gemm_dx.cu -- the trans_rhs grouped GEMM (input gradient), single-CTA and
// CTA-pair variants.
#include "gemm_kernel.cuh"

namespace rd {
cudaError_t launch_gemm_dx(bool pair, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmArgs& args, int grid, cudaStream_t s) {
  return pair ? launch_gemm_impl<kOpDx, false, true>(a, b, args, grid, s)
              : launch_gemm_impl<kOpDx, false, false>(a, b, args, grid, s);
}
}  // namespace rd

// gemm_dx.cu -- the trans_rhs grouped GEMM (input gradient), plain and with
// the fused SiLU-GLU backward epilogue, single-CTA and CTA-pair variants.
#include "gemm_kernel.cuh"

namespace rd {
cudaError_t launch_gemm_dx(bool pair, bool glu_bwd, const CUtensorMap& a, const CUtensorMap& b,
                           const GemmArgs& args, int grid, cudaStream_t s) {
  if (pair)
    return glu_bwd ? launch_gemm_impl<kOpDx, kEpiGluBwd, true>(a, b, args, grid, s)
                   : launch_gemm_impl<kOpDx, kEpiNone, true>(a, b, args, grid, s);
  return glu_bwd ? launch_gemm_impl<kOpDx, kEpiGluBwd, false>(a, b, args, grid, s)
                 : launch_gemm_impl<kOpDx, kEpiNone, false>(a, b, args, grid, s);
}
}  // namespace rd

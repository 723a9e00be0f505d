// gemm_fwd.cu -- forward grouped GEMM (plain and with the fused SiLU-GLU
// epilogue), single-CTA and CTA-pair variants.
#include "gemm_kernel.cuh"

namespace rd {
cudaError_t launch_gemm_fwd(bool glu, bool pair, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmArgs& args, int grid, cudaStream_t s) {
  if (pair)
    return glu ? launch_gemm_impl<kOpFwd, kEpiGlu, true>(a, b, args, grid, s)
               : launch_gemm_impl<kOpFwd, kEpiNone, true>(a, b, args, grid, s);
  return glu ? launch_gemm_impl<kOpFwd, kEpiGlu, false>(a, b, args, grid, s)
             : launch_gemm_impl<kOpFwd, kEpiNone, false>(a, b, args, grid, s);
}
}  // namespace rd

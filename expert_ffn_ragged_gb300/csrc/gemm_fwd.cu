// gemm_fwd.cu -- forward grouped GEMM (plain and with the fused SiLU-GLU epilogue).
#include "gemm_kernel.cuh"

namespace rd {
cudaError_t launch_gemm_fwd(bool glu, const CUtensorMap& a, const CUtensorMap& b,
                            const GemmArgs& args, int grid, cudaStream_t s) {
  return glu ? launch_gemm_impl<kOpFwd, true>(a, b, args, grid, s)
             : launch_gemm_impl<kOpFwd, false>(a, b, args, grid, s);
}
}  // namespace rd

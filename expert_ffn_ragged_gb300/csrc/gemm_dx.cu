// gemm_dx.cu -- the trans_rhs grouped GEMM (input gradient).
#include "gemm_kernel.cuh"

namespace rd {
cudaError_t launch_gemm_dx(const CUtensorMap& a, const CUtensorMap& b, const GemmArgs& args,
                           int grid, cudaStream_t s) {
  return launch_gemm_impl<kOpDx, false>(a, b, args, grid, s);
}
}  // namespace rd

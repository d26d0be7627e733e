// Tensor-core skinny-GEMM instantiations for q4 weights (see gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace dfl {
cudaError_t launch_gemv_q4(int epi, int nt, const GemvArgs& a, int grid, size_t smem, cudaStream_t s) {
  return launch_gemv_fmt<FMT_Q4>(epi, nt, a, grid, smem, s);
}
}  // namespace dfl

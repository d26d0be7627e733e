// Tensor-core skinny-GEMM instantiations for bf16 weights (see gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace dfl {
cudaError_t launch_gemv_bf16(int epi, int nt, const GemvArgs& a, int grid, size_t smem, cudaStream_t s) {
  return launch_gemv_fmt<FMT_BF16>(epi, nt, a, grid, smem, s);
}
}  // namespace dfl

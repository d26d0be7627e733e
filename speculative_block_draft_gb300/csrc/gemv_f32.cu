// CUDA-core fp32 instantiations and the format dispatcher (see gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace dfl {

cudaError_t launch_gemv_q4(int epi, int nt, const GemvArgs& a, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_gemv_bf16(int epi, int nt, const GemvArgs& a, int grid, size_t smem, cudaStream_t s);

size_t gemv_smem_bytes(int fmt, int R, int gps, int x_lo) {
  if (fmt == FMT_F32) return 0;
  const int rp = R <= 8 ? 8 : (R <= 16 ? 16 : 32);
  const int w = gemv_warps(rp / 8);
  size_t b = (size_t)w * kStages * kStageBytes;        // weight rings
  b += (size_t)rp * (gps * 128 + 16) * (x_lo ? 2 : 1); // activation slice (and its f16 remainder)
  if (fmt == FMT_Q4) b += (size_t)rp * gps * 4;        // per-group activation sums
  b += kMaxRows * 4;                                   // row scales
  b += (size_t)w * kMaxRows * sizeof(LmState);         // vocab reduction scratch
  b += (size_t)2 * w * 32 * (rp / 2) * 4;              // split-strip pieces (2 per warp x 32 lanes x NT*4)
  b += 16 + (1 + w * kStages) * 8;                     // mbarriers
  return b;
}

cudaError_t launch_gemv(int fmt, int epi, int nt, const GemvArgs& a, int grid, cudaStream_t s) {
  const size_t smem = gemv_smem_bytes(fmt, a.R, a.gps, a.x_lo_off != 0);
  switch (fmt) {
    case FMT_Q4: return launch_gemv_q4(epi, nt, a, grid, smem, s);
    case FMT_BF16: return launch_gemv_bf16(epi, nt, a, grid, smem, s);
    case FMT_F32: return launch_gemv_fmt<FMT_F32>(epi, nt, a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfl

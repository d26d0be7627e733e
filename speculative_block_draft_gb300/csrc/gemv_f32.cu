// CUDA-core fp32 instantiations and the format dispatcher (see gemv_impl.cuh).
#include "gemv_impl.cuh"

namespace dfl {

cudaError_t launch_gemv_q4(int epi, int nt, const GemvArgs& a, int grid, size_t smem, cudaStream_t s);
cudaError_t launch_gemv_bf16(int epi, int nt, const GemvArgs& a, int grid, size_t smem, cudaStream_t s);

size_t gemv_smem_bytes(int fmt, int R, int gps, int x_lo, int lm, int cpart_cap) {
  if (fmt == FMT_F32) return 0;
  const int rp = R <= 8 ? 8 : (R <= 16 ? 16 : 32);
  const int w = gemv_warps(rp / 8);
  size_t b = (size_t)w * kStages * kStageBytes;        // weight rings
  b += (size_t)rp * (gps * 128 + 16) * (x_lo ? 2 : 1); // activation slice (and its f16 remainder)
  if (fmt == FMT_Q4) b += (size_t)rp * gps * 4;        // per-group activation sums
  b += kMaxRows * 4;                                   // row scales
  if (lm) b += (size_t)w * kMaxRows * sizeof(LmState); // vocab reduction scratch (LM head)
  b += (size_t)2 * w * 32 * (rp / 2) * 4;              // split-strip pieces (2 per warp x 32 lanes x NT*4)
  b += (size_t)cpart_cap * 32 * (rp / 2) * 4;          // cluster K split: partial tiles
  b += 16 + (2 + w * kStages) * 8;                     // mbarriers
  return b;
}

// Final vocab reduction: one CTA per activation row merges n_parts states (stride kMaxRows rows
// apart): thread j takes parts j, j + blockDim, ... in order (eight loads in flight), then a
// pairwise tree; the order is fixed, so the result is reproducible. Writes the greedy token and
// the softmax probability of that token.
__global__ void __launch_bounds__(256) lm_reduce_kernel(const float* __restrict__ parts, int n_parts,
                                                        int32_t* tok_out, float* conf_out, int out_stride) {
  __shared__ LmState sm[256];
  const int c = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  LmState acc{-INFINITY, 0.f, 0x7fffffff};
  for (int b0 = threadIdx.x; b0 < n_parts; b0 += 8 * blockDim.x) {
    LmState o[8];
#pragma unroll
    for (int q = 0; q < 8; q++) {
      const int b = b0 + q * blockDim.x;
      const float* src = parts + ((size_t)b * kMaxRows + c) * 3;
      o[q] = b < n_parts ? LmState{__ldcg(src), __ldcg(src + 1), __float_as_int(__ldcg(src + 2))}
                         : LmState{-INFINITY, 0.f, 0x7fffffff};
    }
#pragma unroll
    for (int q = 0; q < 8; q++) lm_merge(acc, o[q]);
  }
  sm[threadIdx.x] = acc;
  __syncthreads();
  for (int off = blockDim.x / 2; off > 0; off >>= 1) {
    if ((int)threadIdx.x < off) lm_merge(sm[threadIdx.x], sm[threadIdx.x + off]);
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    tok_out[(size_t)c * out_stride] = sm[0].i;
    if (conf_out) conf_out[(size_t)c * out_stride] = 1.0f / sm[0].s;
  }
}

cudaError_t launch_lm_reduce(const float* parts, int n_parts, int rows, int32_t* tok_out, float* conf_out,
                             int out_stride, cudaStream_t s) {
  return launch_pdl(lm_reduce_kernel, dim3(rows), dim3(256), 0, s, parts, n_parts, tok_out, conf_out, out_stride);
}

cudaError_t launch_gemv(int fmt, int epi, int nt, const GemvArgs& a, int grid, cudaStream_t s) {
  const size_t smem = gemv_smem_bytes(fmt, a.R, a.gps, a.x_lo_off != 0, epi == EPI_LMHEAD,
                                     a.cluster2 ? a.cpart_cap : 0);
  switch (fmt) {
    case FMT_Q4: return launch_gemv_q4(epi, nt, a, grid, smem, s);
    case FMT_BF16: return launch_gemv_bf16(epi, nt, a, grid, smem, s);
    case FMT_F32: return launch_gemv_fmt<FMT_F32>(epi, nt, a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfl

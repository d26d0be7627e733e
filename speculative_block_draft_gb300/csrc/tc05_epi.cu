// Epilogues of the round's projections when they run on the many-row tcgen05 contraction. The K
// slices' partial tiles are summed in slice order and handed, one 16-row strip per warp, to the
// same strip epilogues the skinny GEMV fuses: context rows x ctx_norm with sums of squares,
// row-norm scale, Q/K/V split, residual with next norm input and sums of squares, gated FFN, and
// vocab states. One launch covers every row chunk of a projection (grid.y = chunk); row c of
// chunk j is contraction row row_base[j] + map_row(xmap_j, c).
#include "gemm_tc05.h"
#include "gemv_impl.cuh"

namespace dfl {

namespace {

template <int NT, int EPI>
__global__ void __launch_bounds__(kF32Warps * 32)
    tc05_epi_kernel(const __grid_constant__ Tc05EpiChunks ch, const float* __restrict__ part, int slices, int npad,
                    int n_out_pad) {
  constexpr int RP = NT * 8;
  const GemvArgs& a = ch.a[blockIdx.y];   // this CTA's row chunk
  const int row_base = ch.row_base[blockIdx.y];
  __shared__ float srow[kMaxRows];
  __shared__ LmState sm_lm[kF32Warps * kMaxRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  pdl_launch_dependents();
  pdl_wait();   // the partial tiles and the row norms' sums of squares come from earlier kernels
  compute_row_scales(a, srow, RP);
  __syncthreads();
  LmState lm[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int p = 0; p < 2; p++) lm[nt][p] = LmState{-INFINITY, 0.f, 0x7fffffff};
  const size_t slice_stride = (size_t)npad * n_out_pad;   // part[slice][strip][row][16]
  for (int sl = blockIdx.x * kF32Warps + warp; sl < a.n_strips; sl += gridDim.x * kF32Warps) {
    const int strip = a.strip0 + sl;
    float y[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int p = 0; p < 2; p++) {
        const int c = nt * 8 + 2 * t + p;
        float y0 = 0.f, y1 = 0.f;
        if (c < a.R) {
          const float* src = part + ((size_t)strip * npad + row_base + map_row(a.xmap, c)) * 16 + g;
          for (int s = 0; s < slices; s++) {
            y0 += __ldcg(src + s * slice_stride);
            y1 += __ldcg(src + s * slice_stride + 8);
          }
        }
        y[nt][p] = y0;
        y[nt][2 + p] = y1;
      }
    EpiPre<NT> pre;
    epi_preload<EPI, NT, __half>(a, strip, pre);
    strip_epilogue<EPI, NT, __half>(a, strip, y, srow, lm, 0, pre);
  }
  if constexpr (EPI == EPI_LMHEAD) lm_finish<NT>(a, lm, sm_lm);
}

template <int EPI>
cudaError_t launch_epi(int nt, const Tc05EpiChunks& ch, const float* part, int slices, int npad, int n_out_pad,
                       int grid, cudaStream_t s) {
  const dim3 g(grid, ch.n);
  const dim3 b(kF32Warps * 32);
  switch (nt) {
    case 1: return launch_pdl(tc05_epi_kernel<1, EPI>, g, b, 0, s, ch, part, slices, npad, n_out_pad);
    case 2: return launch_pdl(tc05_epi_kernel<2, EPI>, g, b, 0, s, ch, part, slices, npad, n_out_pad);
    case 3: return launch_pdl(tc05_epi_kernel<3, EPI>, g, b, 0, s, ch, part, slices, npad, n_out_pad);
    case 4: return launch_pdl(tc05_epi_kernel<4, EPI>, g, b, 0, s, ch, part, slices, npad, n_out_pad);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_tc05_epilogue(int epi, int nt, const Tc05EpiChunks& ch, const float* part, int slices, int npad,
                                 int n_out_pad, int grid, cudaStream_t s) {
  if (ch.n < 1 || ch.n > kTcMaxChunks) return cudaErrorInvalidValue;
  switch (epi) {
    case EPI_CTX: return launch_epi<EPI_CTX>(nt, ch, part, slices, npad, n_out_pad, grid, s);
    case EPI_QKV: return launch_epi<EPI_QKV>(nt, ch, part, slices, npad, n_out_pad, grid, s);
    case EPI_RESID: return launch_epi<EPI_RESID>(nt, ch, part, slices, npad, n_out_pad, grid, s);
    case EPI_SWIGLU: return launch_epi<EPI_SWIGLU>(nt, ch, part, slices, npad, n_out_pad, grid, s);
    case EPI_LMHEAD: return launch_epi<EPI_LMHEAD>(nt, ch, part, slices, npad, n_out_pad, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfl

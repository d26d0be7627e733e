// Epilogues of the round's projections when they run on the many-row tcgen05 contraction. The K
// slices' partial tiles are summed in slice order and handed, one 16-row strip per warp, to the
// same strip epilogues the skinny GEMV fuses (the rows' norm scales computed once per projection by
// a one-CTA-per-chunk kernel before it), grid.z over the problems of a grouped launch: context rows x ctx_norm with sums of squares,
// row-norm scale, Q/K/V split, residual with next norm input and sums of squares, gated FFN, and
// vocab states. One launch covers every row chunk of a projection (grid.y = chunk); row c of
// chunk j is contraction row row_base[j] + map_row(xmap_j, c).
#include "gemm_tc05.h"
#include "gemv_impl.cuh"

namespace dfl {

namespace {

// One input plane per layer for the grouped context K/V: plane i of row r = (x_r * ctx_norm) *
// attn_norm_i, from the context epilogue's single plane (f16 and its f16 remainder), split again
// into f16 and remainder exactly as the skinny GEMV's K/V launch rescales its staged input. Plane 0
// overwrites the input in place (each element is read, then written, by the same thread).
__global__ void __launch_bounds__(256) tc05_kv_planes_kernel(__half* xw, long long lo_off, const float* attn_norm,
                                                             int rows, int d, int n_layers, long long plane) {
  pdl_launch_dependents();
  pdl_wait();   // the context epilogue wrote the input plane
  const int per_row = d / 8;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < (long long)rows * per_row;
       idx += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(idx / per_row), k8 = (int)(idx % per_row) * 8;
    const size_t off = (size_t)r * d + k8;
    const uint4 h4 = *reinterpret_cast<const uint4*>(xw + off);
    const uint4 l4 = *reinterpret_cast<const uint4*>(xw + lo_off + off);
    const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w}, lw[4] = {l4.x, l4.y, l4.z, l4.w};
    float v[8];
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const float2 fh = __half22float2(*reinterpret_cast<const __half2*>(&hw[q]));
      const float2 fl = __half22float2(*reinterpret_cast<const __half2*>(&lw[q]));
      v[2 * q] = fh.x + fl.x;
      v[2 * q + 1] = fh.y + fl.y;
    }
    for (int i = n_layers - 1; i >= 0; i--) {   // plane 0 last: it is the input
      const float4 a0 = *reinterpret_cast<const float4*>(attn_norm + (size_t)i * d + k8);
      const float4 a1 = *reinterpret_cast<const float4*>(attn_norm + (size_t)i * d + k8 + 4);
      const float w[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      uint32_t oh[4], ol[4];
#pragma unroll
      for (int q = 0; q < 4; q++) {
        const float va = v[2 * q] * w[2 * q], vb = v[2 * q + 1] * w[2 * q + 1];
        const __half ha = from_f<__half>(va), hb = from_f<__half>(vb);
        oh[q] = pack_f16x2(__half2float(ha), __half2float(hb));
        ol[q] = pack_f16x2(va - __half2float(ha), vb - __half2float(hb));
      }
      *reinterpret_cast<uint4*>(xw + (size_t)i * plane + off) = make_uint4(oh[0], oh[1], oh[2], oh[3]);
      *reinterpret_cast<uint4*>(xw + lo_off + (size_t)i * plane + off) = make_uint4(ol[0], ol[1], ol[2], ol[3]);
    }
  }
}

// The rows' norm scales of every chunk, once per projection (a CTA per chunk), instead of in each
// of the epilogue's CTAs: they sum hundreds of per-strip partials per row.
__global__ void __launch_bounds__(kF32Warps * 32)
    tc05_rowscale_kernel(const __grid_constant__ Tc05EpiChunks ch, float* __restrict__ srow_out) {
  __shared__ float srow[kMaxRows];
  pdl_launch_dependents();
  pdl_wait();   // the sums of squares come from earlier kernels
  compute_row_scales(ch.a[blockIdx.x], srow, kMaxRows);
  __syncthreads();
  if (threadIdx.x < kMaxRows) srow_out[blockIdx.x * kMaxRows + threadIdx.x] = srow[threadIdx.x];
}

template <int NT, int EPI>
__global__ void __launch_bounds__(kF32Warps * 32)
    tc05_epi_kernel(const __grid_constant__ Tc05EpiChunks ch, const float* __restrict__ part, int slices, int npad,
                    int n_out_pad, const float* __restrict__ srow_in, size_t part_layer_stride) {
  const GemvArgs& a = ch.a[blockIdx.y];   // this CTA's row chunk
  const int lyr = blockIdx.z;             // problem of a grouped launch (context K/V of every layer)
  part += (size_t)lyr * part_layer_stride;
  const int row_base = ch.row_base[blockIdx.y];
  __shared__ float srow[kMaxRows];
  __shared__ LmState sm_lm[kF32Warps * kMaxRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  pdl_launch_dependents();
  pdl_wait();   // the partial tiles and the row scales come from earlier kernels
  if (threadIdx.x < kMaxRows) srow[threadIdx.x] = srow_in[blockIdx.y * kMaxRows + threadIdx.x];
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
          const float* src = part + ((size_t)sl * npad + row_base + map_row(a.xmap, c)) * 16 + g;
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
    strip_epilogue<EPI, NT, __half>(a, strip, y, srow, lm, lyr, pre);
  }
  if constexpr (EPI == EPI_LMHEAD) lm_finish<NT>(a, lm, sm_lm);
}

// The LM head's epilogue on the contraction's partial tiles, for every row chunk in one pass: a CTA
// takes a range of strips (16 vocab entries each) and a thread one (chunk, row) pair (two threads
// per pair, alternate strips, when there are at most 128 pairs), so that a warp reads whole 64-byte
// row pieces of a strip, consecutive in memory; four strips' loads are in flight per thread. Each
// thread folds its logits (partial sums over the K slices, times the row's norm scale; written out
// when asked for) into a (max, sum, index) state; the CTA's state per row goes to the chunk's slice
// of vocab states, merged later per row by lm_reduce_kernel. Same arithmetic per logit as the
// generic epilogue; ties keep the lowest index.
constexpr int kLmThreads = 256;
__global__ void __launch_bounds__(kLmThreads)
    tc05_lm_epi_kernel(const __grid_constant__ Tc05EpiChunks ch, const float* __restrict__ part, int slices, int npad,
                       int n_out_pad, const float* __restrict__ srow_in, int n_pairs, int n_split) {
  __shared__ LmState sm[kLmThreads];
  pdl_launch_dependents();
  pdl_wait();   // the partial tiles and the row scales come from earlier kernels
  const int t = threadIdx.x;
  const int q = t % n_pairs, sp = t / n_pairs;   // (chunk, row) pair and strip parity of this thread
  const bool active = t < n_pairs * n_split;
  int j = 0, c = q;
  while (j + 1 < ch.n && c >= ch.a[j].R) {
    c -= ch.a[j].R;
    j++;
  }
  const GemvArgs& a = ch.a[j];
  const EpiArgs& e = a.e;
  const int row = ch.row_base[j] + map_row(a.xmap, c);
  const float sc = active ? srow_in[j * kMaxRows + c] : 0.f;
  const size_t slice_stride = (size_t)npad * n_out_pad;
  const int per = (a.n_strips + gridDim.x - 1) / gridDim.x;
  const int s_beg = blockIdx.x * per, s_end = min(a.n_strips, s_beg + per);
  LmState st{-INFINITY, 0.f, 0x7fffffff};
  float* lrow = e.logits ? e.logits + (size_t)c * (e.logit_row_stride ? e.logit_row_stride : e.vocab) : nullptr;
  if (active) {
    constexpr int U = 4;
    for (int s0 = s_beg + sp; s0 < s_end; s0 += U * n_split) {
      float4 v[U][4];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int sl = s0 + u * n_split;
        const float4* src = reinterpret_cast<const float4*>(part + ((size_t)sl * npad + row) * 16);
#pragma unroll
        for (int w = 0; w < 4; w++) v[u][w] = sl < s_end ? __ldcg(src + w) : make_float4(0.f, 0.f, 0.f, 0.f);
        for (int z = 1; z < slices; z++) {
          if (sl >= s_end) break;
#pragma unroll
          for (int w = 0; w < 4; w++) {
            const float4 o = __ldcg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) +
                                                                     z * slice_stride) + w);
            v[u][w].x += o.x;
            v[u][w].y += o.y;
            v[u][w].z += o.z;
            v[u][w].w += o.w;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int sl = s0 + u * n_split;
        if (sl >= s_end) break;
        const float y[16] = {v[u][0].x, v[u][0].y, v[u][0].z, v[u][0].w, v[u][1].x, v[u][1].y, v[u][1].z, v[u][1].w,
                             v[u][2].x, v[u][2].y, v[u][2].z, v[u][2].w, v[u][3].x, v[u][3].y, v[u][3].z, v[u][3].w};
        const int n0 = (a.strip0 + sl) * 16 - e.row_base;
#pragma unroll
        for (int k = 0; k < 16; k++) {
          const int n = n0 + k;
          if (n < 0 || n >= e.n_rows) continue;
          const float l = y[k] * sc;
          if (lrow) lrow[n] = l;
          lm_push(st, l, n);
        }
      }
    }
  }
  // merge the strip parities of a pair, then write the CTA's state per row
  sm[t] = st;
  __syncthreads();
  if (active && sp == 0) {
    for (int o = 1; o < n_split; o++) lm_merge(st, sm[t + o * n_pairs]);
    float* dst = e.lm_part + ((size_t)blockIdx.x * kMaxRows + c) * 3;
    dst[0] = st.m;
    dst[1] = st.s;
    dst[2] = __int_as_float(st.i);
  }
}

// Q/K/V and gated-FFN epilogues on the contraction's partial tiles, one thread per (row, strip): it
// reads the strip's 16 outputs of its row (64 contiguous bytes per K slice, consecutive rows in
// consecutive threads), scales them by the row's norm scale and writes them with 16-byte stores.
// Same arithmetic per element as the strip epilogues.
template <int EPI>
__global__ void __launch_bounds__(256)
    tc05_rowstrip_epi_kernel(const __grid_constant__ Tc05EpiChunks ch, const float* __restrict__ part, int slices,
                             int npad, int n_out_pad, const float* __restrict__ srow_in, int n_pairs) {
  static_assert(EPI == EPI_QKV || EPI == EPI_SWIGLU, "row-by-strip epilogues: Q/K/V and the gated FFN");
  pdl_launch_dependents();
  pdl_wait();   // the partial tiles and the row scales come from earlier kernels
  const int n_strips = ch.a[0].n_strips;
  const long long total = (long long)n_pairs * n_strips;
  const size_t slice_stride = (size_t)npad * n_out_pad;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int sl = (int)(idx / n_pairs);
    int c = (int)(idx - (long long)sl * n_pairs), j = 0;
    while (j + 1 < ch.n && c >= ch.a[j].R) {
      c -= ch.a[j].R;
      j++;
    }
    const GemvArgs& a = ch.a[j];
    const EpiArgs& e = a.e;
    const int row = ch.row_base[j] + map_row(a.xmap, c);
    const float sc = srow_in[j * kMaxRows + c];
    const float4* src = reinterpret_cast<const float4*>(part + ((size_t)sl * npad + row) * 16);
    // the K slices in order, four slices' loads in flight at a time
    float4 v4[4] = {make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f),
                    make_float4(0.f, 0.f, 0.f, 0.f), make_float4(0.f, 0.f, 0.f, 0.f)};
    for (int z0 = 0; z0 < slices; z0 += 4) {
      float4 t[4][4];
#pragma unroll
      for (int u = 0; u < 4; u++)
#pragma unroll
        for (int w = 0; w < 4; w++)
          t[u][w] = z0 + u < slices
                        ? __ldcg(reinterpret_cast<const float4*>(reinterpret_cast<const float*>(src) +
                                                                 (z0 + u) * slice_stride) + w)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int u = 0; u < 4; u++)
#pragma unroll
        for (int w = 0; w < 4; w++) {
          v4[w].x += t[u][w].x;
          v4[w].y += t[u][w].y;
          v4[w].z += t[u][w].z;
          v4[w].w += t[u][w].w;
        }
    }
    float y[16];
#pragma unroll
    for (int w = 0; w < 4; w++) {
      y[4 * w] = v4[w].x * sc;
      y[4 * w + 1] = v4[w].y * sc;
      y[4 * w + 2] = v4[w].z * sc;
      y[4 * w + 3] = v4[w].w * sc;
    }
    const int strip = a.strip0 + sl;
    const int n0 = strip * 16 - e.row_base;   // first output feature of the strip
    if constexpr (EPI == EPI_SWIGLU) {
      // strip rows 0-7 are gate rows, 8-15 the matching up rows; outputs strip * 8 + k
      const int j0 = strip * 8;
      float o[8];
#pragma unroll
      for (int k = 0; k < 8; k++) {
        const float g = y[k];
        const float ga = e.ffn_act == DFLASH_FFN_GELU
                             ? 0.5f * g * (1.0f + tanhf(0.7978845608028654f * fmaf(0.044715f * g, g * g, g)))
                             : g / (1.0f + __expf(-g));
        o[k] = ga * y[k + 8];
      }
      __half* dst = static_cast<__half*>(e.act) + (size_t)c * e.inter + j0;
      if (j0 + 8 <= e.inter) {
        uint32_t pk[4];
#pragma unroll
        for (int q = 0; q < 4; q++) pk[q] = pack_f16x2(__half2float(from_f<__half>(o[2 * q])),
                                                       __half2float(from_f<__half>(o[2 * q + 1])));
        *reinterpret_cast<uint4*>(dst) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
      } else {
        for (int k = 0; k < 8 && j0 + k < e.inter; k++) dst[k] = from_f<__half>(o[k]);
      }
    } else if constexpr (EPI == EPI_QKV) {
      // qd and kvd are multiples of 16: a strip lies in one of q, k, v
      __half* dst;
      if (n0 < e.qd) dst = static_cast<__half*>(e.q) + (size_t)c * e.qd + n0;
      else if (n0 < e.qd + e.kvd) dst = static_cast<__half*>(e.kb) + (size_t)c * e.kvd + n0 - e.qd;
      else dst = static_cast<__half*>(e.vb) + (size_t)c * e.kvd + n0 - e.qd - e.kvd;
      if (n0 + 16 <= e.n_rows) {
        uint32_t pk[8];
#pragma unroll
        for (int q = 0; q < 8; q++) pk[q] = pack_f16x2(__half2float(from_f<__half>(y[2 * q])),
                                                       __half2float(from_f<__half>(y[2 * q + 1])));
        reinterpret_cast<uint4*>(dst)[0] = make_uint4(pk[0], pk[1], pk[2], pk[3]);
        reinterpret_cast<uint4*>(dst)[1] = make_uint4(pk[4], pk[5], pk[6], pk[7]);
      } else {
        for (int k = 0; k < 16 && n0 + k < e.n_rows; k++) dst[k] = from_f<__half>(y[k]);
      }
    }
  }
}

template <int EPI>
cudaError_t launch_epi(int nt, const Tc05EpiChunks& ch, const float* part, int slices, int npad, int n_out_pad,
                       int grid, float* srow, int n_layers, size_t part_layer_stride, cudaStream_t s) {
  const dim3 g(grid, ch.n, n_layers);
  const dim3 b(kF32Warps * 32);
  const cudaError_t e = launch_pdl(tc05_rowscale_kernel, dim3(ch.n), b, 0, s, ch, srow);
  if (e != cudaSuccess) return e;
  if (EPI == EPI_LMHEAD) {
    bool plain = true;   // the dedicated kernel: no logit bias, one output range for every chunk
    int pairs = 0;
    for (int j = 0; j < ch.n; j++) {
      plain = plain && !ch.a[j].e.logit_bias && ch.a[j].strip0 == ch.a[0].strip0 &&
              ch.a[j].n_strips == ch.a[0].n_strips && ch.a[j].R <= kMaxRows;
      pairs += ch.a[j].R;
    }
    if (plain && pairs >= 1 && pairs <= kLmThreads && n_layers == 1)
      return launch_pdl(tc05_lm_epi_kernel, dim3(grid), dim3(kLmThreads), 0, s, ch, part, slices, npad, n_out_pad,
                        static_cast<const float*>(srow), pairs, kLmThreads / pairs > 1 ? 2 : 1);
  }
  // the row-by-strip kernel for Q/K/V and the gated FFN (measured faster); the residual epilogues
  // (O, down: several K slices) stay on the strip kernel, which was faster there
  if constexpr (EPI == EPI_QKV || EPI == EPI_SWIGLU) {
    int pairs = 0;
    bool same = true;
    for (int j = 0; j < ch.n; j++) {
      pairs += ch.a[j].R;
      same = same && ch.a[j].strip0 == ch.a[0].strip0 && ch.a[j].n_strips == ch.a[0].n_strips;
    }
    if (same && n_layers == 1 && pairs >= 1) {
      const long long total = (long long)pairs * ch.a[0].n_strips;
      const int blocks = (int)std::min<long long>(2048, (total + 255) / 256);
      return launch_pdl(tc05_rowstrip_epi_kernel<EPI>, dim3(blocks), dim3(256), 0, s, ch, part, slices, npad,
                        n_out_pad, static_cast<const float*>(srow), pairs);
    }
  }
  switch (nt) {
    case 1:
      return launch_pdl(tc05_epi_kernel<1, EPI>, g, b, 0, s, ch, part, slices, npad, n_out_pad, srow,
                        part_layer_stride);
    case 2:
      return launch_pdl(tc05_epi_kernel<2, EPI>, g, b, 0, s, ch, part, slices, npad, n_out_pad, srow,
                        part_layer_stride);
    case 3:
      return launch_pdl(tc05_epi_kernel<3, EPI>, g, b, 0, s, ch, part, slices, npad, n_out_pad, srow,
                        part_layer_stride);
    case 4:
      return launch_pdl(tc05_epi_kernel<4, EPI>, g, b, 0, s, ch, part, slices, npad, n_out_pad, srow,
                        part_layer_stride);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_tc05_kv_planes(void* xw, long long lo_off, const float* attn_norm, int rows, int d, int n_layers,
                                  long long plane, cudaStream_t s) {
  if (rows < 1 || d % 8 || n_layers < 1) return cudaErrorInvalidValue;
  const long long work = (long long)rows * (d / 8);
  const int blocks = (int)std::min<long long>(1024, (work + 255) / 256);
  return launch_pdl(tc05_kv_planes_kernel, dim3(blocks), dim3(256), 0, s, static_cast<__half*>(xw), lo_off,
                    attn_norm, rows, d, n_layers, plane);
}

cudaError_t launch_tc05_epilogue(int epi, int nt, const Tc05EpiChunks& ch, const float* part, int slices, int npad,
                                 int n_out_pad, int grid, float* srow, int n_layers, size_t part_layer_stride,
                                 cudaStream_t s) {
  if (ch.n < 1 || ch.n > kTcMaxChunks || n_layers < 1) return cudaErrorInvalidValue;
#define DFL_EPI_CASE(E) \
  case E: return launch_epi<E>(nt, ch, part, slices, npad, n_out_pad, grid, srow, n_layers, part_layer_stride, s);
  switch (epi) {
    DFL_EPI_CASE(EPI_CTX)
    DFL_EPI_CASE(EPI_QKV)
    DFL_EPI_CASE(EPI_KV)
    DFL_EPI_CASE(EPI_RESID)
    DFL_EPI_CASE(EPI_SWIGLU)
    DFL_EPI_CASE(EPI_LMHEAD)
    default: return cudaErrorInvalidValue;
  }
#undef DFL_EPI_CASE
}

}  // namespace dfl

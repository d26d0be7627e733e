// Skinny GEMM Y[R][N] = X[R][K] W[N][K]^T for the drafter's projections, R <= 32 activation
// rows, with the RMSNorm scale, residual, SwiGLU, cache-append and vocab argmax epilogues fused.
//
// Tensor-core path (bf16 / 4-bit weights), one CTA per SM:
//  * A CTA owns one K slice and a range of 16-row strips. It stages its activation slice
//    X[R][slice] (f16, plus its f16 remainder where the input carries one) into shared memory
//    with 1-D bulk copies (TMA) once.
//  * Its warps stream weights through private rings of kStages shared-memory stages filled by
//    cp.async.bulk. The CTA's (strip, 64-input group) tiles are cut, in strip-major order, into
//    one contiguous range per warp, so warps stream without synchronising and are balanced to
//    within one tile; a strip cut between warps is summed once, after the stream, in warp
//    order through shared memory.
//  * 4-bit codes become f16 with one lop3 per register (plus a shift for three of four): the
//    re-laid-out word of a lane holds rows g and g+8 in alternating nibbles, so row g decodes
//    to 128 + q (magic 0x5800) and row g+8 to 1024 + 16 q (magic 0x6400, no shift). mma.sync
//    m16n8k16 (weights = A, 16 rows; f16 activations = B, 8 columns per n-tile) accumulates per
//    64-input group in fp32, and the group-64 affine code is folded once per group:
//    sum_k (s q_k + b) x_k equals
//      row g  :  s      * sum (128 + q) x    + (b - 128 s) * sum x
//      row g+8:  s / 16 * sum (1024 + 16q) x + (b -  64 s) * sum x
//    so the MMA sees exact integers; the offsets stay small next to q (17x, 8.5x) because the
//    fp32 group sum loses that factor when they are removed. bf16 weights are stored as f16.
//  * When a strip's K is split in two, the two slice CTAs form a 2-CTA cluster: partial tiles
//    are pushed into the owning CTA's shared memory (distributed shared memory), and after one
//    cluster barrier the owner sums them in slice order and runs the epilogue. Wider K splits
//    write partial tiles to global memory; after its last strip every CTA settles its tickets,
//    and the last slice to arrive (acquire-release ticket, no waiting) sums the partials in
//    slice order and runs the epilogue.
// CUDA-core path (fp32 weights and activations): one warp per strip, fp32 FMA.
#pragma once

#include <cuda_bf16.h>
#include <math.h>

#include <type_traits>

#include "common.cuh"

namespace dfl {

struct LmState {
  float m, s;
  int i;
};

__device__ __forceinline__ void lm_merge(LmState& a, const LmState& b) {
  if (b.m > a.m || (b.m == a.m && b.i < a.i)) {
    const float s = (a.m == -INFINITY) ? b.s : b.s + a.s * __expf(a.m - b.m);
    a.m = b.m;
    a.i = b.i;
    a.s = s;
  } else {
    if (b.m != -INFINITY) a.s += b.s * __expf(b.m - a.m);
  }
}

__device__ __forceinline__ void lm_push(LmState& st, float v, int n) {
  if (v > st.m) {
    st.s = (st.m == -INFINITY) ? 1.0f : st.s * __expf(st.m - v) + 1.0f;
    st.m = v;
    st.i = n;
  } else {
    st.s += __expf(v - st.m);
    if (v == st.m && n < st.i) st.i = n;
  }
}

__device__ __forceinline__ int map_row(const RowMap& m, int r) {
  return (r / m.per) * m.stride + m.off + r % m.per;
}

template <typename XT>
__device__ __forceinline__ void store_act(void* base, size_t idx, float v) {
  static_cast<XT*>(base)[idx] = from_f<XT>(v);
}

// Per-row RMSNorm scale from the producer's per-strip sum-of-squares partials (one warp per
// row; sixteen loads per lane in flight at a time, summed in a fixed order).
__device__ __forceinline__ void compute_row_scales(const GemvArgs& a, float* srow, int nrows) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nw = blockDim.x >> 5;
  const int two = a.norm_mode == NORM_CTX ? 2 : 1;
  for (int r = warp; r < nrows; r += nw) {
    float s = 1.0f;
    if (r < a.R && a.norm_mode != NORM_NONE) {
      const float* base = a.ssq + (size_t)map_row(a.xmap, r) * a.ssq_ld * two;
      float sa = 0.f, sb = 0.f;
      for (int p0 = 0; p0 < a.ssq_parts; p0 += 16 * 32) {
        float va[16], vb[16];
#pragma unroll
        for (int j = 0; j < 16; j++) {
          const int p = p0 + j * 32 + lane;
          const bool in = p < a.ssq_parts;
          va[j] = in ? __ldcg(base + (size_t)p * two) : 0.f;
          vb[j] = in && two == 2 ? __ldcg(base + (size_t)p * 2 + 1) : 0.f;
        }
#pragma unroll
        for (int j = 0; j < 16; j++) {
          sa += va[j];
          sb += vb[j];
        }
      }
      sa = warp_sum(sa);
      if (a.norm_mode == NORM_ONE) {
        s = rsqrtf(sa * a.inv_dim + a.eps);
      } else {
        sb = warp_sum(sb);
        const float inv1 = rsqrtf(sa * a.inv_dim + a.eps);
        s = inv1 * rsqrtf(inv1 * inv1 * sb * a.inv_dim + a.eps);
      }
    }
    if (lane == 0) srow[r] = s;
  }
}

// Inputs an epilogue reads from global memory (residual rows, norm weights). They are loaded
// before any store of the epilogue (a load after a store that may alias it would wait for that
// store, one L2 round trip per element), and on the K-split path together with the partials.
template <int NT>
struct EpiPre {
  float hv[NT][2][2];                 // residual rows (RESID)
  float wn[2];                        // next norm weights of rows nr0, nr1 (RESID)
  float cn[2];                        // context norm weights of rows nr0, nr1 (CTX)
  float an[DFLASH_MAX_LAYERS][2];     // per-layer norm weights of rows nr0, nr1 (CTX, CUDA-core path)
};

// XT = float is the CUDA-core path, which alone writes one context row per layer (EPI_CTX).
template <int EPI, int NT, typename XT>
__device__ __forceinline__ void epi_preload(const GemvArgs& a, int strip, EpiPre<NT>& pre) {
  if constexpr (EPI == EPI_RESID || EPI == EPI_CTX) {
    const EpiArgs& e = a.e;
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const int nr0 = strip * 16 + g - e.row_base, nr1 = nr0 + 8;
    const bool v0 = nr0 >= 0 && nr0 < e.n_rows, v1 = nr1 >= 0 && nr1 < e.n_rows;
    if constexpr (EPI == EPI_RESID) {
      pre.wn[0] = (e.wnext && v0) ? e.wnext[nr0] : 1.f;
      pre.wn[1] = (e.wnext && v1) ? e.wnext[nr1] : 1.f;
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int p = 0; p < 2; p++)
#pragma unroll
          for (int h = 0; h < 2; h++) {
            const int c = nt * 8 + 2 * t + p;
            const int nr = h ? nr1 : nr0;
            pre.hv[nt][p][h] = (c < a.R && (h ? v1 : v0)) ? e.h[(size_t)c * e.ldo + nr] : 0.f;
          }
    } else {
      pre.cn[0] = v0 ? e.ctx_norm[nr0] : 0.f;
      pre.cn[1] = v1 ? e.ctx_norm[nr1] : 0.f;
      if (std::is_same<XT, float>::value && e.attn_norms) {
#pragma unroll
        for (int i = 0; i < DFLASH_MAX_LAYERS; i++) {
          pre.an[i][0] = (i < e.n_layers && v0) ? e.attn_norms[(size_t)i * e.ldo + nr0] : 0.f;
          pre.an[i][1] = (i < e.n_layers && v1) ? e.attn_norms[(size_t)i * e.ldo + nr1] : 0.f;
        }
      }
    }
  }
}

// Epilogue of one complete 16-row strip. Lane (g, t) holds, for n-tile nt, rows strip*16+g
// (y[nt][0..1]) and strip*16+g+8 (y[nt][2..3]) at activation columns nt*8+2t and nt*8+2t+1.
template <int EPI, int NT, typename XT>
__device__ __forceinline__ void strip_epilogue(const GemvArgs& a, int strip, float (&y)[NT][4],
                                               const float* srow, LmState (&lm)[NT][2], int lyr,
                                               const EpiPre<NT>& pre) {
  const EpiArgs& e = a.e;
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int nr0 = strip * 16 + g - e.row_base, nr1 = nr0 + 8;
  LmState lm_strip_state[NT][2];
  const bool v0 = nr0 >= 0 && nr0 < e.n_rows, v1 = nr1 >= 0 && nr1 < e.n_rows;
#pragma unroll
  for (int nt = 0; nt < NT; nt++) {
#pragma unroll
    for (int p = 0; p < 2; p++) {
      const int c = nt * 8 + 2 * t + p;
      const bool cv = c < a.R;
      const float sc = srow[c];
      const float ya = y[nt][p] * sc, yb = y[nt][2 + p] * sc;
      if constexpr (EPI == EPI_STORE) {
        if (cv) {
          const size_t base = (size_t)c * e.ldo;
          if (e.out_f32) {
            if (v0) static_cast<float*>(e.out)[base + nr0] = ya;
            if (v1) static_cast<float*>(e.out)[base + nr1] = yb;
          } else {
            if (v0) store_act<XT>(e.out, base + nr0, ya);
            if (v1) store_act<XT>(e.out, base + nr1, yb);
          }
        }
      } else if constexpr (EPI == EPI_QKV) {
        if (cv) {
#pragma unroll
          for (int h = 0; h < 2; h++) {
            const int nr = h ? nr1 : nr0;
            const float v = h ? yb : ya;
            if (!(h ? v1 : v0)) continue;
            if (nr < e.qd) store_act<XT>(e.q, (size_t)c * e.qd + nr, v);
            else if (nr < e.qd + e.kvd) store_act<XT>(e.kb, (size_t)c * e.kvd + nr - e.qd, v);
            else store_act<XT>(e.vb, (size_t)c * e.kvd + nr - e.qd - e.kvd, v);
          }
        }
      } else if constexpr (EPI == EPI_KV) {
        if (cv) {
#pragma unroll
          for (int h = 0; h < 2; h++) {
            const int nr = h ? nr1 : nr0;
            if (!(h ? v1 : v0)) continue;
            const float v = h ? yb : ya;
            const int half = nr >= e.kvd;
            const int f = nr - half * e.kvd;
            if (!in_bounds(e.kv_slot[c] >= 0 && e.kv_pos[c] >= 0 && e.kv_pos[c] < e.cap, a.err)) continue;
            const size_t idx =
                (((size_t)e.kv_slot[c] * e.n_kv + f / e.hd) * e.cap + e.kv_pos[c]) * e.hd + f % e.hd;
            store_act<XT>(static_cast<uint8_t*>(half ? e.vc : e.kc) + (size_t)lyr * e.kv_grp_stride, idx, v);
          }
        }
      } else if constexpr (EPI == EPI_SWIGLU) {
        const int j = strip * 8 + g;
        if (cv && j < e.inter) {
          float g_act;
          if (e.ffn_act == DFLASH_FFN_GELU)   // tanh approximation: 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3)))
            g_act = 0.5f * ya * (1.0f + tanhf(0.7978845608028654f * fmaf(0.044715f * ya, ya * ya, ya)));
          else
            g_act = ya / (1.0f + __expf(-ya));
          store_act<XT>(e.act, (size_t)c * e.inter + j, g_act * yb);
        }
      } else if constexpr (EPI == EPI_LMHEAD) {
        // Which CTA finishes a split strip varies between runs, so split launches keep one
        // state per strip (merged later in strip order) to stay bit-reproducible.
        LmState& st = a.n_slices > 1 ? lm_strip_state[nt][p] : lm[nt][p];
        if (a.n_slices > 1) st = LmState{-INFINITY, 0.f, 0x7fffffff};
        if (cv) {
          const size_t row = (size_t)c * (e.logit_row_stride ? e.logit_row_stride : e.vocab);
          if (v0) {
            const float l = e.logit_bias ? ya + e.logit_bias[row + nr0] : ya;
            if (e.logits) e.logits[row + nr0] = l;
            lm_push(st, l, nr0);
          }
          if (v1) {
            const float l = e.logit_bias ? yb + e.logit_bias[row + nr1] : yb;
            if (e.logits) e.logits[row + nr1] = l;
            lm_push(st, l, nr1);
          }
        }
      }
    }
  }
  if constexpr (EPI == EPI_LMHEAD) {
    if (a.n_slices > 1) {
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int p = 0; p < 2; p++)
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            LmState other;
            other.m = __shfl_xor_sync(0xffffffffu, lm_strip_state[nt][p].m, o);
            other.s = __shfl_xor_sync(0xffffffffu, lm_strip_state[nt][p].s, o);
            other.i = __shfl_xor_sync(0xffffffffu, lm_strip_state[nt][p].i, o);
            lm_merge(lm_strip_state[nt][p], other);
          }
      if (g == 0) {
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
          for (int p = 0; p < 2; p++) {
            float* dst = e.lm_strip + ((size_t)(strip - a.strip0) * kMaxRows + nt * 8 + 2 * t + p) * 3;
            dst[0] = lm_strip_state[nt][p].m;
            dst[1] = lm_strip_state[nt][p].s;
            dst[2] = __int_as_float(lm_strip_state[nt][p].i);
          }
      }
    }
  }
  if constexpr (EPI == EPI_RESID || EPI == EPI_CTX) {
    // residual update / context rows, then this strip's sum-of-squares partial per column
    const auto& hv = pre.hv;
    const auto& wn = pre.wn;
    const auto& cn = pre.cn;
    const auto& an = pre.an;
    float sq[NT][2][2];
#pragma unroll
    for (int nt = 0; nt < NT; nt++) {
#pragma unroll
      for (int p = 0; p < 2; p++) {
        const int c = nt * 8 + 2 * t + p;
        const bool cv = c < a.R;
        const float sc = srow[c];
        float s0 = 0.f, s1 = 0.f;
#pragma unroll
        for (int h = 0; h < 2; h++) {
          const int nr = h ? nr1 : nr0;
          if (!cv || !(h ? v1 : v0)) continue;
          const float v = y[nt][2 * h + p] * sc;
          if constexpr (EPI == EPI_RESID) {
            const size_t idx = (size_t)c * e.ldo + nr;
            const float hn = hv[nt][p][h] + v;
            e.h[idx] = hn;
            store_act_split<XT>(e.xnext, idx, e.x_lo_off, hn * wn[h]);
            s0 += hn * hn;
          } else if (!std::is_same<XT, float>::value || !e.attn_norms) {
            // one row x * ctx_norm; the consumer applies attn_norm_i
            store_act_split<XT>(e.xw, (size_t)c * e.ldo + nr, e.x_lo_off, v * cn[h]);
            s0 += v * v;
            s1 += (v * cn[h]) * (v * cn[h]);
          } else {
#pragma unroll
            for (int i = 0; i < DFLASH_MAX_LAYERS; i++)
              if (i < e.n_layers)
                store_act_split<XT>(e.xw, ((size_t)i * e.xw_rows + c) * e.ldo + nr, e.x_lo_off,
                                    v * cn[h] * an[i][h]);
            s0 += v * v;
            s1 += (v * cn[h]) * (v * cn[h]);
          }
        }
        sq[nt][p][0] = s0;
        sq[nt][p][1] = s1;
      }
    }
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int p = 0; p < 2; p++)
#pragma unroll
        for (int q = 0; q < 2; q++)
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) sq[nt][p][q] += __shfl_xor_sync(0xffffffffu, sq[nt][p][q], o);
    if (g == 0) {
      const int part = strip - e.row_base / 16;
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int p = 0; p < 2; p++) {
          const int c = nt * 8 + 2 * t + p;
          if (c >= a.R) continue;
          if constexpr (EPI == EPI_RESID) {
            e.ssq_out[(size_t)c * e.ssq_ld + part] = sq[nt][p][0];
          } else {
            e.ssq_out[((size_t)c * e.ssq_ld + part) * 2 + 0] = sq[nt][p][0];
            e.ssq_out[((size_t)c * e.ssq_ld + part) * 2 + 1] = sq[nt][p][1];
          }
        }
    }
  }
}

// Vocab reduction of the LM-head epilogue, GEMV side: lanes -> warps -> one (max, sum, index)
// state per CTA and column in e.lm_part (one K slice), or nothing more when K is split (the
// epilogue already wrote one state per strip to e.lm_strip). lm_reduce_kernel merges them.
template <int NT>
__device__ __forceinline__ void lm_finish(const GemvArgs& a, LmState (&lm)[NT][2], LmState* sm_lm) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int nw = blockDim.x >> 5;
  if (a.n_slices > 1) return;
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int p = 0; p < 2; p++)
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        LmState other;
        other.m = __shfl_xor_sync(0xffffffffu, lm[nt][p].m, o);
        other.s = __shfl_xor_sync(0xffffffffu, lm[nt][p].s, o);
        other.i = __shfl_xor_sync(0xffffffffu, lm[nt][p].i, o);
        lm_merge(lm[nt][p], other);
      }
  if (g == 0) {
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int p = 0; p < 2; p++) sm_lm[warp * kMaxRows + nt * 8 + 2 * t + p] = lm[nt][p];
  }
  __syncthreads();
  const EpiArgs& e = a.e;
  if ((int)threadIdx.x < a.R) {
    LmState acc{-INFINITY, 0.f, 0x7fffffff};
    for (int w = 0; w < nw; w++) lm_merge(acc, sm_lm[w * kMaxRows + threadIdx.x]);
    float* dst = e.lm_part + ((size_t)blockIdx.x * kMaxRows + threadIdx.x) * 3;
    dst[0] = acc.m;
    dst[1] = acc.s;
    dst[2] = __int_as_float(acc.i);
  }
}

// ------------------------------------------------------------------------------------------------
// Tensor-core kernel (bf16 or 4-bit weights, bf16 activations)
// ------------------------------------------------------------------------------------------------
#ifndef DFL_RING_AFTER
#define DFL_RING_AFTER 1   // where the ring's remaining stages are requested (see the kernel)
#endif

template <int FMT, int NT, int EPI>
__global__ void __launch_bounds__(gemv_warps(NT) * 32, 1) gemv_tc_kernel(const __grid_constant__ GemvArgs a) {
  using XT = __half;
  constexpr int kWarps = gemv_warps(NT);   // shadows the NT = 1 default
  constexpr int kGemvThreads = kWarps * 32;
  constexpr int GS = FMT == FMT_Q4 ? kQ4GroupsPerStage : kBf16GroupsPerStage;
  constexpr int GB = FMT == FMT_Q4 ? kQ4GroupBytes : kBf16GroupBytes;
  constexpr int RP = NT * 8;
  constexpr int NT4 = NT * 4;
  extern __shared__ __align__(1024) uint8_t sm[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;

  const int lyr = a.grp_n > 1 ? (int)blockIdx.x / a.grp_ctas : 0;   // problem of a grouped launch
  const int bid = (int)blockIdx.x - lyr * a.grp_ctas;
  const uint8_t* Wb = a.w + (size_t)lyr * a.grp_w_stride;
  const uint8_t* Xb = static_cast<const uint8_t*>(a.x) + (size_t)lyr * a.grp_x_stride * 2;
  const int sgl = lyr * a.n_strips;   // this problem's strips in the partials and tickets
  // slices of a 2-CTA cluster are neighbouring blocks (slice = rank in the cluster)
  const int slice = a.cluster2 ? (bid & 1) : bid / a.ctas_per_slice;
  const int cis = a.cluster2 ? (bid >> 1) : bid % a.ctas_per_slice;
  const int gbeg = slice * a.gps, gend = min(a.groups, gbeg + a.gps), ng = gend - gbeg;
  const int sbeg = (int)((long long)cis * a.n_strips / a.ctas_per_slice);
  const int send = (int)((long long)(cis + 1) * a.n_strips / a.ctas_per_slice);
  const int n_cta = send - sbeg;                 // strips of this CTA
  const int xstride = a.gps * 128 + 16;

  const bool has_lo = a.x_lo_off != 0;
  uint8_t* ring = sm;
  uint8_t* xs = sm + kWarps * kStages * kStageBytes;
  uint8_t* xs_lo = xs + RP * xstride;   // f16 remainder rows (when the input carries them)
  float* xsum = reinterpret_cast<float*>(xs_lo + (has_lo ? RP * xstride : 0));
  float* srow = xsum + (FMT == FMT_Q4 ? RP * a.gps : 0);
  LmState* sm_lm = reinterpret_cast<LmState*>(srow + kMaxRows);
  float* red = reinterpret_cast<float*>(sm_lm + (EPI == EPI_LMHEAD ? kWarps * kMaxRows : 0));
  float* cpart = red + 2 * kWarps * 32 * NT4;   // cluster K split: [strip pair][slice] partial tiles
  uint64_t* bars = reinterpret_cast<uint64_t*>(
      (reinterpret_cast<uintptr_t>(cpart + (a.cluster2 ? a.cpart_cap * 32 * NT4 : 0)) + 15) & ~uintptr_t(15));

  if (threadIdx.x == 0) {
    for (int i = 0; i < 2 + kWarps * kStages; i++) mbar_init(smem_u32(&bars[i]), 1);
    fence_barrier_init();
  }
  __syncthreads();

  // Work of this warp: one contiguous range [t0, t1) of the CTA's n_cta x ng (strip, group)
  // tiles in strip-major order, so every warp streams the same number of tiles with no
  // synchronisation. A range splits at strip boundaries into segments; a segment covering a
  // whole strip is finished at once, a partial one (at most the first and the last of a range)
  // is parked in shared memory and summed after the stream, in warp order, by the warp that
  // owns the strip's last tile.
  const long long T = (long long)n_cta * ng;
  const long long t0 = T * warp / kWarps, t1 = T * (warp + 1) / kWarps;
  const int first_strip = (int)(t0 / ng);
  // issue cursor: stages never cross a strip boundary
  long long i_tile = t0;
  int i_strip = first_strip, i_goff = (int)(t0 % ng);
  int issued = 0;
  auto issue_next = [&]() {
    const int gn = (int)min((long long)min(GS, ng - i_goff), t1 - i_tile);
    in_bounds(sbeg + i_strip < a.n_strips && gbeg + i_goff + gn <= a.groups && gn > 0, lane == 0 ? a.err : nullptr);
    const uint8_t* src = Wb + ((size_t)(a.strip0 + sbeg + i_strip) * a.groups + gbeg + i_goff) * GB;
    const int slot = warp * kStages + issued % kStages;
    if (lane == 0) {
      const uint32_t bar = smem_u32(&bars[1 + slot]);
      mbar_arrive_expect_tx(bar, gn * GB);
      bulk_g2s(smem_u32(ring + (size_t)slot * kStageBytes), src, gn * GB, bar);
    }
    issued++;
    i_tile += gn;
    i_goff += gn;
    if (i_goff == ng) {
      i_goff = 0;
      i_strip++;
    }
  };
  // Weights never change, so some stages are requested before waiting for the previous kernel;
  // the rest follow the activation copies, which are on the critical path.
  for (int q = 0; q < kPrePdlStages && i_tile < t1; q++) issue_next();
  // per-input scales of the slice (constants), eight columns per thread and chunk: read before
  // waiting for the previous kernel
#ifndef DFL_CS_CHUNKS
#define DFL_CS_CHUNKS 2
#endif
  constexpr int kCsChunks = EPI == EPI_KV ? DFL_CS_CHUNKS : 0;   // only the context K/V launch uses them
  float4 csv[kCsChunks > 0 ? kCsChunks : 1][2];
  const float* cs = (EPI == EPI_KV && a.x_colscale)
                        ? a.x_colscale + (size_t)lyr * a.x_colscale_grp_stride + gbeg * 64 : nullptr;
#pragma unroll
  for (int u = 0; u < kCsChunks; u++) {
    const int j = threadIdx.x + u * kGemvThreads;
    const bool in = cs && 8 * j < ng * 64;
    csv[u][0] = in ? *reinterpret_cast<const float4*>(cs + 8 * j) : make_float4(0.f, 0.f, 0.f, 0.f);
    csv[u][1] = in ? *reinterpret_cast<const float4*>(cs + 8 * j + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  if (kL2PrefetchTiles > 0 && lane == 0) {
    // the tiles after the ring's first stages, strip segment by strip segment, into L2: the
    // previous kernel's tail leaves HBM idle, and these loads then hit L2
    long long pt = i_tile + (long long)(kStages - kPrePdlStages) * GS;
    int budget = kL2PrefetchTiles;
    if (pt < t1) {
      int ps = (int)(pt / ng), pg = (int)(pt % ng);
      while (budget > 0 && pt < t1) {
        const int n = (int)min((long long)min(ng - pg, budget), t1 - pt);
        prefetch_l2(Wb + ((size_t)(a.strip0 + sbeg + ps) * a.groups + gbeg + pg) * GB, n * GB);
        pt += n;
        budget -= n;
        pg += n;
        if (pg == ng) {
          pg = 0;
          ps++;
        }
      }
    }
  }
  pdl_launch_dependents();
  pdl_wait();   // from here on, everything earlier kernels wrote is visible
  if (DFL_RING_AFTER == 0)
    for (int q = kPrePdlStages; q < kStages && i_tile < t1; q++) issue_next();

  // activation slice -> shared (bulk copies of at most 2 KB, started at a different piece in
  // every CTA so the CTAs do not all read the same L2 lines at once), pad rows zeroed
  const int k0 = gbeg * 64, kbytes = ng * 128;
  if (warp == 0) {
    const uint32_t bar = smem_u32(&bars[0]);
    if (lane == 0) mbar_arrive_expect_tx(bar, a.R * kbytes * (has_lo ? 2 : 1));
    __syncwarp();
    const int ppr = (kbytes + 2047) / 2048, n_pc = a.R * ppr;
    const int rot = blockIdx.x % n_pc;
    for (int i = lane; i < n_pc; i += 32) {
      const int j = i + rot < n_pc ? i + rot : i + rot - n_pc;
      const int r = j / ppr, off = (j - r * ppr) * 2048, len = min(2048, kbytes - off);
      const uint8_t* row = Xb + ((size_t)map_row(a.xmap, r) * a.ldx + k0) * 2 + off;
      bulk_g2s(smem_u32(xs + (size_t)r * xstride + off), row, len, bar);
      if (has_lo) bulk_g2s(smem_u32(xs_lo + (size_t)r * xstride + off), row + a.x_lo_off * 2, len, bar);
    }
  }
  for (int r = a.R + warp; r < RP; r += kWarps) {   // pad rows
    for (int c = lane; c < kbytes / 16; c += 32) {
      *reinterpret_cast<uint4*>(xs + (size_t)r * xstride + c * 16) = make_uint4(0, 0, 0, 0);
      if (has_lo) *reinterpret_cast<uint4*>(xs_lo + (size_t)r * xstride + c * 16) = make_uint4(0, 0, 0, 0);
    }
  }
  if (DFL_RING_AFTER == 1)
    for (int q = kPrePdlStages; q < kStages && i_tile < t1; q++) issue_next();
  compute_row_scales(a, srow, RP);
  if (DFL_RING_AFTER == 2)
    for (int q = kPrePdlStages; q < kStages && i_tile < t1; q++) issue_next();
  bool ok = mbar_wait_bounded(smem_u32(&bars[0]), 0, a.err, kErrTimeoutGemv);
  if (a.stall_cta1 == (int)blockIdx.x + 1 && threadIdx.x == 0)   // test hook: no copy or thread ends this wait
    ok = mbar_wait_bounded(smem_u32(&bars[1 + kWarps * kStages]), 0, a.err, kErrTimeoutGemv) && ok;
  ok = __syncthreads_and(ok);
  if (a.x_bf16 && ok) {  // caller-side bf16 rows (context taps) -> f16 in place
    for (int r = warp; r < a.R; r += kWarps) {
      uint32_t* rp = reinterpret_cast<uint32_t*>(xs + (size_t)r * xstride);
      for (int i = lane; i < kbytes / 4; i += 32) {
        const uint32_t u = rp[i];
        const float lo = __uint_as_float(u << 16), hi = __uint_as_float(u & 0xFFFF0000u);
        rp[i] = pack_f16x2(fminf(fmaxf(lo, -kF16Max), kF16Max), fminf(fmaxf(hi, -kF16Max), kF16Max));
      }
    }
    __syncthreads();
  }
  if (EPI == EPI_KV && cs && ok) {
    // per-input scale (a layer's norm weights) of the staged slice: x = (hi + lo) * w, split again
    auto scale_cols = [&](int j, const float4& w0, const float4& w1) {
      const float w[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
      for (int r = 0; r < a.R; r++) {
        uint4* ph = reinterpret_cast<uint4*>(xs + (size_t)r * xstride) + j;
        uint4* pl = reinterpret_cast<uint4*>(xs_lo + (size_t)r * xstride) + j;
        const uint4 h4 = *ph;
        const uint4 l4 = has_lo ? *pl : make_uint4(0, 0, 0, 0);
        const uint32_t hw[4] = {h4.x, h4.y, h4.z, h4.w}, lw[4] = {l4.x, l4.y, l4.z, l4.w};
        uint32_t oh[4], ol[4];
#pragma unroll
        for (int q = 0; q < 4; q++) {
          const float2 fh = __half22float2(*reinterpret_cast<const __half2*>(&hw[q]));
          const float2 fl = __half22float2(*reinterpret_cast<const __half2*>(&lw[q]));
          const float va = (fh.x + fl.x) * w[2 * q], vb = (fh.y + fl.y) * w[2 * q + 1];
          const __half ha = from_f<__half>(va), hb = from_f<__half>(vb);
          oh[q] = pack_f16x2(__half2float(ha), __half2float(hb));
          ol[q] = pack_f16x2(va - __half2float(ha), vb - __half2float(hb));
        }
        *ph = make_uint4(oh[0], oh[1], oh[2], oh[3]);
        if (has_lo) *pl = make_uint4(ol[0], ol[1], ol[2], ol[3]);
      }
    };
#pragma unroll
    for (int u = 0; u < kCsChunks; u++) {
      const int j = threadIdx.x + u * kGemvThreads;
      if (8 * j < ng * 64) scale_cols(j, csv[u][0], csv[u][1]);
    }
    for (int j = threadIdx.x + kCsChunks * kGemvThreads; 8 * j < ng * 64; j += kGemvThreads)
      scale_cols(j, *reinterpret_cast<const float4*>(cs + 8 * j), *reinterpret_cast<const float4*>(cs + 8 * j + 4));
    __syncthreads();
  }
  if (FMT == FMT_Q4 && ok) {
    // per (group, activation row) sums of hi + lo: an MMA against an all-ones A operand, with
    // the B fragments read exactly as the weight MMAs read them
    const uint32_t one2 = 0x3C003C00u;
    for (int item = warp; item < ng * NT; item += kWarps) {
      const int gl = item / NT, nt = item - gl * NT;
      const uint8_t* xr = xs + (size_t)(nt * 8 + g) * xstride + (gl * 64 + 16 * t) * 2;
      const uint4 x01 = *reinterpret_cast<const uint4*>(xr);
      const uint4 x23 = *reinterpret_cast<const uint4*>(xr + 16);
      float acc[4] = {0.f, 0.f, 0.f, 0.f};
      mma_f16(acc, one2, one2, one2, one2, x01.x, x01.y);
      mma_f16(acc, one2, one2, one2, one2, x01.z, x01.w);
      mma_f16(acc, one2, one2, one2, one2, x23.x, x23.y);
      mma_f16(acc, one2, one2, one2, one2, x23.z, x23.w);
      if (has_lo) {
        const uint8_t* xl = xs_lo + (size_t)(nt * 8 + g) * xstride + (gl * 64 + 16 * t) * 2;
        const uint4 l01 = *reinterpret_cast<const uint4*>(xl);
        const uint4 l23 = *reinterpret_cast<const uint4*>(xl + 16);
        mma_f16(acc, one2, one2, one2, one2, l01.x, l01.y);
        mma_f16(acc, one2, one2, one2, one2, l01.z, l01.w);
        mma_f16(acc, one2, one2, one2, one2, l23.x, l23.y);
        mma_f16(acc, one2, one2, one2, one2, l23.z, l23.w);
      }
      if (g == 0) *reinterpret_cast<float2*>(xsum + gl * RP + nt * 8 + 2 * t) = make_float2(acc[0], acc[1]);
    }
  }
  __syncthreads();

  LmState lm[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int p = 0; p < 2; p++) lm[nt][p] = LmState{-INFINITY, 0.f, 0x7fffffff};

  // a finished strip: epilogue now, or publish this CTA's partial of a K-split strip
  auto finish = [&](int strip_local, float (&y)[NT][4]) {
    if (a.cluster2) {
      // strip j of the pair's range is reduced by CTA (j & 1); its two slice partials sit side by
      // side in that CTA's shared memory, written locally or through the cluster
      const int j = strip_local - sbeg, owner = j & 1;
      float* slot = cpart + ((size_t)((j >> 1) * 2 + slice) * 32 + lane) * NT4;
      if (owner == slice) {
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
          *reinterpret_cast<float4*>(slot + nt * 4) = make_float4(y[nt][0], y[nt][1], y[nt][2], y[nt][3]);
      } else {
        const uint32_t remote = map_shared_rank(smem_u32(slot), (uint32_t)owner);
#pragma unroll
        for (int nt = 0; nt < NT; nt++) st_cluster_v4(remote + nt * 16, make_float4(y[nt][0], y[nt][1], y[nt][2], y[nt][3]));
      }
    } else if (a.n_slices > 1) {
      float* part = a.partials + (((size_t)(sgl + strip_local) * a.n_slices + slice) * 32 + lane) * NT4;
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
        *reinterpret_cast<float4*>(part + nt * 4) = make_float4(y[nt][0], y[nt][1], y[nt][2], y[nt][3]);
    } else {
      EpiPre<NT> pre;
      epi_preload<EPI, NT, XT>(a, a.strip0 + strip_local, pre);
      strip_epilogue<EPI, NT, XT>(a, a.strip0 + strip_local, y, srow, lm, lyr, pre);
    }
  };
  auto piece = [&](int w, int slot) -> float* { return red + ((size_t)(w * 2 + slot) * 32 + lane) * NT4; };

  int consumed = 0;
  // stream this warp's range: stage q covers groups [c_goff, c_goff + gn) of strip c_strip
  auto stream = [&](auto lo_tag) {
    constexpr bool LO = decltype(lo_tag)::value;
    long long c_tile = t0;
    int c_strip = first_strip, c_goff = (int)(t0 % ng), seg_start = c_goff;
    float y[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int j = 0; j < 4; j++) y[nt][j] = 0.f;
    for (int q = 0; ok && c_tile < t1; q++) {
      const int slot = warp * kStages + q % kStages;
      bool w_ok = mbar_wait_bounded(smem_u32(&bars[1 + slot]), (q / kStages) & 1, a.err, kErrTimeoutGemv);
      w_ok = __all_sync(0xffffffffu, w_ok);
      if (!w_ok) {
        ok = false;
        break;
      }
      consumed = q + 1;
      const int gn = (int)min((long long)min(GS, ng - c_goff), t1 - c_tile);
      const uint8_t* stg = ring + (size_t)slot * kStageBytes;
      auto group = [&](int gi) {
        const int gl = c_goff + gi;
        if constexpr (FMT == FMT_Q4) {
          const uint8_t* gp = stg + gi * kQ4GroupBytes;
          const uint4 A = *reinterpret_cast<const uint4*>(gp + lane * 16);
          const uint32_t sb0 = *reinterpret_cast<const uint32_t*>(gp + 512 + 4 * g);
          const uint32_t sb1 = *reinterpret_cast<const uint32_t*>(gp + 512 + 4 * (g + 8));
          const float s0 = __uint_as_float(sb0 << 16), s1 = __uint_as_float(sb1 << 16);
          const float b0 = fmaf(-128.f, s0, __uint_as_float(sb0 & 0xFFFF0000u));
          const float b1 = fmaf(-64.f, s1, __uint_as_float(sb1 & 0xFFFF0000u));
          const float s1q = s1 * 0.0625f;
          const uint32_t u[4] = {A.x, A.y, A.z, A.w};
          uint32_t af[4][4];
#pragma unroll
          for (int j = 0; j < 4; j++) {
            af[j][0] = nib128_to_f16x2(u[j] << 3);
            af[j][1] = nib_hi_to_f16x2(u[j]);
            af[j][2] = nib128_to_f16x2(u[j] >> 5);
            af[j][3] = nib_hi_to_f16x2(u[j] >> 8);
          }
#pragma unroll
          for (int nt = 0; nt < NT; nt++) {
            const uint8_t* xr = xs + (size_t)(nt * 8 + g) * xstride + (gl * 64 + 16 * t) * 2;
            const uint4 x01 = *reinterpret_cast<const uint4*>(xr);
            const uint4 x23 = *reinterpret_cast<const uint4*>(xr + 16);
            float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
            mma_f16(acc0, af[0][0], af[0][1], af[0][2], af[0][3], x01.x, x01.y);
            mma_f16(acc1, af[1][0], af[1][1], af[1][2], af[1][3], x01.z, x01.w);
            mma_f16(acc0, af[2][0], af[2][1], af[2][2], af[2][3], x23.x, x23.y);
            mma_f16(acc1, af[3][0], af[3][1], af[3][2], af[3][3], x23.z, x23.w);
            if constexpr (LO) {   // the same exact weights against the activations' f16 remainder
              const uint8_t* xl = xs_lo + (size_t)(nt * 8 + g) * xstride + (gl * 64 + 16 * t) * 2;
              const uint4 l01 = *reinterpret_cast<const uint4*>(xl);
              const uint4 l23 = *reinterpret_cast<const uint4*>(xl + 16);
              mma_f16(acc0, af[0][0], af[0][1], af[0][2], af[0][3], l01.x, l01.y);
              mma_f16(acc1, af[1][0], af[1][1], af[1][2], af[1][3], l01.z, l01.w);
              mma_f16(acc0, af[2][0], af[2][1], af[2][2], af[2][3], l23.x, l23.y);
              mma_f16(acc1, af[3][0], af[3][1], af[3][2], af[3][3], l23.z, l23.w);
            }
            const float2 xab = *reinterpret_cast<const float2*>(xsum + gl * RP + nt * 8 + 2 * t);
            y[nt][0] = fmaf(s0, acc0[0] + acc1[0], fmaf(b0, xab.x, y[nt][0]));
            y[nt][1] = fmaf(s0, acc0[1] + acc1[1], fmaf(b0, xab.y, y[nt][1]));
            y[nt][2] = fmaf(s1q, acc0[2] + acc1[2], fmaf(b1, xab.x, y[nt][2]));
            y[nt][3] = fmaf(s1q, acc0[3] + acc1[3], fmaf(b1, xab.y, y[nt][3]));
          }
        } else {
          const uint8_t* gp = stg + gi * kBf16GroupBytes;
          uint4 A[4];
#pragma unroll
          for (int j = 0; j < 4; j++) A[j] = *reinterpret_cast<const uint4*>(gp + j * 512 + lane * 16);
#pragma unroll
          for (int nt = 0; nt < NT; nt++) {
            const uint8_t* xr = xs + (size_t)(nt * 8 + g) * xstride + (gl * 64 + 16 * t) * 2;
            const uint4 x01 = *reinterpret_cast<const uint4*>(xr);
            const uint4 x23 = *reinterpret_cast<const uint4*>(xr + 16);
            mma_f16(y[nt], A[0].x, A[0].y, A[0].z, A[0].w, x01.x, x01.y);
            mma_f16(y[nt], A[1].x, A[1].y, A[1].z, A[1].w, x01.z, x01.w);
            mma_f16(y[nt], A[2].x, A[2].y, A[2].z, A[2].w, x23.x, x23.y);
            mma_f16(y[nt], A[3].x, A[3].y, A[3].z, A[3].w, x23.z, x23.w);
            if constexpr (LO) {
              const uint8_t* xl = xs_lo + (size_t)(nt * 8 + g) * xstride + (gl * 64 + 16 * t) * 2;
              const uint4 l01 = *reinterpret_cast<const uint4*>(xl);
              const uint4 l23 = *reinterpret_cast<const uint4*>(xl + 16);
              mma_f16(y[nt], A[0].x, A[0].y, A[0].z, A[0].w, l01.x, l01.y);
              mma_f16(y[nt], A[1].x, A[1].y, A[1].z, A[1].w, l01.z, l01.w);
              mma_f16(y[nt], A[2].x, A[2].y, A[2].z, A[2].w, l23.x, l23.y);
              mma_f16(y[nt], A[3].x, A[3].y, A[3].z, A[3].w, l23.z, l23.w);
            }
          }
        }
      };
      if (EPI == EPI_LMHEAD && NT == 1 && gn == GS) {
        // LM head, a whole stage: straight-line code the compiler can interleave across groups
        // (measured faster there; the other projections ran slower with it)
#pragma unroll
        for (int gi = 0; gi < GS; gi++) group(gi);
      } else {
#pragma unroll
        for (int gi = 0; gi < GS; gi++) {
          if (gi >= gn) break;
          group(gi);
        }
      }
      // every lane is done reading this slot before the copy engine refills it
      fence_proxy_async();
      __syncwarp();
      if (i_tile < t1) issue_next();
      c_tile += gn;
      c_goff += gn;
      if (c_goff == ng || c_tile == t1) {   // end of a segment
        if (seg_start == 0 && c_goff == ng) {
          finish(sbeg + c_strip, y);
        } else {
          float* dst = piece(warp, c_strip == first_strip ? 0 : 1);
#pragma unroll
          for (int nt = 0; nt < NT; nt++)
            *reinterpret_cast<float4*>(dst + nt * 4) = make_float4(y[nt][0], y[nt][1], y[nt][2], y[nt][3]);
        }
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
          for (int j = 0; j < 4; j++) y[nt][j] = 0.f;
        if (c_goff == ng) {
          c_goff = 0;
          c_strip++;
        }
        seg_start = c_goff;
      }
    }
  };
  if (has_lo) stream(std::true_type{});
  else stream(std::false_type{});
  ok = __syncthreads_and(ok);

  // strips split between warps: the warp owning a strip's last tile sums the pieces in warp order
  if (ok && t1 > t0) {
    const long long s_first_tile = (long long)first_strip * ng;
    if (t0 > s_first_tile && s_first_tile + ng <= t1) {
      int wa = warp;
      while (wa > 0 && T * wa / kWarps > s_first_tile) wa--;
      float y[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int j = 0; j < 4; j++) y[nt][j] = 0.f;
      for (int w = wa; w <= warp; w++) {
        const long long w0 = T * w / kWarps, w1 = T * (w + 1) / kWarps;
        if (w1 == w0) continue;
        const float* src = piece(w, (int)(w0 / ng) == first_strip ? 0 : 1);
#pragma unroll
        for (int nt = 0; nt < NT; nt++) {
          const float4 v = *reinterpret_cast<const float4*>(src + nt * 4);
          y[nt][0] += v.x;
          y[nt][1] += v.y;
          y[nt][2] += v.z;
          y[nt][3] += v.w;
        }
      }
      finish(sbeg + first_strip, y);
    }
  }

  if (!ok && lane == 0) {
    // leave no copy in flight into this CTA's shared memory
    if (threadIdx.x == 0) mbar_wait_bounded(smem_u32(&bars[0]), 0, nullptr, 0);
    for (int q = consumed; q < issued; q++) {
      const int slot = warp * kStages + q % kStages;
      mbar_wait_bounded(smem_u32(&bars[1 + slot]), (q / kStages) & 1, nullptr, 0);
    }
  }

  if (a.cluster2) {
    // both CTAs of the pair reach this barrier on every path (a CTA that gave up still arrives),
    // so neither can wait for a partner that left
    EpiPre<NT> pre;
    const int o0 = warp;
    if (2 * o0 + slice < n_cta) epi_preload<EPI, NT, XT>(a, a.strip0 + sbeg + 2 * o0 + slice, pre);
    cluster_sync();
    for (int o = o0; ok && 2 * o + slice < n_cta; o += kWarps) {
      const int strip_local = sbeg + 2 * o + slice;
      if (o != o0) epi_preload<EPI, NT, XT>(a, a.strip0 + strip_local, pre);
      const float* p0 = cpart + ((size_t)(o * 2 + 0) * 32 + lane) * NT4;
      const float* p1 = cpart + ((size_t)(o * 2 + 1) * 32 + lane) * NT4;
      float y[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; nt++) {   // slice 0 + slice 1, in that order
        const float4 u = *reinterpret_cast<const float4*>(p0 + nt * 4);
        const float4 v = *reinterpret_cast<const float4*>(p1 + nt * 4);
        y[nt][0] = u.x + v.x;
        y[nt][1] = u.y + v.y;
        y[nt][2] = u.z + v.z;
        y[nt][3] = u.w + v.w;
      }
      strip_epilogue<EPI, NT, XT>(a, a.strip0 + strip_local, y, srow, lm, lyr, pre);
    }
  } else if (ok && a.n_slices > 1) {
    // every partial of this CTA is written (by whichever warp finished the strip) before any
    // ticket is taken; the last slice to arrive at a strip sums all slices in slice order and
    // runs the epilogue
    __syncthreads();
    for (int si0 = warp; si0 < n_cta; si0 += 32 * kWarps) {
      // one ticket per lane (strips si0 + kWarps * lane), all in flight at once
      const int my_si = si0 + kWarps * lane;
      int prev = -1;
      if (my_si < n_cta) prev = atom_add_acq_rel_gpu(&a.tickets[sgl + sbeg + my_si], 1);
      unsigned last_mask = __ballot_sync(0xffffffffu, prev == a.n_slices - 1);
      __syncwarp();   // the acquiring lane's view extends to the lanes that read the partials
      while (last_mask) {
      const int j = __ffs(last_mask) - 1;
      last_mask &= last_mask - 1;
      const int strip_local = sbeg + si0 + kWarps * j;
      EpiPre<NT> pre;   // issued with the partial loads below: one round trip for both
      epi_preload<EPI, NT, XT>(a, a.strip0 + strip_local, pre);
      float y[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; nt++)
#pragma unroll
        for (int jj = 0; jj < 4; jj++) y[nt][jj] = 0.f;
      for (int s0 = 0; s0 < a.n_slices; s0 += 8) {
        float4 v[8][NT];   // eight slices' loads in flight, then summed in slice order
#pragma unroll
        for (int q = 0; q < 8; q++) {
          const float* src = a.partials + (((size_t)(sgl + strip_local) * a.n_slices + s0 + q) * 32 + lane) * NT4;
#pragma unroll
          for (int nt = 0; nt < NT; nt++)
            v[q][nt] = s0 + q < a.n_slices ? __ldcg(reinterpret_cast<const float4*>(src + nt * 4))
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int q = 0; q < 8; q++) {
          if (s0 + q >= a.n_slices) break;
#pragma unroll
          for (int nt = 0; nt < NT; nt++) {
            y[nt][0] += v[q][nt].x;
            y[nt][1] += v[q][nt].y;
            y[nt][2] += v[q][nt].z;
            y[nt][3] += v[q][nt].w;
          }
        }
      }
      if (lane == 0) a.tickets[sgl + strip_local] = 0;
      strip_epilogue<EPI, NT, XT>(a, a.strip0 + strip_local, y, srow, lm, lyr, pre);
      }
    }
  }
  if constexpr (EPI == EPI_LMHEAD) lm_finish<NT>(a, lm, sm_lm);
}

// ------------------------------------------------------------------------------------------------
// CUDA-core kernel (fp32 weights and activations): one warp per strip
// ------------------------------------------------------------------------------------------------
template <int NT, int EPI>
__global__ void __launch_bounds__(kF32Warps * 32) gemv_f32_kernel(const __grid_constant__ GemvArgs a) {
  constexpr int RP = NT * 8;
  __shared__ float srow[kMaxRows];
  __shared__ LmState sm_lm[kF32Warps * kMaxRows];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  compute_row_scales(a, srow, RP);
  __syncthreads();
  const float* X = static_cast<const float*>(a.x);
  const float* W = reinterpret_cast<const float*>(a.w);
  LmState lm[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; nt++)
#pragma unroll
    for (int p = 0; p < 2; p++) lm[nt][p] = LmState{-INFINITY, 0.f, 0x7fffffff};

  for (int sl = blockIdx.x * kF32Warps + warp; sl < a.n_strips; sl += gridDim.x * kF32Warps) {
    const int strip = a.strip0 + sl;
    float y[NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int j = 0; j < 4; j++) y[nt][j] = 0.f;
    for (int m = 0; m < 16; m++) {
      const float* wr = W + (size_t)(strip * 16 + m) * a.k;
      float part[RP];
#pragma unroll
      for (int c = 0; c < RP; c++) part[c] = 0.f;
      for (int k = lane; k < a.k; k += 32) {
        const float w = wr[k];
#pragma unroll
        for (int c = 0; c < RP; c++)
          if (c < a.R) part[c] = fmaf(w, X[(size_t)map_row(a.xmap, c) * a.ldx + k], part[c]);
      }
#pragma unroll
      for (int c = 0; c < RP; c++) {
        const float v = warp_sum(part[c]);
        if ((c % 8) / 2 == t) {
          if (m == g) y[c / 8][c & 1] = v;
          if (m == g + 8) y[c / 8][2 + (c & 1)] = v;
        }
      }
    }
    EpiPre<NT> pre;
    epi_preload<EPI, NT, float>(a, strip, pre);
    strip_epilogue<EPI, NT, float>(a, strip, y, srow, lm, 0, pre);
  }
  if constexpr (EPI == EPI_LMHEAD) lm_finish<NT>(a, lm, sm_lm);
}

template <int FMT, int NT>
cudaError_t launch_gemv_fmt_nt(int epi, const GemvArgs& a, int grid, size_t smem, cudaStream_t s) {
#define DFL_CASE(E)                                                                              \
  case E: {                                                                                      \
    if constexpr (FMT == FMT_F32) {                                                              \
      gemv_f32_kernel<NT, E><<<grid, kF32Warps * 32, 0, s>>>(a);                                 \
    } else {                                                                                     \
      auto k = gemv_tc_kernel<FMT, NT, E>;                                                       \
      static std::atomic<int> smem_set[kMaxDevices];                                             \
      cudaError_t err = ensure_smem_limit(k, smem, smem_set);                                    \
      if (err != cudaSuccess) return err;                                                        \
      return launch_pdl_cluster(k, dim3(grid), dim3(gemv_warps(NT) * 32), smem, s, a.cluster2 ? 2 : 1, a); \
    }                                                                                            \
    return cudaGetLastError();                                                                   \
  }
  switch (epi) {
    DFL_CASE(EPI_STORE)
    DFL_CASE(EPI_CTX)
    DFL_CASE(EPI_KV)
    DFL_CASE(EPI_QKV)
    DFL_CASE(EPI_RESID)
    DFL_CASE(EPI_SWIGLU)
    DFL_CASE(EPI_LMHEAD)
    default:
      return cudaErrorInvalidValue;
  }
#undef DFL_CASE
}

template <int FMT>
cudaError_t launch_gemv_fmt(int epi, int nt, const GemvArgs& a, int grid, size_t smem, cudaStream_t s) {
  switch (nt) {
    case 1: return launch_gemv_fmt_nt<FMT, 1>(epi, a, grid, smem, s);
    case 2: return launch_gemv_fmt_nt<FMT, 2>(epi, a, grid, smem, s);
    case 4: return launch_gemv_fmt_nt<FMT, 4>(epi, a, grid, smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfl

// Small kernels of the draft round: weight re-layout (once, at create), block construction,
// embedding gather and greedy acceptance.
#include <cuda_fp16.h>

#include "common.cuh"

namespace dfl {

namespace {

// logical matrix row n -> (source, source row); false for padding rows
__device__ __forceinline__ bool resolve_row(const RepackArgs& a, int n, int& src, int& row) {
  if (a.interleave) {
    const int strip = n / 16, m = n % 16;
    src = m < 8 ? 0 : 1;
    row = strip * 8 + (m % 8);
    return row < a.src[src].rows;
  }
  for (int s = 0; s < a.n_src; s++) {
    if (n < a.src[s].rows) {
      src = s;
      row = n;
      return true;
    }
    n -= a.src[s].rows;
  }
  return false;
}

__device__ __forceinline__ uint32_t q4_code(const RepackArgs& a, int n, int k) {
  int s, r;
  if (!resolve_row(a, n, s, r)) return 0u;
  const uint32_t w = static_cast<const uint32_t*>(a.src[s].data)[(size_t)r * (a.k / 8) + k / 8];
  return (w >> (4 * (k % 8))) & 15u;
}

// bf16 weight -> f16 bits (exact for |w| in the f16 normal range; the tensor-core path runs f16)
__device__ __forceinline__ uint32_t bf16_as_f16_bits(const RepackArgs& a, int n, int k) {
  int s, r;
  if (!resolve_row(a, n, s, r)) return 0u;
  const float w = bf16_bits_to_float(static_cast<const uint16_t*>(a.src[s].data)[(size_t)r * a.k + k]);
  return __half_as_ushort(__float2half_rn(w));
}

// Destination layouts (per 16-row strip, per 64-input group; k0 = 64*grp + 16*t + 4*j for
// lane = 4*g + t and mma step j):
//  q4  : 144 words. Word lane*4 + j packs the 8 codes lane (g,t) feeds mma j, nibble positions
//        0..7 = (g,k0) (g+8,k0) (g,k0+2) (g+8,k0+2) (g,k0+1) (g+8,k0+1) (g,k0+3) (g+8,k0+3),
//        so that (w >> 4i) & 0x000F000F yields A register i. Words 128 + m hold row m's
//        (scale | bias << 16) bf16 pair.
//  bf16: 512 words of f16 pairs. Word j*128 + lane*4 + i is A register i of mma j:
//        i=0 (g,k0..k0+1), 1 (g+8,k0..k0+1), 2 (g,k0+2..k0+3), 3 (g+8,k0+2..k0+3).
//  f32 : row-major rows.
__global__ void repack_kernel(const __grid_constant__ RepackArgs a) {
  const int groups = a.k / 64;
  const size_t words_per = a.fmt == FMT_Q4 ? 144 : 512;
  const size_t total = a.fmt == FMT_F32 ? (size_t)a.n_strips * 16 * a.k : (size_t)a.n_strips * groups * words_per;
  for (size_t w = blockIdx.x * (size_t)blockDim.x + threadIdx.x; w < total; w += (size_t)gridDim.x * blockDim.x) {
    if (a.fmt == FMT_F32) {
      const int n = (int)(w / a.k), k = (int)(w % a.k);
      int s, r;
      float v = 0.f;
      if (resolve_row(a, n, s, r)) v = static_cast<const float*>(a.src[s].data)[(size_t)r * a.k + k];
      reinterpret_cast<float*>(a.dst)[w] = v;
      continue;
    }
    const int strip = (int)(w / (groups * words_per));
    const int rem = (int)(w % (groups * words_per));
    const int grp = rem / (int)words_per, wi = rem % (int)words_per;
    uint32_t out = 0;
    if (a.fmt == FMT_Q4) {
      if (wi < 128) {
        const int lane = wi / 4, j = wi % 4, g = lane / 4, t = lane % 4;
        const int k0 = grp * 64 + 16 * t + 4 * j;
        const int r0 = strip * 16 + g, r1 = r0 + 8;
        const uint32_t c[8] = {q4_code(a, r0, k0),     q4_code(a, r1, k0),     q4_code(a, r0, k0 + 2),
                               q4_code(a, r1, k0 + 2), q4_code(a, r0, k0 + 1), q4_code(a, r1, k0 + 1),
                               q4_code(a, r0, k0 + 3), q4_code(a, r1, k0 + 3)};
#pragma unroll
        for (int p = 0; p < 8; p++) out |= c[p] << (4 * p);
      } else {
        const int n = strip * 16 + (wi - 128);
        int s, r;
        if (resolve_row(a, n, s, r)) {
          const size_t gi = (size_t)r * groups + grp;
          out = (uint32_t)a.src[s].scale[gi] | ((uint32_t)a.src[s].bias[gi] << 16);
        }
      }
    } else {
      const int j = wi / 128, lane = (wi % 128) / 4, i = wi % 4, g = lane / 4, t = lane % 4;
      const int k0 = grp * 64 + 16 * t + 4 * j + ((i >> 1) << 1);
      const int row = strip * 16 + g + ((i & 1) << 3);
      out = bf16_as_f16_bits(a, row, k0) | (bf16_as_f16_bits(a, row, k0 + 1) << 16);
    }
    reinterpret_cast<uint32_t*>(a.dst)[w] = out;
  }
}

// grid (column chunks of kBlockCols, block rows): row 0 of a request is its anchor's embedding
// (or tok_proj of it) plus block_pos[0]; row k >= 1 is mask_emb[k-1] + block_pos[k]. Writes the
// residual h, the next input h * attn_norm_0 and one sum-of-squares part per chunk.
template <typename XT>
__global__ void __launch_bounds__(256) block_init_kernel(const __grid_constant__ BlockArgs a) {
  // kBlockCols columns of one block row per CTA, four per thread. The constant inputs (mask
  // embedding, block positions, first norm) are read before waiting for the previous kernel; only
  // row 0 (the anchor's embedding) needs data of this round.
  constexpr int kPer = kBlockCols / 256;
  const int r = blockIdx.y, chunk = blockIdx.x, b = r / a.gamma, k = r % a.gamma;
  __shared__ float red[8];
  const int j0 = chunk * kBlockCols + threadIdx.x;
  float bp[kPer], an[kPer], base[kPer];
#pragma unroll
  for (int u = 0; u < kPer; u++) {
    const int j = j0 + u * 256;
    const bool in = j < a.d;
    bp[u] = in ? a.block_pos[(size_t)k * a.d + j] : 0.f;
    an[u] = in ? a.attn_norm0[j] : 0.f;
    base[u] = (in && k > 0) ? a.mask_emb[(size_t)(k - 1) * a.d + j] : 0.f;
  }
  pdl_launch_dependents();
  pdl_wait();
  if (k == 0) {
    int tok = a.anchor[b];
    if (!in_bounds(tok >= 0 && tok < a.vocab, threadIdx.x == 0 && chunk == 0 ? a.err : nullptr))
      tok = tok < 0 ? 0 : a.vocab - 1;   // clamped: no read outside the table
#pragma unroll
    for (int u = 0; u < kPer; u++) {
      const int j = j0 + u * 256;
      if (j < a.d)
        base[u] = a.tokrow ? a.tokrow[(size_t)b * a.d + j]
                           : load_weight(a.fmt, a.emb, a.emb_scale, a.emb_bias, a.H, tok, j);
    }
  }
  float ss = 0.f;
#pragma unroll
  for (int u = 0; u < kPer; u++) {
    const int j = j0 + u * 256;
    if (j >= a.d) continue;
    const float v = base[u] + bp[u];
    a.h[(size_t)r * a.d + j] = v;
    store_act_split<XT>(a.xn, (size_t)r * a.d + j, a.xn_lo_off, v * an[u]);
    ss += v * v;
  }
  ss = warp_sum(ss);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) s += red[w];
    a.ssq[(size_t)r * a.ssq_ld + chunk] = s;
  }
}

template <typename XT>
__global__ void __launch_bounds__(256) embed_gather_kernel(const __grid_constant__ BlockArgs a) {
  const int b = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  int tok = a.anchor[b];
  if (!in_bounds(tok >= 0 && tok < a.vocab, threadIdx.x == 0 ? a.err : nullptr))
    tok = tok < 0 ? 0 : a.vocab - 1;   // clamped: no read outside the table
  for (int j = threadIdx.x; j < a.H; j += blockDim.x)
    static_cast<XT*>(a.emb_out)[(size_t)b * a.H + j] =
        from_f<XT>(load_weight(a.fmt, a.emb, a.emb_scale, a.emb_bias, a.H, tok, j));
}

// One warp per request: first mismatch via ballot.
// keep (nullable): per request, only the first keep[b] drafts are verified (pruned blocks).
// hist (nullable): hist[a] counts the blocks whose accepted length is a (0 <= a <= n).
__global__ void accept_kernel(int n, const int32_t* draft, const int32_t* keep, const int32_t* target,
                              int32_t* accept_len, int32_t* next_anchor, unsigned long long* hist, unsigned* err) {
  const int b = blockIdx.x, lane = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  int cap = n;
  if (keep) {
    cap = keep[b];
    if (!in_bounds(cap >= 0 && cap <= n, lane == 0 ? err : nullptr))
      cap = cap < 0 ? 0 : n;   // clamped: no read outside target's row
  }
  const bool miss = lane < cap && draft[(size_t)b * n + lane] != target[(size_t)b * (n + 1) + lane];
  const unsigned mask = __ballot_sync(0xffffffffu, miss);
  const int acc = mask ? __ffs(mask) - 1 : cap;
  if (lane == 0) {
    accept_len[b] = acc;
    next_anchor[b] = target[(size_t)b * (n + 1) + acc];
    if (hist) atomicAdd(hist + acc, 1ull);
  }
}

// Draft-length pruning: one warp per request; the first position k >= 1 whose confidence is
// below its threshold ends the block.
__global__ void draft_lengths_kernel(int n, const float* conf, const float* thresholds, float min_conf,
                                     int32_t* keep) {
  const int b = blockIdx.x, lane = threadIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  bool drop = false;
  if (lane >= 1 && lane < n) {
    const float th = thresholds ? thresholds[lane] : min_conf;
    drop = conf[(size_t)b * n + lane] < th;
  }
  const unsigned mask = __ballot_sync(0xffffffffu, drop);
  if (lane == 0) keep[b] = mask ? __ffs(mask) - 1 : n;
}

// Markov head input for draft k of every request: the W1 row of the previous token, as f16 plus
// its f16 remainder (the row is a stored weight, so hi + lo carries it to ~22 bits).
template <typename XT>
__global__ void __launch_bounds__(256) markov_gather_kernel(int k, int n, int rank, int vocab, int fmt,
                                                            const void* w1, const uint16_t* w1_scale,
                                                            const uint16_t* w1_bias, const int32_t* anchor,
                                                            const int32_t* draft, XT* x, size_t lo_off,
                                                            unsigned* err) {
  const int b = blockIdx.x;
  pdl_launch_dependents();
  pdl_wait();
  int prev = k == 0 ? anchor[b] : draft[(size_t)b * n + k - 1];
  if (!in_bounds(prev >= 0 && prev < vocab, threadIdx.x == 0 ? err : nullptr))
    prev = prev < 0 ? 0 : vocab - 1;   // clamped: no read outside the table
  for (int i = threadIdx.x; i < rank; i += blockDim.x)
    store_act_split<XT>(x, (size_t)b * rank + i, lo_off, load_weight(fmt, w1, w1_scale, w1_bias, rank, prev, i));
}

}  // namespace

cudaError_t launch_markov_gather(int n_req, int k, int n, int rank, int vocab, int fmt, const void* w1,
                                 const uint16_t* w1_scale, const uint16_t* w1_bias, const int32_t* anchor,
                                 const int32_t* draft, void* x, size_t lo_off, unsigned* err, cudaStream_t s) {
  if (fmt == FMT_F32)   // the CUDA-core path keeps fp32 activations
    return launch_pdl(markov_gather_kernel<float>, dim3(n_req), dim3(256), 0, s, k, n, rank, vocab, fmt, w1,
                      w1_scale, w1_bias, anchor, draft, static_cast<float*>(x), (size_t)0, err);
  return launch_pdl(markov_gather_kernel<__half>, dim3(n_req), dim3(256), 0, s, k, n, rank, vocab, fmt, w1,
                    w1_scale, w1_bias, anchor, draft, static_cast<__half*>(x), lo_off, err);
}

cudaError_t launch_draft_lengths(int n_req, int n, const float* conf, const float* thresholds, float min_conf,
                                 int32_t* keep, cudaStream_t s) {
  return launch_pdl(draft_lengths_kernel, dim3(n_req), dim3(32), 0, s, n, conf, thresholds, min_conf, keep);
}

cudaError_t launch_repack(const RepackArgs& a, cudaStream_t s) {
  repack_kernel<<<1024, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_block_init(const BlockArgs& a, cudaStream_t s) {
  const dim3 grid((a.d + kBlockCols - 1) / kBlockCols, a.n_req * a.gamma);
  if (a.act_f32) return launch_pdl(block_init_kernel<float>, grid, dim3(256), 0, s, a);
  return launch_pdl(block_init_kernel<__half>, grid, dim3(256), 0, s, a);
}

cudaError_t launch_embed_gather(const BlockArgs& a, cudaStream_t s) {
  if (a.act_f32) return launch_pdl(embed_gather_kernel<float>, dim3(a.n_req), dim3(256), 0, s, a);
  return launch_pdl(embed_gather_kernel<__half>, dim3(a.n_req), dim3(256), 0, s, a);
}

cudaError_t launch_accept(int n_req, int n, const int32_t* draft, const int32_t* keep, const int32_t* target,
                          int32_t* accept_len, int32_t* next_anchor, unsigned long long* hist, unsigned* err,
                          cudaStream_t s) {
  return launch_pdl(accept_kernel, dim3(n_req), dim3(32), 0, s, n, draft, keep, target, accept_len, next_anchor,
                    hist, err);
}

}  // namespace dfl

// Block attention of the KV-injection layer (Eq 3 of the dflash.ts page): the gamma block rows of
// one request attend, with NO causal mask, over [context rows in the window ++ all gamma block
// rows]; query head h reads K/V head h / (Hq/Hkv).
//
// Tensor-core path (f16 cache): grid = (kv head, key split, request), flash-decoding style.
//  * The CTA's query rows are the GQA group x gamma rows of one KV head (<= 64 rows, one 16-row
//    m-tile per warp), held in shared memory.
//  * Context K/V tiles of 64 rows x head_dim come from the per-layer ring cache
//    [slot][Hkv][cap][hd] through 4-D TMA copies (one for K, one for V, every 64-column part of
//    the head as its own sub-tile) with the 128-byte swizzle (two stages), so
//    ldmatrix reads are bank-conflict free. A tile never crosses the ring's wrap point; rows past
//    the ring end read as zeros and are masked.
//  * The last split also takes the 16-row block tile (K_d, V_d of this block, not cached).
//  * S = Q K^T and O += P V run on mma.sync m16n8k16 (f16 in, fp32 accumulate) with an online
//    softmax in fp32 (base-2 exponent, scores pre-scaled by log2(e)/sqrt(hd)).
//  * Each split writes (O, m, l); a second, wide kernel (one CTA per query row) merges the splits
//    in split order and writes the f16 attention output.
// CUDA-core path (fp32 cache): one warp per (query head, block row), online softmax over keys.
#include <cuda_fp16.h>
#include <math.h>

#include "common.cuh"

namespace dfl {

namespace {

constexpr int kAttnWarps = 8;   // two groups of four m-tile warps, each taking half of every key tile
constexpr int kGroupWarps = 4;
constexpr int kTileKeys = 64;
constexpr int kSub = 64 * 128;     // one 64-row x 128-byte swizzled sub-tile
constexpr int kBlkSub = 16 * 128;  // one 16-row x 128-byte swizzled sub-tile

__device__ __forceinline__ uint32_t swz(int row, int chunk) {  // byte offset in a sub-tile
  return row * 128 + ((chunk ^ (row & 7)) << 4);
}

// S[nb] for NKEY keys: Q rows of this warp's m-tile against the key tile.
template <int HD, int NKEY>
__device__ __forceinline__ void qk_tile(uint32_t q_base, uint32_t k_base, int sub_bytes, int mt, int lane,
                                        float (&S)[NKEY / 8][4], int key0 = 0) {
#pragma unroll
  for (int nb = 0; nb < NKEY / 8; nb++)
#pragma unroll
    for (int j = 0; j < 4; j++) S[nb][j] = 0.f;
#pragma unroll
  for (int kk = 0; kk < HD / 16; kk++) {
    const int sub = (kk * 16) / 64, chunk0 = ((kk * 16) % 64) / 8;
    uint32_t a0, a1, a2, a3;
    {
      const int row = mt * 16 + (lane & 15);
      const int chunk = chunk0 + (lane >> 4);
      ldmatrix_x4(q_base + sub * kSub + swz(row, chunk), a0, a1, a2, a3);
    }
#pragma unroll
    for (int nb = 0; nb < NKEY / 8; nb += 2) {
      const int key = key0 + nb * 8 + (lane & 7) + ((lane >> 4) << 3);
      const int chunk = chunk0 + ((lane >> 3) & 1);
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4(k_base + sub * sub_bytes + swz(key, chunk), b0, b1, b2, b3);
      mma_f16(S[nb], a0, a1, a2, a3, b0, b1);
      mma_f16(S[nb + 1], a0, a1, a2, a3, b2, b3);
    }
  }
}

// nvalid counts from key0 (the first of the NKEY keys of this call)
template <int HD, int NKEY>
__device__ __forceinline__ void softmax_pv(float (&S)[NKEY / 8][4], int nvalid, float scale_log2, uint32_t v_base,
                                           int sub_bytes, int lane, float (&m_run)[2], float (&l_run)[2],
                                           float (&O)[HD / 8][4], int key0 = 0) {
  const int t = lane & 3;
  float mt[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nb = 0; nb < NKEY / 8; nb++)
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const int key = nb * 8 + 2 * t + (j & 1);
      const float s = key < nvalid ? S[nb][j] * scale_log2 : -INFINITY;
      S[nb][j] = s;
      mt[j >> 1] = fmaxf(mt[j >> 1], s);
    }
#pragma unroll
  for (int h = 0; h < 2; h++) {
    mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 1));
    mt[h] = fmaxf(mt[h], __shfl_xor_sync(0xffffffffu, mt[h], 2));
  }
  float alpha[2], base[2];
#pragma unroll
  for (int h = 0; h < 2; h++) {
    const float mn = fmaxf(m_run[h], mt[h]);
    base[h] = mn == -INFINITY ? 0.f : mn;
    alpha[h] = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - mn);
    m_run[h] = mn;
    l_run[h] *= alpha[h];
  }
#pragma unroll
  for (int nb = 0; nb < NKEY / 8; nb++)
#pragma unroll
    for (int j = 0; j < 4; j++) {
      const float p = exp2f(S[nb][j] - base[j >> 1]);
      S[nb][j] = p;
      l_run[j >> 1] += p;
    }
#pragma unroll
  for (int nd = 0; nd < HD / 8; nd++) {
    O[nd][0] *= alpha[0];
    O[nd][1] *= alpha[0];
    O[nd][2] *= alpha[1];
    O[nd][3] *= alpha[1];
  }
#pragma unroll
  for (int kb = 0; kb < NKEY / 16; kb++) {
    const uint32_t a0 = pack_f16x2(S[2 * kb][0], S[2 * kb][1]);
    const uint32_t a1 = pack_f16x2(S[2 * kb][2], S[2 * kb][3]);
    const uint32_t a2 = pack_f16x2(S[2 * kb + 1][0], S[2 * kb + 1][1]);
    const uint32_t a3 = pack_f16x2(S[2 * kb + 1][2], S[2 * kb + 1][3]);
#pragma unroll
    for (int nd = 0; nd < HD / 8; nd += 2) {
      const int key = key0 + kb * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
      const int col8 = nd + (lane >> 4);  // 8-element column block of head_dim
      const int sub = col8 / 8, chunk = col8 % 8;
      uint32_t b0, b1, b2, b3;
      ldmatrix_x4_trans(v_base + sub * sub_bytes + swz(key, chunk), b0, b1, b2, b3);
      mma_f16(O[nd], a0, a1, a2, a3, b0, b1);
      mma_f16(O[nd + 1], a0, a1, a2, a3, b2, b3);
    }
  }
}

// Online combination of one key split (m, l, unnormalised O) into the running (M, L, O).
__device__ __forceinline__ void merge_split(float2 ml, float4 v, float& mx, float& L, float4& acc) {
  if (ml.x == -INFINITY) return;
  const float mn = fmaxf(mx, ml.x);
  const float so = mx == -INFINITY ? 0.f : exp2f(mx - mn), w = exp2f(ml.x - mn);
  L = fmaf(w, ml.y, L * so);
  acc.x = fmaf(w, v.x, acc.x * so);
  acc.y = fmaf(w, v.y, acc.y * so);
  acc.z = fmaf(w, v.z, acc.z * so);
  acc.w = fmaf(w, v.w, acc.w * so);
  mx = mn;
}

template <int HD>
__global__ void __launch_bounds__(kAttnWarps * 32) attn_tc_kernel(const __grid_constant__ AttnArgs a,
                                                                  const __grid_constant__ CUtensorMap kmap,
                                                                  const __grid_constant__ CUtensorMap vmap) {
  constexpr int NSUB = HD / 64;
  extern __shared__ __align__(1024) uint8_t sm[];
  // layout: Q [NSUB][64 rows] | K/V stages 2 x {K [NSUB][64], V [NSUB][64]} | block K, V [NSUB][16] | bars
  uint8_t* q_s = sm;
  uint8_t* stage_s = q_s + NSUB * kSub;
  uint8_t* bk_s = stage_s + 2 * 2 * NSUB * kSub;
  uint8_t* bv_s = bk_s + NSUB * kBlkSub;
  uint64_t* bars = reinterpret_cast<uint64_t*>(bv_s + NSUB * kBlkSub);

  const int kvh = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const AttnReq rq = a.req[b];
  const int grp = a.hq / a.hkv;
  const int M = grp * a.gamma;

  // context keys of this request: ring run 1 then run 2, tiled by 64
  const int P = rq.ctx_len;
  const int lo = (a.window > 0 && P > a.window) ? P - a.window : 0;
  const int nw = P - lo;
  const int s_lo = lo % a.cap;
  const int len1 = min(nw, a.cap - s_lo), len2 = nw - len1;
  const int T1 = (len1 + kTileKeys - 1) / kTileKeys, T2 = (len2 + kTileKeys - 1) / kTileKeys;
  const int T = T1 + T2;
  const int tb = (int)((long long)split * T / a.n_splits), te = (int)((long long)(split + 1) * T / a.n_splits);
  const int n_tiles = te - tb;
  const bool with_block = split == a.n_splits - 1;
  in_bounds(rq.slot >= 0 && rq.slot < a.max_batch && s_lo + len1 <= a.cap, threadIdx.x == 0 ? a.err : nullptr);
  const int plane = a.plane0 + rq.slot * a.hkv + kvh;

  auto tile_info = [&](int ti, int& slot0, int& nvalid) {
    if (ti < T1) {
      slot0 = s_lo + ti * kTileKeys;
      nvalid = min(kTileKeys, len1 - ti * kTileKeys);
    } else {
      slot0 = (ti - T1) * kTileKeys;
      nvalid = min(kTileKeys, len2 - (ti - T1) * kTileKeys);
    }
  };
  auto issue = [&](int i) {  // thread 0: context tile tb + i -> stage i % 2
    int slot0, nv;
    tile_info(tb + i, slot0, nv);
    const uint32_t bar = smem_u32(&bars[i & 1]);
    uint8_t* ks = stage_s + (i & 1) * 2 * NSUB * kSub;
    uint8_t* vs = ks + NSUB * kSub;
    mbar_arrive_expect_tx(bar, 2 * NSUB * kSub);
    // one copy each for K and V: all NSUB 64-column sub-tiles of the 64 keys (a copy has a fixed
    // cost of its own in the copy engine, so fewer, larger copies keep the tiles coming)
    tma_load_4d(smem_u32(ks), &kmap, 0, slot0, 0, plane, bar);
    tma_load_4d(smem_u32(vs), &vmap, 0, slot0, 0, plane, bar);
  };

  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bars[0]), 1);
    mbar_init(smem_u32(&bars[1]), 1);
    fence_barrier_init();
  }
  pdl_launch_dependents();
  pdl_wait();   // the cache rows and Q/K/V of this round were written by earlier kernels
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < min(2, n_tiles); i++) issue(i);
  }

  // Q rows (query row i = head-in-group * gamma + block row), pad rows zero; every load of a
  // thread is issued before its first shared-memory store
  constexpr int kThreads = kAttnWarps * 32;
  constexpr int kQPer = 64 * (HD / 8) / kThreads;
  const __half* qg = static_cast<const __half*>(a.q);
  uint4 qv[kQPer];
#pragma unroll
  for (int u = 0; u < kQPer; u++) {
    const int idx = threadIdx.x + u * kThreads;
    const int i = idx / (HD / 8), c8 = idx % (HD / 8);
    qv[u] = make_uint4(0, 0, 0, 0);
    if (i < M) {
      const int h = kvh * grp + i / a.gamma, k = i % a.gamma;
      qv[u] = *reinterpret_cast<const uint4*>(qg + (size_t)(rq.row0 + k) * a.qd + h * HD + c8 * 8);
    }
  }
  constexpr int kBPer = (16 * (HD / 8) + kThreads - 1) / kThreads;
  uint4 kv[kBPer], vv[kBPer];
  if (with_block) {
    const __half* kg = static_cast<const __half*>(a.kb);
    const __half* vg = static_cast<const __half*>(a.vb);
#pragma unroll
    for (int u = 0; u < kBPer; u++) {
      const int idx = threadIdx.x + u * kThreads;
      const int k = idx / (HD / 8), c8 = idx % (HD / 8);
      kv[u] = vv[u] = make_uint4(0, 0, 0, 0);
      if (idx < 16 * (HD / 8) && k < a.gamma) {
        const size_t off = (size_t)(rq.row0 + k) * a.kvd + kvh * HD + c8 * 8;
        kv[u] = *reinterpret_cast<const uint4*>(kg + off);
        vv[u] = *reinterpret_cast<const uint4*>(vg + off);
      }
    }
  }
#pragma unroll
  for (int u = 0; u < kQPer; u++) {
    const int idx = threadIdx.x + u * kThreads;
    const int i = idx / (HD / 8), c8 = idx % (HD / 8);
    *reinterpret_cast<uint4*>(q_s + (c8 / 8) * kSub + swz(i, c8 % 8)) = qv[u];
  }
  if (with_block) {
#pragma unroll
    for (int u = 0; u < kBPer; u++) {
      const int idx = threadIdx.x + u * kThreads;
      if (idx >= 16 * (HD / 8)) continue;
      const int k = idx / (HD / 8), c8 = idx % (HD / 8);
      const uint32_t o = (c8 / 8) * kBlkSub + swz(k, c8 % 8);
      *reinterpret_cast<uint4*>(bk_s + o) = kv[u];
      *reinterpret_cast<uint4*>(bv_s + o) = vv[u];
    }
  }
  __syncthreads();

  const int n_mt = (M + 15) / 16;
  const int mt = warp % kGroupWarps, kg = warp / kGroupWarps;   // m-tile, key half
  const bool active = mt < n_mt;
  float O[HD / 8][4];
#pragma unroll
  for (int nd = 0; nd < HD / 8; nd++)
#pragma unroll
    for (int j = 0; j < 4; j++) O[nd][j] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  const uint32_t q_base = smem_u32(q_s);

  int failed_at = -1;
  for (int i = 0; i < n_tiles; i++) {
    bool w = mbar_wait_bounded(smem_u32(&bars[i & 1]), (i >> 1) & 1, a.err, kErrTimeoutAttn);
    if (!__syncthreads_and(w)) {
      failed_at = i;
      break;
    }
    int slot0, nv;
    tile_info(tb + i, slot0, nv);
    if (active) {
      constexpr int kHalf = kTileKeys / 2;
      const uint32_t ks = smem_u32(stage_s + (i & 1) * 2 * NSUB * kSub);
      float S[kHalf / 8][4];
      qk_tile<HD, kHalf>(q_base, ks, kSub, mt, lane, S, kg * kHalf);
      softmax_pv<HD, kHalf>(S, nv - kg * kHalf, a.scale_log2, ks + NSUB * kSub, kSub, lane, m_run, l_run, O,
                            kg * kHalf);
    }
    __syncthreads();
    if (threadIdx.x == 0 && i + 2 < n_tiles) issue(i + 2);
  }
  if (failed_at >= 0) {
    if (threadIdx.x == 0)  // leave no copy in flight: tiles failed_at and failed_at + 1 may be
      for (int i = failed_at; i < min(failed_at + 2, n_tiles); i++)
        mbar_wait_bounded(smem_u32(&bars[i & 1]), (i >> 1) & 1, nullptr, 0);
    return;
  }
  if (with_block && active && kg == 0) {
    float S[2][4];
    qk_tile<HD, 16>(q_base, smem_u32(bk_s), kBlkSub, mt, lane, S);
    softmax_pv<HD, 16>(S, a.gamma, a.scale_log2, smem_u32(bv_s), kBlkSub, lane, m_run, l_run, O);
  }
#pragma unroll
  for (int h = 0; h < 2; h++) {
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 1);
    l_run[h] += __shfl_xor_sync(0xffffffffu, l_run[h], 2);
  }
  // merge the two key halves: group 1 parks (O, m, l) in the free stage buffers, group 0 folds
  // them into its own state (the stage buffers hold at least 4 warps x 32 lanes x (HD/2 + 4) floats)
  {
    constexpr int kPer = HD / 2 + 4;
    float* park = reinterpret_cast<float*>(stage_s) + ((size_t)mt * 32 + lane) * kPer;
    __syncthreads();   // every warp is done with the last tile
    if (kg == 1 && active) {
#pragma unroll
      for (int nd = 0; nd < HD / 8; nd++)
        *reinterpret_cast<float4*>(park + nd * 4) = make_float4(O[nd][0], O[nd][1], O[nd][2], O[nd][3]);
      *reinterpret_cast<float4*>(park + HD / 2) = make_float4(m_run[0], m_run[1], l_run[0], l_run[1]);
    }
    __syncthreads();
    if (kg == 0 && active) {
      const float4 ml = *reinterpret_cast<const float4*>(park + HD / 2);
      const float mo[2] = {ml.x, ml.y}, lo[2] = {ml.z, ml.w};
      float sa[2], sb[2];
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const float mn = fmaxf(m_run[h], mo[h]);
        sa[h] = m_run[h] == -INFINITY ? 0.f : exp2f(m_run[h] - mn);
        sb[h] = mo[h] == -INFINITY ? 0.f : exp2f(mo[h] - mn);
        m_run[h] = mn;
        l_run[h] = l_run[h] * sa[h] + lo[h] * sb[h];
      }
#pragma unroll
      for (int nd = 0; nd < HD / 8; nd++) {
        const float4 v = *reinterpret_cast<const float4*>(park + nd * 4);
        O[nd][0] = O[nd][0] * sa[0] + v.x * sb[0];
        O[nd][1] = O[nd][1] * sa[0] + v.y * sb[0];
        O[nd][2] = O[nd][2] * sa[1] + v.z * sb[1];
        O[nd][3] = O[nd][3] * sa[1] + v.w * sb[1];
      }
    }
  }

  __half* out = static_cast<__half*>(a.out);
  if (a.n_splits == 1) {
    if (active && kg == 0) {
#pragma unroll
      for (int h = 0; h < 2; h++) {
        const int i = mt * 16 + g + 8 * h;
        if (i >= M) continue;
        const int head = kvh * grp + i / a.gamma, k = i % a.gamma;
        const float inv = 1.0f / l_run[h];
        __half* o = out + (size_t)(rq.row0 + k) * a.qd + head * HD;
#pragma unroll
        for (int nd = 0; nd < HD / 8; nd++)
          *reinterpret_cast<uint32_t*>(o + nd * 8 + 2 * t) = pack_f16x2(O[nd][2 * h] * inv, O[nd][2 * h + 1] * inv);
      }
    }
    return;
  }

  // split partials (unnormalised O, running max m and sum l, base 2); attn_merge_kernel combines them
  const int pair = b * a.hkv + kvh;
  const size_t pidx = (size_t)pair * a.n_splits + split;
  if (active && kg == 0) {
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const int i = mt * 16 + g + 8 * h;
      float* po = a.part_o + (pidx * 64 + i) * HD;
#pragma unroll
      for (int nd = 0; nd < HD / 8; nd++)
        *reinterpret_cast<float2*>(po + nd * 8 + 2 * t) = make_float2(O[nd][2 * h], O[nd][2 * h + 1]);
      if (t == 0) *reinterpret_cast<float2*>(&a.part_ml[(pidx * 64 + i) * 2]) = make_float2(m_run[h], l_run[h]);
    }
  }
}

// Combine the key splits of one query row: grid (request * kv head, query row), one float4 of
// head_dim per thread. Splits are taken in order, sixteen at a time with all their loads in
// flight, and combined online: O = sum_s 2^(m_s - M) O_s / sum_s 2^(m_s - M) l_s, M the running
// maximum.
template <int HD>
__global__ void __launch_bounds__(HD / 4) attn_merge_kernel(const __grid_constant__ AttnArgs a) {
  pdl_launch_dependents();
  pdl_wait();
  const int pair = blockIdx.x, i = blockIdx.y, c4 = threadIdx.x;
  const int b = pair / a.hkv, kvh = pair % a.hkv, grp = a.hq / a.hkv;
  const size_t pbase = (size_t)pair * a.n_splits;
  float mx = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < a.n_splits; s0 += 16) {
    float2 ml[16];
    float4 v[16];
#pragma unroll
    for (int q = 0; q < 16; q++) {
      const int s2 = s0 + q;
      const bool in = s2 < a.n_splits;
      ml[q] = in ? __ldcg(reinterpret_cast<const float2*>(&a.part_ml[((pbase + s2) * 64 + i) * 2]))
                 : make_float2(-INFINITY, 0.f);
      v[q] = in ? __ldcg(reinterpret_cast<const float4*>(a.part_o + ((pbase + s2) * 64 + i) * HD) + c4)
                : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int q = 0; q < 16; q++) merge_split(ml[q], v[q], mx, L, acc);
  }
  const float inv = 1.0f / L;
  const int head = kvh * grp + i / a.gamma, k = i % a.gamma;
  __half* o = static_cast<__half*>(a.out) + (size_t)(a.req[b].row0 + k) * a.qd + head * HD + c4 * 4;
  *reinterpret_cast<uint2*>(o) = make_uint2(pack_f16x2(acc.x * inv, acc.y * inv), pack_f16x2(acc.z * inv, acc.w * inv));
}

// fp32 path: warp per (query head, block row)
__global__ void __launch_bounds__(128) attn_f32_kernel(const __grid_constant__ AttnArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y;
  const int pair = blockIdx.x * 4 + warp;  // = head * gamma + k
  if (pair >= a.hq * a.gamma) return;
  const int head = pair / a.gamma, k = pair % a.gamma;
  const AttnReq rq = a.req[b];
  const int grp = a.hq / a.hkv, kvh = head / grp, hd = a.hd;
  const float* q = static_cast<const float*>(a.q) + (size_t)(rq.row0 + k) * a.qd + head * hd;
  const float* kc = static_cast<const float*>(a.kc) + ((size_t)rq.slot * a.hkv + kvh) * a.cap * hd;
  const float* vc = static_cast<const float*>(a.vc) + ((size_t)rq.slot * a.hkv + kvh) * a.cap * hd;
  const float* kb = static_cast<const float*>(a.kb);
  const float* vb = static_cast<const float*>(a.vb);
  const int P = rq.ctx_len;
  const int lo = (a.window > 0 && P > a.window) ? P - a.window : 0;
  const int nw = P - lo, nkeys = nw + a.gamma;
  const float scale = rsqrtf((float)hd);
  float m = -INFINITY, l = 0.f, o[8];  // hd <= 256: lane holds c = lane + 32 j
#pragma unroll
  for (int j = 0; j < 8; j++) o[j] = 0.f;
  for (int j0 = 0; j0 < nkeys; j0 += 32) {
    const int j = j0 + lane;
    const float* kr = nullptr;
    if (j < nw) kr = kc + (size_t)((lo + j) % a.cap) * hd;
    else if (j < nkeys) kr = kb + (size_t)(rq.row0 + j - nw) * a.kvd + kvh * hd;
    float s = -INFINITY;
    if (kr) {
      s = 0.f;
      for (int c = 0; c < hd; c++) s = fmaf(q[c], kr[c], s);
      s *= scale;
    }
    float cm = s;
    for (int o2 = 16; o2 > 0; o2 >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
    const float mn = fmaxf(m, cm);
    const float alpha = m == -INFINITY ? 0.f : expf(m - mn);
    const float p = kr ? expf(s - mn) : 0.f;
    l = l * alpha + warp_sum(p);
    m = mn;
#pragma unroll
    for (int jj = 0; jj < 8; jj++) o[jj] *= alpha;
    for (int src = 0; src < 32 && j0 + src < nkeys; src++) {
      const float ps = __shfl_sync(0xffffffffu, p, src);
      const int js = j0 + src;
      const float* vr = js < nw ? vc + (size_t)((lo + js) % a.cap) * hd
                                : vb + (size_t)(rq.row0 + js - nw) * a.kvd + kvh * hd;
#pragma unroll
      for (int jj = 0; jj < 8; jj++) {
        const int c = lane + 32 * jj;
        if (c < hd) o[jj] = fmaf(ps, vr[c], o[jj]);
      }
    }
  }
  float* out = static_cast<float*>(a.out) + (size_t)(rq.row0 + k) * a.qd + head * hd;
#pragma unroll
  for (int jj = 0; jj < 8; jj++) {
    const int c = lane + 32 * jj;
    if (c < hd) out[c] = o[jj] / l;
  }
}

}  // namespace

size_t attn_smem_bytes(int hd) {
  const int nsub = hd / 64;
  return (size_t)nsub * kSub + 2 * 2 * nsub * kSub + 2 * nsub * kBlkSub + 64;
}

cudaError_t launch_attn_tc(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t s) {
  const dim3 grid(a.hkv, a.n_splits, a.n_req);
  const size_t smem = attn_smem_bytes(a.hd);
  cudaError_t err;
#define DFL_ATTN(HD)                                                                                \
  {                                                                                                 \
    static std::atomic<int> smem_set[kMaxDevices];                                                  \
    err = ensure_smem_limit(attn_tc_kernel<HD>, smem, smem_set);                                    \
    if (err != cudaSuccess) return err;                                                             \
  }                                                                                                 \
  return launch_pdl(attn_tc_kernel<HD>, grid, dim3(kAttnWarps * 32), smem, s, a, kmap, vmap);
  switch (a.hd) {
    case 64: { DFL_ATTN(64) }
    case 128: { DFL_ATTN(128) }
    case 256: { DFL_ATTN(256) }
    default: return cudaErrorInvalidValue;
  }
#undef DFL_ATTN
}

cudaError_t launch_attn_merge(const AttnArgs& a, cudaStream_t s) {
  const dim3 grid(a.n_req * a.hkv, (a.hq / a.hkv) * a.gamma);
  switch (a.hd) {
    case 64: return launch_pdl(attn_merge_kernel<64>, grid, dim3(16), 0, s, a);
    case 128: return launch_pdl(attn_merge_kernel<128>, grid, dim3(32), 0, s, a);
    case 256: return launch_pdl(attn_merge_kernel<256>, grid, dim3(64), 0, s, a);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_attn_f32(const AttnArgs& a, cudaStream_t s) {
  const dim3 grid((a.hq * a.gamma + 3) / 4, a.n_req);
  attn_f32_kernel<<<grid, 128, 0, s>>>(a);
  return cudaGetLastError();
}

}  // namespace dfl

// The draft round's skinny projections (at most 32 activation rows) on the fifth-generation
// tensor cores, with the GEMV's fused epilogues: one launch per projection, HBM-bound.
//
// The (128-row tile, 64-input group) units of the matrix, in tile-major order, are cut into one
// contiguous range per CTA (one CTA per SM), so every CTA streams the same number of weight bytes.
// Fourteen warps:
//  * warp 0 (one thread) requests the range's 4-bit (strip, group) tiles with bulk copies into a
//    deep ring -- the first stages before waiting for the previous kernel, since weights never
//    change -- and each unit's activation rows (f16, plus the f16 remainder where given) with 2-D
//    tensor copies in the 128-byte swizzle;
//  * warps 2-9 (one 16-row strip each) dequantise the codes to f16 weights, w = s q + b with one
//    rounding, into the MMA's swizzled K-major A tile;
//  * warp 1 allocates tensor memory; one of its threads issues tcgen05.mma kind::f16 (M = 128,
//    N = the contraction rows padded to 16, K = 16), accumulating each segment (the units of one
//    tile inside the range) in one of two fp32 accumulators;
//  * warps 10-13 (tensor-memory lane quarters 2, 3, 0, 1) read a finished segment's accumulator.
//    A segment that covers its whole tile goes through a shared-memory tile to the GEMV's strip
//    epilogues (two strips per warp). A tile cut between CTAs is stored as partial pieces (at most
//    two per CTA: its first and last segments); the last CTA to arrive at the tile's ticket sums
//    the pieces in CTA order and runs the epilogue, so the result does not depend on who arrives
//    last.
// Every mbarrier wait is bounded (error word + early exit); tensor memory is freed at the end.
#include <cuda.h>
#include <cuda_fp16.h>

#include "gemm_tc05.h"
#include "gemv_impl.cuh"
#include "tc05.cuh"

namespace dfl {

namespace {

constexpr int kPjWarps = 14;
constexpr int kPjThreads = kPjWarps * 32;
constexpr int kPjEpiWarp0 = 10;                           // epilogue warps 10-13
constexpr int kPjChains = 4;                              // independent accumulators per segment (one per K step)
constexpr int kPjStrips = 8;                              // 16-row strips per 128-row tile
constexpr int kPjKG = 4;                                  // groups per raw stage (per-strip copies of 2304 B)
constexpr int kPjWStage = kPjStrips * kPjKG * kQ4GroupBytes;   // 18 KB: a raw stage's weights
constexpr int kPjAStage = 128 * 128;                      // 16 KB: one unit, f16
constexpr uint32_t kPjEpiBar = 1;                         // named barrier of the epilogue warps

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 bits_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// (c + q0, c + q1) -> s * (q0, q1) + b in f16 with one rounding; q exact after the subtraction
__device__ __forceinline__ uint32_t dequant2(uint32_t v, __half2 c, __half2 s, __half2 b) {
  return h2_bits(__hfma2(__hsub2(bits_h2(v), c), s, b));
}

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync %0, %1;" ::"r"(kPjEpiBar), "r"(4 * 32) : "memory"); }

// First unit of CTA c when T units are cut into n contiguous ranges.
__device__ __forceinline__ long long range_start(long long T, int n, int c) { return T * c / n; }

// The CTA whose range holds unit u.
__device__ __forceinline__ int cta_of_unit(long long T, int n, long long u) {
  int c = (int)((u * n) / T);
  while (c + 1 < n && range_start(T, n, c + 1) <= u) c++;
  while (c > 0 && range_start(T, n, c) > u) c--;
  return c;
}

// The raw stages of a CTA's range: stage j holds up to kPjKG consecutive groups of one tile (one
// bulk copy of n x 576 B per strip, since a strip's groups are contiguous in the stored layout).
struct StageWalk {
  long long v;   // first unit of the stage
  int j;         // stage index within the range
  int i;         // unit index (within the range) of v
  int mt, g, n;  // tile, first group and units of the stage
  __device__ __forceinline__ void set(long long u1, int groups) {
    mt = (int)(v / groups);
    g = (int)(v - (long long)mt * groups);
    n = (int)min((long long)min(kPjKG, groups - g), u1 - v);
  }
  __device__ __forceinline__ void next(long long u1, int groups) {
    v += n;
    i += n;
    j++;
    if (v < u1) set(u1, groups);
  }
};

template <int EPI, int NT, int NP>
__global__ void __launch_bounds__(kPjThreads, 1) proj_tc05_kernel(const __grid_constant__ ProjArgs pa) {
  const GemvArgs& a = pa.g;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // A stages (pa.sa): dequantised weights of one unit. Raw stages (pa.sw): the 4-bit tiles of up to
  // kPjKG units and, after them, those units' activation tiles, so both share one lookahead.
  const uint32_t raw_bytes = kPjWStage + kPjKG * pa.x_stage;   // a multiple of 1024
  uint8_t* aring = sm;                                          // pa.sa x 16 KB (1024-aligned)
  uint8_t* wring = aring + pa.sa * kPjAStage;                   // pa.sw x raw_bytes (1024-aligned)
  float* tile = reinterpret_cast<float*>(wring + (size_t)pa.sw * raw_bytes);   // [128][NP] fp32
  float* srow = tile + 128 * NP;                                // kMaxRows row scales
  uint64_t* bars = reinterpret_cast<uint64_t*>(srow + kMaxRows);
  uint64_t* full_w = bars;                                      // weights and activations landed
  uint64_t* empty_w = full_w + pa.sw;                           // decoders and MMAs done with a raw stage
  uint64_t* full_a = empty_w + pa.sw;                           // an A stage written
  uint64_t* freed = full_a + pa.sa;                             // an A stage's MMAs completed
  uint64_t* acc_full = freed + pa.sa;
  uint64_t* acc_empty = acc_full + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_empty + 2);
  int* flag = reinterpret_cast<int*>(tmem_slot + 1);           // last-arriver decision, broadcast
  int* okflag = flag + 1;                                       // accumulator wait result, broadcast

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long T = (long long)pa.mtiles * pa.groups;
  const long long u0 = range_start(T, gridDim.x, blockIdx.x), u1 = range_start(T, gridDim.x, blockIdx.x + 1);
  const int n_units = (int)(u1 - u0);

  if (threadIdx.x == 0) {
    for (int i = 0; i < pa.sw; i++) {
      mbar_init(smem_u32(&full_w[i]), 1);
      mbar_init(smem_u32(&empty_w[i]), kPjStrips + 1);   // eight dequantising warps + the MMA commit
    }
    for (int i = 0; i < pa.sa; i++) {
      mbar_init(smem_u32(&full_a[i]), kPjStrips);
      mbar_init(smem_u32(&freed[i]), 1);                  // the MMA commit
    }
    for (int b = 0; b < 2; b++) {
      mbar_init(smem_u32(&acc_full[b]), 1);               // the MMA commit
      mbar_init(smem_u32(&acc_empty[b]), 4);              // the four epilogue warps
    }
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), (uint32_t)pa.tmem_cols);
    tmem_relinquish();
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_launch_dependents();

  // The copy and MMA warps run their loops with all 32 lanes (one lane issues): a lone lane whose
  // warp-mates wait at a block barrier is scheduled far too rarely for an issue loop.
  if (warp == 0) {
    // ---- copies ------------------------------------------------------------------------------------
    if (n_units > 0) {
      bool ok = true;
      int nw = 0;   // stages whose copies were issued
      auto weights = [&](const StageWalk& st, int sw) {
        if (lane != 0) return;
        in_bounds(st.mt < pa.mtiles && st.g + st.n <= pa.groups && st.n > 0, a.err);
        const int strips = min(kPjStrips, pa.n_strips - st.mt * kPjStrips);
        const uint32_t fw = smem_u32(&full_w[sw]);
        mbar_arrive_expect_tx(fw, (uint32_t)(strips * st.n * kQ4GroupBytes + st.n * pa.x_stage));
        for (int s = 0; s < strips; s++)
          bulk_g2s(smem_u32(wring + (size_t)sw * raw_bytes + s * (kPjKG * kQ4GroupBytes)),
                   pa.w + ((size_t)(st.mt * kPjStrips + s) * pa.groups + st.g) * kQ4GroupBytes,
                   (uint32_t)(st.n * kQ4GroupBytes), fw);
      };
      auto acts = [&](const StageWalk& st, int sw) {
        if (lane != 0) return;
        const uint32_t fw = smem_u32(&full_w[sw]);
        for (int gi = 0; gi < st.n; gi++) {
          const uint32_t xst = smem_u32(wring + (size_t)sw * raw_bytes + kPjWStage + gi * pa.x_stage);
          tma_load_2d(xst, &pa.xmap, (st.g + gi) * 64, 0, fw);
          if (pa.has_lo) tma_load_2d(xst + NP * 128, &pa.xlmap, (st.g + gi) * 64, 0, fw);
        }
      };
      // weights never change: the first stages' weights go out before waiting for the previous
      // kernel, their activations after it
      StageWalk st{u0, 0, 0};
      st.set(u1, pa.groups);
      StageWalk first = st;
      for (; st.v < u1 && st.j < pa.sw; st.next(u1, pa.groups)) {
        weights(st, st.j);
        nw = st.j + 1;
      }
      pdl_wait();
      for (StageWalk q = first; q.v < u1 && q.j < pa.sw; q.next(u1, pa.groups)) acts(q, q.j);
      __syncwarp();
      for (; st.v < u1 && ok; st.next(u1, pa.groups)) {
        const int sw = st.j % pa.sw;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&empty_w[sw]), ((st.j / pa.sw) + 1) & 1, a.err,
                                                       kErrTimeoutProj));
        if (!ok) break;
        weights(st, sw);
        acts(st, sw);
        __syncwarp();
        nw = st.j + 1;
      }
      // leave no copy in flight into this CTA's shared memory, also when a consumer gave up
      for (int j = nw > pa.sw ? nw - pa.sw : 0; j < nw; j++)
        mbar_wait_bounded(smem_u32(&full_w[j % pa.sw]), (j / pa.sw) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    // ---- MMA issue: per segment (the range's units of one tile) kPjChains accumulators, K step kk
    // of every unit into chain kk, so consecutive MMAs do not wait for each other's results
    if (n_units > 0) {
      const uint32_t idesc = umma_idesc_f16_f32(128, NP);
      bool ok = true;
      int issued = 0, seg = -1, first_of_seg = 1;
      StageWalk st{u0, 0, 0};
      st.set(u1, pa.groups);
      for (; st.v < u1 && ok; st.next(u1, pa.groups)) {
        const int sw = st.j % pa.sw;
        for (int gi = 0; gi < st.n && ok; gi++) {
          const int i = st.i + gi, g = st.g + gi, sa = i % pa.sa;
          if (i == 0 || g == 0) {   // a new segment
            seg++;
            first_of_seg = 1;
            if (seg >= 2)
              ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&acc_empty[seg & 1]), ((seg >> 1) + 1) & 1,
                                                             a.err, kErrTimeoutProj));
          }
          // the decoders wrote this A stage after the raw stage (weights and activations) landed
          ok = ok && __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full_a[sa]), (i / pa.sa) & 1, a.err,
                                                               kErrTimeoutProj));
          if (!ok) break;
          tc05_fence_after();
          if (lane == 0) {
            const uint32_t d = tmem + (uint32_t)((seg & 1) * kPjChains * NP);
            const uint32_t abase = smem_u32(aring + sa * kPjAStage);
            const uint32_t xbase = smem_u32(wring + (size_t)sw * raw_bytes + kPjWStage + gi * pa.x_stage);
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
              const uint64_t ad = umma_desc_sw128(abase + 32 * kk);
              const uint32_t dk = d + (uint32_t)(kk * NP);
              umma_f16_ss(dk, ad, umma_desc_sw128(xbase + 32 * kk), idesc, first_of_seg ? 0u : 1u);
              if (pa.has_lo) umma_f16_ss(dk, ad, umma_desc_sw128(xbase + NP * 128 + 32 * kk), idesc, 1u);
            }
            umma_commit(smem_u32(&freed[sa]));
            if (gi + 1 == st.n) umma_commit(smem_u32(&empty_w[sw]));   // its activations were read
            if (i + 1 == n_units || g + 1 == pa.groups) umma_commit(smem_u32(&acc_full[seg & 1]));
          }
          __syncwarp();
          first_of_seg = 0;
          issued = i + 1;
        }
      }
      // nothing of this CTA may still be running on the tensor core when its memory is freed
      if (issued > 0)
        mbar_wait_bounded(smem_u32(&freed[(issued - 1) % pa.sa]), ((issued - 1) / pa.sa) & 1, a.err,
                          kErrTimeoutProj);
    }
  } else if (warp < kPjEpiWarp0) {
    // ---- dequantise: 4-bit codes -> f16 weights, swizzled K-major A tile ---------------------------
    const int s = warp - 2, g8 = lane >> 2, t = lane & 3;
    const __half2 c1024 = __float2half2_rn(1024.f), c64 = __float2half2_rn(64.f);
    bool ok = n_units > 0;
    StageWalk st{u0, 0, 0};
    if (ok) st.set(u1, pa.groups);
    for (; st.v < u1 && ok; st.next(u1, pa.groups)) {
      const int sw = st.j % pa.sw;
      const int strips = min(kPjStrips, pa.n_strips - st.mt * kPjStrips);
      ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full_w[sw]), (st.j / pa.sw) & 1, a.err, kErrTimeoutProj));
      if (!ok) break;
      const uint8_t* sp = wring + (size_t)sw * raw_bytes + s * (kPjKG * kQ4GroupBytes);
      __half2 sg, bg, s8, b8;
      for (int gi = 0; gi < st.n && ok; gi++) {
        const int i = st.i + gi, sa = i % pa.sa;
        if (i >= pa.sa)
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&freed[sa]), ((i / pa.sa) + 1) & 1, a.err,
                                                         kErrTimeoutProj));
        if (!ok) break;
        const uint8_t* gp = sp + gi * kQ4GroupBytes;
        const uint32_t ast = smem_u32(aring + sa * kPjAStage);
        uint32_t rg[4][2], r8[4][2];
        if (s < strips) {
          const uint4 W = *reinterpret_cast<const uint4*>(gp + lane * 16);
          const uint32_t sbg = *reinterpret_cast<const uint32_t*>(gp + 512 + 4 * g8);
          const uint32_t sb8 = *reinterpret_cast<const uint32_t*>(gp + 512 + 4 * (g8 + 8));
          sg = __float2half2_rn(__uint_as_float(sbg << 16));
          bg = __float2half2_rn(__uint_as_float(sbg & 0xFFFF0000u));
          s8 = __float2half2_rn(__uint_as_float(sb8 << 16));
          b8 = __float2half2_rn(__uint_as_float(sb8 & 0xFFFF0000u));
          const uint32_t w4[4] = {W.x, W.y, W.z, W.w};
#pragma unroll
          for (int j = 0; j < 4; j++) {
            // word j of lane (g, t): inputs k0 = 16 t + 4 j .. k0 + 3 of rows g and g + 8, nibbles
            // (g,k0) (g+8,k0) (g,k0+2) (g+8,k0+2) (g,k0+1) (g+8,k0+1) (g,k0+3) (g+8,k0+3) from bit 0
            const uint32_t w = w4[j], w8 = w >> 8;
            rg[j][0] = dequant2(lop3_and_or(w, 0x000F000Fu, 0x64006400u), c1024, sg, bg);    // 1024 + q
            rg[j][1] = dequant2(lop3_and_or(w8, 0x000F000Fu, 0x64006400u), c1024, sg, bg);
            r8[j][0] = dequant2(lop3_and_or(w, 0x00F000F0u, 0x54005400u), c64, s8, b8);      // 64 + q
            r8[j][1] = dequant2(lop3_and_or(w8, 0x00F000F0u, 0x54005400u), c64, s8, b8);
          }
        } else {
#pragma unroll
          for (int j = 0; j < 4; j++) rg[j][0] = rg[j][1] = r8[j][0] = r8[j][1] = 0u;
        }
        // 16-byte chunk c of row r lives at r * 128 + ((c ^ (r % 8)) * 16); r % 8 == g here
        const uint32_t row_g = ast + (uint32_t)(s * 16 + g8) * 128, row_8 = row_g + 8 * 128;
        const uint32_t c0 = (uint32_t)(((2 * t) ^ g8) << 4), c1 = (uint32_t)(((2 * t + 1) ^ g8) << 4);
        st_shared_v4(row_g + c0, rg[0][0], rg[0][1], rg[1][0], rg[1][1]);
        st_shared_v4(row_g + c1, rg[2][0], rg[2][1], rg[3][0], rg[3][1]);
        st_shared_v4(row_8 + c0, r8[0][0], r8[0][1], r8[1][0], r8[1][1]);
        st_shared_v4(row_8 + c1, r8[2][0], r8[2][1], r8[3][0], r8[3][1]);
        fence_proxy_async();   // generic stores read by the tensor core
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&full_a[sa]));
      }
      if (!ok) break;
      fence_proxy_async();     // this warp's reads of the raw stage come before its refill
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&empty_w[sw]));
    }
  } else {
    // ---- epilogue warps ------------------------------------------------------------------------------
    const int ew = warp - kPjEpiWarp0, quarter = warp & 3;
    const int n = quarter * 32 + lane;                     // tile row = tensor-memory lane
    const int et = threadIdx.x - kPjEpiWarp0 * 32;         // 0..127
    pdl_wait();
    // per-row RMSNorm scales of the epilogue's rows (from the producers' sum-of-squares partials)
    {
      const int two = a.norm_mode == NORM_CTX ? 2 : 1;
      for (int r = ew; r < NT * 8; r += 4) {
        float sc = 1.0f;
        if (r < a.R && a.norm_mode != NORM_NONE) {
          const float* base = a.ssq + (size_t)map_row(a.xmap, r) * a.ssq_ld * two;
          float sa0 = 0.f, sb0 = 0.f;
          for (int p = lane; p < a.ssq_parts; p += 32) {
            sa0 += __ldcg(base + (size_t)p * two);
            if (two == 2) sb0 += __ldcg(base + (size_t)p * 2 + 1);
          }
          sa0 = warp_sum(sa0);
          if (a.norm_mode == NORM_ONE) {
            sc = rsqrtf(sa0 * a.inv_dim + a.eps);
          } else {
            sb0 = warp_sum(sb0);
            const float inv1 = rsqrtf(sa0 * a.inv_dim + a.eps);
            sc = inv1 * rsqrtf(inv1 * inv1 * sb0 * a.inv_dim + a.eps);
          }
        }
        if (lane == 0) srow[r] = sc;
      }
    }
    epi_bar();
    LmState lm[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; nt++)
#pragma unroll
      for (int p = 0; p < 2; p++) lm[nt][p] = LmState{-INFINITY, 0.f, 0x7fffffff};
    // the tile in shared memory -> the strip epilogues of this warp's two strips
    auto run_tile = [&](int mt) {
      epi_bar();   // every row of the tile is in shared memory
      const int g = lane >> 2, t = lane & 3;
#pragma unroll 1
      for (int j = 0; j < 2; j++) {
        const int sl = 2 * ew + j, strip = mt * kPjStrips + sl;
        if (strip >= pa.n_strips) break;
        float y[NT][4];
#pragma unroll
        for (int nt = 0; nt < NT; nt++)
#pragma unroll
          for (int p = 0; p < 2; p++) {
            const int c = nt * 8 + 2 * t + p;
            const int col = c < a.R ? pa.row_base + map_row(a.xmap, c) : 0;
            y[nt][p] = tile[(sl * 16 + g) * NP + col];
            y[nt][2 + p] = tile[(sl * 16 + g + 8) * NP + col];
          }
        EpiPre<NT> pre;
        epi_preload<EPI, NT, __half>(a, strip, pre);
        strip_epilogue<EPI, NT, __half>(a, strip, y, srow, lm, 0, pre);
      }
      epi_bar();   // the tile may be overwritten
    };
    bool ok = n_units > 0;
    int seg = 0;
    for (long long u = u0; u < u1 && ok; seg++) {
      const int mt = (int)(u / pa.groups);
      const long long tb = (long long)mt * pa.groups, te = tb + pa.groups;
      const long long su1 = min(u1, te);
      const bool whole = u == tb && su1 == te;
      const int b = seg & 1;
      // one warp waits and the barrier hands the result to all four warps, so that they take the
      // same number of named barriers whatever happens
      if (ew == 0) {
        const bool w_ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&acc_full[b]), (seg >> 1) & 1, a.err,
                                                                    kErrTimeoutProj));
        if (lane == 0) *okflag = w_ok;
      }
      epi_bar();
      ok = *okflag != 0;
      if (!ok) break;
      tc05_fence_after();
      // the segment's result: its chains summed in chain order
      float v[NP];
      const uint32_t taddr = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(b * kPjChains * NP);
#pragma unroll
      for (int h = 0; h < NP; h += 16) {
        float w[16];
        tmem_ld16(taddr + h, w);
#pragma unroll
        for (int e = 0; e < 16; e++) v[h + e] = w[e];
#pragma unroll
        for (int ch = 1; ch < kPjChains; ch++) {
          tmem_ld16(taddr + (uint32_t)(ch * NP + h), w);
#pragma unroll
          for (int e = 0; e < 16; e++) v[h + e] += w[e];
        }
      }
      tc05_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&acc_empty[b]));
      if (whole) {
#pragma unroll
        for (int c = 0; c < NP; c += 4)
          *reinterpret_cast<float4*>(&tile[n * NP + c]) = make_float4(v[c], v[c + 1], v[c + 2], v[c + 3]);
        run_tile(mt);
      } else {
        // partial piece: slot 0 = this CTA's first segment, 1 = its last
        const int slot = u == u0 ? 0 : 1;
        float* piece = pa.partials + ((size_t)blockIdx.x * 2 + slot) * NP * 128;
#pragma unroll
        for (int c = 0; c < NP; c++) piece[c * 128 + n] = v[c];
        epi_bar();   // every row of the piece is written (released by the ticket below)
        if (et == 0) {
          const int c_first = cta_of_unit(T, gridDim.x, tb), c_last = cta_of_unit(T, gridDim.x, te - 1);
          const int prev = atom_add_acq_rel_gpu(&pa.tickets[mt], 1);
          const bool last = prev == c_last - c_first;
          if (last) pa.tickets[mt] = 0;
          *flag = last ? c_first * 2 + 1 : 0;   // odd: this CTA finishes the tile; c_first recovered
        }
        epi_bar();
        const int f = *flag;
        if (f) {
          // sum the pieces in CTA order: CTA c's piece of this tile is its first segment when its
          // range starts inside the tile, else its last
          __threadfence();
          const int c_first = f >> 1, c_last = cta_of_unit(T, gridDim.x, te - 1);
          float acc[NP];
#pragma unroll
          for (int c = 0; c < NP; c++) acc[c] = 0.f;
          for (int cc = c_first; cc <= c_last; cc++) {
            const int sl2 = range_start(T, gridDim.x, cc) >= tb ? 0 : 1;
            const float* pp = pa.partials + ((size_t)cc * 2 + sl2) * NP * 128;
#pragma unroll
            for (int c = 0; c < NP; c++) acc[c] += __ldcg(pp + c * 128 + n);
          }
#pragma unroll
          for (int c = 0; c < NP; c += 4)
            *reinterpret_cast<float4*>(&tile[n * NP + c]) = make_float4(acc[c], acc[c + 1], acc[c + 2], acc[c + 3]);
          run_tile(mt);
        }
      }
      u = su1;
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc05_fence_after();
    tmem_dealloc(tmem, (uint32_t)pa.tmem_cols);
  }
}

template <int EPI>
cudaError_t launch_proj_epi(int nt, int np, const ProjArgs& pa, int grid, size_t smem, cudaStream_t s) {
#define DFL_PJ(NTV, NPV)                                                                            \
  if (nt == NTV && np == NPV) {                                                                     \
    static std::atomic<int> smem_set[kMaxDevices];                                                  \
    const cudaError_t e = ensure_smem_limit(proj_tc05_kernel<EPI, NTV, NPV>, smem, smem_set);       \
    if (e != cudaSuccess) return e;                                                                 \
    return launch_pdl(proj_tc05_kernel<EPI, NTV, NPV>, dim3(grid), dim3(kPjThreads), smem, s, pa); \
  }
  DFL_PJ(1, 16)
  DFL_PJ(2, 16)
  DFL_PJ(1, 32)
  DFL_PJ(2, 32)
  DFL_PJ(4, 32)
#undef DFL_PJ
  return cudaErrorInvalidValue;
}

}  // namespace

ProjPlan plan_proj_tc05(int n_strips, int groups, int rows, int x_lo, int n_sm) {
  ProjPlan p{};
  if (n_strips < 1 || groups < 1 || rows < 1 || rows > kProjMaxRows || n_sm < 1) return p;
  p.npad = rows <= 16 ? 16 : 32;
  p.mtiles = (n_strips + kPjStrips - 1) / kPjStrips;
  const long long T = (long long)p.mtiles * groups;
  p.grid = (int)std::min<long long>(n_sm, T);
  p.x_stage = (uint32_t)p.npad * 128u * (x_lo ? 2u : 1u);
  p.sa = 4;                                // dequantised A stages
  p.sx = 0;
  p.tmem_cols = 2 * kPjChains * p.npad;    // two segments in flight, kPjChains accumulators each
  const size_t fixed = 1024 /* alignment slack */ + (size_t)p.sa * kPjAStage + (size_t)128 * p.npad * 4 +
                       kMaxRows * 4 + (size_t)(2 * p.sa + 4) * 8 + 16;
  const size_t per_stage = kPjWStage + (size_t)kPjKG * p.x_stage + 16;   // a raw stage and its two barriers
  const size_t room = kTcSmemMax > fixed ? kTcSmemMax - fixed : 0;
  p.sw = (int)std::min<size_t>(8, room / per_stage);
  if (p.sw < 2) return ProjPlan{};
  p.smem = fixed + (size_t)p.sw * per_stage;
  p.partial_floats = (size_t)p.grid * 2 * p.npad * 128;
  return p;
}

cudaError_t launch_proj_tc05(int epi, int nt, const ProjArgs& pa, const ProjPlan& p, cudaStream_t s) {
  switch (epi) {
    case EPI_QKV: return launch_proj_epi<EPI_QKV>(nt, p.npad, pa, p.grid, p.smem, s);
    case EPI_RESID: return launch_proj_epi<EPI_RESID>(nt, p.npad, pa, p.grid, p.smem, s);
    case EPI_SWIGLU: return launch_proj_epi<EPI_SWIGLU>(nt, p.npad, pa, p.grid, p.smem, s);
    case EPI_LMHEAD: return launch_proj_epi<EPI_LMHEAD>(nt, p.npad, pa, p.grid, p.smem, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace dfl

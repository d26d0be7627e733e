// Many-row contraction Y[r][n] = sum_k X[r][k] W[n][k] over a stored 4-bit drafter matrix on the
// fifth-generation tensor cores (tcgen05), for batches of activation rows (up to 160) where the
// skinny mma.sync GEMV runs into the legacy tensor path's ceiling.
//
// One CTA per (group of up to kTcTiles 128-row output tiles, K slice), eleven warps. The tiles of a
// CTA share every activation tile: it is loaded once per 64-input group for all of them, which
// divides the activation traffic from L2 and the number of activation loads in flight by the
// tile count.
//  * warp 0 streams the CTA's 4-bit (strip, group) tiles, kTcKW 64-input groups of all its tiles
//    per tensor copy, and keeps the following ones coming into L2 with tensor prefetches; warp 10
//    streams the activation rows (f16, plus the f16 remainder where given), one or two groups per
//    tensor copy in the 128-byte swizzle (4-D maps: a grouped launch's layer is the outer
//    coordinate, grid.y);
//  * warps 2-9 (strip w of every tile) dequantise the codes to f16 weights, w = s q + b with one
//    rounding (the code q is made exact in f16 from its nibble with a magic-number lop3 and one
//    exact subtraction, then one fused f16 multiply-add with the row's scale and bias), and store
//    them as the MMAs' K-major A tiles in the same swizzle (the stored word order of a lane covers
//    whole 16-byte chunks of a row);
//  * warp 1 allocates tensor memory and, converged, issues tcgen05.mma kind::f16 through one
//    elected lane (M = 128 output rows, N = the activation rows padded to 16, K = 16), one fp32
//    accumulator per tile over the whole K slice, then commits to the stages' mbarriers;
//  * warps 4-7 (tensor-memory lane quarters 0-3) finally read the accumulators and store the
//    slice's partial tiles, strip-major ([slice][strip][row][16]).
// The copy and MMA warps run their loops with all 32 lanes (one lane issues): a lone lane whose
// warp-mates wait at a block barrier is scheduled far too rarely for an issue loop. Every mbarrier
// wait is bounded (error word + early exit); tensor memory is freed at the end. The K slices'
// partial tiles are summed in slice order by the reduction kernel below (dflash_rows_matmul) or by
// the draft round's epilogues (tc05_epi.cu). The launch shape (tiles per CTA, K slices, ring
// depths) comes from plan_tc05's cost model.
#include <cuda.h>

#include <algorithm>
#include <array>
#include <map>
#include <mutex>
#include <vector>
#include <cuda_fp16.h>

#include "common.cuh"
#include "gemm_tc05.h"
#include "tc05.cuh"

namespace dfl {

namespace {

constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcStrips = 8;                                      // 16-row strips per 128-row tile
constexpr int kTcTileW = kTcStrips * kQ4GroupBytes;               // 4608 B: one group of one tile, raw
constexpr int kTcTileA = 128 * 128;                               // 16 KB: one group of one tile, f16

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 bits_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// (c + q0, c + q1) -> s * (q0, q1) + b in f16 with one rounding; q exact after the subtraction
__device__ __forceinline__ uint32_t dequant2(uint32_t v, __half2 c, __half2 s, __half2 b) {
  return h2_bits(__hfma2(__hsub2(bits_h2(v), c), s, b));
}

// Ring position: stage index and the parity of its current fill.
struct RingPos {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int n) {
    if (++stage == n) {
      stage = 0;
      phase ^= 1u;
    }
  }
};

template <bool LO>
__global__ void __launch_bounds__(kTcThreads, 1) tc05_q4_kernel(const __grid_constant__ Tc05Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int cb = a.tiles_big;                                   // tiles of the largest CTA: ring strides
  const uint32_t a_stage = (uint32_t)cb * kTcTileA, w_stage = (uint32_t)(kTcKW * cb * kTcTileW);
  uint8_t* aring = sm;                                          // a.sa x a_stage (1024-aligned)
  uint8_t* xring = aring + (size_t)a.sa * a_stage;              // a.sx x a.x_stage (1024-aligned)
  uint8_t* wring = xring + (size_t)a.sx * a.x_stage;            // a.sw x w_stage
  uint64_t* bars = reinterpret_cast<uint64_t*>(wring + (size_t)a.sw * w_stage);
  uint64_t* full_w = bars;
  uint64_t* empty_w = full_w + kTcMaxSW;
  uint64_t* full_x = empty_w + kTcMaxSW;
  uint64_t* empty_x = full_x + kTcMaxSX;
  uint64_t* full_a = empty_x + kTcMaxSX;
  uint64_t* empty_a = full_a + kTcMaxSA;
  uint64_t* acc_done = empty_a + kTcMaxSA;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // CTA -> (tile group, K slice); the first a.groups_big tile groups hold tiles_big tiles, the
  // rest tiles_small (the last one possibly fewer)
  const int tg = blockIdx.x % a.tgroups, slice = blockIdx.x / a.tgroups;
  const int layer = blockIdx.y;   // grouped launches: one problem (layer) per grid row
  const int mt0 = tg < a.groups_big ? tg * cb : a.groups_big * cb + (tg - a.groups_big) * a.tiles_small;
  const int n_tiles = min(tg < a.groups_big ? cb : a.tiles_small, a.mtiles - mt0);
  const int g0 = slice * a.gps, ng = min(a.groups, g0 + a.gps) - g0;
  // copies: raw weights kTcKW groups at a time (W step), activations a.kx groups at a time (x step)
  const int kx = a.kx;
  const int nsw = (ng + kTcKW - 1) / kTcKW, nsx = (ng + kx - 1) / kx;

  if (threadIdx.x == 0) {
    for (int i = 0; i < a.sw; i++) {
      mbar_init(smem_u32(&full_w[i]), 1);
      mbar_init(smem_u32(&empty_w[i]), kTcStrips);   // the eight decoder warps
    }
    for (int i = 0; i < a.sx; i++) {
      mbar_init(smem_u32(&full_x[i]), 1);
      mbar_init(smem_u32(&empty_x[i]), 1);            // the MMA commit
    }
    for (int i = 0; i < a.sa; i++) {
      mbar_init(smem_u32(&full_a[i]), kTcStrips);     // the eight decoder warps
      mbar_init(smem_u32(&empty_a[i]), 1);            // the MMA commit
    }
    mbar_init(smem_u32(acc_done), 1);                 // the last MMA commit
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), (uint32_t)a.tmem_cols);
    tmem_relinquish();
  }
  tc05_fence_before();
  __syncthreads();
  tc05_fence_after();
  const uint32_t tmem = *tmem_slot;

  // Launched with programmatic dependent launch: the next kernel may start its prologue now, and
  // this one may have started while the previous kernel drained. Nothing earlier kernels wrote
  // (activation rows, the partial-tile scratch an earlier epilogue reads) is touched before
  // pdl_wait(); the constant weights of the first stages are requested before it.
  pdl_launch_dependents();
  if (warp == 0) {
    // ---- copies: raw 4-bit tiles -------------------------------------------------------------------
    if (ng > 0) {
      // One tensor copy per W step: kTcKW groups of the 8 strips of each of the CTA's tiles (a box
      // as tall as the CTA's tile count; strips and groups past the matrix read as zero, and a
      // short last CTA reads only strips past the matrix beyond its own). Few large copies: each
      // copy has a fixed cost of its own in the copy engine, whatever its size.
      const bool big = tg < a.groups_big;
      const CUtensorMap* wm = big ? &a.wmap : &a.wmap_small;
      const uint32_t w_bytes = (uint32_t)(kTcKW * (big ? cb : a.tiles_small) * kTcTileW);   // whole box
      auto issue_w = [&](int j, int stage) {
        if (lane == 0) {
          in_bounds(mt0 < a.mtiles && g0 + j * kTcKW < a.groups, a.err);
          const uint32_t fw = smem_u32(&full_w[stage]);
          mbar_arrive_expect_tx(fw, w_bytes);
          tma_load_4d(smem_u32(wring + stage * w_stage), wm, 0, g0 + j * kTcKW, a.w_strip0 + mt0 * kTcStrips, layer,
                      fw);
        }
        __syncwarp();
      };
      const int pre = min(a.sw, nsw);
      for (int j = 0; j < pre; j++) issue_w(j, j);
      // and the next a.pf steps into L2, so that the ring's copies find them there: the ring alone
      // holds too few bytes per SM to cover HBM latency under a full stream
      int npf = pre;
      auto prefetch_next = [&]() {
        if (lane == 0 && npf < nsw) tma_prefetch_4d(wm, 0, g0 + npf * kTcKW, a.w_strip0 + mt0 * kTcStrips, layer);
        npf++;
      };
      while (npf < min(nsw, pre + a.pf)) prefetch_next();
      pdl_wait();
      bool ok = true;
      RingPos pw;
      for (int j = 0; j < pre; j++) pw.next(a.sw);
      int nw = pre;   // fills issued
      for (int j = pre; j < nsw && ok; j++) {
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&empty_w[pw.stage]), pw.phase ^ 1u, a.err,
                                                       kErrTimeoutTc05));
        if (!ok) break;
        issue_w(j, pw.stage);
        nw = j + 1;
        prefetch_next();
        pw.next(a.sw);
      }
      // leave no copy in flight into this CTA's shared memory, also when a consumer gave up:
      // the last fill of every stage has completed (earlier fills of a stage completed before
      // its refill was issued); after a normal run these waits return at once
      for (int j = nw > a.sw ? nw - a.sw : 0; j < nw; j++)
        mbar_wait_bounded(smem_u32(&full_w[j % a.sw]), (j / a.sw) & 1, nullptr, 0);
    } else {
      pdl_wait();
    }
  } else if (warp == kTcWarps - 1) {
    // ---- copies: activation tiles (a warp of their own, so that neither stream waits on the
    // other's free stages) ------------------------------------------------------------------------
    pdl_wait();
    if (ng > 0) {
      bool ok = true;
      RingPos px;
      int nx = 0;   // fills issued
      for (int k = 0; k < nsx && ok; k++) {
        if (k >= a.sx)
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&empty_x[px.stage]), px.phase ^ 1u, a.err,
                                                         kErrTimeoutTc05));
        if (!ok) break;
        if (lane == 0) {
          const uint32_t fx = smem_u32(&full_x[px.stage]);
          uint8_t* xst = xring + (size_t)px.stage * a.x_stage;
          mbar_arrive_expect_tx(fx, a.x_tx);
          tma_load_4d(smem_u32(xst), &a.xmap, 0, 0, g0 + k * kx, layer, fx);
          if (LO) tma_load_4d(smem_u32(xst + kx * a.npad * 128), &a.xlmap, 0, 0, g0 + k * kx, layer, fx);
        }
        __syncwarp();
        nx = k + 1;
        px.next(a.sx);
      }
      for (int j = nx > a.sx ? nx - a.sx : 0; j < nx; j++)
        mbar_wait_bounded(smem_u32(&full_x[j % a.sx]), (j / a.sx) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    pdl_wait();
    // ---- MMA issue: accumulator t (tensor-memory columns t * npad ...) for tile t ----------------
    // The whole warp runs the loop; one elected lane issues each MMA and commit. Descriptors are
    // the rings' base descriptors plus start-address offsets (16-byte units in the low field;
    // shared-memory addresses stay below 2^18, so the field never carries).
    if (ng > 0) {
      const uint32_t idesc = umma_idesc_f16_f32(128, a.npad);
      const uint64_t a_base = umma_desc_sw128(smem_u32(aring)), x_base = umma_desc_sw128(smem_u32(xring));
      const uint32_t a_step = a_stage >> 4, x_step = a.x_stage >> 4, x_tile = (uint32_t)a.npad * 8u;
      const uint32_t lo_off = (uint32_t)kx * x_tile;   // the remainder rows follow the kx tiles
      bool ok = true;
      RingPos pa, px;
      int issued = 0;
      for (int i = 0; i < ng && ok; i++) {
        const int kxi = i % kx;   // group within the x step
        const bool x_last = kxi == kx - 1 || i + 1 == ng;
        ok = __all_sync(0xffffffffu,
                        mbar_wait_bounded(smem_u32(&full_a[pa.stage]), pa.phase, a.err, kErrTimeoutTc05) &&
                            mbar_wait_bounded(smem_u32(&full_x[px.stage]), px.phase, a.err, kErrTimeoutTc05));
        if (!ok) break;
        tc05_fence_after();
        const uint64_t ad = a_base + (uint64_t)(pa.stage * a_step);
        const uint64_t xd = x_base + (uint64_t)(px.stage * x_step + kxi * x_tile);
#pragma unroll
        for (int t = 0; t < kTcTiles; t++) {
          if (t < n_tiles) {
            const uint32_t d = tmem + (uint32_t)(t * a.npad);
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
              const uint64_t adk = ad + (uint64_t)(t * (kTcTileA >> 4) + 2 * kk);
              umma_f16_ss_warp(d, adk, xd + (uint64_t)(2 * kk), idesc, (i > 0 || kk > 0) ? 1u : 0u);
              if (LO) umma_f16_ss_warp(d, adk, xd + (uint64_t)(lo_off + 2 * kk), idesc, 1u);
            }
          }
        }
        umma_commit_warp(smem_u32(&empty_a[pa.stage]));
        if (x_last) umma_commit_warp(smem_u32(&empty_x[px.stage]));
        if (i + 1 == ng) umma_commit_warp(smem_u32(acc_done));
        issued = i + 1;
        pa.next(a.sa);
        if (x_last) px.next(a.sx);
      }
      // nothing of this CTA may still be running on the tensor core when its memory is freed
      if (issued > 0) mbar_wait_bounded(smem_u32(&empty_a[(issued - 1) % a.sa]), ((issued - 1) / a.sa) & 1, a.err,
                                        kErrTimeoutTc05);
    }
  } else {
    pdl_wait();
    // ---- dequantise: 4-bit codes -> f16 weights, swizzled K-major A tiles -------------------------
    // Warp s (0-7) takes strip s of every tile. All of a group's words are read first, then
    // converted and stored, so the tiles' shared-memory latencies overlap.
    const int s = warp - 2, g8 = lane >> 2, t4 = lane & 3;
    const __half2 c1024 = __float2half2_rn(1024.f), c64 = __float2half2_rn(64.f);
    bool ok = true;
    RingPos pw, pa;
    for (int i = 0; i < ng && ok; i++) {
      const int kwi = i % kTcKW;   // group within the W step
      const bool w_last = kwi == kTcKW - 1 || i + 1 == ng;
      ok = mbar_wait_bounded(smem_u32(&full_w[pw.stage]), pw.phase, a.err, kErrTimeoutTc05) &&
           (i < a.sa || mbar_wait_bounded(smem_u32(&empty_a[pa.stage]), pa.phase ^ 1u, a.err, kErrTimeoutTc05));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      uint4 W[kTcTiles];
      uint32_t sbg[kTcTiles], sb8[kTcTiles];
#pragma unroll
      for (int t = 0; t < kTcTiles; t++) {
        if (t < n_tiles) {
          const uint8_t* gp = wring + pw.stage * w_stage + ((t * kTcStrips + s) * kTcKW + kwi) * kQ4GroupBytes;
          W[t] = *reinterpret_cast<const uint4*>(gp + lane * 16);
          sbg[t] = *reinterpret_cast<const uint32_t*>(gp + 512 + 4 * g8);
          sb8[t] = *reinterpret_cast<const uint32_t*>(gp + 512 + 4 * (g8 + 8));
        }
      }
#pragma unroll
      for (int t = 0; t < kTcTiles; t++) {
        if (t < n_tiles) {
          const uint32_t ast = smem_u32(aring + pa.stage * a_stage + t * kTcTileA);
          const __half2 sg = __float2half2_rn(__uint_as_float(sbg[t] << 16));
          const __half2 bg = __float2half2_rn(__uint_as_float(sbg[t] & 0xFFFF0000u));
          const __half2 s8 = __float2half2_rn(__uint_as_float(sb8[t] << 16));
          const __half2 b8 = __float2half2_rn(__uint_as_float(sb8[t] & 0xFFFF0000u));
          const uint32_t w4[4] = {W[t].x, W[t].y, W[t].z, W[t].w};
          uint32_t rg[4][2], r8[4][2];
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
          // 16-byte chunk c of row r lives at r * 128 + ((c ^ (r % 8)) * 16); r % 8 == g here
          const uint32_t row_g = ast + (uint32_t)(s * 16 + g8) * 128, row_8 = row_g + 8 * 128;
          const uint32_t c0 = (uint32_t)(((2 * t4) ^ g8) << 4), c1 = (uint32_t)(((2 * t4 + 1) ^ g8) << 4);
          st_shared_v4(row_g + c0, rg[0][0], rg[0][1], rg[1][0], rg[1][1]);
          st_shared_v4(row_g + c1, rg[2][0], rg[2][1], rg[3][0], rg[3][1]);
          st_shared_v4(row_8 + c0, r8[0][0], r8[0][1], r8[1][0], r8[1][1]);
          st_shared_v4(row_8 + c1, r8[2][0], r8[2][1], r8[3][0], r8[3][1]);
        }
      }
      // the generic-proxy stores are read by the tensor core, and the raw stage is refilled by the
      // copy engine (both async proxy)
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&full_a[pa.stage]));
        if (w_last) mbar_arrive(smem_u32(&empty_w[pw.stage]));
      }
      if (w_last) pw.next(a.sw);
      pa.next(a.sa);
    }
    if (warp >= 4 && warp < 8 && ok && ng > 0) {
      // ---- the slice's partial tiles: tensor memory -> part[slice][strip][column][16] -----------
      // (a strip's 16 outputs of one activation row are 64 contiguous bytes, and a strip's rows
      // follow each other: the epilogues read whole strips)
      const int quarter = warp & 3, n = quarter * 32 + lane;   // tile row = tensor-memory lane
      ok = mbar_wait_bounded(smem_u32(acc_done), 0, a.err, kErrTimeoutTc05);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc05_fence_after();
        const size_t strips_pad = (size_t)a.n_out_pad / 16;
        for (int t = 0; t < n_tiles; t++) {
          const size_t strip = (size_t)(mt0 + t) * kTcStrips + n / 16;
          float* out = a.part + (size_t)layer * a.part_layer_stride + ((size_t)slice * strips_pad + strip) * a.npad * 16 +
                       (n & 15);
          const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(t * a.npad);
          for (int ch = 0; ch < a.npad / 16; ch++) {
            float v[16];
            tmem_ld16(tb + (uint32_t)(ch * 16), v);
#pragma unroll
            for (int e = 0; e < 16; e++) out[(size_t)(ch * 16 + e) * 16] = v[e];
          }
        }
        tc05_fence_before();
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc05_fence_after();
    tmem_dealloc(tmem, (uint32_t)a.tmem_cols);
  }
}

// Y[r][n] = sum over slices, in slice order, of the partial tiles; n in the matrix's natural row
// order (gate/up: the stored strips interleave 8 gate rows and 8 up rows, `half` gate rows).
__global__ void __launch_bounds__(256) tc05_reduce_kernel(const float* __restrict__ part, int slices, int npad,
                                                          int n_out_pad, int rows, int n_out, int half, float* y,
                                                          int ldy) {
  const long long total = (long long)rows * n_out;
  for (long long idx = blockIdx.x * (long long)blockDim.x + threadIdx.x; idx < total;
       idx += (long long)gridDim.x * blockDim.x) {
    const int r = (int)(idx / n_out), nn = (int)(idx - (long long)r * n_out);
    int p = nn;
    if (half > 0) p = nn < half ? 16 * (nn / 8) + nn % 8 : 16 * ((nn - half) / 8) + 8 + (nn - half) % 8;
    float acc = 0.f;
    const size_t strips_pad = (size_t)n_out_pad / 16;
    for (int s = 0; s < slices; s++) acc += part[(((size_t)s * strips_pad + p / 16) * npad + r) * 16 + p % 16];
    y[(size_t)r * ldy + nn] = acc;
  }
}

// Caller-side bf16 rows (context taps) -> f16, as the skinny GEMV stages them (round to
// nearest, clamped to the f16 range). n_pairs element pairs.
__global__ void __launch_bounds__(256) tc05_bf16_to_f16_kernel(const uint32_t* __restrict__ src, long long n_pairs,
                                                               uint32_t* __restrict__ dst) {
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n_pairs;
       i += (long long)gridDim.x * blockDim.x) {
    const uint32_t u = src[i];
    const float lo = __uint_as_float(u << 16), hi = __uint_as_float(u & 0xFFFF0000u);
    dst[i] = pack_f16x2(fminf(fmaxf(lo, -kF16Max), kF16Max), fminf(fmaxf(hi, -kF16Max), kF16Max));
  }
}

}  // namespace

cudaError_t launch_bf16_to_f16(const void* src, long long n_elems, void* dst, cudaStream_t s) {
  const long long pairs = n_elems / 2;
  const int blocks = (int)std::min<long long>(4096, (pairs + 255) / 256);
  if (blocks < 1) return cudaSuccess;
  tc05_bf16_to_f16_kernel<<<blocks, 256, 0, s>>>(static_cast<const uint32_t*>(src), pairs,
                                                  static_cast<uint32_t*>(dst));
  return cudaGetLastError();
}

namespace {

// Shared memory of a CTA with cb tiles, sa f16 stages, sw raw stages (kTcKW groups each) and sx
// activation stages.
size_t tc05_smem(int cb, int sa, int sw, int sx, uint32_t x_stage) {
  return 1024 /* alignment slack */ + (size_t)sa * cb * kTcTileA + (size_t)sw * kTcKW * cb * kTcTileW +
         (size_t)sx * x_stage + (size_t)(2 * kTcMaxSW + 2 * kTcMaxSX + 2 * kTcMaxSA + 1) * 8 + 16;
}

// Ring depths of a CTA with cb tiles: as many f16 stages as fit in ~96 KB (the dequantisation of
// group i + sa can only start when the MMAs of group i have completed, so the stage count divides
// that round trip); activation copies of two groups where three or more groups then fit, else of
// one; the rest of shared memory as raw stages (kTcKW groups each, at least two: with the L2
// prefetch they cover HBM latency).
struct Depths {
  int sa = 0, sw = 0, sx = 0, kx = 0;
  uint32_t x_stage = 0;
};

Depths pick_depths(int cb, int npad, int x_lo) {
  const int sa_max = std::max(2, std::min(kTcMaxSA, 6 / cb));
  const size_t w_stage = (size_t)kTcKW * cb * kTcTileW;
  for (int sa = sa_max; sa >= 2; sa--)
    for (int kx = 2; kx >= 1; kx--) {
      const uint32_t xs = (uint32_t)(kx * npad * 128 * (x_lo ? 2 : 1));
      for (int sx = kTcMaxSX; sx >= 2; sx--) {
        if (kx * sx < 3) continue;
        const size_t base = tc05_smem(cb, sa, 0, sx, xs);
        if (base >= kTcSmemMax) continue;
        const int sw = (int)std::min<size_t>(kTcMaxSW, (kTcSmemMax - base) / w_stage);
        if (sw >= 2) return Depths{sa, sw, sx, kx, xs};
      }
    }
  const uint32_t xs = (uint32_t)(npad * 128 * (x_lo ? 2 : 1));   // large tiles and rows: whatever fits
  const size_t base = tc05_smem(cb, 2, 0, 2, xs);
  if (base < kTcSmemMax && (kTcSmemMax - base) / w_stage >= 1)
    return Depths{2, (int)std::min<size_t>(kTcMaxSW, (kTcSmemMax - base) / w_stage), 2, 1, xs};
  return Depths{};
}

// Cost model of one launch, in SM cycles, for choosing a plan (constants measured on this kernel
// with per-CTA clock stamps). Per 64-input group, a CTA with nt tiles takes the largest of: the
// dequantisation (~290 cycles per tile), the MMAs' issue (~50 + 0.19 N cycles per M = 128, K = 16
// instruction), the round trip dequantise -> MMA -> completion -> next dequantisation into the
// same stage divided by the f16 stages, the tiles' share of HBM and the activation tile's share of
// L2 bandwidth; plus ~150 cycles of waits. Per CTA: ~7000 cycles of start-up and pipeline fill
// and the store of its partial tiles; per extra K slice the partial tiles written and read once
// more. CTAs are dispatched in index order to the SM that frees first (one CTA per SM fits).
struct CostModel {
  double dq, mma, chain, hbm_tile, l2_x, copies, per_group, per_cta, per_tile_out, hbm_bytes_per_cycle;
  int sa;
};

CostModel cost_model(int npad, int x_lo, int n_sm, const Depths& dp) {
  CostModel c{};
  const int sa = dp.sa;
  const uint32_t x_stage = dp.x_stage / dp.kx;   // per group
  const double hbm = 6.6e12 / 2.07e9;   // bytes per SM cycle, whole GPU
  const double l2 = 12e12 / 2.07e9;
  c.dq = 290.0;
  c.mma = 4.0 * (x_lo ? 2.0 : 1.0) * (50.0 + 0.19 * npad);
  c.chain = 1100.0;
  c.hbm_tile = kTcTileW / (hbm / n_sm);
  c.l2_x = x_stage / (l2 / n_sm);
  c.copies = 540.0 * (1.0 / kTcKW + (x_lo ? 2.0 : 1.0) / dp.kx);   // the copy engine's fixed cost per copy
  c.per_group = 150.0;
  c.per_cta = 7000.0;
  c.per_tile_out = 16.0 * npad;
  c.hbm_bytes_per_cycle = hbm;
  c.sa = sa;
  return c;
}

double group_cycles(const CostModel& c, int nt) {
  const double d = c.dq * nt, m = c.mma * nt;
  return c.per_group + std::max({d, m, (d + m + c.chain) / c.sa, c.hbm_tile * nt, c.l2_x, c.copies});
}

double makespan(const CostModel& c, int n_sm, int mtiles, int cb, int nb, int cs, int groups, int gps) {
  const int slices = (groups + gps - 1) / gps;
  const int rest = mtiles - nb * cb;
  const int tgroups = nb + (rest > 0 ? (rest + cs - 1) / cs : 0);
  std::vector<double> sm(n_sm, 0.0);   // a binary heap of SM free times
  auto cmp = [](double x, double y) { return x > y; };
  double end = 0.0;
  for (int b = 0; b < tgroups * slices; b++) {
    const int tg = b % tgroups, sl = b / tgroups;
    const int mt0 = tg < nb ? tg * cb : nb * cb + (tg - nb) * cs;
    const int nt = std::min(tg < nb ? cb : cs, mtiles - mt0);
    const int ng = std::min(groups, (sl + 1) * gps) - sl * gps;
    const double cost = c.per_cta + ng * group_cycles(c, nt) + nt * c.per_tile_out;
    std::pop_heap(sm.begin(), sm.end(), cmp);
    sm.back() += cost;
    end = std::max(end, sm.back());
    std::push_heap(sm.begin(), sm.end(), cmp);
  }
  return end;
}

}  // namespace

Tc05Plan plan_tc05_uncached(int n_strips, int groups, int npad, int x_lo, int n_sm) {
  Tc05Plan p{};
  const int mtiles = (n_strips + kTcStrips - 1) / kTcStrips;
  // Candidates: every CTA with c tiles (c = 3, 2, 1) and s K slices (each >= 4 groups long), or,
  // with one slice, k x n_sm CTAs of three tiles followed by CTAs of two.
  struct Cand {
    int cb, nb, cs, gps;
    double t;
  } best{0, 0, 0, 0, 0.0};
  auto consider = [&](int cb, int nb, int cs, int gps) {
    const Depths dp = pick_depths(cb, npad, x_lo);
    if (dp.sa == 0) return;
    const CostModel cm = cost_model(npad, x_lo, n_sm, dp);
    double t = makespan(cm, n_sm, mtiles, cb, nb, cs, groups, gps);
    const int slices = (groups + gps - 1) / gps;
    t += (slices - 1) * (double)npad * mtiles * 128 * 8.0 / cm.hbm_bytes_per_cycle;   // partials re-read
    if (best.cb == 0 || t < best.t * 0.99) best = Cand{cb, nb, cs, gps, t};
  };
  for (int c = kTcTiles; c >= 1; c--) {
    if (c * npad > 512 || (c > 1 && c > mtiles)) continue;   // accumulators must fit tensor memory
    const int tg = (mtiles + c - 1) / c;
    for (int s = 1; s <= std::max(1, std::min(groups / 4, 64)); s++) {
      const int gps = (groups + s - 1) / s;
      if (s > 1 && (groups + gps - 1) / gps != s) continue;   // same slicing as a smaller s
      if (s > 1 && (long long)tg * s > n_sm) break;   // a K split fills at most one wave of CTAs
      consider(c, tg, c, gps);
    }
  }
  if (kTcTiles * npad <= 512)
    for (int k = 1; (long long)k * n_sm * kTcTiles < mtiles; k++) consider(kTcTiles, k * n_sm, 2, groups);
  if (best.cb == 0) return p;
  p.npad = npad;
  p.mtiles = mtiles;
  p.tiles_big = best.cb;
  p.groups_big = best.nb;
  p.tiles_small = best.cs;
  p.gps = best.gps;
  p.slices = (groups + p.gps - 1) / p.gps;
  const int rest = mtiles - p.groups_big * p.tiles_big;
  p.tgroups = p.groups_big + (rest > 0 ? (rest + p.tiles_small - 1) / p.tiles_small : 0);
  p.grid = p.tgroups * p.slices;
  const Depths dp = pick_depths(p.tiles_big, npad, x_lo);
  p.x_stage = dp.x_stage;   // a multiple of 2048 B
  p.x_tx = p.x_stage;
  p.sa = dp.sa;
  p.sw = dp.sw;
  p.sx = dp.sx;
  p.kx = dp.kx;
  // L2 prefetch distance: about kTcBytesInFlight of weights per SM requested ahead, ring included
  if (p.sw == 0) return Tc05Plan{};
  p.smem = tc05_smem(p.tiles_big, p.sa, p.sw, p.sx, p.x_stage);
  const int in_flight = (int)(kTcBytesInFlight / ((size_t)kTcKW * p.tiles_big * kTcTileW));   // W steps
  p.pf = std::max(0, in_flight - p.sw);
  int cols = 32;
  while (cols < p.tiles_big * npad) cols *= 2;
  p.tmem_cols = cols;
  p.part_off = 0;
  p.srow_off = (size_t)p.slices * npad * mtiles * 128 * 4;
  p.scratch = p.srow_off + (size_t)kTcMaxChunks * kMaxRows * 4;
  return p;
}

// Plans depend on the activation rows only through npad; a launch asks for one per projection, so
// they are kept (a few dozen shapes per drafter).
Tc05Plan plan_tc05(int n_strips, int groups, int rows, int x_lo, int n_sm) {
  if (n_strips < 1 || groups < 1 || rows < 1 || rows > kTcMaxRows || n_sm < 1) return Tc05Plan{};
  const int npad = (rows + 15) / 16 * 16;
  static std::mutex mu;
  static std::map<std::array<int, 5>, Tc05Plan> cache;
  const std::array<int, 5> key{n_strips, groups, npad, x_lo ? 1 : 0, n_sm};
  {
    std::lock_guard<std::mutex> lock(mu);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  const Tc05Plan p = plan_tc05_uncached(n_strips, groups, npad, x_lo, n_sm);
  std::lock_guard<std::mutex> lock(mu);
  if (cache.size() < 4096) cache.emplace(key, p);
  return p;
}

void tc05_fill_args(const Tc05Plan& p, int has_lo, Tc05Args& a) {
  a.npad = p.npad;
  a.gps = p.gps;
  a.mtiles = p.mtiles;
  a.tgroups = p.tgroups;
  a.tiles_big = p.tiles_big;
  a.groups_big = p.groups_big;
  a.tiles_small = p.tiles_small;
  a.has_lo = has_lo;
  a.n_out_pad = p.mtiles * 128;
  a.sx = p.sx;
  a.sw = p.sw;
  a.sa = p.sa;
  a.pf = p.pf;
  a.kx = p.kx;
  if (a.n_layers < 1) a.n_layers = 1;
  a.tmem_cols = p.tmem_cols;
  a.x_stage = p.x_stage;
  a.x_tx = p.x_tx;
}

cudaError_t launch_tc05_parts(const Tc05Args& a, const Tc05Plan& p, cudaStream_t s) {
  static std::atomic<int> smem_set[2][kMaxDevices];
  cudaError_t e;
  if (a.has_lo) {
    e = ensure_smem_limit(tc05_q4_kernel<true>, p.smem, smem_set[1]);
    if (e != cudaSuccess) return e;
    return launch_pdl(tc05_q4_kernel<true>, dim3(p.grid, a.n_layers), dim3(kTcThreads), p.smem, s, a);
  }
  e = ensure_smem_limit(tc05_q4_kernel<false>, p.smem, smem_set[0]);
  if (e != cudaSuccess) return e;
  return launch_pdl(tc05_q4_kernel<false>, dim3(p.grid, a.n_layers), dim3(kTcThreads), p.smem, s, a);
}

cudaError_t launch_tc05(const Tc05Args& a, const Tc05Plan& p, int rows, int n_out, int half, float* y, int ldy,
                        cudaStream_t s) {
  const cudaError_t e = launch_tc05_parts(a, p, s);
  if (e != cudaSuccess) return e;
  const long long total = (long long)rows * n_out;
  const int blocks = (int)std::min<long long>(4096, (total + 255) / 256);
  tc05_reduce_kernel<<<blocks, 256, 0, s>>>(a.part, p.slices, p.npad, a.n_out_pad, rows, n_out, half, y, ldy);
  return cudaGetLastError();
}

}  // namespace dfl

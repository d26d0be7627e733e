// Many-row contraction Y[r][n] = sum_k X[r][k] W[n][k] over a stored 4-bit drafter matrix on the
// fifth-generation tensor cores (tcgen05), for batches of activation rows (up to 160) where the
// skinny mma.sync GEMV runs into the legacy tensor path's ceiling.
//
// One CTA per (group of up to kTcTiles 128-row output tiles, K slice), ten warps. The tiles of a
// CTA share every activation tile: it is loaded once per 64-input group for all of them, which
// divides the activation traffic from L2 and the number of activation loads in flight by the
// tile count.
//  * warp 0 streams, per 64-input group, each tile's eight 4-bit (strip, group) tiles with one 3-D
//    tensor copy, and the group's activation rows (f16, plus the f16 remainder where given) with
//    2-D tensor copies in the 128-byte swizzle;
//  * warps 2-9 (strip w of every tile) dequantise the codes to f16 weights, w = s q + b with one
//    rounding (the code q is made exact in f16 from its nibble with a magic-number lop3 and one
//    exact subtraction, then one fused f16 multiply-add with the row's scale and bias), and store
//    them as the MMAs' K-major A tiles in the same swizzle (the stored word order of a lane covers
//    whole 16-byte chunks of a row);
//  * warp 1 allocates tensor memory and one of its lanes issues tcgen05.mma kind::f16 (M = 128
//    output rows, N = the activation rows padded to 16, K = 16), one fp32 accumulator per tile
//    over the whole K slice, then commits to the stages' mbarriers;
//  * warps 4-7 (tensor-memory lane quarters 0-3) finally read the accumulators and store the
//    slice's partial tiles.
// The copy and MMA warps run their loops with all 32 lanes (one lane issues): a lone lane whose
// warp-mates wait at a block barrier is scheduled far too rarely for an issue loop. Every mbarrier
// wait is bounded (error word + early exit); tensor memory is freed at the end. The K slices'
// partial tiles are summed in slice order by a separate kernel.
#include <cuda.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "gemm_tc05.h"
#include "tc05.cuh"

namespace dfl {

namespace {

constexpr int kTcThreads = kTcWarps * 32;
constexpr int kTcStrips = 8;                                      // 16-row strips per 128-row tile
constexpr int kTcTileW = kTcStrips * kQ4GroupBytes;               // 4608 B: one group of one tile, raw
constexpr int kTcWStage = kTcTiles * kTcTileW;                    // one group of a CTA's tiles, raw
constexpr int kTcTileA = 128 * 128;                               // 16 KB: one group of one tile, f16
constexpr int kTcAStage = kTcTiles * kTcTileA;

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

__device__ __forceinline__ uint32_t h2_bits(__half2 v) { return *reinterpret_cast<uint32_t*>(&v); }
__device__ __forceinline__ __half2 bits_h2(uint32_t v) { return *reinterpret_cast<__half2*>(&v); }

// (c + q0, c + q1) -> s * (q0, q1) + b in f16 with one rounding; q exact after the subtraction
__device__ __forceinline__ uint32_t dequant2(uint32_t v, __half2 c, __half2 s, __half2 b) {
  return h2_bits(__hfma2(__hsub2(bits_h2(v), c), s, b));
}

__global__ void __launch_bounds__(kTcThreads, 1) tc05_q4_kernel(const __grid_constant__ Tc05Args a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* aring = sm;                                          // kTcSA x kTcAStage (1024-aligned)
  uint8_t* xring = aring + kTcSA * kTcAStage;                   // a.sx x a.x_stage (1024-aligned)
  uint8_t* wring = xring + (size_t)a.sx * a.x_stage;            // kTcSW x kTcWStage
  uint64_t* bars = reinterpret_cast<uint64_t*>(wring + kTcSW * kTcWStage);
  uint64_t* full_w = bars;
  uint64_t* empty_w = full_w + kTcSW;
  uint64_t* full_x = empty_w + kTcSW;
  uint64_t* empty_x = full_x + kTcMaxSX;
  uint64_t* full_a = empty_x + kTcMaxSX;
  uint64_t* empty_a = full_a + kTcSA;
  uint64_t* acc_done = empty_a + kTcSA;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_done + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tg = blockIdx.x % a.tgroups, slice = blockIdx.x / a.tgroups;
  const int mt0 = tg * kTcTiles, n_tiles = min(kTcTiles, a.mtiles - mt0);
  const int g0 = slice * a.gps, ng = min(a.groups, g0 + a.gps) - g0;
  auto strips_of = [&](int t) { return min(kTcStrips, a.n_strips - (mt0 + t) * kTcStrips); };

  if (threadIdx.x == 0) {
    for (int i = 0; i < kTcSW; i++) {
      mbar_init(smem_u32(&full_w[i]), 1);
      mbar_init(smem_u32(&empty_w[i]), kTcStrips);   // the eight decoder warps
    }
    for (int i = 0; i < a.sx; i++) {
      mbar_init(smem_u32(&full_x[i]), 1);
      mbar_init(smem_u32(&empty_x[i]), 1);            // the MMA commit
    }
    for (int i = 0; i < kTcSA; i++) {
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

  if (warp == 0) {
    // ---- copies: raw 4-bit tiles and activation tiles --------------------------------------------
    if (ng > 0) {
      const uint32_t w_bytes = (uint32_t)(n_tiles * kTcTileW);   // whole boxes, zero-filled rows included
      bool ok = true;
      int nw = 0, nx = 0;   // stages whose copies were issued
      for (int i = 0; i < ng && ok; i++) {
        const int g = g0 + i, sw = i % kTcSW, sx = i % a.sx;
        if (i >= kTcSW)
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&empty_w[sw]), ((i / kTcSW) + 1) & 1, a.err,
                                                         kErrTimeoutTc05));
        if (!ok) break;
        if (lane == 0) {
          in_bounds(mt0 < a.mtiles && g < a.groups, a.err);
          const uint32_t fw = smem_u32(&full_w[sw]);
          mbar_arrive_expect_tx(fw, w_bytes);
          // one tensor copy per tile: its 8 strips' tiles of group g (strips past the matrix: zeros)
          for (int t = 0; t < n_tiles; t++)
            tma_load_3d(smem_u32(wring + sw * kTcWStage + t * kTcTileW), &a.wmap, 0, g, (mt0 + t) * kTcStrips, fw);
        }
        __syncwarp();
        nw = i + 1;
        if (i >= a.sx)
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&empty_x[sx]), ((i / a.sx) + 1) & 1, a.err,
                                                         kErrTimeoutTc05));
        if (!ok) break;
        if (lane == 0) {
          const uint32_t fx = smem_u32(&full_x[sx]);
          uint8_t* xst = xring + (size_t)sx * a.x_stage;
          mbar_arrive_expect_tx(fx, a.x_tx);
          tma_load_2d(smem_u32(xst), &a.xmap, g * 64, 0, fx);
          if (a.has_lo) tma_load_2d(smem_u32(xst + a.npad * 128), &a.xlmap, g * 64, 0, fx);
        }
        __syncwarp();
        nx = i + 1;
      }
      // leave no copy in flight into this CTA's shared memory, also when a consumer gave up:
      // the last fill of every stage has completed (earlier fills of a stage completed before
      // its refill was issued); after a normal run these waits return at once
      for (int j = nw > kTcSW ? nw - kTcSW : 0; j < nw; j++)
        mbar_wait_bounded(smem_u32(&full_w[j % kTcSW]), (j / kTcSW) & 1, nullptr, 0);
      for (int j = nx > a.sx ? nx - a.sx : 0; j < nx; j++)
        mbar_wait_bounded(smem_u32(&full_x[j % a.sx]), (j / a.sx) & 1, nullptr, 0);
    }
  } else if (warp == 1) {
    // ---- MMA issue: accumulator t (tensor-memory columns t * npad ...) for tile t ----------------
    if (ng > 0) {
      const uint32_t idesc = umma_idesc_f16_f32(128, a.npad);
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < ng && ok; i++) {
        const int sa = i % kTcSA, sx = i % a.sx;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&full_a[sa]), (i / kTcSA) & 1, a.err, kErrTimeoutTc05) &&
                                     mbar_wait_bounded(smem_u32(&full_x[sx]), (i / a.sx) & 1, a.err, kErrTimeoutTc05));
        if (!ok) break;
        tc05_fence_after();
        if (lane == 0) {
          const uint32_t xbase = smem_u32(xring + (size_t)sx * a.x_stage);
          for (int t = 0; t < n_tiles; t++) {
            const uint32_t abase = smem_u32(aring + sa * kTcAStage + t * kTcTileA);
            const uint32_t d = tmem + (uint32_t)(t * a.npad);
#pragma unroll
            for (int kk = 0; kk < 4; kk++) {
              const uint64_t ad = umma_desc_sw128(abase + 32 * kk);
              umma_f16_ss(d, ad, umma_desc_sw128(xbase + 32 * kk), idesc, (i > 0 || kk > 0) ? 1u : 0u);
              if (a.has_lo) umma_f16_ss(d, ad, umma_desc_sw128(xbase + a.npad * 128 + 32 * kk), idesc, 1u);
            }
          }
          umma_commit(smem_u32(&empty_a[sa]));
          umma_commit(smem_u32(&empty_x[sx]));
          if (i + 1 == ng) umma_commit(smem_u32(acc_done));
        }
        __syncwarp();
        issued = i + 1;
      }
      // nothing of this CTA may still be running on the tensor core when its memory is freed
      if (issued > 0) mbar_wait_bounded(smem_u32(&empty_a[(issued - 1) % kTcSA]), ((issued - 1) / kTcSA) & 1, a.err,
                                        kErrTimeoutTc05);
    }
  } else {
    // ---- dequantise: 4-bit codes -> f16 weights, swizzled K-major A tiles -------------------------
    const int s = warp - 2, g8 = lane >> 2, t4 = lane & 3;
    const __half2 c1024 = __float2half2_rn(1024.f), c64 = __float2half2_rn(64.f);
    bool ok = true;
    for (int i = 0; i < ng && ok; i++) {
      const int sw = i % kTcSW, sa = i % kTcSA;
      ok = mbar_wait_bounded(smem_u32(&full_w[sw]), (i / kTcSW) & 1, a.err, kErrTimeoutTc05) &&
           (i < kTcSA || mbar_wait_bounded(smem_u32(&empty_a[sa]), ((i / kTcSA) + 1) & 1, a.err, kErrTimeoutTc05));
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      for (int t = 0; t < n_tiles; t++) {
        const uint8_t* gp = wring + sw * kTcWStage + (t * kTcStrips + s) * kQ4GroupBytes;
        const uint32_t ast = smem_u32(aring + sa * kTcAStage + t * kTcTileA);
        uint32_t rg[4][2], r8[4][2];
        if (s < strips_of(t)) {
          const uint4 W = *reinterpret_cast<const uint4*>(gp + lane * 16);
          const uint32_t sbg = *reinterpret_cast<const uint32_t*>(gp + 512 + 4 * g8);
          const uint32_t sb8 = *reinterpret_cast<const uint32_t*>(gp + 512 + 4 * (g8 + 8));
          const __half2 sg = __float2half2_rn(__uint_as_float(sbg << 16));
          const __half2 bg = __float2half2_rn(__uint_as_float(sbg & 0xFFFF0000u));
          const __half2 s8 = __float2half2_rn(__uint_as_float(sb8 << 16));
          const __half2 b8 = __float2half2_rn(__uint_as_float(sb8 & 0xFFFF0000u));
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
        const uint32_t c0 = (uint32_t)(((2 * t4) ^ g8) << 4), c1 = (uint32_t)(((2 * t4 + 1) ^ g8) << 4);
        st_shared_v4(row_g + c0, rg[0][0], rg[0][1], rg[1][0], rg[1][1]);
        st_shared_v4(row_g + c1, rg[2][0], rg[2][1], rg[3][0], rg[3][1]);
        st_shared_v4(row_8 + c0, r8[0][0], r8[0][1], r8[1][0], r8[1][1]);
        st_shared_v4(row_8 + c1, r8[2][0], r8[2][1], r8[3][0], r8[3][1]);
      }
      // the generic-proxy stores are read by the tensor core, and the raw stage is refilled by the
      // copy engine (both async proxy)
      fence_proxy_async();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&full_a[sa]));
        mbar_arrive(smem_u32(&empty_w[sw]));
      }
    }
    if (warp >= 4 && warp < 8 && ok && ng > 0) {
      // ---- the slice's partial tiles: tensor memory -> part[slice][column][output row] ----------
      const int quarter = warp & 3, n = quarter * 32 + lane;   // tile row = tensor-memory lane
      ok = mbar_wait_bounded(smem_u32(acc_done), 0, a.err, kErrTimeoutTc05);
      ok = __all_sync(0xffffffffu, ok);
      if (ok) {
        tc05_fence_after();
        for (int t = 0; t < n_tiles; t++) {
          float* out = a.part + (size_t)slice * a.npad * a.n_out_pad + (size_t)(mt0 + t) * 128 + n;
          const uint32_t tb = tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(t * a.npad);
          for (int ch = 0; ch < a.npad / 16; ch++) {
            float v[16];
            tmem_ld16(tb + (uint32_t)(ch * 16), v);
#pragma unroll
            for (int e = 0; e < 16; e++) out[(size_t)(ch * 16 + e) * a.n_out_pad] = v[e];
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
    for (int s = 0; s < slices; s++) acc += part[((size_t)s * npad + r) * n_out_pad + p];
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

Tc05Plan plan_tc05(int n_strips, int groups, int rows, int x_lo, int n_sm) {
  Tc05Plan p{};
  if (n_strips < 1 || groups < 1 || rows < 1 || rows > kTcMaxRows || n_sm < 1) return p;
  p.npad = (rows + 15) / 16 * 16;
  p.mtiles = (n_strips + kTcStrips - 1) / kTcStrips;
  p.tgroups = (p.mtiles + kTcTiles - 1) / kTcTiles;
  // K slices: enough CTAs to cover the SMs, each slice at least 4 groups long
  const int want = (n_sm + p.tgroups - 1) / p.tgroups;
  const int s = std::max(1, std::min(want, groups / 4));
  p.gps = (groups + s - 1) / s;
  p.slices = (groups + p.gps - 1) / p.gps;
  p.grid = p.tgroups * p.slices;
  p.x_stage = (uint32_t)p.npad * 128u * (x_lo ? 2u : 1u);   // a multiple of 2048 B
  p.x_tx = p.x_stage;
  const size_t fixed = 1024 /* alignment slack */ + (size_t)kTcSA * kTcAStage + (size_t)kTcSW * kTcWStage +
                       (size_t)(2 * kTcSW + 2 * kTcMaxSX + 2 * kTcSA + 1) * 8 + 16;
  const size_t room = kTcSmemMax > fixed ? kTcSmemMax - fixed : 0;
  p.sx = (int)std::min<size_t>(kTcMaxSX, room / p.x_stage);
  if (p.sx < 2) return Tc05Plan{};
  p.smem = fixed + (size_t)p.sx * p.x_stage;
  int cols = 32;
  while (cols < kTcTiles * p.npad) cols *= 2;
  p.tmem_cols = cols;
  p.part_off = 0;
  p.scratch = (size_t)p.slices * p.npad * p.mtiles * 128 * 4;
  return p;
}

cudaError_t launch_tc05_parts(const Tc05Args& a, const Tc05Plan& p, cudaStream_t s) {
  static std::atomic<int> smem_set[kMaxDevices];
  cudaError_t e;
  e = ensure_smem_limit(tc05_q4_kernel, p.smem, smem_set);
  if (e != cudaSuccess) return e;
  tc05_q4_kernel<<<p.grid, kTcThreads, p.smem, s>>>(a);
  return cudaGetLastError();
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

// Device helpers for sm_103a: mbarriers, bulk / tensor copies (TMA), mma.sync fragments,
// bf16 packing and a bounded wait that reports instead of hanging.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "internal.h"

namespace dfl {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later async-proxy
// (TMA) writes to the same bytes.
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of an mbarrier for a bounded time. On timeout, set `code` in the device
// error word err[0] and return false: the caller stops issuing work and leaves. The limit is
// err[1] microseconds when that word is nonzero (a test setting), else 1 s; a wait without an
// error word (err == nullptr: draining a CTA's own copies before it leaves) always allows 1 s.
// The first ~20000 cycles (~10 us) poll the barrier alone: reading the limit word is a global
// load, and a pipeline's ordinary short waits must not each pay a memory round trip for it (under
// a full HBM stream that is a microsecond). Limits are therefore at least ~10 us.
constexpr long long kWaitFastCycles = 20000;
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, unsigned* err,
                                                  unsigned code) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long c0 = clock64();
  do {
    if (mbar_try_wait(bar, parity)) return true;
  } while (clock64() - c0 < kWaitFastCycles);
  const uint64_t t0 = global_timer_ns();
  const unsigned limit_us = err ? *reinterpret_cast<volatile unsigned*>(err + 1) : 0u;
  const uint64_t limit_ns = limit_us ? (uint64_t)limit_us * 1000ull : 1000000000ull;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > limit_ns) {
      if (err) atomicOr(err, code);
      return false;
    }
  }
}

// Device bounds checks of debug builds (compiled with -DDFL_DEBUG_CHECKS): in_bounds(cond, err)
// returns cond, and a false cond also sets kErrBounds in the error word, which dflash_check_errors
// reports as DFLASH_EBOUNDS. Release builds compile the report away and keep only the caller's own
// guard (a clamp or a skipped access), so both builds compute the same results on valid inputs.
__device__ __forceinline__ bool in_bounds(bool cond, unsigned* err) {
#ifdef DFL_DEBUG_CHECKS
  if (!cond && err) atomicOr(err, kErrBounds);
#else
  (void)err;
#endif
  return cond;
}

// 1-D bulk copy global -> shared, completing on an mbarrier (16-byte aligned, size % 16 == 0).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// Bulk prefetch of global bytes into L2 (16-byte aligned, size % 16 == 0); nothing waits for it.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 3-D tiled tensor copy global -> shared (TMA), completing on an mbarrier.
// Tiled tensor prefetch of one 4-D box into L2; nothing waits for it.
__device__ __forceinline__ void tma_prefetch_4d(const CUtensorMap* map, int x, int y, int z, int w) {
  asm volatile("cp.async.bulk.prefetch.tensor.4d.L2.global.tile [%0, {%1, %2, %3, %4}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z), "r"(w)
               : "memory");
}

// Tiled tensor prefetch of one 3-D box into L2; nothing waits for it.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int x, int y, int z,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// D = A * B + D, m16n8k16, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                            uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldmatrix_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                                  uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// (a & b) | c in one instruction.
__device__ __forceinline__ uint32_t lop3_and_or(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t r;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// 4-bit codes -> f16x2 with one lop3 each; both forms are exact and the caller undoes the offset
// (and the factor 16) in fp32, once per 64-input group:
//   codes at bits 3-6 / 19-22 with 0x5800 (128.0, ulp 1/8) -> 128 + q
//   codes at bits 4-7 / 20-23 with 0x6400 (1024.0, ulp 1)  -> 1024 + 16 q   (no shift needed)
// The offsets are kept small relative to q (about 17x and 8.5x) because the fp32 group sum loses
// that factor when the offset is removed.
__device__ __forceinline__ uint32_t nib128_to_f16x2(uint32_t u_at_bit3) {
  return lop3_and_or(u_at_bit3, 0x00780078u, 0x58005800u);
}
__device__ __forceinline__ uint32_t nib_hi_to_f16x2(uint32_t u) { return lop3_and_or(u, 0x00F000F0u, 0x64006400u); }

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

constexpr float kF16Max = 65504.0f;

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__half>(__half v) { return __half2float(v); }

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>  // saturating: activations never become inf
__device__ __forceinline__ __half from_f<__half>(float v) {
  return __float2half_rn(fminf(fmaxf(v, -kF16Max), kF16Max));
}

// Store an activation; for f16 with lo_off != 0 also store the rounding remainder v - f16(v) at
// base[idx + lo_off], so that hi + lo carries v to about 22 bits.
template <typename T>
__device__ __forceinline__ void store_act_split(void* base, size_t idx, size_t lo_off, float v) {
  const T hi = from_f<T>(v);
  static_cast<T*>(base)[idx] = hi;
  if constexpr (sizeof(T) == 2) {
    if (lo_off) static_cast<T*>(base)[idx + lo_off] = from_f<T>(v - to_f<T>(hi));
  }
}

// Element k of row n of a matrix in its caller-side storage format (used for gathers).
__device__ __forceinline__ float load_weight(int fmt, const void* data, const uint16_t* scale,
                                             const uint16_t* bias, int n_in, int64_t n, int k) {
  if (fmt == FMT_F32) return static_cast<const float*>(data)[n * n_in + k];
  if (fmt == FMT_BF16) return bf16_bits_to_float(static_cast<const uint16_t*>(data)[n * n_in + k]);
  const uint32_t word = static_cast<const uint32_t*>(data)[n * (n_in / 8) + k / 8];
  const float q = static_cast<float>((word >> (4 * (k % 8))) & 15u);
  const int64_t g = n * (n_in / 64) + k / 64;
  return fmaf(bf16_bits_to_float(scale[g]), q, bf16_bits_to_float(bias[g]));
}

// Programmatic dependent launch: let the next kernel of the stream start launching, and wait
// until every earlier kernel of the stream has completed and its writes are visible.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Ticket for "last one to arrive does the follow-up work": an atomic add at GPU scope with
// acquire-release semantics. Callers pass a CTA barrier first, so the writes of every thread of
// the CTA are released with it (cumulativity through the barrier), and the thread that sees the
// final count acquires everything the other CTAs released.
__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// ---- thread-block clusters (distributed shared memory) ----
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in CTA `rank` of this cluster.
__device__ __forceinline__ uint32_t map_shared_rank(uint32_t smem_addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_v4(uint32_t addr, float4 v) {
  asm volatile("st.shared::cluster.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "f"(v.x), "f"(v.y), "f"(v.z),
               "f"(v.w)
               : "memory");
}

// Every thread of every CTA of the cluster arrives (releasing its earlier shared-memory writes,
// remote ones included) and waits for all the others (acquiring theirs).
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

}  // namespace dfl

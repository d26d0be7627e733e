// Internal declarations shared by the host side (abi.cu) and the kernels (gemv.cu, attn.cu,
// misc.cu) of the DFlash draft-round library. Not part of the public ABI (include/dflash.h).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <stdint.h>

#include <utility>

#include "../../include/dflash.h"

namespace dfl {

// ---- GEMV (skinny GEMM) geometry ---------------------------------------------------------------
// Weights are re-laid-out at create time into 16-row strips. Per strip and per 64-input group:
//   q4   : 576 B = 512 B of nibbles in mma.sync A-fragment order (16 B per lane) + 16 x (scale, bias)
//   bf16 : 2048 B = 4 k16 steps x 32 lanes x 16 B, A-fragment order, values stored as f16
//   f32  : row-major float rows (CUDA-core path), strips of 16 consecutive logical rows
#ifndef DFL_GEMV_WARPS
#define DFL_GEMV_WARPS 16
#endif
#ifndef DFL_GEMV_STAGES
#define DFL_GEMV_STAGES 2
#endif
#ifndef DFL_Q4_GROUPS_PER_STAGE
#define DFL_Q4_GROUPS_PER_STAGE 6
#endif
constexpr int kWarps = DFL_GEMV_WARPS;    // consumer warps per tensor-core GEMV CTA
constexpr int kStages = DFL_GEMV_STAGES;  // ring depth per warp (bulk copies in flight)
#ifndef DFL_PRE_PDL_STAGES
#define DFL_PRE_PDL_STAGES 1
#endif
// stages per warp requested before waiting for the previous kernel (the rest after)
constexpr int kPrePdlStages = DFL_PRE_PDL_STAGES < kStages ? DFL_PRE_PDL_STAGES : kStages;
#ifndef DFL_L2_PREFETCH_TILES
#define DFL_L2_PREFETCH_TILES 0
#endif
// weight tiles per warp, beyond its ring, prefetched into L2 before waiting for the previous kernel
constexpr int kL2PrefetchTiles = DFL_L2_PREFETCH_TILES;
constexpr int kQ4GroupBytes = 576;
constexpr int kBf16GroupBytes = 2048;
constexpr int kQ4GroupsPerStage = DFL_Q4_GROUPS_PER_STAGE;
constexpr int kBf16GroupsPerStage = (kQ4GroupsPerStage * kQ4GroupBytes) / kBf16GroupBytes > 0
                                        ? (kQ4GroupsPerStage * kQ4GroupBytes) / kBf16GroupBytes : 1;
constexpr int kStageBytes = kQ4GroupsPerStage * kQ4GroupBytes > kBf16GroupsPerStage * kBf16GroupBytes
                                ? kQ4GroupsPerStage * kQ4GroupBytes : kBf16GroupsPerStage * kBf16GroupBytes;
constexpr int kMaxRows = 32;              // activation rows per launch (4 n-tiles of 8)
constexpr int kMaxCtxChunk = 32;          // context rows per projection chunk
// Warps per tensor-core GEMV CTA by n-tile count: more activation columns need more registers
// per thread (one CTA per SM, 64K registers).
__host__ __device__ constexpr int gemv_warps(int nt) { return nt == 1 ? kWarps : (nt == 2 ? 12 : 8); }
constexpr int kF32Warps = 8;

enum Fmt { FMT_F32 = 0, FMT_BF16 = 1, FMT_Q4 = 2 };
enum Epi { EPI_STORE = 0, EPI_CTX = 1, EPI_KV = 2, EPI_QKV = 3, EPI_RESID = 4, EPI_SWIGLU = 5, EPI_LMHEAD = 6 };
enum NormMode { NORM_NONE = 0, NORM_ONE = 1, NORM_CTX = 2 };

// Device error word bits.
constexpr unsigned kErrTimeoutGemv = 1u;
constexpr unsigned kErrTimeoutAttn = 2u;
constexpr unsigned kErrBounds = 16u;   // a device bounds check failed (builds with DFL_DEBUG_CHECKS)

struct RowMap {      // activation row r of a launch reads source row (r/per)*stride + off + r%per
  int per, stride, off;
};

struct EpiArgs {
  int row_base;      // first logical matrix row of the epilogue's output space
  int n_rows;        // valid output features (rows >= row_base + n_rows are padding)
  // EPI_STORE
  void* out; int ldo; int out_f32;
  // EPI_RESID: h[r][n] += y; xnext[r][n] = act(h[r][n] * wnext[n]); ssq_out[r*ssq_ld + strip]
  float* h; const float* wnext; void* xnext; float* ssq_out; int ssq_ld;
  size_t x_lo_off;   // EPI_RESID / EPI_CTX: also write the f16 remainder this many elements on
  // EPI_CTX: x = y; xw[i][r][n] = act(x*ctx_norm*attn_norm_i); ssq_out[(r*ssq_ld+strip)*2+{0,1}]
  const float* ctx_norm; const float* attn_norms; int n_layers; void* xw; int xw_rows;
  // EPI_QKV
  void* q; void* kb; void* vb; int qd, kvd;
  // EPI_KV (append to a ring of cap rows per (slot, kv head)); cache layout [slot][Hkv][cap][hd]
  void* kc; void* vc; int cap, hd, n_kv;
  long long kv_grp_stride;   // bytes between the caches of consecutive layers (grouped launches)
  int kv_slot[kMaxRows];
  int kv_pos[kMaxRows];
  // EPI_SWIGLU (gated FFN: silu(g) * u, or gelu_tanh(g) * u when ffn_act == DFLASH_FFN_GELU)
  void* act; int inter; int ffn_act;
  // EPI_LMHEAD
  float* logits; int vocab;
  const float* logit_bias;    // added to every logit before the argmax (Markov head), or null
  long long logit_row_stride; // elements between activation rows in logits / logit_bias (0: vocab)
  float* lm_part;    // one K slice: per-CTA (max, sum, index) per column, merged by lm_reduce_kernel
  float* lm_strip;   // split-K launches: per-strip (max, sum, index) per column, merged in strip order
};

struct GemvArgs {
  const uint8_t* w;        // packed matrix base
  // Grouped launch: grp_n equally shaped problems side by side in the grid (grp_ctas CTAs each);
  // problem j uses w + j * grp_w_stride (bytes) and x + j * grp_x_stride (elements). grp_n = 1:
  // one problem.
  int grp_n, grp_ctas;
  long long grp_w_stride, grp_x_stride;
  // K split over a 2-CTA cluster (n_slices == 2): blockIdx pairs are the two slices of the same
  // strips; partials meet in the owning CTA's shared memory (cpart_cap strip slots per CTA).
  int cluster2, cpart_cap;
  int strip0, n_strips;    // strip range of this launch
  int k, groups;           // inputs and 64-input groups
  int n_slices, gps;       // K slices per strip, groups per slice
  int ctas_per_slice;
  int R;                   // activation rows (<= kMaxRows)
  const void* x; int ldx; RowMap xmap;
  int x_bf16;              // tensor-core path: x rows are bf16 (converted to f16 after staging)
  const float* x_colscale; // tensor-core path: optional per-input scale of x (problem j: + j * stride)
  long long x_colscale_grp_stride;
  long long x_lo_off;      // tensor-core path: f16 remainder rows at x + x_lo_off elements (0: none)
  int norm_mode; const float* ssq; int ssq_ld; int ssq_parts; float inv_dim; float eps;
  float* partials; int* tickets;
  unsigned* err;
  int stall_cta1;          // test hook: CTA stall_cta1 - 1 also waits on a barrier nothing completes (0: none)
  EpiArgs e;
};

// ---- attention ---------------------------------------------------------------------------------
struct AttnReq {
  int slot;      // cache slot of the request
  int ctx_len;   // context length P
  int row0;      // first block row of the request
};

struct AttnArgs {
  const void* q; const void* kb; const void* vb; void* out;   // q/out [rows][qd], kb/vb [rows][kvd]
  const void* kc; const void* vc;                             // layer base of the cache
  int qd, kvd, hd, hq, hkv, gamma, window, cap, max_batch;
  int plane0;                                                 // layer * max_batch * hkv
  int n_req, n_splits;
  float scale_log2;                                           // log2(e) / sqrt(hd)
  float* part_o; float* part_ml;
  unsigned* err;
  AttnReq req[DFLASH_MAX_BATCH];
};

// ---- misc --------------------------------------------------------------------------------------
struct RepackSrc {
  const void* data; const uint16_t* scale; const uint16_t* bias; int rows;
};

struct RepackArgs {
  RepackSrc src[3]; int n_src;
  int interleave;          // 1: strip rows 0-7 from src[0] (gate), 8-15 from src[1] (up)
  int fmt, k, n_strips;
  uint8_t* dst;
};

constexpr int kBlockCols = 1024;           // block-init columns per CTA (one ssq part each)

struct BlockArgs {
  int n_req, gamma, d, H, vocab, fmt, act_f32;
  const int32_t* anchor;
  const void* emb; const uint16_t* emb_scale; const uint16_t* emb_bias;
  const float* tokrow;        // [n_req][d] tok_proj(E[anchor]) when d != H
  const float* mask_emb; const float* block_pos; const float* attn_norm0;
  float* h; void* xn; float* ssq; int ssq_ld;
  size_t xn_lo_off;           // f16 remainder of xn at this element offset (0: none)
  void* emb_out;              // gather mode: [n_req][H] activation rows
  unsigned* err;              // device error word (bounds checks of debug builds)
};

// Raise a kernel's dynamic shared-memory limit to at least `bytes` on the current device (the
// attribute is per device). `cache` holds the limit set so far, per device ordinal.
constexpr int kMaxDevices = 64;
template <typename K>
inline cudaError_t ensure_smem_limit(K kernel, size_t bytes, std::atomic<int>* cache) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if ((int)bytes <= cache[dev].load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) cache[dev].store((int)bytes, std::memory_order_relaxed);
  return e;
}

// Launch with programmatic stream serialization: the kernel may start while the previous kernel
// of the stream drains; it must call pdl_wait() before reading anything earlier kernels wrote.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t s, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  int n = 0;
#ifndef DFL_NO_PDL
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  n++;
#endif
  if (cluster_x > 1) {   // grid.x must be a multiple of cluster_x
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    n++;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  return launch_pdl_cluster(kernel, grid, block, smem, s, 1, std::forward<Args>(args)...);
}

// ---- launchers (return cudaGetLastError of the launch) -----------------------------------------
cudaError_t launch_gemv(int fmt, int epi, int nt, const GemvArgs& a, int grid, cudaStream_t s);
// Final greedy token + confidence per row from n_parts (max, sum, index) states kMaxRows rows apart;
// row c's results go to tok_out[c * out_stride], conf_out[c * out_stride].
cudaError_t launch_lm_reduce(const float* parts, int n_parts, int rows, int32_t* tok_out, float* conf_out,
                             int out_stride, cudaStream_t s);
// Markov head input of draft k: x[b] = W1[prev] (f16, remainder at x + lo_off), prev = anchor[b] for
// k == 0, else draft[b * n + k - 1].
cudaError_t launch_markov_gather(int n_req, int k, int n, int rank, int vocab, int fmt, const void* w1,
                                 const uint16_t* w1_scale, const uint16_t* w1_bias, const int32_t* anchor,
                                 const int32_t* draft, void* x, size_t lo_off, unsigned* err, cudaStream_t s);
size_t gemv_smem_bytes(int fmt, int R, int gps, int x_lo, int lm, int cpart_cap);
cudaError_t launch_attn_tc(const AttnArgs& a, const CUtensorMap& kmap, const CUtensorMap& vmap,
                           cudaStream_t s);
size_t attn_smem_bytes(int hd);
cudaError_t launch_attn_merge(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_attn_f32(const AttnArgs& a, cudaStream_t s);
cudaError_t launch_repack(const RepackArgs& a, cudaStream_t s);
cudaError_t launch_block_init(const BlockArgs& a, cudaStream_t s);
cudaError_t launch_embed_gather(const BlockArgs& a, cudaStream_t s);
cudaError_t launch_accept(int n_req, int n, const int32_t* draft, const int32_t* keep, const int32_t* target,
                          int32_t* accept_len, int32_t* next_anchor, unsigned long long* hist, unsigned* err,
                          cudaStream_t s);
cudaError_t launch_draft_lengths(int n_req, int n, const float* conf, const float* thresholds, float min_conf,
                                 int32_t* keep, cudaStream_t s);

}  // namespace dfl

// Host-side declarations of the many-row tcgen05 contraction (gemm_tc05.cu), shared with abi.cu.
#pragma once

#include <cuda_fp16.h>

#include "internal.h"

namespace dfl {

constexpr unsigned kErrTimeoutTc05 = 4u;  // device error word bit of this kernel's bounded waits

constexpr int kTcWarps = 11;              // weight copies, MMA issue, 8 dequantising warps (4 of them also the
                                          // epilogue), activation copies
constexpr int kTcMaxRows = 160;           // activation rows per call (the MMA's N, padded to 16)
constexpr int kTcTiles = 3;               // 128-row output tiles per CTA, at most (3 x 160 accumulator columns <= 512)
#ifndef DFL_TC_KW
#define DFL_TC_KW 1
#endif
constexpr int kTcKW = DFL_TC_KW;          // 64-input groups per raw-weight copy (and stage)
constexpr int kTcMaxSW = 8;               // raw 4-bit stages (kTcKW groups of a CTA's tiles each), at most
constexpr size_t kTcBytesInFlight = 96 * 1024;   // weights requested ahead per SM (ring + L2 prefetch)
constexpr int kTcMaxSA = 6;               // dequantised f16 A stages, at most
constexpr int kTcMaxSX = 4;               // activation stages, at most
constexpr size_t kTcSmemMax = 232448;     // dynamic shared memory a CTA may opt into (227 KB)

struct Tc05Args {
  CUtensorMap xmap, xlmap;   // activation rows (f16) and their f16 remainder as [layer][k / 64][rows][64]:
                             // box 64 x npad x kx x 1, 128-byte swizzle (kx groups per copy)
  CUtensorMap wmap;          // the stored 4-bit matrix as [layer][strip][group][144 words]: box 144 x kTcKW
                             // x (8 x tiles_big) x 1, kTcKW groups of a big CTA's tiles per copy (rows
                             // and groups past the matrix read as zero);
  CUtensorMap wmap_small;    // the same with box 144 x kTcKW x (8 x tiles_small) x 1
  const uint8_t* w;          // stored 4-bit matrix: [strip][group] tiles of kQ4GroupBytes
  float* part;               // [slices][n_out_pad / 16][npad][16] partial tiles (scratch): per 16-row
                             // strip of the stored order, each activation row's 16 outputs
  unsigned* err;
  int n_strips, groups, npad, gps, mtiles, has_lo, n_out_pad, sx, sw, sa, pf, kx, tmem_cols;
  // CTA b covers tile group b % tgroups and K slice b / tgroups; the first groups_big tile groups
  // hold tiles_big consecutive 128-row tiles, the others tiles_small (the last possibly fewer)
  int tgroups, tiles_big, groups_big, tiles_small;
  uint32_t x_stage, x_tx;
  // grouped launches (grid.y = n_layers): the same plan over n_layers equally spaced matrices and
  // activation planes; partial tiles of layer l at part + l * part_layer_stride. w_strip0: the
  // first stored strip of the row range the contraction covers (a part of a larger matrix).
  int n_layers, w_strip0;
  size_t part_layer_stride;
};

struct Tc05Plan {
  int npad = 0, mtiles = 0, slices = 0, gps = 0, grid = 0, sx = 0, sw = 0, sa = 0, pf = 0, kx = 0, tmem_cols = 0;   // npad == 0: no plan
  int tgroups = 0, tiles_big = 0, groups_big = 0, tiles_small = 0;
  uint32_t x_stage = 0, x_tx = 0;
  size_t smem = 0, part_off = 0, srow_off = 0, scratch = 0;   // scratch: partial tiles, then row scales
};

// The launch shape with the shortest modelled time: tiles per CTA, K slices, ring depths.
Tc05Plan plan_tc05(int n_strips, int groups, int rows, int x_lo, int n_sm);

// Copies the plan's shape into the kernel arguments (maps, pointers and sizes are the caller's).
void tc05_fill_args(const Tc05Plan& p, int has_lo, Tc05Args& a);

// The contraction: partial tiles [slices][n_out_pad / 16][npad][16] in a.part (stored row order).
cudaError_t launch_tc05_parts(const Tc05Args& a, const Tc05Plan& p, cudaStream_t s);

// launch_tc05_parts, then the ordered slice reduction into y [rows][ldy] (natural row order of
// the matrix; half > 0: a gate/up matrix with `half` gate rows).
cudaError_t launch_tc05(const Tc05Args& a, const Tc05Plan& p, int rows, int n_out, int half, float* y, int ldy,
                        cudaStream_t s);

// bf16 -> f16 of n_elems (even) contiguous elements, as the skinny GEMV converts context taps.
cudaError_t launch_bf16_to_f16(const void* src, long long n_elems, void* dst, cudaStream_t s);

// A draft-round projection's epilogue (EPI_CTX, EPI_QKV, EPI_KV, EPI_RESID, EPI_SWIGLU or EPI_LMHEAD) from the
// partial tiles, through the skinny GEMV's strip epilogues, for up to kTcMaxChunks row chunks in
// one launch (grid.y = chunk): ch.a[j] describes chunk j as for the GEMV (a.R <= kMaxRows rows,
// nt = n-tiles of 8 for the largest chunk) with a.n_slices == 1; its row c is contraction row
// ch.row_base[j] + map_row(ch.a[j].xmap, c). LM head: one vocab state per CTA and row in each
// chunk's a.e.lm_part.
constexpr int kTcMaxChunks = 8;   // ceil(160 / (gamma * floor(32 / gamma))) for gamma in 2..16
struct Tc05EpiChunks {
  GemvArgs a[kTcMaxChunks];
  int row_base[kTcMaxChunks];
  int n;
};
// One f16 (+ remainder) input plane per layer, planes `plane` elements apart, for the grouped
// context K/V: plane i = plane 0 (x * ctx_norm, in place) * attn_norm_i, rows [0, rows) of width d.
cudaError_t launch_tc05_kv_planes(void* xw, long long lo_off, const float* attn_norm, int rows, int d, int n_layers,
                                  long long plane, cudaStream_t s);

// srow: kTcMaxChunks x kMaxRows floats of scratch for the rows' norm scales. n_layers > 1: a grouped
// launch (EPI_KV over every layer), layer l's partial tiles at part + l * part_layer_stride; strips
// of the partial tiles count from the chunks' strip0.
cudaError_t launch_tc05_epilogue(int epi, int nt, const Tc05EpiChunks& ch, const float* part, int slices, int npad,
                                 int n_out_pad, int grid, float* srow, int n_layers, size_t part_layer_stride,
                                 cudaStream_t s);

// ---- skinny projections of the draft round on tcgen05 (proj_tc05.cu) ---------------------------
constexpr unsigned kErrTimeoutProj = 8u;  // device error word bit of its bounded waits
constexpr int kProjMaxRows = 32;          // contraction rows (the MMA's N: 16 or 32)

struct ProjArgs {
  CUtensorMap xmap, xlmap;   // contraction rows (f16) and their f16 remainder: box 64 x npad, 128-byte swizzle
  GemvArgs g;                // the epilogue (rows, row map, norms, outputs) as for the GEMV
  const uint8_t* w;          // stored 4-bit matrix: [strip][group] tiles of kQ4GroupBytes
  float* partials;           // [grid][2][npad][128] pieces of tiles cut between CTAs
  int* tickets;              // [mtiles] arrivals, zero between launches
  int n_strips, groups, mtiles, npad, has_lo, sa, sx, sw, tmem_cols;
  int row_base;              // contraction row of the epilogue's row map origin
  uint32_t x_stage;
};

struct ProjPlan {
  int npad = 0, mtiles = 0, grid = 0, sa = 0, sx = 0, sw = 0, tmem_cols = 0;   // npad == 0: no plan
  uint32_t x_stage = 0;
  size_t smem = 0, partial_floats = 0;
};

ProjPlan plan_proj_tc05(int n_strips, int groups, int rows, int x_lo, int n_sm);

// One projection: EPI_QKV, EPI_RESID, EPI_SWIGLU or EPI_LMHEAD (nt = n-tiles of 8 epilogue rows).
cudaError_t launch_proj_tc05(int epi, int nt, const ProjArgs& pa, const ProjPlan& p, cudaStream_t s);

}  // namespace dfl

// Host side of the C ABI in include/dflash.h: validation, workspace layout, weight re-layout at
// create, launch planning and the three calls of a draft round.
#include <cuda.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <new>

#include "gemm_tc05.h"
#include "internal.h"

using namespace dfl;

namespace {

struct PackedMat {
  uint8_t* w = nullptr;
  int n_rows = 0;    // logical rows
  int n_strips = 0;  // ceil(n_rows / 16)
  int k = 0, groups = 0;
};

struct GemvPlan {
  int n_slices, gps, ctas_per_slice, grid;
  int cluster2 = 0, cpart_cap = 0;   // 2-way K split inside 2-CTA clusters
};

}  // namespace

struct dflash_handle {
  dflash_config cfg;
  int fmt = 0, act_f32 = 0, act_bytes = 2;
  int d = 0, H = 0, qd = 0, kvd = 0, I = 0, L = 0, G = 0, V = 0, mH = 0, cap = 0;
  int nd = 0;   // drafts per block: gamma - 1, or gamma when drafting from every block row
  int n_sm = 148, r_blk = 0, ssq_ld = 0;
  size_t ws_bytes = 0;

  PackedMat wc, qkv[DFLASH_MAX_LAYERS], wo[DFLASH_MAX_LAYERS], gu[DFLASH_MAX_LAYERS], down[DFLASH_MAX_LAYERS],
      tok, outp, lm;
  PackedMat mk;                 // Markov head W2^T [V][r] (markov_rank > 0)
  dflash_matrix mk_w1{};        // Markov head W1 [V][r], borrowed
  float* mk_base = nullptr;     // [max_batch][n_draft][V] head logits before the Markov bias
  void* mk_x = nullptr;         // [max_batch][r] W1 rows (f16 + remainder, or fp32)
  dflash_matrix embed{};
  float *ctx_norm = nullptr, *mask_emb = nullptr, *block_pos = nullptr, *out_norm = nullptr;
  float *attn_norm = nullptr, *ff_norm = nullptr;  // [L][d]
  void *kc = nullptr, *vc = nullptr;               // [L][max_batch][Hkv][cap][hd]
  float* h = nullptr;
  void *xn = nullptr, *q = nullptr, *kb = nullptr, *vb = nullptr, *attn = nullptr, *act = nullptr, *hout = nullptr,
       *emb = nullptr, *xw = nullptr;
  float *tokrow = nullptr, *ssq = nullptr, *ssq_ctx = nullptr;
  float* partials = nullptr;
  int* tickets = nullptr;
  float* lm_part = nullptr;
  float* lm_strip = nullptr;
  float *att_o = nullptr, *att_ml = nullptr;
  unsigned* err = nullptr;
  unsigned long long* acc_hist = nullptr;   // [DFLASH_MAX_GAMMA + 1] blocks per accepted length
  size_t partial_floats = 0;
  int ticket_count = 0, lm_grid_max = 0, att_pairs_max = 0;
  // many-row draft calls on the tcgen05 contraction (config large_batch_tc05)
  int tc05_on = 0, tc05_rows = 0;
  int xw_rows = 0;   // context rows per input plane of xw (and rows of ssq_ctx)
  uint8_t* tc05_scratch = nullptr;
  size_t tc05_scratch_bytes = 0;
  void* tc05_taps = nullptr;    // [kTcMaxRows][n_taps * H] f16: context taps converted for TMA
  // draft calls of <= 32 rows on the tcgen05 projection kernel (config skinny_tc05)
  int pj_on = 0;
  float* pj_partials = nullptr;  // [n_sm][2][32][128] pieces of tiles cut between CTAs
  CUtensorMap kmap{}, vmap{};

  int64_t ctx_len[DFLASH_MAX_BATCH] = {};
  dflash_stats stats{};
  uint64_t launches = 0;
  cudaEvent_t probe_start = nullptr, probe_stop = nullptr;
  int probe_kernel = 0;         // DFLASH_PROBE_* the events go around (used once)
  int stall_armed = 0, stall_active = 0;   // test hook: CTA + 1 that stalls in the next / this draft call
};

namespace {

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int packed_bytes_per_strip(int fmt, int k) {
  if (fmt == FMT_Q4) return (k / 64) * kQ4GroupBytes;
  if (fmt == FMT_BF16) return (k / 64) * kBf16GroupBytes;
  return 16 * k * 4;
}

int nt_for(int R) { return R <= 8 ? 1 : (R <= 16 ? 2 : 4); }

// Split of one launch over the SMs. Every warp of a CTA works on every strip of that CTA, so the
// time of a launch is about (strips per CTA) x (groups per K slice); a K split over several
// CTAs costs a partial tile per strip, counted here as one extra group.
#ifndef DFL_CLUSTER_SPLIT
#define DFL_CLUSTER_SPLIT 1
#endif

// allow_cluster: the launch may split K in two inside 2-CTA clusters (partials meet in shared
// memory through the cluster instead of global memory and tickets); lm: the LM-head epilogue.
GemvPlan plan_gemv(const dflash_handle* h, int n_strips, int groups, int R, int x_lo, int n_sm,
                   int allow_cluster = 0, int lm = 0) {
  GemvPlan p{};
  if (h->fmt == FMT_F32) {
    p.n_slices = 1;
    p.gps = groups;
    p.ctas_per_slice = std::max(1, std::min((n_strips + kF32Warps - 1) / kF32Warps, 4 * n_sm));
    p.grid = p.ctas_per_slice;
    return p;
  }
  constexpr size_t kSmemLimit = 225 * 1024;
  long best = -1;
  for (int s = 1; s <= std::max(1, std::min(16, groups / gemv_warps(nt_for(R)))); s++) {
    const int gps = (groups + s - 1) / s;
    if (gemv_smem_bytes(h->fmt, R, gps, x_lo, lm, 0) > kSmemLimit) continue;
    const int slices = (groups + gps - 1) / gps;
    const int ctas = std::max(1, std::min(n_strips, n_sm / slices));
    const long per_cta = (n_strips + ctas - 1) / ctas;
    const long cost = per_cta * (gps + (slices > 1 ? 1 : 0));
    if (best < 0 || cost < best) {
      best = cost;
      p.n_slices = slices;
      p.gps = gps;
      p.ctas_per_slice = ctas;
    }
  }
  if (best < 0) {  // the activation slice must shrink further: split K until it fits
    int gps = groups;
    while (gps > 1 && gemv_smem_bytes(h->fmt, R, gps, x_lo, lm, 0) > kSmemLimit) gps = (gps + 1) / 2;
    p.gps = gps;
    p.n_slices = (groups + gps - 1) / gps;
    p.ctas_per_slice = std::max(1, std::min(n_strips, n_sm / p.n_slices));
  }
  p.grid = p.n_slices * p.ctas_per_slice;
  if (DFL_CLUSTER_SPLIT && allow_cluster && groups >= 2 && n_sm >= 2 && n_strips >= 2) {
    // two slices per 2-CTA cluster: taken when it fits and costs at most a little more streaming
    // than the best plan (it saves the split-K round trips at the end)
    const int gps2 = (groups + 1) / 2, pairs = std::min(n_sm / 2, n_strips);
    const int cap = (n_strips + pairs - 1) / pairs, cap_even = (cap + 1) & ~1;
    const long cost2 = (long)cap * gps2;
    if (gemv_smem_bytes(h->fmt, R, gps2, x_lo, lm, cap_even) <= kSmemLimit && (best < 0 || cost2 * 100 <= best * 115)) {
      p.n_slices = 2;
      p.gps = gps2;
      p.ctas_per_slice = pairs;
      p.grid = 2 * pairs;
      p.cluster2 = 1;
      p.cpart_cap = cap_even;
    }
  }
  return p;
}

struct Carver {
  uint8_t* base;
  size_t off = 0;
  template <typename T>
  T* take(size_t bytes) {
    off = round_up(off, 256);
    T* p = base ? reinterpret_cast<T*>(base + off) : nullptr;
    off += bytes;
    return p;
  }
};

bool valid_config(const dflash_config* c) {
  if (!c) return false;
  if (c->n_layers < 1 || c->n_layers > DFLASH_MAX_LAYERS) return false;
  if (c->d <= 0 || c->d % 64 || c->inter <= 0 || c->inter % 64 || c->target_hidden <= 0 || c->target_hidden % 64)
    return false;
  if (c->n_taps < 1 || c->vocab < 2 || c->gamma < 2 || c->gamma > DFLASH_MAX_GAMMA) return false;
  if (c->n_q_heads < 1 || c->n_kv_heads < 1 || c->n_q_heads % c->n_kv_heads) return false;
  if (c->head_dim != 64 && c->head_dim != 128 && c->head_dim != 256) return false;
  if (c->n_q_heads * c->head_dim != c->d) return false;
  if (c->window < 0 || c->max_batch < 1 || c->max_batch > DFLASH_MAX_BATCH || c->ctx_capacity < 1) return false;
  if (c->window > 0 && c->ctx_capacity < c->window) return false;
  if (!(c->eps >= 0.f)) return false;
  if (c->ffn_act != DFLASH_FFN_SWIGLU && c->ffn_act != DFLASH_FFN_GELU) return false;
  if (c->draft_all_rows != 0 && c->draft_all_rows != 1) return false;
  if (c->markov_rank < 0 || c->markov_rank > 1024 || c->markov_rank % 64) return false;
  if (c->large_batch_tc05 != 0 && c->large_batch_tc05 != 1) return false;
  if (c->skinny_tc05 != 0 && c->skinny_tc05 != 1) return false;
  if (c->wdtype < DFLASH_F32 || c->wdtype > DFLASH_Q4G64) return false;
  if (c->adtype == DFLASH_F32) {
    if (c->wdtype != DFLASH_F32) return false;
  } else if (c->adtype == DFLASH_BF16) {
    if (c->wdtype == DFLASH_F32) return false;
    if ((c->n_q_heads / c->n_kv_heads) * c->gamma > 64) return false;  // query rows per KV head
  } else {
    return false;
  }
  return true;
}

// Lay out the workspace; with base == nullptr only sizes are computed.
#ifndef DFL_ATTN_TILES_PER_SPLIT
#define DFL_ATTN_TILES_PER_SPLIT 2
#endif

// Which projections also read the f16 remainder of their input. Rounding the inputs of the
// projections that feed the attention scores (Q, K, V of the block and of the context rows) is
// amplified by the softmax; with those and gate-up covered, the rms logit error of the 4-bit
// 5120-wide drafter drops by 30% at no measured cost. out_proj and the LM head do not need it.
#ifndef DFL_LO_MASK
#define DFL_LO_MASK 11
#endif
enum { LO_QKV = 1, LO_GU = 2, LO_LM = 4, LO_CTXKV = 8, LO_OUTPROJ = 16 };
long long lo_if(int bit, size_t off) { return (DFL_LO_MASK & bit) ? (long long)off : 0; }

// The grouped context K/V contraction of `rows` context rows: the K/V strips of every layer's
// Q/K/V matrix, planned as one layer's problem on its share of the SMs.
Tc05Plan plan_kv_tc05(const dflash_handle* h, int rows) {
  return plan_tc05((2 * h->kvd) / 16, h->qkv[0].groups, rows, (DFL_LO_MASK & LO_CTXKV) ? 1 : 0,
                   std::max(1, h->n_sm / std::max(1, h->L)));
}

size_t carve(dflash_handle* h, uint8_t* base) {
  const dflash_config& c = h->cfg;
  Carver cv{base};
  auto mat = [&](PackedMat& m, int rows, int k) {
    m.n_rows = rows;
    m.n_strips = (rows + 15) / 16;
    m.k = k;
    m.groups = k / 64;
    m.w = cv.take<uint8_t>((size_t)m.n_strips * packed_bytes_per_strip(h->fmt, k));
  };
  mat(h->wc, h->d, h->mH);
  for (int i = 0; i < h->L; i++) {
    mat(h->qkv[i], h->qd + 2 * h->kvd, h->d);
    mat(h->wo[i], h->d, h->qd);
    mat(h->gu[i], 2 * h->I, h->d);
    mat(h->down[i], h->d, h->I);
  }
  if (h->d != h->H) {
    mat(h->tok, h->d, h->H);
    mat(h->outp, h->H, h->d);
  }
  mat(h->lm, h->V, h->H);
  if (c.markov_rank) mat(h->mk, h->V, c.markov_rank);

  const size_t ab = h->act_bytes;
  h->ctx_norm = cv.take<float>(h->d * 4);
  h->mask_emb = cv.take<float>((size_t)(h->G - 1) * h->d * 4);
  h->block_pos = cv.take<float>((size_t)h->G * h->d * 4);
  h->out_norm = cv.take<float>(h->d * 4);
  h->attn_norm = cv.take<float>((size_t)h->L * h->d * 4);
  h->ff_norm = cv.take<float>((size_t)h->L * h->d * 4);
  const size_t state_begin = round_up(cv.off, 256);
  const size_t cache_elems = (size_t)h->L * c.max_batch * c.n_kv_heads * h->cap * c.head_dim;
  h->kc = cv.take<void>(cache_elems * ab);
  h->vc = cv.take<void>(cache_elems * ab);
  const int R = h->r_blk;
  h->h = cv.take<float>((size_t)R * h->d * 4);
  h->xn = cv.take<void>((size_t)R * h->d * ab * 2);   // f16 values, then their f16 remainders
  h->q = cv.take<void>((size_t)R * h->qd * ab);
  h->kb = cv.take<void>((size_t)R * h->kvd * ab);
  h->vb = cv.take<void>((size_t)R * h->kvd * ab);
  h->attn = cv.take<void>((size_t)R * h->qd * ab);
  h->act = cv.take<void>((size_t)R * h->I * ab);
  h->hout = cv.take<void>((size_t)R * h->H * ab);
  h->emb = cv.take<void>((size_t)c.max_batch * h->H * ab);
  h->tokrow = cv.take<float>((size_t)c.max_batch * h->d * 4);
  h->ssq_ld = (h->d + 15) / 16;
  h->ssq = cv.take<float>((size_t)R * h->ssq_ld * 4);
  // a context call on the tcgen05 contraction projects up to kTcMaxRows rows' context K/V of every
  // layer in one grouped launch, from one input plane per layer
  const bool tc_possible = c.large_batch_tc05 && h->fmt == FMT_Q4 && !h->act_f32 && h->d == h->H && !c.markov_rank &&
                           std::min(c.max_batch * h->G, kTcMaxRows) > kMaxRows;
  h->xw_rows = tc_possible ? kTcMaxRows : kMaxCtxChunk;
  h->ssq_ctx = cv.take<float>((size_t)h->xw_rows * h->ssq_ld * 2 * 4);
  h->xw = cv.take<void>((size_t)h->L * h->xw_rows * h->d * ab * 2);
  if (c.markov_rank) {
    h->mk_base = cv.take<float>((size_t)c.max_batch * h->nd * h->V * 4);
    h->mk_x = cv.take<void>((size_t)c.max_batch * c.markov_rank * ab * 2);
  }

  // split-K partials / tickets: the largest plan over every matrix and row count
  size_t pf = 0;
  int tk = 0, lmg = 0;
  auto consider = [&](const PackedMat& m, int strips) {
    for (int r : {8, 16, 32})
      for (int lo : {0, 1}) {
        const GemvPlan p = plan_gemv(h, strips, m.groups, r, lo, h->n_sm, 0, &m == &h->lm);
        if (p.n_slices > 1) pf = std::max(pf, (size_t)strips * p.n_slices * 32 * nt_for(r) * 4);
        lmg = std::max(lmg, p.grid);
      }
    tk = std::max(tk, strips);
  };
  // the context K/V of every layer in one grouped launch
  if (h->L > 1)
    for (int r : {8, 16, 32})
      for (int lo : {0, 1}) {
        const int strips = (2 * h->kvd) / 16;
        const GemvPlan p = plan_gemv(h, strips, h->qkv[0].groups, r, lo, std::max(1, h->n_sm / h->L));
        if (p.n_slices > 1) pf = std::max(pf, (size_t)h->L * strips * p.n_slices * 32 * nt_for(r) * 4);
        tk = std::max(tk, h->L * strips);
      }
  consider(h->wc, h->wc.n_strips);
  for (int i = 0; i < h->L; i++) {
    consider(h->qkv[i], h->qkv[i].n_strips);
    consider(h->qkv[i], (2 * h->kvd) / 16);
    consider(h->wo[i], h->wo[i].n_strips);
    consider(h->gu[i], h->gu[i].n_strips);
    consider(h->down[i], h->down[i].n_strips);
  }
  if (h->d != h->H) {
    consider(h->tok, h->tok.n_strips);
    consider(h->outp, h->outp.n_strips);
  }
  consider(h->lm, h->lm.n_strips);
  h->partial_floats = pf;
  h->ticket_count = tk;
  h->lm_grid_max = lmg;
  h->partials = cv.take<float>(std::max<size_t>(pf, 4) * 4);
  h->tickets = cv.take<int>((size_t)tk * 4);
  // vocab states per CTA and row; a many-row draft call on the tcgen05 contraction keeps one slice
  // per row chunk
  const int lm_slices = tc_possible ? kTcMaxChunks : 1;
  h->lm_part = cv.take<float>((size_t)lmg * kMaxRows * 3 * 4 * lm_slices);
  h->lm_strip = cv.take<float>((size_t)tk * kMaxRows * 3 * 4);
  // attention split partials: n_req * Hkv * splits stays below ~2 waves of CTAs (see draft)
  h->att_pairs_max = std::max(4 * h->n_sm, c.max_batch * c.n_kv_heads);
  h->att_o = cv.take<float>((size_t)h->att_pairs_max * 64 * c.head_dim * 4);
  h->att_ml = cv.take<float>((size_t)h->att_pairs_max * 64 * 2 * 4);
  h->err = cv.take<unsigned>(8);   // [0] error bits, [1] wait limit in us (0: 1 s)
  h->acc_hist = cv.take<unsigned long long>((DFLASH_MAX_GAMMA + 1) * 8);
  // the tcgen05 contraction's scratch: the largest plan over the block projections and the head
  h->tc05_on = 0;
  h->tc05_rows = std::min(c.max_batch * h->G, kTcMaxRows);
  if (tc_possible) {
    size_t sc = 0;
    // every row count a many-row call can have (33 .. tc05_rows): the plan's K slices may grow as
    // the rows shrink
    auto need = [&](const PackedMat& m, int lo) {
      for (int r = kMaxRows + 1; r <= h->tc05_rows + 15; r += 16) {
        const Tc05Plan p = plan_tc05(m.n_strips, m.groups, std::min(r, h->tc05_rows), lo, h->n_sm);
        sc = std::max(sc, p.scratch);
      }
    };
    need(h->qkv[0], 1);
    need(h->wo[0], 0);
    need(h->gu[0], 1);
    need(h->down[0], 0);
    need(h->lm, 1);
    for (int r = kMaxRows + 1; r <= kTcMaxRows + 15; r += 16) {   // context rows, in chunks of up to 160
      const int rr = std::min(r, kTcMaxRows);
      const Tc05Plan pc = plan_tc05(h->wc.n_strips, h->wc.groups, rr, 0, h->n_sm);
      sc = std::max(sc, pc.scratch);
      const Tc05Plan pk = plan_kv_tc05(h, rr);   // every layer's context K/V, grouped
      sc = std::max(sc, (size_t)h->L * pk.srow_off + (pk.scratch - pk.srow_off));
    }
    h->tc05_on = sc > 0;
    h->tc05_scratch_bytes = sc;
    h->tc05_scratch = cv.take<uint8_t>(sc);
    h->tc05_taps = cv.take<void>((size_t)kTcMaxRows * h->mH * 2);
  }
  h->pj_on = c.skinny_tc05 && h->fmt == FMT_Q4 && !h->act_f32;
  if (h->pj_on) h->pj_partials = cv.take<float>((size_t)h->n_sm * 2 * kProjMaxRows * 128 * 4);
  (void)state_begin;
  return round_up(cv.off, 256);
}

void init_dims(dflash_handle* h, const dflash_config* c) {
  h->cfg = *c;
  h->fmt = c->wdtype == DFLASH_Q4G64 ? FMT_Q4 : (c->wdtype == DFLASH_BF16 ? FMT_BF16 : FMT_F32);
  h->act_f32 = c->adtype == DFLASH_F32;
  h->act_bytes = h->act_f32 ? 4 : 2;
  h->d = c->d;
  h->H = c->target_hidden;
  h->qd = c->n_q_heads * c->head_dim;
  h->kvd = c->n_kv_heads * c->head_dim;
  h->I = c->inter;
  h->L = c->n_layers;
  h->G = c->gamma;
  h->nd = c->gamma - 1 + c->draft_all_rows;
  h->V = c->vocab;
  h->mH = c->n_taps * c->target_hidden;
  // ring rows: at least the requested capacity, a multiple of the 64-row attention tile
  h->cap = (int)round_up((size_t)std::max(c->ctx_capacity, 64), 64);
  h->r_blk = c->max_batch * c->gamma;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? DFLASH_OK : DFLASH_ECUDA; }

bool disabled_by_env() {
  const char* v = getenv("DFLASH_DISABLE");
  return v && v[0] == '1';
}

typedef CUresult (*EncodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiled tensor_map_encoder() {
  static std::atomic<EncodeTiled> encode{nullptr};
  EncodeTiled e = encode.load(std::memory_order_acquire);
  if (!e) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return nullptr;
    e = reinterpret_cast<EncodeTiled>(fn);
    encode.store(e, std::memory_order_release);
  }
  return e;
}

// f16 activation rows [rows][ld] as 2-D tiles of 64 inputs x box_rows rows in the 128-byte
// swizzle (the K-major operand layout of the tcgen05 MMA); rows past `rows` read as zero.
int make_rows_map(const void* base, int k, int rows, int ld, int box_rows, CUtensorMap* map) {
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return DFLASH_ECUDA;
  const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_ECUDA;
}

// Activation rows (f16 [rows][ld], `layers` planes layer_stride bytes apart) as a 4-D map
// [layer][k / 64][rows][64]: box 64 x box_rows x kx x 1 with the 128-byte swizzle, i.e. kx
// consecutive 64-input groups of one plane per copy, each a K-major tile of box_rows rows of 128 B
// (rows past `rows` read as zero).
int make_rows_map_groups(const void* base, int k, int rows, int ld, int box_rows, int kx, int layers,
                         size_t layer_stride, CUtensorMap* map) {
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return DFLASH_ECUDA;
  const cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(k / 64), (cuuint64_t)layers};
  const cuuint64_t strides[3] = {(cuuint64_t)ld * 2, 128,
                                 (cuuint64_t)(layers > 1 ? layer_stride : round_up((size_t)rows * ld * 2, 16))};
  const cuuint32_t box[4] = {64, (cuuint32_t)box_rows, (cuuint32_t)kx, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_ECUDA;
}

// A stored 4-bit matrix ([strip][group] tiles of 576 B; `layers` matrices layer_stride bytes apart)
// as a 4-D map of 32-bit words [layer][n_strips][groups][144], box 144 x kw x (8 * tiles) x 1: kw
// consecutive groups of `tiles` consecutive 128-row output tiles of one matrix per copy; strips
// and groups past the matrix read as zero.
int make_q4_tile_map(const PackedMat& m, int tiles, int kw, int layers, size_t layer_stride, CUtensorMap* map) {
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return DFLASH_ECUDA;
  const size_t mat_bytes = (size_t)m.n_strips * m.groups * kQ4GroupBytes;
  const cuuint64_t dims[4] = {(cuuint64_t)(kQ4GroupBytes / 4), (cuuint64_t)m.groups, (cuuint64_t)m.n_strips,
                              (cuuint64_t)layers};
  const cuuint64_t strides[3] = {(cuuint64_t)kQ4GroupBytes, (cuuint64_t)m.groups * kQ4GroupBytes,
                                 (cuuint64_t)(layers > 1 ? layer_stride : round_up(mat_bytes, 16))};
  const cuuint32_t box[4] = {kQ4GroupBytes / 4, (cuuint32_t)kw, (cuuint32_t)(8 * tiles), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<uint8_t*>(m.w), dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_ECUDA;
}

int make_cache_map(dflash_handle* h, void* base, CUtensorMap* map) {
  EncodeTiled encode = tensor_map_encoder();
  if (!encode) return DFLASH_ECUDA;
  const dflash_config& c = h->cfg;
  // [plane][cap][head_dim] viewed as [plane][head_dim / 64][cap][64]: one copy brings a 64-key tile
  // with every 64-column part of the head (each a 64-row x 128-byte swizzled sub-tile)
  const cuuint64_t dims[4] = {64, (cuuint64_t)h->cap, (cuuint64_t)(c.head_dim / 64),
                              (cuuint64_t)h->L * c.max_batch * c.n_kv_heads};
  const cuuint64_t strides[3] = {(cuuint64_t)c.head_dim * 2, 128, (cuuint64_t)h->cap * c.head_dim * 2};
  const cuuint32_t box[4] = {64, 64, (cuuint32_t)(c.head_dim / 64), 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, base, dims, strides, box, estr,
                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH_OK : DFLASH_ECUDA;
}

bool mat_ok(const dflash_matrix& m, int fmt) {
  if (!m.data) return false;
  if (fmt == FMT_Q4 && (!m.scale || !m.bias)) return false;
  return true;
}

RepackSrc src_of(const dflash_matrix& m, int rows) {
  return RepackSrc{m.data, static_cast<const uint16_t*>(m.scale), static_cast<const uint16_t*>(m.bias), rows};
}

int repack(dflash_handle* h, const PackedMat& dst, const RepackSrc* srcs, int n_src, int interleave, cudaStream_t s) {
  RepackArgs a{};
  for (int i = 0; i < n_src; i++) a.src[i] = srcs[i];
  a.n_src = n_src;
  a.interleave = interleave;
  a.fmt = h->fmt;
  a.k = dst.k;
  a.n_strips = dst.n_strips;
  a.dst = dst.w;
  h->launches++;
  return status_of(launch_repack(a, s));
}

// ---- one GEMV over rows [0, R) ------------------------------------------------------------------
struct GemvCall {
  const PackedMat* m;
  int strip0 = 0, n_strips = -1;
  int R = 0;
  const void* x = nullptr;
  int ldx = 0;
  RowMap xmap{1 << 30, 0, 0};
  int x_bf16 = 0;
  long long x_lo_off = 0;   // f16 remainder rows of x (tensor-core path only)
  int norm_mode = NORM_NONE;
  const float* ssq = nullptr;
  int ssq_ld = 0, ssq_parts = 0;
  float inv_dim = 1.f;
  int epi = EPI_STORE;
  EpiArgs e{};
  int grp_n = 1;                 // grouped launch of grp_n equally shaped problems
  long long grp_w_stride = 0, grp_x_stride = 0;
  const float* x_colscale = nullptr;
  long long x_colscale_grp_stride = 0;
};

// Live per-kernel timing (dflash_set_probe): events around the first launch of the chosen kind.
void probe_begin(dflash_handle* h, int kind, cudaStream_t s) {
  if (h->probe_start && h->probe_kernel == kind) cudaEventRecord(h->probe_start, s);
}
void probe_end(dflash_handle* h, int kind, cudaStream_t s) {
  if (h->probe_stop && h->probe_kernel == kind) {
    cudaEventRecord(h->probe_stop, s);
    h->probe_start = h->probe_stop = nullptr;
  }
}

size_t xn_lo(const dflash_handle* h) { return h->act_f32 ? 0 : (size_t)h->r_blk * h->d; }
size_t xw_lo(const dflash_handle* h) { return h->act_f32 ? 0 : (size_t)h->L * h->xw_rows * h->d; }


int run_gemv(dflash_handle* h, GemvCall& c, cudaStream_t s, GemvPlan* plan_out = nullptr) {
  const PackedMat& m = *c.m;
  const int strips = c.n_strips < 0 ? m.n_strips : c.n_strips;
  if (c.R <= 0 || strips <= 0) return DFLASH_OK;
  if (h->act_f32) c.x_lo_off = 0;
  const int grp = h->act_f32 ? 1 : std::max(1, c.grp_n);
  const GemvPlan p = plan_gemv(h, strips, m.groups, c.R, c.x_lo_off != 0, std::max(1, h->n_sm / grp),
                               !h->act_f32 && c.epi != EPI_LMHEAD, c.epi == EPI_LMHEAD);
  if (plan_out) *plan_out = p;
  GemvArgs a{};
  a.w = m.w;
  a.grp_n = grp;
  a.grp_ctas = p.grid;
  a.grp_w_stride = c.grp_w_stride;
  a.grp_x_stride = c.grp_x_stride;
  a.cluster2 = p.cluster2;
  a.cpart_cap = p.cpart_cap;
  a.x_colscale = h->act_f32 ? nullptr : c.x_colscale;
  a.x_colscale_grp_stride = c.x_colscale_grp_stride;
  a.strip0 = c.strip0;
  a.n_strips = strips;
  a.k = m.k;
  a.groups = m.groups;
  a.n_slices = p.n_slices;
  a.gps = p.gps;
  a.ctas_per_slice = p.ctas_per_slice;
  a.R = c.R;
  a.x = c.x;
  a.ldx = c.ldx;
  a.xmap = c.xmap;
  a.x_bf16 = c.x_bf16;
  a.x_lo_off = c.x_lo_off;
  a.norm_mode = c.norm_mode;
  a.ssq = c.ssq;
  a.ssq_ld = c.ssq_ld;
  a.ssq_parts = c.ssq_parts;
  a.inv_dim = c.inv_dim;
  a.eps = h->cfg.eps;
  a.partials = h->partials;
  a.tickets = h->tickets;
  a.err = h->err;
  a.stall_cta1 = h->fmt == FMT_F32 ? 0 : h->stall_active;
  a.e = c.e;
  if (c.epi == EPI_LMHEAD) {
    a.e.lm_part = h->lm_part;
    a.e.lm_strip = h->lm_strip;
  }
  h->launches++;
  return status_of(launch_gemv(h->fmt, c.epi, nt_for(c.R), a, p.grid * grp, s));
}

// Many-row draft calls: one tcgen05 contraction over rows [0, rows) of x (f16 [rows][ldx], the
// f16 remainder at element offset lo_off when nonzero) into the handle's scratch (partial tiles).
int run_tc05_parts(dflash_handle* h, const PackedMat& m, int rows, const void* x, int ldx, long long lo_off,
                   cudaStream_t s, Tc05Plan* out) {
  const Tc05Plan p = plan_tc05(m.n_strips, m.groups, rows, lo_off != 0, h->n_sm);
  if (p.npad == 0 || p.scratch > h->tc05_scratch_bytes) return DFLASH_EINVAL;
  const void* xl = lo_off ? static_cast<const void*>(static_cast<const __half*>(x) + lo_off) : nullptr;
  Tc05Args a{};
  if (make_rows_map_groups(x, m.k, rows, ldx, p.npad, p.kx, 1, 0, &a.xmap) != DFLASH_OK) return DFLASH_ECUDA;
  if (xl && make_rows_map_groups(xl, m.k, rows, ldx, p.npad, p.kx, 1, 0, &a.xlmap) != DFLASH_OK) return DFLASH_ECUDA;
  if (make_q4_tile_map(m, p.tiles_big, kTcKW, 1, 0, &a.wmap) != DFLASH_OK ||
      make_q4_tile_map(m, p.tiles_small, kTcKW, 1, 0, &a.wmap_small) != DFLASH_OK)
    return DFLASH_ECUDA;
  a.w = m.w;
  a.part = reinterpret_cast<float*>(h->tc05_scratch + p.part_off);
  a.err = h->err;
  a.n_strips = m.n_strips;
  a.groups = m.groups;
  tc05_fill_args(p, xl != nullptr, a);
  *out = p;
  h->launches += 1;
  return status_of(launch_tc05_parts(a, p, s));
}

// The epilogue arguments of one row chunk of a projection (described as for run_gemv) on the
// contraction's partial tiles; an LM-head chunk's vocab states go to its own slice of lm_part.
GemvArgs tc05_epi_args(dflash_handle* h, const GemvCall& c, int chunk, int grid) {
  const PackedMat& m = *c.m;
  GemvArgs a{};
  a.w = m.w;
  a.strip0 = c.epi == EPI_KV ? c.strip0 : 0;   // the context K/V strips of a Q/K/V matrix
  a.n_strips = c.epi == EPI_KV ? c.n_strips : m.n_strips;
  a.k = m.k;
  a.groups = m.groups;
  a.n_slices = 1;
  a.gps = m.groups;
  a.ctas_per_slice = 1;
  a.R = c.R;
  a.xmap = c.xmap;
  a.norm_mode = c.norm_mode;
  a.ssq = c.ssq;
  a.ssq_ld = c.ssq_ld;
  a.ssq_parts = c.ssq_parts;
  a.inv_dim = c.inv_dim;
  a.eps = h->cfg.eps;
  a.err = h->err;
  a.e = c.e;
  if (c.epi == EPI_LMHEAD) {
    a.e.lm_part = h->lm_part + (size_t)chunk * grid * kMaxRows * 3;
    a.e.lm_strip = h->lm_strip;
  }
  return a;
}

int tc05_epi_grid(const dflash_handle* h, const GemvCall& c) {
  const int strips = c.epi == EPI_KV ? c.n_strips : c.m->n_strips;
  const int grid = (strips + kF32Warps - 1) / kF32Warps;
  return std::max(1, std::min(grid, c.epi == EPI_LMHEAD ? h->lm_grid_max : 4 * h->n_sm));
}

// The epilogues of n row chunks of one projection from the contraction's partial tiles, one launch;
// chunk j's row c is contraction row r0[j] + map_row(calls[j].xmap, c).
int run_tc05_epi_chunks(dflash_handle* h, const GemvCall* calls, const int* r0, int n, const Tc05Plan& p,
                        cudaStream_t s, int* grid_out = nullptr) {
  if (n <= 0) return DFLASH_OK;
  if (n > kTcMaxChunks) return DFLASH_EINVAL;
  static thread_local Tc05EpiChunks ch;   // ~6 KB of launch arguments
  const int grid = tc05_epi_grid(h, calls[0]);
  int nt = 1;
  for (int j = 0; j < n; j++) {
    ch.a[j] = tc05_epi_args(h, calls[j], j, grid);
    ch.row_base[j] = r0[j];
    nt = std::max(nt, nt_for(calls[j].R));
  }
  ch.n = n;
  if (grid_out) *grid_out = grid;
  h->launches += 2;   // the rows' norm scales, then the epilogue
  return status_of(launch_tc05_epilogue(calls[0].epi, nt, ch,
                                        reinterpret_cast<const float*>(h->tc05_scratch + p.part_off), p.slices,
                                        p.npad, p.mtiles * 128, grid,
                                        reinterpret_cast<float*>(h->tc05_scratch + p.srow_off), 1, 0, s));
}

// The epilogue of one chunk of a projection (the context projection's chunks).
int run_tc05_epi(dflash_handle* h, const GemvCall& c, const Tc05Plan& p, int row_base, cudaStream_t s) {
  if (c.R <= 0) return DFLASH_OK;
  return run_tc05_epi_chunks(h, &c, &row_base, 1, p, s);
}

// The context K/V of `rows` context rows for every layer, on the tcgen05 contraction: one launch
// makes layer i's input plane of xw (x * ctx_norm * attn_norm_i, f16 and its remainder) from the
// context epilogue's plane, one grouped launch contracts the K/V strips of each layer's Q/K/V
// matrix with its plane, then one epilogue launch (grid.z = layer)
// that scales by the rows' norm and appends to each layer's ring cache. calls[j] describes chunk j
// (contraction rows r0[j] ...) as for the GEMV.
int run_tc05_kv(dflash_handle* h, int rows, const GemvCall* calls, const int* r0, int n, cudaStream_t s) {
  const int L = h->L;
  const Tc05Plan p = plan_kv_tc05(h, rows);
  if (p.npad == 0 || n < 1 || n > kTcMaxChunks) return DFLASH_EINVAL;
  const size_t layer_bytes = p.srow_off;   // one layer's partial tiles
  if ((size_t)L * layer_bytes + (p.scratch - p.srow_off) > h->tc05_scratch_bytes) return DFLASH_EINVAL;
  const PackedMat& m = h->qkv[0];
  const int lo = (DFL_LO_MASK & LO_CTXKV) ? 1 : 0;
  const size_t plane = (size_t)h->xw_rows * h->d * 2;   // bytes between the layers' input planes
  const size_t w_stride = L > 1 ? (size_t)(h->qkv[1].w - h->qkv[0].w) : 0;
  Tc05Args a{};
  if (make_rows_map_groups(h->xw, h->d, rows, h->d, p.npad, p.kx, L, plane, &a.xmap) != DFLASH_OK) return DFLASH_ECUDA;
  if (lo && make_rows_map_groups(static_cast<const __half*>(h->xw) + xw_lo(h), h->d, rows, h->d, p.npad, p.kx, L,
                                 plane, &a.xlmap) != DFLASH_OK)
    return DFLASH_ECUDA;
  if (make_q4_tile_map(m, p.tiles_big, kTcKW, L, w_stride, &a.wmap) != DFLASH_OK ||
      make_q4_tile_map(m, p.tiles_small, kTcKW, L, w_stride, &a.wmap_small) != DFLASH_OK)
    return DFLASH_ECUDA;
  h->launches++;
  int st = status_of(launch_tc05_kv_planes(h->xw, (long long)xw_lo(h), h->attn_norm, rows, h->d, L,
                                           (long long)h->xw_rows * h->d, s));
  if (st) return st;
  a.w = m.w;
  a.part = reinterpret_cast<float*>(h->tc05_scratch);
  a.err = h->err;
  a.n_strips = (2 * h->kvd) / 16;
  a.groups = m.groups;
  tc05_fill_args(p, lo, a);
  a.n_layers = L;
  a.w_strip0 = h->qd / 16;
  a.part_layer_stride = layer_bytes / 4;
  h->launches++;
  st = status_of(launch_tc05_parts(a, p, s));
  if (st) return st;
  static thread_local Tc05EpiChunks ch;
  const int grid = tc05_epi_grid(h, calls[0]);
  int nt = 1;
  for (int j = 0; j < n; j++) {
    ch.a[j] = tc05_epi_args(h, calls[j], j, grid);
    ch.row_base[j] = r0[j];
    nt = std::max(nt, nt_for(calls[j].R));
  }
  ch.n = n;
  h->launches += 2;   // the rows' norm scales, then the epilogue
  return status_of(launch_tc05_epilogue(EPI_KV, nt, ch, a.part, p.slices, p.npad, p.mtiles * 128, grid,
                                        reinterpret_cast<float*>(h->tc05_scratch + (size_t)L * layer_bytes), L,
                                        layer_bytes / 4, s));
}

// One projection of a draft call of at most kProjMaxRows block rows on the tcgen05 projection
// kernel: the contraction runs over rows [0, rows) of x (f16 [rows][ldx], the f16 remainder at
// element offset lo_off when nonzero); the epilogue (described as for run_gemv) reads contraction
// row row_base + map_row(c.xmap, r) for its row r.
int run_proj(dflash_handle* h, const GemvCall& c, int rows, const void* x, int ldx, long long lo_off, int row_base,
             cudaStream_t s) {
  const PackedMat& m = *c.m;
  if (c.R <= 0) return DFLASH_OK;
  const ProjPlan p = plan_proj_tc05(m.n_strips, m.groups, rows, lo_off != 0, h->n_sm);
  if (p.npad == 0 || p.grid > h->n_sm || p.mtiles > h->ticket_count) return DFLASH_EINVAL;
  ProjArgs pa{};
  const void* xl = lo_off ? static_cast<const void*>(static_cast<const __half*>(x) + lo_off) : nullptr;
  if (make_rows_map(x, m.k, rows, ldx, p.npad, &pa.xmap) != DFLASH_OK) return DFLASH_ECUDA;
  if (xl && make_rows_map(xl, m.k, rows, ldx, p.npad, &pa.xlmap) != DFLASH_OK) return DFLASH_ECUDA;
  GemvArgs& a = pa.g;
  a.w = m.w;
  a.strip0 = 0;
  a.n_strips = m.n_strips;
  a.k = m.k;
  a.groups = m.groups;
  a.n_slices = c.epi == EPI_LMHEAD ? 2 : 1;   // LM head: one vocab state per strip, merged in strip order
  a.gps = m.groups;
  a.ctas_per_slice = 1;
  a.R = c.R;
  a.xmap = c.xmap;
  a.norm_mode = c.norm_mode;
  a.ssq = c.ssq;
  a.ssq_ld = c.ssq_ld;
  a.ssq_parts = c.ssq_parts;
  a.inv_dim = c.inv_dim;
  a.eps = h->cfg.eps;
  a.err = h->err;
  a.e = c.e;
  if (c.epi == EPI_LMHEAD) {
    a.e.lm_part = h->lm_part;
    a.e.lm_strip = h->lm_strip;
  }
  pa.w = m.w;
  pa.partials = h->pj_partials;
  pa.tickets = h->tickets;
  pa.n_strips = m.n_strips;
  pa.groups = m.groups;
  pa.mtiles = p.mtiles;
  pa.npad = p.npad;
  pa.has_lo = xl != nullptr;
  pa.sa = p.sa;
  pa.sx = p.sx;
  pa.sw = p.sw;
  pa.tmem_cols = p.tmem_cols;
  pa.row_base = row_base;
  pa.x_stage = p.x_stage;
  h->launches++;
  return status_of(launch_proj_tc05(c.epi, nt_for(c.R), pa, p, s));
}

}  // namespace

extern "C" {

size_t dflash_workspace_bytes(const dflash_config* cfg) {
  if (!valid_config(cfg)) return 0;
  dflash_handle* h = new (std::nothrow) dflash_handle();
  if (!h) return 0;
  init_dims(h, cfg);
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, dev);
  const size_t b = carve(h, nullptr);
  delete h;
  return b;
}

int dflash_create(const dflash_config* cfg, const dflash_weights* w, void* workspace, size_t workspace_bytes,
                  void* stream, dflash_handle** out) {
  if (!out) return DFLASH_EINVAL;
  *out = nullptr;
  if (!valid_config(cfg) || !w || !workspace || (reinterpret_cast<uintptr_t>(workspace) & 255)) return DFLASH_EINVAL;
  dflash_handle* h = new (std::nothrow) dflash_handle();
  if (!h) return DFLASH_EINVAL;
  init_dims(h, cfg);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    delete h;
    return DFLASH_ECUDA;
  }
  const size_t need = carve(h, nullptr);
  if (workspace_bytes < need) {
    delete h;
    return DFLASH_ECAPACITY;
  }
  h->ws_bytes = carve(h, static_cast<uint8_t*>(workspace));
  for (int i = 2; i < h->L; i++)   // grouped launches rely on equally spaced per-layer matrices
    if (h->qkv[i].w - h->qkv[0].w != i * (h->qkv[1].w - h->qkv[0].w)) {
      delete h;
      return DFLASH_EINVAL;
    }

  const int f = h->fmt;
  bool ok = mat_ok(w->w_c, f) && mat_ok(w->embed, f) && mat_ok(w->lm_head, f) && w->ctx_norm && w->block_pos &&
            w->out_norm && (h->G < 2 || w->mask_emb);
  if (h->d != h->H) ok = ok && mat_ok(w->tok_proj, f) && mat_ok(w->out_proj, f);
  if (cfg->markov_rank) ok = ok && mat_ok(w->markov_w1, f) && mat_ok(w->markov_w2t, f);
  for (int i = 0; i < h->L && ok; i++) {
    const dflash_layer_weights& l = w->layer[i];
    ok = mat_ok(l.wq, f) && mat_ok(l.wk, f) && mat_ok(l.wv, f) && mat_ok(l.wo, f) && mat_ok(l.w_gate, f) &&
         mat_ok(l.w_up, f) && mat_ok(l.w_down, f) && l.attn_norm && l.ff_norm;
  }
  if (!ok) {
    delete h;
    return DFLASH_EINVAL;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int st = DFLASH_OK;
  auto chk = [&](int r) {
    if (st == DFLASH_OK) st = r;
  };
  // zero everything after the weights (caches, activations, tickets, error word)
  chk(status_of(cudaMemsetAsync(h->kc, 0, h->ws_bytes - (static_cast<uint8_t*>(h->kc) - static_cast<uint8_t*>(workspace)), s)));
  {
    RepackSrc a = src_of(w->w_c, h->d);
    chk(repack(h, h->wc, &a, 1, 0, s));
  }
  for (int i = 0; i < h->L; i++) {
    const dflash_layer_weights& l = w->layer[i];
    RepackSrc qkv[3] = {src_of(l.wq, h->qd), src_of(l.wk, h->kvd), src_of(l.wv, h->kvd)};
    chk(repack(h, h->qkv[i], qkv, 3, 0, s));
    RepackSrc o = src_of(l.wo, h->d);
    chk(repack(h, h->wo[i], &o, 1, 0, s));
    RepackSrc gu[2] = {src_of(l.w_gate, h->I), src_of(l.w_up, h->I)};
    chk(repack(h, h->gu[i], gu, 2, 1, s));
    RepackSrc dn = src_of(l.w_down, h->d);
    chk(repack(h, h->down[i], &dn, 1, 0, s));
    chk(status_of(cudaMemcpyAsync(h->attn_norm + (size_t)i * h->d, l.attn_norm, h->d * 4, cudaMemcpyDefault, s)));
    chk(status_of(cudaMemcpyAsync(h->ff_norm + (size_t)i * h->d, l.ff_norm, h->d * 4, cudaMemcpyDefault, s)));
  }
  if (h->d != h->H) {
    RepackSrc t = src_of(w->tok_proj, h->d), o = src_of(w->out_proj, h->H);
    chk(repack(h, h->tok, &t, 1, 0, s));
    chk(repack(h, h->outp, &o, 1, 0, s));
  }
  {
    RepackSrc l = src_of(w->lm_head, h->V);
    chk(repack(h, h->lm, &l, 1, 0, s));
  }
  if (cfg->markov_rank) {
    RepackSrc mk = src_of(w->markov_w2t, h->V);
    chk(repack(h, h->mk, &mk, 1, 0, s));
    h->mk_w1 = w->markov_w1;
  }
  chk(status_of(cudaMemcpyAsync(h->ctx_norm, w->ctx_norm, h->d * 4, cudaMemcpyDefault, s)));
  if (h->G > 1)
    chk(status_of(cudaMemcpyAsync(h->mask_emb, w->mask_emb, (size_t)(h->G - 1) * h->d * 4, cudaMemcpyDefault, s)));
  chk(status_of(cudaMemcpyAsync(h->block_pos, w->block_pos, (size_t)h->G * h->d * 4, cudaMemcpyDefault, s)));
  chk(status_of(cudaMemcpyAsync(h->out_norm, w->out_norm, h->d * 4, cudaMemcpyDefault, s)));
  h->embed = w->embed;
  if (!h->act_f32 && st == DFLASH_OK) {
    chk(make_cache_map(h, h->kc, &h->kmap));
    chk(make_cache_map(h, h->vc, &h->vmap));
  }
  if (st != DFLASH_OK) {
    delete h;
    return st;
  }
  *out = h;
  return DFLASH_OK;
}

int dflash_project_ctx(dflash_handle* h, int n_req, const int32_t* req_ids, const int32_t* n_new, const void* taps,
                       void* stream) {
  if (!h || n_req < 0 || n_req > h->cfg.max_batch) return DFLASH_EINVAL;
  if (n_req == 0) return DFLASH_OK;
  if (!req_ids || !n_new) return DFLASH_EINVAL;
  bool seen[DFLASH_MAX_BATCH] = {};
  int64_t total = 0;
  for (int i = 0; i < n_req; i++) {
    const int r = req_ids[i];
    if (r < 0 || r >= h->cfg.max_batch || seen[r] || n_new[i] < 0) return DFLASH_EINVAL;
    seen[r] = true;
    total += n_new[i];
    if (h->cfg.window == 0 && h->ctx_len[r] + n_new[i] > h->cfg.ctx_capacity) return DFLASH_ECAPACITY;
  }
  if (total == 0) return DFLASH_OK;
  if (!taps) return DFLASH_EINVAL;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t ab = h->act_bytes;
  const uint8_t* tp = static_cast<const uint8_t*>(taps);
  const int parts = h->ssq_ld;
  const size_t layer_cache = (size_t)h->cfg.max_batch * h->cfg.n_kv_heads * h->cap * h->cfg.head_dim * ab;

  // rows in call order: (slot, position)
  int req_i = 0, j_in = 0;
  int64_t row = 0;
  // many rows: W_c runs once per kTcMaxRows rows on the tcgen05 contraction (a whole number of
  // chunks), then each chunk's epilogue and its context K/V launch as below
  const bool tc = h->tc05_on && total > kMaxCtxChunk;
  // the grouped context K/V appends a whole block's rows in one launch, so no request may wrap its
  // ring within the call (later rows must overwrite earlier ones in order: the chunked path then)
  int max_new = 0;
  for (int i = 0; i < n_req; i++) max_new = std::max(max_new, (int)n_new[i]);
  const bool tc_kv = tc && max_new <= h->cap;
  Tc05Plan wcp{};
  int64_t tc_row0 = 0;
  int tc_rows = 0;
  GemvCall kv_calls[kTcMaxChunks];   // the tcgen05 block's context K/V epilogues, one per 32-row chunk
  int kv_r0[kTcMaxChunks], n_kv = 0;
  while (row < total) {
    if (tc && (row == 0 || row - tc_row0 >= kTcMaxRows)) {
      tc_row0 = row;
      const int rows = (int)std::min<int64_t>(kTcMaxRows, total - row);
      tc_rows = rows;
      n_kv = 0;
      probe_begin(h, DFLASH_PROBE_WC, s);   // the block's W_c: contraction and every chunk's epilogue
      h->launches++;
      int st = status_of(launch_bf16_to_f16(tp + (size_t)row * h->mH * ab, (long long)rows * h->mH, h->tc05_taps, s));
      if (!st) st = run_tc05_parts(h, h->wc, rows, h->tc05_taps, h->mH, 0, s, &wcp);
      if (st) return st;
    }
    const int rc = (int)std::min<int64_t>(kMaxCtxChunk, total - row);
    int slots[kMaxCtxChunk], pos[kMaxCtxChunk];
    for (int r = 0; r < rc; r++) {
      while (j_in >= n_new[req_i]) {
        req_i++;
        j_in = 0;
      }
      slots[r] = req_ids[req_i];
      pos[r] = (int)((h->ctx_len[req_ids[req_i]] + j_in) % h->cap);
      j_in++;
    }
    // Eq 2: x = W_c taps; epilogue writes x*ctx_norm*attn_norm_i for every layer + sums of squares
    GemvCall c1;
    c1.m = &h->wc;
    c1.R = rc;
    c1.x = tp + (size_t)row * h->mH * ab;
    c1.ldx = h->mH;
    c1.x_bf16 = !h->act_f32;   // caller taps are bf16; the tensor-core path computes in f16
    c1.epi = EPI_CTX;
    c1.e.row_base = 0;
    c1.e.n_rows = h->d;
    c1.e.ldo = h->d;
    c1.e.ctx_norm = h->ctx_norm;
    // tensor-core path: one row x * ctx_norm, the K/V launch applies attn_norm_i to its input
    // (the tcgen05 block: its rows at their offset in the block, every layer's plane made from
    // them before the grouped K/V); CUDA-core path: one input row per layer
    const size_t blk = tc_kv ? (size_t)(row - tc_row0) : 0;
    c1.e.attn_norms = h->act_f32 ? h->attn_norm : nullptr;
    c1.e.n_layers = h->L;
    c1.e.xw = static_cast<uint8_t*>(h->xw) + blk * h->d * ab;
    c1.e.xw_rows = h->xw_rows;
    c1.e.x_lo_off = xw_lo(h);
    c1.e.ssq_out = h->ssq_ctx + blk * h->ssq_ld * 2;
    c1.e.ssq_ld = h->ssq_ld;
    if (!tc) probe_begin(h, DFLASH_PROBE_WC, s);
    int st = tc ? run_tc05_epi(h, c1, wcp, (int)(row - tc_row0), s) : run_gemv(h, c1, s);
    if (st) return st;
    if (!tc || row + rc == tc_row0 + tc_rows) probe_end(h, DFLASH_PROBE_WC, s);
    // per layer: K_i, V_i of RMSNorm_attn_i(RMSNorm_ctx(x)), appended to the ring cache; the
    // tensor-core path runs every layer in one grouped launch over the same input rows (the
    // layers' packed Q/K/V matrices and caches are equally spaced; attn_norm_i scales the input)
    const bool grouped = !h->act_f32;
    for (int i = 0; i < (grouped ? 1 : h->L); i++) {
      GemvCall c2;
      if (!h->act_f32 && !tc_kv) {
        c2.grp_n = h->L;
        c2.grp_w_stride = h->L > 1 ? h->qkv[1].w - h->qkv[0].w : 0;
        c2.grp_x_stride = 0;   // the same input rows, scaled per layer by attn_norm_i
        c2.x_colscale = h->attn_norm;
        c2.x_colscale_grp_stride = h->d;
        c2.e.kv_grp_stride = (long long)layer_cache;
      }
      c2.m = &h->qkv[i];
      c2.strip0 = h->qd / 16;
      c2.n_strips = (2 * h->kvd) / 16;
      c2.R = rc;
      c2.x = static_cast<const uint8_t*>(h->xw) + (grouped ? 0 : (size_t)i * h->xw_rows * h->d * ab);
      c2.ldx = h->d;
      c2.x_lo_off = lo_if(LO_CTXKV, xw_lo(h));
      c2.norm_mode = NORM_CTX;
      c2.ssq = h->ssq_ctx + blk * h->ssq_ld * 2;
      c2.ssq_ld = h->ssq_ld;
      c2.ssq_parts = parts;
      c2.inv_dim = 1.f / h->d;
      c2.epi = EPI_KV;
      c2.e.row_base = h->qd;
      c2.e.n_rows = 2 * h->kvd;
      c2.e.kc = static_cast<uint8_t*>(h->kc) + i * layer_cache;
      c2.e.vc = static_cast<uint8_t*>(h->vc) + i * layer_cache;
      c2.e.cap = h->cap;
      c2.e.hd = h->cfg.head_dim;
      c2.e.n_kv = h->cfg.n_kv_heads;
      c2.e.kvd = h->kvd;
      for (int r = 0; r < rc; r++) {
        c2.e.kv_slot[r] = slots[r];
        c2.e.kv_pos[r] = pos[r];
      }
      if (tc_kv) {
        // every layer's K/V of the whole tcgen05 block at once, after its last chunk
        c2.e.kv_grp_stride = (long long)layer_cache;
        kv_calls[n_kv] = c2;
        kv_r0[n_kv] = (int)blk;
        n_kv++;
        if (row + rc == tc_row0 + tc_rows) {
          probe_begin(h, DFLASH_PROBE_CTX_KV, s);
          st = run_tc05_kv(h, tc_rows, kv_calls, kv_r0, n_kv, s);
          if (st) return st;
          probe_end(h, DFLASH_PROBE_CTX_KV, s);
        }
        continue;
      }
      probe_begin(h, DFLASH_PROBE_CTX_KV, s);
      st = run_gemv(h, c2, s);
      if (st) return st;
      probe_end(h, DFLASH_PROBE_CTX_KV, s);
    }
    row += rc;
  }
  for (int i = 0; i < n_req; i++) h->ctx_len[req_ids[i]] += n_new[i];
  h->stats.ctx_rows += (uint64_t)total;
  return DFLASH_OK;
}

int dflash_draft_block(dflash_handle* h, int n_req, const int32_t* req_ids, const int32_t* anchor, float temperature,
                       int32_t* draft, float* conf, float* logits, void* stream) {
  if (!h) return DFLASH_EINVAL;
  if (temperature != 0.0f || disabled_by_env()) {
    h->stats.declined++;
    return DFLASH_DECLINED;
  }
  if (n_req < 0 || n_req > h->cfg.max_batch) return DFLASH_EINVAL;
  if (n_req == 0) return DFLASH_OK;
  if (!req_ids || !anchor || !draft) return DFLASH_EINVAL;
  bool seen[DFLASH_MAX_BATCH] = {};
  for (int i = 0; i < n_req; i++) {
    const int r = req_ids[i];
    if (r < 0 || r >= h->cfg.max_batch || seen[r]) return DFLASH_EINVAL;
    seen[r] = true;
  }
  // an armed stall (test hook) applies to this call's projection launches only
  struct StallScope {
    dflash_handle* h;
    explicit StallScope(dflash_handle* hh) : h(hh) {
      h->stall_active = h->stall_armed;
      h->stall_armed = 0;
    }
    ~StallScope() { h->stall_active = 0; }
  } stall_scope(h);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const dflash_config& c = h->cfg;
  const size_t ab = h->act_bytes;
  const int G = h->G, n = h->nd, d = h->d;   // n drafting rows per request: the last n block rows
  const int parts = h->ssq_ld;
  const size_t layer_cache = (size_t)c.max_batch * c.n_kv_heads * h->cap * c.head_dim * ab;
  auto off = [&](void* p, size_t rows, size_t width) -> void* {
    return static_cast<uint8_t*>(p) + rows * width * ab;
  };
  int st = DFLASH_OK;

  // block construction
  BlockArgs ba{};
  ba.n_req = n_req;
  ba.gamma = G;
  ba.d = d;
  ba.H = h->H;
  ba.vocab = h->V;
  ba.fmt = h->fmt;
  ba.act_f32 = h->act_f32;
  ba.anchor = anchor;
  ba.emb = h->embed.data;
  ba.emb_scale = static_cast<const uint16_t*>(h->embed.scale);
  ba.emb_bias = static_cast<const uint16_t*>(h->embed.bias);
  ba.mask_emb = h->mask_emb;
  ba.block_pos = h->block_pos;
  ba.attn_norm0 = h->attn_norm;
  ba.h = h->h;
  ba.xn = h->xn;
  ba.ssq = h->ssq;
  ba.ssq_ld = h->ssq_ld;
  ba.xn_lo_off = xn_lo(h);
  ba.emb_out = h->emb;
  ba.err = h->err;
  if (d != h->H) {
    h->launches++;
    if ((st = status_of(launch_embed_gather(ba, s)))) return st;
    for (int b0 = 0; b0 < n_req; b0 += kMaxRows) {
      const int rb = std::min(kMaxRows, n_req - b0);
      GemvCall ct;
      ct.m = &h->tok;
      ct.R = rb;
      ct.x = off(h->emb, b0, h->H);
      ct.ldx = h->H;
      ct.epi = EPI_STORE;
      ct.e.n_rows = d;
      ct.e.out = h->tokrow + (size_t)b0 * d;
      ct.e.ldo = d;
      ct.e.out_f32 = 1;
      if ((st = run_gemv(h, ct, s))) return st;
    }
    ba.tokrow = h->tokrow;
  }
  h->launches++;
  if ((st = status_of(launch_block_init(ba, s)))) return st;

  const int req_per_chunk = std::max(1, kMaxRows / G);
  // many rows: each projection runs once over all block rows on the tcgen05 contraction, then
  // its epilogue per chunk (the chunks' row scales, residuals and outputs are those of the GEMV)
  const int rows_all = n_req * G;
  const bool tc = h->tc05_on && rows_all > kMaxRows && rows_all <= h->tc05_rows;
  // at most 32 rows: each projection is one launch of the tcgen05 projection kernel (config
  // skinny_tc05), its contraction over all block rows, its epilogue over the chunk's rows
  const bool pj = h->pj_on && rows_all <= kProjMaxRows;
  Tc05Plan tp{};
  const void* px = nullptr;   // the projection's input rows and remainder offset (pj)
  int pldx = 0;
  long long plo = 0;
  // tcgen05 contraction: a projection's row chunks are collected and get one epilogue launch
  GemvCall tc_calls[kTcMaxChunks];
  int tc_r0[kTcMaxChunks], tc_n = 0;
  auto project = [&](GemvCall& c, int r0) {
    if (pj) return run_proj(h, c, rows_all, px, pldx, plo, r0, s);
    if (!tc) return run_gemv(h, c, s);
    if (tc_n == kTcMaxChunks) return (int)DFLASH_EINVAL;
    tc_calls[tc_n] = c;
    tc_r0[tc_n++] = r0;
    return (int)DFLASH_OK;
  };
  auto flush = [&](int* grid_out = nullptr) {
    const int n_chunks = tc_n;
    tc_n = 0;
    return tc ? run_tc05_epi_chunks(h, tc_calls, tc_r0, n_chunks, tp, s, grid_out) : (int)DFLASH_OK;
  };
  for (int i = 0; i < h->L; i++) {
    const int in_parts = i == 0 ? (d + kBlockCols - 1) / kBlockCols : parts;
    // Q, K_d, V_d of RMSNorm_attn_i(H_d)
    if (i == 0) probe_begin(h, DFLASH_PROBE_QKV, s);
    if (tc && (st = run_tc05_parts(h, h->qkv[i], rows_all, h->xn, d, lo_if(LO_QKV, xn_lo(h)), s, &tp))) return st;
    px = h->xn, pldx = d, plo = lo_if(LO_QKV, xn_lo(h));
    for (int b0 = 0; b0 < n_req; b0 += req_per_chunk) {
      const int nb = std::min(req_per_chunk, n_req - b0), r0 = b0 * G;
      GemvCall cq;
      cq.m = &h->qkv[i];
      cq.R = nb * G;
      cq.x = off(h->xn, r0, d);
      cq.ldx = d;
      cq.x_lo_off = lo_if(LO_QKV, xn_lo(h));
      cq.norm_mode = NORM_ONE;
      cq.ssq = h->ssq + (size_t)r0 * h->ssq_ld;
      cq.ssq_ld = h->ssq_ld;
      cq.ssq_parts = in_parts;
      cq.inv_dim = 1.f / d;
      cq.epi = EPI_QKV;
      cq.e.n_rows = h->qd + 2 * h->kvd;
      cq.e.q = off(h->q, r0, h->qd);
      cq.e.kb = off(h->kb, r0, h->kvd);
      cq.e.vb = off(h->vb, r0, h->kvd);
      cq.e.qd = h->qd;
      cq.e.kvd = h->kvd;
      if ((st = project(cq, r0))) return st;
    }
    if ((st = flush())) return st;
    if (i == 0) probe_end(h, DFLASH_PROBE_QKV, s);
    // attention over [windowed context ++ block], no causal mask
    {
      AttnArgs aa{};
      aa.q = h->q;
      aa.kb = h->kb;
      aa.vb = h->vb;
      aa.out = h->attn;
      aa.kc = static_cast<uint8_t*>(h->kc) + i * layer_cache;
      aa.vc = static_cast<uint8_t*>(h->vc) + i * layer_cache;
      aa.qd = h->qd;
      aa.kvd = h->kvd;
      aa.hd = c.head_dim;
      aa.hq = c.n_q_heads;
      aa.hkv = c.n_kv_heads;
      aa.gamma = G;
      aa.window = c.window;
      aa.cap = h->cap;
      aa.max_batch = c.max_batch;
      aa.plane0 = i * c.max_batch * c.n_kv_heads;
      aa.n_req = n_req;
      aa.scale_log2 = (float)(1.4426950408889634 / sqrt((double)c.head_dim));
      aa.part_o = h->att_o;
      aa.part_ml = h->att_ml;
      aa.err = h->err;
      int max_tiles = 0;
      for (int b = 0; b < n_req; b++) {
        const int64_t P = h->ctx_len[req_ids[b]];
        const int64_t nw = c.window > 0 ? std::min<int64_t>(P, c.window) : P;
        aa.req[b] = AttnReq{req_ids[b], (int)P, b * G};
        max_tiles = std::max(max_tiles, (int)((nw + 63) / 64) + 1);
      }
      if (h->act_f32) {
        aa.n_splits = 1;
        h->launches++;
        if ((st = status_of(launch_attn_f32(aa, s)))) return st;
      } else {
        // about DFL_ATTN_TILES_PER_SPLIT 64-key tiles per split, up to two CTAs per SM
        const int pairs = n_req * c.n_kv_heads;
        int splits = std::max(1, (2 * h->n_sm + pairs - 1) / pairs);
        splits = std::min(splits, std::max(1, (max_tiles + DFL_ATTN_TILES_PER_SPLIT - 1) / DFL_ATTN_TILES_PER_SPLIT));
        splits = std::max(1, std::min(std::min(splits, 64), h->att_pairs_max / pairs));
        aa.n_splits = splits;
        if (i == 0) probe_begin(h, DFLASH_PROBE_ATTN, s);
        h->launches++;
        if ((st = status_of(launch_attn_tc(aa, h->kmap, h->vmap, s)))) return st;
        if (splits > 1) {
          h->launches++;
          if ((st = status_of(launch_attn_merge(aa, s)))) return st;
        }
        if (i == 0) probe_end(h, DFLASH_PROBE_ATTN, s);
      }
    }
    if (i == 0) probe_begin(h, DFLASH_PROBE_O, s);
    if (tc && (st = run_tc05_parts(h, h->wo[i], rows_all, h->attn, h->qd, 0, s, &tp))) return st;
    px = h->attn, pldx = h->qd, plo = 0;
    for (int b0 = 0; b0 < n_req; b0 += req_per_chunk) {
      const int nb = std::min(req_per_chunk, n_req - b0), r0 = b0 * G;
      // H_d += W_o attn; next input = H_d * ff_norm_i (+ sums of squares)
      GemvCall co;
      co.m = &h->wo[i];
      co.R = nb * G;
      co.x = off(h->attn, r0, h->qd);
      co.ldx = h->qd;
      co.epi = EPI_RESID;
      co.e.n_rows = d;
      co.e.ldo = d;
      co.e.h = h->h + (size_t)r0 * d;
      co.e.wnext = h->ff_norm + (size_t)i * d;
      co.e.xnext = off(h->xn, r0, d);
      co.e.x_lo_off = xn_lo(h);
      co.e.ssq_out = h->ssq + (size_t)r0 * h->ssq_ld;
      co.e.ssq_ld = h->ssq_ld;
      if ((st = project(co, r0))) return st;
    }
    if ((st = flush())) return st;
    if (i == 0) probe_end(h, DFLASH_PROBE_O, s);
    if (i == 0) probe_begin(h, DFLASH_PROBE_GATE_UP, s);
    if (tc && (st = run_tc05_parts(h, h->gu[i], rows_all, h->xn, d, lo_if(LO_GU, xn_lo(h)), s, &tp))) return st;
    px = h->xn, pldx = d, plo = lo_if(LO_GU, xn_lo(h));
    for (int b0 = 0; b0 < n_req; b0 += req_per_chunk) {
      const int nb = std::min(req_per_chunk, n_req - b0), r0 = b0 * G;
      // a = act(W_gate n2) * (W_up n2), n2 = RMSNorm_ff_i(H_d); act = SiLU or GELU (tanh form)
      GemvCall cg;
      cg.m = &h->gu[i];
      cg.R = nb * G;
      cg.x = off(h->xn, r0, d);
      cg.ldx = d;
      cg.x_lo_off = lo_if(LO_GU, xn_lo(h));
      cg.norm_mode = NORM_ONE;
      cg.ssq = h->ssq + (size_t)r0 * h->ssq_ld;
      cg.ssq_ld = h->ssq_ld;
      cg.ssq_parts = parts;
      cg.inv_dim = 1.f / d;
      cg.epi = EPI_SWIGLU;
      cg.e.n_rows = 2 * h->I;
      cg.e.act = off(h->act, r0, h->I);
      cg.e.inter = h->I;
      cg.e.ffn_act = c.ffn_act;
      if ((st = project(cg, r0))) return st;
    }
    if ((st = flush())) return st;
    if (i == 0) probe_end(h, DFLASH_PROBE_GATE_UP, s);
    if (i == 0) probe_begin(h, DFLASH_PROBE_DOWN, s);
    if (tc && (st = run_tc05_parts(h, h->down[i], rows_all, h->act, h->I, 0, s, &tp))) return st;
    px = h->act, pldx = h->I, plo = 0;
    for (int b0 = 0; b0 < n_req; b0 += req_per_chunk) {
      const int nb = std::min(req_per_chunk, n_req - b0), r0 = b0 * G;
      // H_d += W_down a; next input = H_d * (attn_norm_{i+1} | out_norm)
      GemvCall cd;
      cd.m = &h->down[i];
      cd.R = nb * G;
      cd.x = off(h->act, r0, h->I);
      cd.ldx = h->I;
      cd.epi = EPI_RESID;
      cd.e.n_rows = d;
      cd.e.ldo = d;
      cd.e.h = h->h + (size_t)r0 * d;
      cd.e.wnext = i + 1 < h->L ? h->attn_norm + (size_t)(i + 1) * d : h->out_norm;
      cd.e.xnext = off(h->xn, r0, d);
      cd.e.x_lo_off = xn_lo(h);
      cd.e.ssq_out = h->ssq + (size_t)r0 * h->ssq_ld;
      cd.e.ssq_ld = h->ssq_ld;
      if ((st = project(cd, r0))) return st;
    }
    if ((st = flush())) return st;
    if (i == 0) probe_end(h, DFLASH_PROBE_DOWN, s);
  }

  // out_norm (+ out_proj), borrowed LM head, greedy token and softmax confidence (drafting rows)
  const int lm_req_per_chunk = std::max(1, kMaxRows / n);
  probe_begin(h, DFLASH_PROBE_LM_HEAD, s);
  // many rows (d == H, no Markov head): the head over every block row once; the epilogue reads
  // the drafting rows through the chunk's row map
  if (tc && (st = run_tc05_parts(h, h->lm, rows_all, h->xn, d, lo_if(LO_LM, xn_lo(h)), s, &tp))) return st;
  for (int b0 = 0; b0 < n_req; b0 += lm_req_per_chunk) {
    const int nb = std::min(lm_req_per_chunk, n_req - b0);
    const int r0 = b0 * G, l0 = b0 * n, R = nb * n;
    GemvCall cl;
    cl.m = &h->lm;
    cl.R = R;
    if (d != h->H) {
      GemvCall cp;
      cp.m = &h->outp;
      cp.R = R;
      cp.x = off(h->xn, r0, d);
      cp.ldx = d;
      cp.x_lo_off = lo_if(LO_OUTPROJ, xn_lo(h));
      cp.xmap = RowMap{n, G, G - n};
      cp.norm_mode = NORM_ONE;
      cp.ssq = h->ssq + (size_t)r0 * h->ssq_ld;
      cp.ssq_ld = h->ssq_ld;
      cp.ssq_parts = parts;
      cp.inv_dim = 1.f / d;
      cp.epi = EPI_STORE;
      cp.e.n_rows = h->H;
      cp.e.out = h->hout;
      cp.e.ldo = h->H;
      if ((st = run_gemv(h, cp, s))) return st;
      cl.x = h->hout;
      cl.ldx = h->H;
    } else {
      cl.x = off(h->xn, r0, d);
      cl.ldx = d;
      cl.x_lo_off = lo_if(LO_LM, xn_lo(h));
      cl.xmap = RowMap{n, G, G - n};
      cl.norm_mode = NORM_ONE;
      cl.ssq = h->ssq + (size_t)r0 * h->ssq_ld;
      cl.ssq_ld = h->ssq_ld;
      cl.ssq_parts = parts;
      cl.inv_dim = 1.f / d;
    }
    cl.epi = EPI_LMHEAD;
    cl.e.n_rows = h->V;
    // with the Markov head the head's logits are only the base of the serial drafts below
    const bool markov = c.markov_rank > 0;
    cl.e.logits = markov ? h->mk_base + (size_t)l0 * h->V : (logits ? logits + (size_t)l0 * h->V : nullptr);
    cl.e.vocab = h->V;
    if (tc) {   // collected: one epilogue launch for every chunk, then one vocab merge per chunk
      if ((st = project(cl, r0))) return st;
      continue;
    }
    GemvPlan lp{};
    const bool pj_lm = pj && d == h->H;
    if (pj_lm) {
      if ((st = run_proj(h, cl, rows_all, h->xn, d, lo_if(LO_LM, xn_lo(h)), r0, s))) return st;
    } else if ((st = run_gemv(h, cl, s, &lp))) {
      return st;
    }
    if (markov) continue;
    // merge the per-CTA (one K slice) or per-strip (K split, projection kernel) vocab states
    const bool split = pj_lm || (h->fmt != FMT_F32 && lp.n_slices > 1);
    h->launches++;
    if ((st = status_of(launch_lm_reduce(split ? h->lm_strip : h->lm_part, split ? h->lm.n_strips : lp.grid, R,
                                         draft + l0, conf ? conf + l0 : nullptr, 1, s))))
      return st;
  }
  if (tc) {
    const int n_chunks = tc_n;
    int epi_grid = 0;
    if ((st = flush(&epi_grid))) return st;
    for (int j = 0; j < n_chunks && !c.markov_rank; j++) {
      const int l0 = (tc_r0[j] / G) * n;
      h->launches++;
      if ((st = status_of(launch_lm_reduce(h->lm_part + (size_t)j * epi_grid * kMaxRows * 3, epi_grid,
                                           tc_calls[j].R, draft + l0, conf ? conf + l0 : nullptr, 1, s))))
        return st;
    }
  }
  if (c.markov_rank) {
    // Markov sequential head (Eq 5 of the dflash.ts page): draft k = argmax(base_k + W1[prev_k] W2),
    // prev_0 = the anchor, prev_k = draft k-1; one gather, one rank-r GEMV (bias + argmax epilogue)
    // and one vocab merge per draft, in order
    const int r = c.markov_rank;
    const size_t lo_off = h->act_f32 ? 0 : (size_t)c.max_batch * r;
    for (int k = 0; k < n; k++) {
      for (int b0 = 0; b0 < n_req; b0 += kMaxRows) {
        const int nb = std::min(kMaxRows, n_req - b0);
        h->launches++;
        if ((st = status_of(launch_markov_gather(nb, k, n, r, h->V, h->fmt, h->mk_w1.data,
                                                 static_cast<const uint16_t*>(h->mk_w1.scale),
                                                 static_cast<const uint16_t*>(h->mk_w1.bias), anchor + b0,
                                                 draft + (size_t)b0 * n, h->mk_x, lo_off, h->err, s))))
          return st;
        GemvCall cm;
        cm.m = &h->mk;
        cm.R = nb;
        cm.x = h->mk_x;
        cm.ldx = r;
        cm.x_lo_off = (long long)lo_off;
        cm.epi = EPI_LMHEAD;
        cm.e.n_rows = h->V;
        cm.e.vocab = h->V;
        cm.e.logit_bias = h->mk_base + ((size_t)b0 * n + k) * h->V;
        cm.e.logit_row_stride = (long long)n * h->V;
        cm.e.logits = logits ? logits + ((size_t)b0 * n + k) * h->V : nullptr;
        GemvPlan mp{};
        if ((st = run_gemv(h, cm, s, &mp))) return st;
        const bool split = h->fmt != FMT_F32 && mp.n_slices > 1;
        h->launches++;
        if ((st = status_of(launch_lm_reduce(split ? h->lm_strip : h->lm_part, split ? h->mk.n_strips : mp.grid, nb,
                                             draft + (size_t)b0 * n + k, conf ? conf + (size_t)b0 * n + k : nullptr,
                                             n, s))))
          return st;
      }
    }
  }
  probe_end(h, DFLASH_PROBE_LM_HEAD, s);
  h->stats.rounds++;
  h->stats.blocks += (uint64_t)n_req;
  return DFLASH_OK;
}

int dflash_accept(dflash_handle* h, int n_req, const int32_t* draft, const int32_t* target, int32_t* accept_len,
                  int32_t* next_anchor, void* stream) {
  if (!h || n_req < 0) return DFLASH_EINVAL;
  if (n_req == 0) return DFLASH_OK;
  if (!draft || !target || !accept_len || !next_anchor) return DFLASH_EINVAL;
  h->launches++;
  h->stats.accept_calls++;
  return status_of(launch_accept(n_req, h->nd, draft, nullptr, target, accept_len, next_anchor, h->acc_hist, h->err,
                                 static_cast<cudaStream_t>(stream)));
}

int dflash_draft_lengths(dflash_handle* h, int n_req, const float* conf, const float* thresholds, float min_conf,
                         int32_t* keep, void* stream) {
  if (!h || n_req < 0) return DFLASH_EINVAL;
  if (n_req == 0) return DFLASH_OK;
  if (!conf || !keep || min_conf != min_conf) return DFLASH_EINVAL;
  h->launches++;
  return status_of(launch_draft_lengths(n_req, h->nd, conf, thresholds, min_conf, keep,
                                        static_cast<cudaStream_t>(stream)));
}

int dflash_accept_kept(dflash_handle* h, int n_req, const int32_t* draft, const int32_t* keep, const int32_t* target,
                       int32_t* accept_len, int32_t* next_anchor, void* stream) {
  if (!h || n_req < 0) return DFLASH_EINVAL;
  if (n_req == 0) return DFLASH_OK;
  if (!draft || !keep || !target || !accept_len || !next_anchor) return DFLASH_EINVAL;
  h->launches++;
  h->stats.accept_calls++;
  return status_of(launch_accept(n_req, h->nd, draft, keep, target, accept_len, next_anchor, h->acc_hist, h->err,
                                 static_cast<cudaStream_t>(stream)));
}

int dflash_reset_request(dflash_handle* h, int req_id) {
  if (!h || req_id < 0 || req_id >= h->cfg.max_batch) return DFLASH_EINVAL;
  h->ctx_len[req_id] = 0;
  return DFLASH_OK;
}

int64_t dflash_ctx_len(const dflash_handle* h, int req_id) {
  if (!h || req_id < 0 || req_id >= h->cfg.max_batch) return -1;
  return h->ctx_len[req_id];
}

int dflash_check_errors(dflash_handle* h, void* stream) {
  if (!h) return DFLASH_EINVAL;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DFLASH_ECUDA;
  unsigned word = 0;
  if (cudaMemcpy(&word, h->err, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return DFLASH_ECUDA;
  if (word) {
    // a kernel gave up part-way (or, in a debug build, a bounds check failed): clear the error word
    // and the arrival counters it may have left
    const unsigned zero = 0;
    if (cudaMemcpy(h->err, &zero, 4, cudaMemcpyHostToDevice) != cudaSuccess ||
        cudaMemset(h->tickets, 0, (size_t)h->ticket_count * 4) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess)
      return DFLASH_ECUDA;
    return (word & kErrBounds) ? DFLASH_EBOUNDS : DFLASH_ETIMEOUT;
  }
  return DFLASH_OK;
}

int dflash_get_stats(const dflash_handle* h, dflash_stats* out) {
  if (!h || !out) return DFLASH_EINVAL;
  *out = h->stats;
  return DFLASH_OK;
}

int dflash_set_probe(dflash_handle* h, int kernel, void* start_event, void* stop_event) {
  if (!h || kernel < DFLASH_PROBE_LM_HEAD || kernel > DFLASH_PROBE_CTX_KV) return DFLASH_EINVAL;
  h->probe_kernel = kernel;
  h->probe_start = static_cast<cudaEvent_t>(start_event);
  h->probe_stop = static_cast<cudaEvent_t>(stop_event);
  return DFLASH_OK;
}

uint64_t dflash_launch_count(const dflash_handle* h) { return h ? h->launches : 0; }

int dflash_accept_histogram(dflash_handle* h, uint64_t* counts, int n_counts, void* stream) {
  if (!h || !counts || n_counts < 1 || n_counts > DFLASH_MAX_GAMMA + 1) return DFLASH_EINVAL;
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DFLASH_ECUDA;
  unsigned long long v[DFLASH_MAX_GAMMA + 1];
  if (cudaMemcpy(v, h->acc_hist, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return DFLASH_ECUDA;
  for (int a = 0; a < n_counts; a++) counts[a] = (uint64_t)v[a];
  return DFLASH_OK;
}

int dflash_set_wait_limit(dflash_handle* h, unsigned limit_us, void* stream) {
  if (!h) return DFLASH_EINVAL;
  return status_of(cudaMemcpyAsync(h->err + 1, &limit_us, 4, cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream)));
}

int dflash_debug_stall(dflash_handle* h, int cta) {
  if (!h) return DFLASH_EINVAL;
  h->stall_armed = cta < 0 ? 0 : cta + 1;
  return DFLASH_OK;
}

int dflash_rows_matmul_plan(int n_out, int k_in, int n_rows, int x_lo, int n_sm, dflash_rows_plan* plan) {
  if (!plan || n_out < 1 || k_in < 64 || k_in % 64 || n_rows < 1 || n_sm < 1) return DFLASH_EINVAL;
  if (n_rows > DFLASH_ROWS_MATMUL_MAX) return DFLASH_ECAPACITY;
  const Tc05Plan p = plan_tc05((n_out + 15) / 16, k_in / 64, n_rows, x_lo != 0, n_sm);
  if (p.npad == 0) return DFLASH_EINVAL;
  plan->n_pad = p.npad;
  plan->m_tiles = p.mtiles;
  plan->k_slices = p.slices;
  plan->groups_per_slice = p.gps;
  plan->grid = p.grid;
  plan->x_stages = p.sx;
  plan->tile_groups = p.tgroups;
  plan->tiles_big = p.tiles_big;
  plan->big_groups = p.groups_big;
  plan->tiles_small = p.tiles_small;
  plan->w_stages = p.sw;
  plan->a_stages = p.sa;
  plan->w_groups = kTcKW;
  plan->x_groups = p.kx;
  plan->smem_bytes = p.smem;
  plan->scratch_bytes = p.scratch;
  return DFLASH_OK;
}

int dflash_rows_matmul(dflash_handle* h, int matrix, int layer, int n_rows, const void* x, const void* x_lo,
                       int ldx, float* y, int ldy, void* scratch, size_t scratch_bytes, void* stream) {
  if (!h || h->fmt != FMT_Q4 || !x || !y || !scratch || n_rows < 1) return DFLASH_EINVAL;
  if (n_rows > DFLASH_ROWS_MATMUL_MAX) return DFLASH_ECAPACITY;
  const bool per_layer = matrix == DFLASH_MAT_QKV || matrix == DFLASH_MAT_O || matrix == DFLASH_MAT_GATEUP ||
                         matrix == DFLASH_MAT_DOWN;
  if (per_layer && (layer < 0 || layer >= h->L)) return DFLASH_EINVAL;
  const PackedMat* m = nullptr;
  switch (matrix) {
    case DFLASH_MAT_CTX: m = &h->wc; break;
    case DFLASH_MAT_QKV: m = &h->qkv[layer]; break;
    case DFLASH_MAT_O: m = &h->wo[layer]; break;
    case DFLASH_MAT_GATEUP: m = &h->gu[layer]; break;
    case DFLASH_MAT_DOWN: m = &h->down[layer]; break;
    case DFLASH_MAT_LM: m = &h->lm; break;
    default: return DFLASH_EINVAL;
  }
  const uintptr_t misalign = reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(x_lo);
  if ((misalign & 15) || (reinterpret_cast<uintptr_t>(scratch) & 255) || ldx < m->k || ldx % 8 || ldy < m->n_rows)
    return DFLASH_EINVAL;
  const Tc05Plan p = plan_tc05(m->n_strips, m->groups, n_rows, x_lo != nullptr, h->n_sm);
  if (p.npad == 0) return DFLASH_EINVAL;
  if (scratch_bytes < p.scratch) return DFLASH_ECAPACITY;
  Tc05Args a{};
  if (make_rows_map_groups(x, m->k, n_rows, ldx, p.npad, p.kx, 1, 0, &a.xmap) != DFLASH_OK) return DFLASH_ECUDA;
  if (x_lo && make_rows_map_groups(x_lo, m->k, n_rows, ldx, p.npad, p.kx, 1, 0, &a.xlmap) != DFLASH_OK)
    return DFLASH_ECUDA;
  if (make_q4_tile_map(*m, p.tiles_big, kTcKW, 1, 0, &a.wmap) != DFLASH_OK ||
      make_q4_tile_map(*m, p.tiles_small, kTcKW, 1, 0, &a.wmap_small) != DFLASH_OK)
    return DFLASH_ECUDA;
  uint8_t* sc = static_cast<uint8_t*>(scratch);
  a.w = m->w;
  a.part = reinterpret_cast<float*>(sc + p.part_off);
  a.err = h->err;
  a.n_strips = m->n_strips;
  a.groups = m->groups;
  tc05_fill_args(p, x_lo != nullptr, a);
  h->launches += 2;
  const int half = matrix == DFLASH_MAT_GATEUP ? h->I : 0;
  return status_of(launch_tc05(a, p, n_rows, m->n_rows, half, y, ldy, static_cast<cudaStream_t>(stream)));
}

void dflash_destroy(dflash_handle* h) { delete h; }

const char* dflash_status_str(int s) {
  switch (s) {
    case DFLASH_OK: return "ok";
    case DFLASH_DECLINED: return "declined (temperature > 0 or DFLASH_DISABLE=1): fall back to plain decoding";
    case DFLASH_EINVAL: return "invalid argument";
    case DFLASH_ECAPACITY: return "capacity exceeded";
    case DFLASH_ECUDA: return "CUDA error";
    case DFLASH_ETIMEOUT: return "a bounded device wait timed out";
    case DFLASH_EBOUNDS: return "a device bounds check failed (debug build)";
    default: return "unknown status";
  }
}

}  // extern "C"

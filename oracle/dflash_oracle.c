/*
 * dflash_oracle.c -- TEST INFRASTRUCTURE ONLY (see dflash_oracle.h). Only the tests, the smoke
 * check and the bench's CPU-baseline arm call it; the CUDA library never does.
 *
 * Sources, by page:
 *  [P3] "@mlx-bun/inference 0.0.0-stage -> 1.0.0", diff of src/models/speculative/dflash.ts:
 *       Eq 2 (context injection), Eq 3 (KV-injection layer), the retained context projection,
 *       the block builder, the borrowed-head logits and greedy drafting.
 *  [P1] "Inco Hacks Native: DFlash 2 Speculation & SSM Prefix Ladders in sanctum-mlx",
 *       section 1 (geometry: block 8 = 1 verify token + 7 proposals, sliding-window drafter)
 *       and section 3 (bs=8 accepted=7 committed=8; accepted=5 committed=6).
 *  [P2] "A Refusal Is Not A Failure", section "What the port taught, besides that"
 *       (is_causal is false; the drafter borrows the target's embedding and output head).
 *  [P3] also: DflashDraftOpts.thresholds / minConf and the drafting loop of forwardRows
 *       (confidence-scheduled draft-length pruning, "Alg 1", single-user form).
 *
 * Readings where the pages leave a step open are stated at each function.
 * Everything is fp64; loops run in the order the definitions are written, each output's sum
 * over k in increasing k. OpenMP only splits independent outputs across threads.
 */
#include "dflash_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static double bf16_value(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* One stored matrix element, dequantised. The 4-bit form is the affine group-64 code
 * w = scale*q + bias with q the 4-bit integer of input k (nibble k%8 of word k/8, low nibble
 * first) and scale/bias the bf16 pair of group k/64 of that row. */
double orc_weight(const orc_mat* m, int n, int k) {
  if (m->fmt == ORC_F32) return (double)((const float*)m->w)[(int64_t)n * m->n_in + k];
  if (m->fmt == ORC_BF16) return bf16_value(((const uint16_t*)m->w)[(int64_t)n * m->n_in + k]);
  uint32_t word = ((const uint32_t*)m->w)[(int64_t)n * (m->n_in / 8) + k / 8];
  int q = (int)((word >> (4 * (k % 8))) & 15u);
  int64_t g = (int64_t)n * (m->n_in / 64) + k / 64;
  return bf16_value(m->scale[g]) * (double)q + bf16_value(m->bias[g]);
}

/* y[r][n] = sum_k W[n][k] x[r][k] for rows r < rows. */
void orc_linear(const orc_mat* m, int rows, const double* x, double* y) {
#pragma omp parallel
  {
    double* wrow = (double*)malloc(sizeof(double) * (size_t)m->n_in);
#pragma omp for schedule(static)
    for (int n = 0; n < m->n_out; n++) {
      for (int k = 0; k < m->n_in; k++) wrow[k] = orc_weight(m, n, k);
      for (int r = 0; r < rows; r++) {
        const double* xr = x + (int64_t)r * m->n_in;
        double acc = 0.0;
        for (int k = 0; k < m->n_in; k++) acc += wrow[k] * xr[k];
        y[(int64_t)r * m->n_out + n] = acc;
      }
    }
    free(wrow);
  }
}

/* RMSNorm as used throughout [P3]: y = x / sqrt(mean(x^2) + eps) * w. */
void orc_rmsnorm(const double* x, const float* w, int n, double eps, double* y) {
  double ss = 0.0;
  for (int i = 0; i < n; i++) ss += x[i] * x[i];
  double inv = 1.0 / sqrt(ss / n + eps);
  for (int i = 0; i < n; i++) y[i] = x[i] * inv * (double)w[i];
}

/* SiLU(x) = x / (1 + e^-x): the gate activation of the SwiGLU feed-forward. */
double orc_silu(double x) { return x / (1.0 + exp(-x)); }

/* The gated-GELU FFN of the dflash.ts page applies "geluApprox" to the gate. Reading: the tanh
 * approximation of GELU (Hendrycks and Gimpel), 0.5 x (1 + tanh(sqrt(2/pi) (x + 0.044715 x^3))). */
double orc_gelu_tanh(double x) {
  const double k = sqrt(2.0 / 3.14159265358979323846);
  return 0.5 * x * (1.0 + tanh(k * (x + 0.044715 * x * x * x)));
}

/* Scaled dot-product attention of [P3] Eq 3 with grouped K/V heads:
 * q [n_q_rows][Hq*hd], k/v [n_keys][Hkv*hd], out [n_q_rows][Hq*hd].
 * Query head h reads key/value head h / (Hq/Hkv) (contiguous groups).
 * Scores scaled by hd^-1/2, softmax over keys with no mask (is_causal false, [P2]).
 * causal_block_start >= 0 is the test-only causal variant: query row i then sees keys
 * [0, causal_block_start + i + 1). */
void orc_attention(int n_q_rows, int n_q_heads, int n_kv_heads, int head_dim, const double* q,
                   int n_keys, const double* k, const double* v, int causal_block_start,
                   double* out) {
  const int qd = n_q_heads * head_dim, kvd = n_kv_heads * head_dim;
  const int group = n_q_heads / n_kv_heads;
  const double scale = 1.0 / sqrt((double)head_dim);
  double* p = (double*)malloc(sizeof(double) * (size_t)(n_keys > 0 ? n_keys : 1));
  for (int i = 0; i < n_q_rows; i++) {
    int seen = n_keys;
    if (causal_block_start >= 0) seen = causal_block_start + i + 1;
    for (int h = 0; h < n_q_heads; h++) {
      const int g = h / group;
      const double* qi = q + (int64_t)i * qd + h * head_dim;
      double mx = -INFINITY;
      for (int j = 0; j < seen; j++) {
        const double* kj = k + (int64_t)j * kvd + g * head_dim;
        double s = 0.0;
        for (int c = 0; c < head_dim; c++) s += qi[c] * kj[c];
        p[j] = s * scale;
        if (p[j] > mx) mx = p[j];
      }
      double z = 0.0;
      for (int j = 0; j < seen; j++) {
        p[j] = exp(p[j] - mx);
        z += p[j];
      }
      double* oi = out + (int64_t)i * qd + h * head_dim;
      for (int c = 0; c < head_dim; c++) {
        double acc = 0.0;
        for (int j = 0; j < seen; j++) acc += p[j] * v[(int64_t)j * kvd + g * head_dim + c];
        oi[c] = acc / z;
      }
    }
  }
  free(p);
}

/* Context rows ([P3] Eq 2 and the retained context projection). For each new row:
 *   x = W_c [H^{l1}; ...; H^{lm}]          (taps concatenated on the feature axis)
 *   H_ctx = RMSNorm(x; ctx_norm)
 *   per layer i: n = RMSNorm(H_ctx; attn_norm_i)  -- the same norm the block rows use
 *                K_i = W_k^i n, V_i = W_v^i n
 * taps [rows][m*H] (exact values of the stored taps); k_out/v_out [L][rows][Hkv*hd].
 * The rows do not depend on the block, so they are computed once per position. */
void orc_ctx_rows(const orc_cfg* c, const orc_weights* w, int rows, const double* taps,
                  double* k_out, double* v_out) {
  const int d = c->d, kvd = c->n_kv_heads * c->head_dim;
  double* x = (double*)malloc(sizeof(double) * (size_t)rows * d);
  double* hctx = (double*)malloc(sizeof(double) * (size_t)rows * d);
  double* nrm = (double*)malloc(sizeof(double) * (size_t)rows * d);
  orc_linear(&w->w_c, rows, taps, x);
  for (int r = 0; r < rows; r++)
    orc_rmsnorm(x + (int64_t)r * d, w->ctx_norm, d, c->eps, hctx + (int64_t)r * d);
  for (int i = 0; i < c->n_layers; i++) {
    for (int r = 0; r < rows; r++)
      orc_rmsnorm(hctx + (int64_t)r * d, w->layer[i].attn_norm, d, c->eps, nrm + (int64_t)r * d);
    orc_linear(&w->layer[i].wk, rows, nrm, k_out + (int64_t)i * rows * kvd);
    orc_linear(&w->layer[i].wv, rows, nrm, v_out + (int64_t)i * rows * kvd);
  }
  free(x);
  free(hctx);
  free(nrm);
}

/* Greedy token and softmax confidence of one logit row:
 * token = argmax (lowest index on ties), conf = softmax(l)[token] = 1 / sum_j exp(l_j - max),
 * margin = max - (largest logit at any other index). */
void orc_argmax_conf(const double* logits, int vocab, int* token, double* conf, double* margin) {
  int best = 0;
  for (int j = 1; j < vocab; j++)
    if (logits[j] > logits[best]) best = j;
  double mx = logits[best], z = 0.0, second = -INFINITY;
  for (int j = 0; j < vocab; j++) {
    z += exp(logits[j] - mx);
    if (j != best && logits[j] > second) second = logits[j];
  }
  *token = best;
  *conf = 1.0 / z;
  *margin = mx - second;
}

/* One drafting pass over a block ([P3] block builder, Eq 3 layers, output norm and the
 * borrowed-head logits; greedy drafting at temperature 0).
 *
 *  H_d[0] = T(E[anchor]) + block_pos[0]; H_d[k] = mask_emb[k-1] + block_pos[k], k = 1..gamma-1
 *    (T = tok_proj when d != H, the identity otherwise: DFlash2 has no embedding of its own)
 *  per layer i:
 *    n = RMSNorm(H_d; attn_norm_i); Q = W_q n; K_d = W_k n; V_d = W_v n
 *    keys/values = [context rows in the window ; K_d/V_d of all gamma block rows]
 *    H_d += W_o Attention(Q, keys, values)
 *    n2 = RMSNorm(H_d; ff_norm_i); H_d += W_down (SiLU(W_gate n2) * (W_up n2))
 *  drafts from rows 1..gamma-1 (row 0 holds the anchor, the token the target verifies):
 *    h = RMSNorm(H_d[k]; out_norm), h = out_proj h when d != H, l = lm_head h, token = argmax l
 *
 * Context: k_ctx/v_ctx [L][n_ctx][Hkv*hd] hold positions 0..n_ctx-1; the window keeps
 * positions [max(0, n_ctx - window), n_ctx) (window 0 keeps them all), the same for every
 * block row. Outputs: logits [gamma-1][V], tokens/conf/margin [gamma-1];
 * trace (optional) [L+1][gamma][d] = H_d before each layer and after the last one. */
int orc_draft(const orc_cfg* c, const orc_weights* w, int anchor, int n_ctx, const double* k_ctx,
              const double* v_ctx, double* logits, int* tokens, double* conf, double* margin,
              double* trace) {
  const int d = c->d, H = c->target_hidden, G = c->gamma, V = c->vocab;
  const int qd = c->n_q_heads * c->head_dim, kvd = c->n_kv_heads * c->head_dim;
  if (anchor < 0 || anchor >= V || G < 2 || n_ctx < 0) return -1;
  const int lo = (c->window > 0 && n_ctx > c->window) ? n_ctx - c->window : 0;
  const int n_win = n_ctx - lo, n_keys = n_win + G;
  const int wide = d > H ? d : H;

  double* hd = (double*)calloc((size_t)G * d, sizeof(double));
  double* nd = (double*)malloc(sizeof(double) * (size_t)G * d);
  double* q = (double*)malloc(sizeof(double) * (size_t)G * qd);
  double* keys = (double*)malloc(sizeof(double) * (size_t)n_keys * kvd);
  double* vals = (double*)malloc(sizeof(double) * (size_t)n_keys * kvd);
  double* att = (double*)malloc(sizeof(double) * (size_t)G * qd);
  double* tmp = (double*)malloc(sizeof(double) * (size_t)G * wide);
  double* gate = (double*)malloc(sizeof(double) * (size_t)G * c->inter);
  double* up = (double*)malloc(sizeof(double) * (size_t)G * c->inter);
  double* e = (double*)malloc(sizeof(double) * (size_t)H);

  /* block construction */
  for (int j = 0; j < H; j++) e[j] = orc_weight(&w->embed, anchor, j);
  if (d != H) {
    orc_linear(&w->tok_proj, 1, e, tmp);
    for (int j = 0; j < d; j++) hd[j] = tmp[j] + (double)w->block_pos[j];
  } else {
    for (int j = 0; j < d; j++) hd[j] = e[j] + (double)w->block_pos[j];
  }
  for (int k = 1; k < G; k++)
    for (int j = 0; j < d; j++)
      hd[(int64_t)k * d + j] =
          (double)w->mask_emb[(int64_t)(k - 1) * d + j] + (double)w->block_pos[(int64_t)k * d + j];

  for (int i = 0; i < c->n_layers; i++) {
    const orc_layer* L = &w->layer[i];
    if (trace) memcpy(trace + (int64_t)i * G * d, hd, sizeof(double) * (size_t)G * d);
    for (int k = 0; k < G; k++)
      orc_rmsnorm(hd + (int64_t)k * d, L->attn_norm, d, c->eps, nd + (int64_t)k * d);
    orc_linear(&L->wq, G, nd, q);
    memcpy(keys, k_ctx + ((int64_t)i * n_ctx + lo) * kvd, sizeof(double) * (size_t)n_win * kvd);
    memcpy(vals, v_ctx + ((int64_t)i * n_ctx + lo) * kvd, sizeof(double) * (size_t)n_win * kvd);
    orc_linear(&L->wk, G, nd, keys + (int64_t)n_win * kvd);
    orc_linear(&L->wv, G, nd, vals + (int64_t)n_win * kvd);
    orc_attention(G, c->n_q_heads, c->n_kv_heads, c->head_dim, q, n_keys, keys, vals,
                  c->causal ? n_win : -1, att);
    orc_linear(&L->wo, G, att, tmp);
    for (int64_t j = 0; j < (int64_t)G * d; j++) hd[j] += tmp[j];
    for (int k = 0; k < G; k++)
      orc_rmsnorm(hd + (int64_t)k * d, L->ff_norm, d, c->eps, nd + (int64_t)k * d);
    orc_linear(&L->w_gate, G, nd, gate);
    orc_linear(&L->w_up, G, nd, up);
    for (int64_t j = 0; j < (int64_t)G * c->inter; j++)
      gate[j] = (c->ffn_act ? orc_gelu_tanh(gate[j]) : orc_silu(gate[j])) * up[j];
    orc_linear(&L->w_down, G, gate, tmp);
    for (int64_t j = 0; j < (int64_t)G * d; j++) hd[j] += tmp[j];
  }
  if (trace) memcpy(trace + (int64_t)c->n_layers * G * d, hd, sizeof(double) * (size_t)G * d);

  /* the drafting rows (1..gamma-1, or all gamma rows: the dflash.ts page's forwardRows drafts a
   * token from every block row) through the output norm (and out_proj), then the borrowed head */
  const int r0 = c->draft_all_rows ? 0 : 1, nrow = G - r0;
  for (int k = r0; k < G; k++)
    orc_rmsnorm(hd + (int64_t)k * d, w->out_norm, d, c->eps, nd + (int64_t)(k - r0) * d);
  if (d != H) {
    orc_linear(&w->out_proj, nrow, nd, tmp);
    orc_linear(&w->lm_head, nrow, tmp, logits);
  } else {
    orc_linear(&w->lm_head, nrow, nd, logits);
  }
  for (int k = 0; k < nrow; k++)
    orc_argmax_conf(logits + (int64_t)k * V, V, tokens + k, conf + k, margin + k);

  free(hd); free(nd); free(q); free(keys); free(vals); free(att); free(tmp);
  free(gate); free(up); free(e);
  return 0;
}

/* Greedy acceptance ([P1] section 3): the target verifies [anchor, d_1..d_n] and returns its
 * greedy tokens t_1..t_{n+1} (target[0..n]). The accepted length a is the length of the
 * longest prefix with draft[k] == target[k]; the bonus token target[a] becomes the next
 * anchor, and a + 1 tokens are committed. */
int orc_accept(int n, const int* draft, const int* target, int* next_anchor) {
  int a = 0;
  while (a < n && draft[a] == target[a]) a++;
  *next_anchor = target[a];
  return a;
}

/* Confidence-scheduled draft-length pruning ([P3], the draft options and the drafting loop of
 * forwardRows): walking the drafts in order, position k >= 1 ends the block when its confidence
 * is below its threshold -- thresholds[k] when a per-position list is given, otherwise min_conf;
 * position 0 is always drafted. Returns the number of drafts kept (1..n). Reading: the
 * confidence is the softmax probability of the drafted token (this drafter has no learned
 * acceptance head), and "below" is the strict comparison the page writes. */
int orc_draft_length(int n, const float* conf, const float* thresholds, float min_conf) {
  for (int k = 1; k < n; k++) {
    const float th = thresholds ? thresholds[k] : min_conf;
    if (conf[k] < th) return k;
  }
  return n;
}

/* Acceptance over a pruned block: the target verifies only the first keep drafts, so the
 * accepted length is the longest matching prefix within them and the bonus token is the
 * target's token right after it. */
int orc_accept_kept(int n, int keep, const int* draft, const int* target, int* next_anchor) {
  int a = 0;
  while (a < keep && a < n && draft[a] == target[a]) a++;
  *next_anchor = target[a];
  return a;
}

/* The Markov sequential head ([P3] Eq 5, the markov branch of forwardRows): the drafts are taken
 * one after another; before the argmax of draft k its logits get the rank-r bias
 *   b_k = W1[prev_k] W2,  prev_0 = the anchor, prev_k = draft k-1,
 * W1 [V][r] (a token embedding), W2 [r][V], stored here as W2^T [V][r] so that b_k = W2^T e.
 * prev_given (NULL for the head's own greedy chain) fixes prev_1.. to given tokens, so that a
 * caller can follow another implementation's chain past a near-tie. */
void orc_markov(const orc_mat* w1, const orc_mat* w2t, int rank, int vocab, int n, int anchor,
                const double* base_logits, const int* prev_given, double* logits, int* tokens,
                double* conf, double* margin) {
  double* e = (double*)malloc(sizeof(double) * (size_t)rank);
  double* bias = (double*)malloc(sizeof(double) * (size_t)vocab);
  int prev = anchor;
  for (int k = 0; k < n; k++) {
    for (int i = 0; i < rank; i++) e[i] = orc_weight(w1, prev, i);
    orc_linear(w2t, 1, e, bias);
    for (int j = 0; j < vocab; j++) logits[(int64_t)k * vocab + j] = base_logits[(int64_t)k * vocab + j] + bias[j];
    orc_argmax_conf(logits + (int64_t)k * vocab, vocab, tokens + k, conf + k, margin + k);
    prev = prev_given ? prev_given[k] : tokens[k];
  }
  free(e);
  free(bias);
}

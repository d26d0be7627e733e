/*
 * dflash_oracle.h -- TEST INFRASTRUCTURE. Plain, slow CPU definition of one DFlash drafting
 * round, used only by the tests, by the smoke check and by the bench's CPU-baseline arm.
 * It shares no code with the CUDA library (speculative_block_draft_gb300/csrc) and must never
 * be linked into it.
 *
 * All arithmetic is fp64. Weights are read in their storage format (fp32, bf16 bits or
 * group-64 affine 4-bit) and dequantised element by element: w = scale*q + bias.
 * Every matrix is stored output-major: W[n_out][n_in], y = W x.
 */
#ifndef DFLASH_ORACLE_H
#define DFLASH_ORACLE_H
#include <stdint.h>

#define ORC_F32 0
#define ORC_BF16 1
#define ORC_Q4G64 2
#define ORC_MAX_LAYERS 16

typedef struct {
  int n_layers, d, n_q_heads, n_kv_heads, head_dim, inter, n_taps, target_hidden, vocab, gamma,
      window;   /* window over context rows; 0 = the whole context */
  double eps;
  int causal;   /* 0 = the method (non-causal block). 1 only for the test that shows the
                   difference a causal mask would make. */
  int ffn_act;  /* 0 = SwiGLU silu(g) * u; 1 = gated GELU gelu(g) * u (tanh approximation) */
  int draft_all_rows;  /* 0 = drafts from block rows 1..gamma-1 (gamma-1 tokens); 1 = from all
                          gamma rows (gamma tokens) */
} orc_cfg;

typedef struct {
  int fmt, n_out, n_in;
  const void* w;          /* f32 [n_out][n_in] | bf16 bits [n_out][n_in] | u32 [n_out][n_in/8] */
  const uint16_t* scale;  /* q4 only: bf16 bits [n_out][n_in/64] */
  const uint16_t* bias;   /* q4 only */
} orc_mat;

typedef struct {
  orc_mat wq, wk, wv, wo, w_gate, w_up, w_down;
  const float *attn_norm, *ff_norm;
} orc_layer;

typedef struct {
  orc_mat w_c, tok_proj, out_proj, embed, lm_head;   /* tok_proj/out_proj used iff d != H */
  const float *ctx_norm, *mask_emb /* [gamma-1][d] */, *block_pos /* [gamma][d] */, *out_norm;
  orc_layer layer[ORC_MAX_LAYERS];
} orc_weights;

double orc_weight(const orc_mat* m, int n, int k);
void orc_linear(const orc_mat* m, int rows, const double* x, double* y);
void orc_rmsnorm(const double* x, const float* w, int n, double eps, double* y);
double orc_silu(double x);
double orc_gelu_tanh(double x);
void orc_attention(int n_q_rows, int n_q_heads, int n_kv_heads, int head_dim, const double* q,
                   int n_keys, const double* k, const double* v, int causal_block_start,
                   double* out);
void orc_ctx_rows(const orc_cfg* c, const orc_weights* w, int rows, const double* taps,
                  double* k_out, double* v_out);
int orc_draft(const orc_cfg* c, const orc_weights* w, int anchor, int n_ctx, const double* k_ctx,
              const double* v_ctx, double* logits, int* tokens, double* conf, double* margin,
              double* trace);
void orc_argmax_conf(const double* logits, int vocab, int* token, double* conf, double* margin);
int orc_accept(int n, const int* draft, const int* target, int* next_anchor);
int orc_draft_length(int n, const float* conf, const float* thresholds, float min_conf);
int orc_accept_kept(int n, int keep, const int* draft, const int* target, int* next_anchor);
void orc_markov(const orc_mat* w1, const orc_mat* w2t, int rank, int vocab, int n, int anchor,
                const double* base_logits, const int* prev_given, double* logits, int* tokens,
                double* conf, double* margin);

#endif

/*
 * dflash.h -- C ABI of the GB300 (sm_103a) DFlash / DFlash2 block-drafter round.
 *
 * One speculative round is three calls on one CUDA stream:
 *   dflash_project_ctx  context rows: Eq 2 of the dflash.ts page (H_ctx = RMSNorm(W_c [H^l1;..;H^lm]))
 *                       and each layer's K_i = W_k^i RMSNorm(H_ctx), V_i = W_v^i RMSNorm(H_ctx),
 *                       appended to a per-layer context K/V cache ("projectContextRows": the rows do
 *                       not depend on the block, so each position is projected once).
 *   dflash_draft_block  the block pass: block rows (anchor embedding + block_pos, mask_emb + block_pos),
 *                       the Eq 3 KV-injection layers (non-causal attention of the block over
 *                       [windowed context ++ block], SwiGLU MLP), out_norm, the borrowed target LM head,
 *                       greedy token and softmax confidence of the drafting rows (1..gamma-1).
 *   dflash_accept       greedy acceptance: longest prefix of drafts equal to the target's greedy
 *                       tokens; the bonus token becomes the next anchor ("Inco Hacks Native: DFlash 2
 *                       Speculation", section 3: bs=8 accepted=7 committed=8).
 *
 * Conventions
 *  - Every projection matrix is output-major W[n_out][n_in] (y = W x) in one storage format:
 *      DFLASH_F32   float      [n_out][n_in]
 *      DFLASH_BF16  bf16 bits  [n_out][n_in]
 *      DFLASH_Q4G64 uint32     [n_out][n_in/8] (nibble i of word j = input 8j+i, low nibble first)
 *                   + scale, bias bf16 bits [n_out][n_in/64]; element = scale*q + bias
 *    Norm weights, mask_emb [gamma-1][d] and block_pos [gamma][d] are float32.
 *  - All pointers passed to the calls below are DEVICE pointers unless stated otherwise.
 *  - Ownership: the caller allocates every device buffer (weights, workspace, inputs, outputs).
 *    The library never calls cudaMalloc/cudaFree. dflash_create copies and re-lays-out the
 *    drafter weights and the target LM head into the workspace; the source weight buffers may be
 *    freed once the create stream has been synchronised. The target embedding table is BORROWED
 *    (the drafter has no embedding of its own, "A Refusal Is Not A Failure", section "What the port
 *    taught"): it must stay alive and unchanged for the handle's lifetime.
 *  - Calls only enqueue work on the given stream and never synchronise, except dflash_check_errors.
 *  - Calls are validated on the host before any launch; a rejected call changes no state.
 *  - Temperature != 0, or the environment variable DFLASH_DISABLE=1, make dflash_draft_block return
 *    DFLASH_DECLINED without doing any work: the caller falls back to plain autoregressive decoding
 *    ("A Refusal Is Not A Failure", section "The rule it earned": an acceleration path may decline a
 *    request, it must never fail one).
 *  - Handles are not thread-safe; use one handle per thread or serialise calls.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_MAX_LAYERS 8
#define DFLASH_MAX_BATCH 64
#define DFLASH_MAX_GAMMA 16

enum dflash_status {
  DFLASH_OK = 0,
  DFLASH_DECLINED = 1,    /* not drafted on purpose (temperature > 0, kill switch); not an error */
  DFLASH_EINVAL = -1,     /* bad shape, null pointer, unsupported combination */
  DFLASH_ECAPACITY = -2,  /* context cache or batch capacity exceeded */
  DFLASH_ECUDA = -3,      /* a CUDA runtime call failed */
  DFLASH_ETIMEOUT = -4,   /* a bounded device-side wait gave up (reported by dflash_check_errors) */
  DFLASH_EBOUNDS = -5,    /* a device bounds check failed (builds with DFL_DEBUG_CHECKS; see below) */
};

enum dflash_dtype { DFLASH_F32 = 0, DFLASH_BF16 = 1, DFLASH_Q4G64 = 2 };
enum dflash_ffn { DFLASH_FFN_SWIGLU = 0, DFLASH_FFN_GELU = 1 };

typedef struct {
  int n_layers;       /* drafter layers L (<= DFLASH_MAX_LAYERS) */
  int d;              /* draft width; n_q_heads * head_dim == d */
  int n_q_heads, n_kv_heads, head_dim;   /* head_dim in {64, 128, 256}; n_q_heads % n_kv_heads == 0 */
  int inter;          /* gated FFN inner width */
  int n_taps;         /* m tapped target layers */
  int target_hidden;  /* H; tok_proj / out_proj exist iff d != H */
  int vocab;          /* V */
  int gamma;          /* block size (2..DFLASH_MAX_GAMMA); n_draft drafts per block (below) */
  int window;         /* sliding window over context rows; 0 = the whole context */
  int max_batch;      /* request slots (<= DFLASH_MAX_BATCH) */
  int ctx_capacity;   /* context rows kept per request and layer. With window > 0 the cache is a
                         ring of this many rows and must hold >= window rows; with window == 0 it
                         bounds the total context length of a request. */
  float eps;          /* RMSNorm epsilon */
  int wdtype;         /* storage of every projection matrix, the embedding and the LM head */
  int adtype;         /* DFLASH_F32: fp32 taps, fp32 cache, CUDA-core fp32 arithmetic (requires
                         wdtype DFLASH_F32). DFLASH_BF16: bf16 taps; internally the tensor-core
                         path runs f16 activations and an f16 context cache with fp32
                         accumulation (bf16 weights are stored as f16 in the workspace). */
  int ffn_act;        /* FFN gate: DFLASH_FFN_SWIGLU silu(g) * u (the workload's MLP), or
                         DFLASH_FFN_GELU gelu(g) * u with the tanh approximation of GELU (the
                         gated-GELU FFN of the dflash.ts page, "geluApprox") */
  int draft_all_rows; /* 0: drafts from block rows 1..gamma-1 (n_draft = gamma-1, the DFlash2 block:
                         one verify token + gamma-1 proposals); 1: from all gamma block rows
                         (n_draft = gamma, the dflash.ts page's forwardRows) */
  int markov_rank;    /* 0: drafts are the argmax of the head's logits. r > 0 (a multiple of 64,
                         <= 1024): the Markov sequential head of the dflash.ts page (Eq 5) --
                         drafts are taken in order and draft k's logits get the bias
                         W1[prev_k] W2 before its argmax (prev_0 = the anchor, prev_k = draft k-1);
                         weights markov_w1 [V][r] and markov_w2t [V][r] (= W2 transposed) */
  int large_batch_tc05; /* 0 (default): dflash_draft_block runs every projection as the skinny GEMV,
                         in launches of at most 32 activation rows. 1: a call with more than 32 and
                         at most DFLASH_ROWS_MATMUL_MAX block rows runs its Q/K/V, O, gate/up, down
                         and LM-head projections once over all its rows on the tcgen05 contraction
                         (as dflash_rows_matmul), followed by the same epilogues; likewise
                         dflash_project_ctx runs W_c once per 160 context rows when a call appends
                         more than 32, and every layer's context K/V of those rows in one grouped
                         launch (the 32-row GEMV chunks instead when a request's ring would wrap
                         within the call, so later rows overwrite earlier ones in order). It
                         applies to 4-bit weights with d == H and no Markov head;
                         other calls use the GEMV. The workspace grows by the contraction's scratch
                         and an f16 copy of 160 tap rows. */
  int skinny_tc05;    /* 0: calls of at most 32 block rows run every projection as the mma.sync
                         GEMV. 1: with 4-bit weights and f16 activations, a dflash_draft_block call
                         of at most 32 block rows runs its Q/K/V, O, gate/up and down projections
                         and (d == H) the LM head each as one tcgen05 launch with the same fused
                         epilogues: weights dequantised to f16 (one rounding) in shared memory,
                         fp32 accumulators in tensor memory. */
} dflash_config;

typedef struct {
  const void* data;   /* see the storage formats above */
  const void* scale;  /* DFLASH_Q4G64 only */
  const void* bias;   /* DFLASH_Q4G64 only */
} dflash_matrix;

typedef struct {
  dflash_matrix wq, wk, wv, wo;        /* [Hq*hd][d], [Hkv*hd][d], [Hkv*hd][d], [d][Hq*hd] */
  dflash_matrix w_gate, w_up, w_down;  /* [inter][d], [inter][d], [d][inter] */
  const float* attn_norm;              /* [d]; used for the block rows AND the context rows */
  const float* ff_norm;                /* [d] */
} dflash_layer_weights;

typedef struct {
  dflash_matrix w_c;        /* [d][n_taps*H]  Eq 2 context projection */
  dflash_matrix tok_proj;   /* [d][H]  only when d != H */
  dflash_matrix out_proj;   /* [H][d]  only when d != H */
  dflash_matrix embed;      /* [V][H]  the target's embedding table (borrowed, see above) */
  dflash_matrix lm_head;    /* [V][H]  the target's output head (copied into the workspace) */
  const float* ctx_norm;    /* [d] */
  const float* mask_emb;    /* [gamma-1][d] */
  const float* block_pos;   /* [gamma][d] */
  const float* out_norm;    /* [d] */
  dflash_layer_weights layer[DFLASH_MAX_LAYERS];
  dflash_matrix markov_w1;  /* [V][r]  Markov head token table (borrowed; markov_rank > 0 only) */
  dflash_matrix markov_w2t; /* [V][r]  W2 of the Markov head, transposed (copied into the workspace) */
} dflash_weights;

typedef struct dflash_handle dflash_handle;

typedef struct {
  uint64_t rounds;          /* successful dflash_draft_block calls */
  uint64_t blocks;          /* request-blocks drafted */
  uint64_t declined;        /* dflash_draft_block calls that returned DFLASH_DECLINED */
  uint64_t ctx_rows;        /* context rows projected */
  uint64_t accept_calls;    /* dflash_accept calls */
} dflash_stats;

/* Bytes of device workspace dflash_create needs for this configuration (0 if invalid). */
size_t dflash_workspace_bytes(const dflash_config* cfg);

/* Validate cfg, lay out the workspace (>= dflash_workspace_bytes, 256-byte aligned, device
 * memory owned by the caller), re-lay-out the weights into it and zero all state, all on
 * `stream` (a cudaStream_t; NULL = legacy default stream). *out receives a host-side handle.
 * A handle belongs to the device current at create: make that device current for every call
 * on it. A handle's calls must be issued in order on one stream (its scratch is shared by all of
 * them); different handles are independent and may run on different devices and threads. */
int dflash_create(const dflash_config* cfg, const dflash_weights* weights, void* workspace,
                  size_t workspace_bytes, void* stream, dflash_handle** out);

/* Append context rows (Eq 2 plus each layer's K/V projection of the retained context).
 * req_ids [n_req], n_new [n_req]: HOST arrays; request slots are 0..max_batch-1, each at most once.
 * taps: device [sum(n_new)][n_taps*H] (fp32 or bf16 per adtype), rows of request i after those of
 * request i-1; row j of request i is context position P_i + j, where P_i is the request's
 * current context length. Every request's P grows by n_new[i].
 * Returns DFLASH_ECAPACITY if window == 0 and a request would exceed ctx_capacity. */
int dflash_project_ctx(dflash_handle* h, int n_req, const int32_t* req_ids, const int32_t* n_new,
                       const void* taps, void* stream);

/* Draft one block per request. req_ids: HOST [n_req]. anchor: device int32 [n_req], the last
 * committed token of each request. Outputs (device): draft int32 [n_req][n_draft] (greedy tokens of
 * the drafting rows: block rows 1..gamma-1, or all gamma rows with draft_all_rows), conf float
 * [n_req][n_draft] (softmax probability of the drafted token; may be NULL), logits float
 * [n_req][n_draft][V] (may be NULL; written only when given). n_draft = gamma-1+draft_all_rows.
 * Attention of each request reads its context rows [max(0, P - window), P) (all when window == 0)
 * and all gamma block rows, with no causal mask. temperature != 0 -> DFLASH_DECLINED. */
int dflash_draft_block(dflash_handle* h, int n_req, const int32_t* req_ids, const int32_t* anchor,
                       float temperature, int32_t* draft, float* conf, float* logits, void* stream);

/* Greedy acceptance for n_req requests (independent of any handle state except gamma).
 * draft int32 [n_req][n_draft], target int32 [n_req][n_draft+1] (the target's greedy tokens after
 * [anchor, d_1..d_{n_draft}]). Outputs: accept_len int32 [n_req] = longest prefix with
 * draft == target; next_anchor int32 [n_req] = target[accept_len]; accept_len + 1 tokens commit. */
int dflash_accept(dflash_handle* h, int n_req, const int32_t* draft, const int32_t* target,
                  int32_t* accept_len, int32_t* next_anchor, void* stream);

/* Confidence-scheduled draft-length pruning ("Alg 1", single-user form, in the dflash.ts page's
 * draft options): draft position k (0-based over the n_draft drafts) is dropped, and the block
 * truncated there, when k >= 1 and conf[k] < thr_k, where thr_k = thresholds[k] if thresholds is
 * given, else min_conf; position 0 is always kept. conf is dflash_draft_block's confidence (the
 * softmax probability of the drafted token; the pages' learned acceptance head is not part of
 * this library). conf: device float [n_req][n_draft]; thresholds: device float [n_draft] or NULL;
 * min_conf: used only when thresholds is NULL (a value <= 0 keeps every position).
 * Output: keep int32 [n_req] (device), 1 <= keep[i] <= n_draft, the number of drafts the target
 * verifies. Pruning never changes what is emitted, only how many positions are verified. */
int dflash_draft_lengths(dflash_handle* h, int n_req, const float* conf, const float* thresholds,
                         float min_conf, int32_t* keep, void* stream);

/* Greedy acceptance over pruned blocks: as dflash_accept with accept_len capped at keep[i]
 * (device int32 [n_req], from dflash_draft_lengths): accept_len = longest prefix with
 * draft == target within the first keep[i] drafts; next_anchor = target[accept_len]. */
int dflash_accept_kept(dflash_handle* h, int n_req, const int32_t* draft, const int32_t* keep,
                       const int32_t* target, int32_t* accept_len, int32_t* next_anchor, void* stream);

/* Forget a request slot's context (its length returns to 0). Host-only; no device work. */
int dflash_reset_request(dflash_handle* h, int req_id);

/* Current context length of a request slot (host mirror), or -1 for a bad slot. */
int64_t dflash_ctx_len(const dflash_handle* h, int req_id);

/* Synchronise `stream`, then read and clear the device error word. Returns DFLASH_EBOUNDS if a
 * device bounds check failed since the last check (only libraries compiled with DFL_DEBUG_CHECKS
 * check: out-of-range anchors, previous Markov tokens and kept-draft counts, which every build
 * clamps; cache slots and ring positions of context appends, which every build skips when out of
 * range; and the weight-tile and cache-plane ranges the kernels compute), DFLASH_ETIMEOUT if a
 * bounded device wait gave up, DFLASH_ECUDA on a CUDA error, else DFLASH_OK. */
int dflash_check_errors(dflash_handle* h, void* stream);

/* ---- failure-handling test hooks ---------------------------------------------------------------
 * The pages' rule that an acceleration path may decline a request but must never fail one (the
 * "A Refusal Is Not A Failure" page, its closing rule) is kept on the device by bounded waits:
 * every wait of a kernel on an mbarrier gives up after a limit, sets a bit of the handle's error
 * word, waits for the CTA's own copies in flight and returns. These two calls let a test make such
 * a wait run out; neither is needed in production.
 *
 * dflash_set_wait_limit: the limit of the kernels' waits from the next launch on, in microseconds
 * (0 restores the default of 1 s). Waits that only drain a CTA's own copies before it leaves
 * always allow 1 s. Enqueued on `stream` (a 4-byte host-to-device copy). Returns DFLASH_EINVAL for
 * a NULL handle, DFLASH_ECUDA on a CUDA error.
 *
 * dflash_debug_stall: in the next dflash_draft_block call only, CTA `cta` of every tensor-core
 * projection launch also waits on an mbarrier that no copy and no thread completes, so that wait
 * runs out after the limit and the launch gives up; the round's outputs are then undefined and
 * dflash_check_errors returns DFLASH_ETIMEOUT (clearing the error word and the split-K tickets
 * the launches left). cta < 0 disarms it. Host-only. Returns DFLASH_EINVAL for a NULL handle. */
int dflash_set_wait_limit(dflash_handle* h, unsigned limit_us, void* stream);
int dflash_debug_stall(dflash_handle* h, int cta);

/* Host-side counters. */
int dflash_get_stats(const dflash_handle* h, dflash_stats* out);

/* Accepted-length histogram of every dflash_accept / dflash_accept_kept call since create (the
 * "Inco Hacks Native" page, section 3, logs each round as bs= accepted= committed=; here
 * counts[a] = blocks whose accepted length was a, and such a block committed a + 1 tokens).
 * Kept on the device by the accept kernel; this call synchronises `stream` and copies
 * counts[0 .. n_counts-1], 1 <= n_counts <= DFLASH_MAX_GAMMA + 1. Returns DFLASH_EINVAL for a
 * NULL handle or counts or a bad n_counts, DFLASH_ECUDA on a CUDA error. */
int dflash_accept_histogram(dflash_handle* h, uint64_t* counts, int n_counts, void* stream);

/* Record two caller-created CUDA events (cudaEvent_t) around the first launch (or launch pair) of
 * one kind in the next dflash_draft_block or dflash_project_ctx call that runs it, for live
 * per-kernel timing: the LM head with its vocab merge; layer 0's Q/K/V projection, attention
 * (with its split merge), O projection, gate/up projection, down projection; the context
 * projection W_c and the context K/V append of the first 32-row chunk. Events are used once,
 * then forgotten. Returns DFLASH_EINVAL for a NULL handle or an unknown kind. */
enum {
  DFLASH_PROBE_LM_HEAD = 0,
  DFLASH_PROBE_QKV = 1,
  DFLASH_PROBE_ATTN = 2,
  DFLASH_PROBE_O = 3,
  DFLASH_PROBE_GATE_UP = 4,
  DFLASH_PROBE_DOWN = 5,
  DFLASH_PROBE_WC = 6,
  DFLASH_PROBE_CTX_KV = 7
};
int dflash_set_probe(dflash_handle* h, int kernel, void* start_event, void* stop_event);

/* Kernel launches issued by this handle since create (all calls), for launch accounting. */
uint64_t dflash_launch_count(const dflash_handle* h);

/* ---- many-row contraction over a stored drafter matrix (tcgen05 tensor cores) -----------------
 * y[r][n] = sum_k x[r][k] W[n][k] for r < n_rows, with W one of the drafter's 4-bit matrices as
 * stored in the handle (the dflash.ts page's linear maps of Eq 2 and Eq 3, the FFN and the
 * borrowed LM head; each weight is the group-64 affine code w = scale * q + bias). It serves
 * batches of activation rows (up to DFLASH_ROWS_MATMUL_MAX rows per call) in one pass over the
 * weights, where the draft round's skinny per-request projections would stream them once per 32
 * rows; the draft round's large_batch_tc05 option runs its projections on it. */
#define DFLASH_ROWS_MATMUL_MAX 160
enum {
  DFLASH_MAT_CTX = 0,    /* W_c [d][n_taps*H] (Eq 2) */
  DFLASH_MAT_QKV = 1,    /* layer's [W_q; W_k; W_v] [qd + 2 kvd][d] (Eq 3) */
  DFLASH_MAT_O = 2,      /* layer's W_o [d][qd] */
  DFLASH_MAT_GATEUP = 3, /* layer's [W_gate; W_up] [2 inter][d]; y columns gate rows first */
  DFLASH_MAT_DOWN = 4,   /* layer's W_down [d][inter] */
  DFLASH_MAT_LM = 5      /* borrowed LM head [vocab][H] */
};

/* Launch geometry and caller scratch of dflash_rows_matmul for a matrix of n_out rows and k_in
 * inputs (k_in % 64 == 0), n_rows activation rows, with (x_lo != 0) or without the activations'
 * f16 remainder, on a device with n_sm SMs: the shape (tiles per CTA, K slices) with the shortest
 * modelled time, CTAs dispatched in index order to the SM that frees first. Host only. Returns DFLASH_OK, DFLASH_EINVAL for bad
 * sizes or a NULL plan, DFLASH_ECAPACITY for n_rows > DFLASH_ROWS_MATMUL_MAX. */
typedef struct {
  int n_pad;            /* activation rows padded to a multiple of 16 (the MMA's N) */
  int m_tiles;          /* 128-row output tiles */
  int k_slices;         /* K slices per tile (their partial tiles are summed in slice order) */
  int groups_per_slice; /* 64-input groups per K slice */
  int grid;             /* CTAs = tile_groups * k_slices */
  int x_stages;         /* activation ring depth */
  int tile_groups;      /* groups of consecutive output tiles, one per CTA and K slice: */
  int tiles_big;        /*   the first big_groups hold tiles_big tiles (1-3), */
  int big_groups;
  int tiles_small;      /*   the others tiles_small (the last possibly fewer) */
  int w_stages;         /* ring depth of the raw 4-bit tiles, w_groups 64-input groups per stage */
  int w_groups;
  int a_stages;         /* ring depth of the dequantised f16 tiles (one group per stage) */
  int x_groups;         /* 64-input groups per activation stage */
  size_t smem_bytes;    /* dynamic shared memory per CTA */
  size_t scratch_bytes; /* scratch dflash_rows_matmul needs */
} dflash_rows_plan;
int dflash_rows_matmul_plan(int n_out, int k_in, int n_rows, int x_lo, int n_sm, dflash_rows_plan* plan);

/* x: device f16 [n_rows][ldx] (ldx >= k_in, ldx % 8 == 0, 16-byte aligned); x_lo: NULL or the
 * f16 remainder of x in the same layout (x + x_lo is the activation). y: device fp32
 * [n_rows][ldy], ldy >= n_out, in the matrix's natural row order. scratch: device, 256-byte
 * aligned, >= the plan's scratch_bytes, owned by the caller and free for the call's duration.
 * layer is ignored for DFLASH_MAT_CTX and DFLASH_MAT_LM. Enqueued on `stream`; nothing is
 * allocated. Returns DFLASH_EINVAL (bad arguments, or a handle whose weights are not 4-bit),
 * DFLASH_ECAPACITY (n_rows > DFLASH_ROWS_MATMUL_MAX or scratch too small), DFLASH_ECUDA. A bounded
 * wait that gives up sets the handle's error word (dflash_check_errors -> DFLASH_ETIMEOUT) and
 * leaves y undefined. */
int dflash_rows_matmul(dflash_handle* h, int matrix, int layer, int n_rows, const void* x, const void* x_lo,
                       int ldx, float* y, int ldy, void* scratch, size_t scratch_bytes, void* stream);

void dflash_destroy(dflash_handle* h);

/* Allocation-free greedy token and softmax confidence for logits the caller already holds.
 * The pages describe no such call; it exists for callers that cannot allocate device memory on
 * their request path (an engine whose memory pool already owns the GPU, or a host process that
 * forbids the library from calling cudaMalloc) and therefore cannot provide a dflash_create
 * workspace. It runs the same vocab reduction as the LM-head epilogue of dflash_draft_block:
 * token[r] = argmax_j logits[r][j] (lowest index on ties), conf[r] = 1 / sum_j exp(l_rj - max)
 * (conf may be NULL). logits: device fp32 [rows][vocab], never NaN; an entry of -inf is masked
 * out (it never wins and adds nothing to the sum), and a row whose every entry is -inf has no
 * greedy token: token -1, conf 0. token: device int32 [rows].
 * It allocates nothing: its scratch is a fixed ~49 KB array inside the library that every
 * device loading the library keeps until the process exits. Limits: rows <= 64
 * (DFLASH_NOALLOC_MAX_ROWS; more returns DFLASH_ECAPACITY), 2 <= vocab < 2^31.
 * The first call on each device looks up that array's device address (with the device
 * current), so make that first call before any stream capture. All calls share the array:
 * calls that can overlap on the GPU (different streams, different threads) race and must be
 * serialised by the caller. No handle is needed. */
#define DFLASH_NOALLOC_MAX_ROWS 64
int dflash_greedy_from_logits_noalloc(const float* logits, int rows, int vocab, int32_t* token, float* conf,
                                      void* stream);

const char* dflash_status_str(int status);

#ifdef __cplusplus
}
#endif
#endif

/*
 * libdtree — path-conditioned draft-tree construction, built depth by depth in
 * batches, for a Domino-style drafter (parallel backbone + GRU low-rank logit
 * correction), on NVIDIA GB300 (sm_103a).
 *
 * The method (sources are three technical summaries):
 *   "Resumen Técnico: Domino" (Metodología): base logits L^base_i = H_i W_lm
 *     from the frozen LM head; a light GRU summarises the preceding draft
 *     tokens into S_{i-1}; a rank-r bottleneck maps [H_i ; S_{i-1}] to a logit
 *     correction Delta L_i; final logits L_i = L^base_i + Delta L_i.
 *   "Resumen Técnico: DominoTree" (Componentes Principales, 2. Top-M): the
 *     correction is evaluated only on the Top-M base candidates of each depth.
 *   "DARTree: Speculative Diffusion Decoding with Autoregressive Draft Trees"
 *     (Metodología 1, depth-wise parallel expansion; 2, deferred pruning and
 *     Lemma 1): all live branches of a depth are corrected in one batch, the W
 *     best children live on, and one global Top-B over score + beta*depth
 *     (beta <= 0) picks the tree handed to tree-attention verification.
 *   Also: the greedy acceptance walk through an emitted tree given the target
 *   model's logits (dt_accept_walk); marginal scoring, the correction left out
 *   (DT_FLAG_MARGINAL); and the node-by-node conditional best-first builder
 *   that depth batching replaces (DT_FLAG_BEST_FIRST).
 *
 * Conventions of every entry point:
 *   - All device pointers are plain CUDA device addresses owned by the caller
 *     unless stated; bf16 data is passed as `const void*` (IEEE bfloat16).
 *   - Weights use the out-by-in row-major layout of torch.nn.Linear weights.
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  They never synchronise except dt_get_device_status and
 *     dt_build_round_host.
 *   - Errors are returned as dt_status; nothing is thrown across the ABI.
 *     Faults detected on the device (an index out of range, a bounded wait that
 *     gave up) are recorded in the context's device status word and reported
 *     by dt_get_device_status.
 *   - Depth i = 1..D (D = block - 1) uses block position i of H; position 0 is
 *     the last verified token (the root) and its hidden state is not used.
 *   - Super-tree node numbering (per request): node 0 is the root; the nodes
 *     created at depth i follow all nodes of depth i-1, ordered by (parent
 *     index, token id).  Node arrays hold dt_node_count(cfg) + 1 entries per
 *     request.
 *   - Tie rules: Top-M and per-branch top-K prefer the lower token id; top-W and
 *     Top-B prefer the lower node index.
 */
#ifndef DTREE_H_
#define DTREE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dt_status {
  DT_OK = 0,
  DT_ERR_INVALID_ARG = 1,   /* null pointer, out-of-range scalar, calls out of order */
  DT_ERR_SHAPE = 2,         /* sizes the kernels do not support (see dt_check_config) */
  DT_ERR_CUDA = 3,          /* a CUDA runtime call failed */
  DT_ERR_OOM = 4,           /* device allocation failed */
  DT_ERR_TIMEOUT = 5,       /* a device-side bounded wait gave up */
  DT_ERR_UNIMPLEMENTED = 6, /* entry point or mode not built */
  DT_ERR_DEVICE = 7         /* device-side check failed (bad index, non-closed tree) */
} dt_status;

/* Round configuration.  D = block - 1 depths. */
typedef struct dt_config {
  int d;      /* backbone hidden size; multiple of 8 */
  int V;      /* vocabulary size */
  int block;  /* block length (root + D masked positions), 2..64 */
  int g;      /* GRU hidden size */
  int r;      /* correction bottleneck rank */
  int M;      /* Top-M candidates per depth, K <= M <= min(V, 512) */
  int K;      /* children kept per branch, 1..32 */
  int W;      /* live branches kept per depth, 1..64 */
  int B;      /* node budget of the emitted tree (root excluded), B <= N */
  int n_req;  /* independent requests per round; n_req * block <= 512 */
  float beta; /* depth bonus of the Top-B key (score + beta * depth); <= 0 */
  float T;    /* temperature dividing the corrected logits; > 0 */
  unsigned flags; /* DT_FLAG_MARGINAL | DT_FLAG_BEST_FIRST | DT_FLAG_SEPARATE_TOPM | DT_FLAG_POSITIVE_BETA, or 0 */
} dt_config;

/* Marginal scoring over the same super-tree: the correction Delta L is left
 * out, so a node's log-probability depends only on its depth and token and
 * every branch of a depth gets the same children (the conditional-versus-
 * marginal ablation of the DominoTree summary, Contribuciones Clave,
 * "Ablación de la Condicionalidad").  No GRU state is kept; the depth chain
 * runs on one CTA. */
#define DT_FLAG_MARGINAL 1u

/* Sequential conditional best-first construction instead of depth batching:
 * the node-by-node builder of the DominoTree summary (Metodología, 1. Montículo
 * de Mejor Primera Búsqueda con Puntuación Condicional).  The root is
 * expanded, then B pops of the frontier node with the largest score +
 * beta * depth (equal keys: the lower node index; nodes are numbered in
 * creation order, an expansion's K children in token order); each popped
 * node below depth D, except the B-th, gets its GRU state and is expanded with
 * the same correction and log-partition.  The tree is the root plus the popped
 * nodes in ascending node index.  W is not used.  Only dt_build_round and
 * dt_build_round_host build in this mode (dt_expand_depth returns
 * DT_ERR_INVALID_ARG); n_req must be 1, M <= 64 with M % 8 == 0, and the
 * frontier (1 + B*K nodes) must fit in shared memory, else dt_create returns
 * DT_ERR_SHAPE.  Combines with DT_FLAG_MARGINAL. */
#define DT_FLAG_BEST_FIRST 2u

/* The rounds of dt_build_round / dt_build_round_host run the Top-M as its own
 * kernel over logits written by the LM-head GEMM.  Without the flag, a round
 * of one request whose LM-head GEMM has a single 16-wide tile of H rows
 * (block <= 16) and M <= 64 keeps each CTA's Top-M inside the GEMM's
 * epilogue as the logits stream by, does not
 * write the logits, and merges the CTAs' lists in a small kernel; the
 * candidates, their order and the log-partition are the same up to the
 * rounding of the partial sums.  dt_plan_string says which one runs.  The
 * stand-alone dt_base_logits and dt_topm calls are not affected. */
#define DT_FLAG_SEPARATE_TOPM 4u

/* Accept beta > 0 (a bonus for depth instead of a penalty).  The pages state
 * the equivalence of the global Top-B with sequential best-first (DARTree,
 * Metodología, 2. Poda Diferida, Equivalencia Teórica, Lemma 1) for
 * beta <= 0 only; with beta > 0 it does not hold: the global Top-B of the
 * depth-batched builder may select a node without its parent (the tree/mask
 * step then reports DT_DEV_TREE and the selection, dt_prune_topB's output,
 * is still the B largest keys), while the best-first builder
 * (DT_FLAG_BEST_FIRST), whose heap only reaches a node through its parent,
 * always emits a tree.  Without the flag, beta > 0 is DT_ERR_INVALID_ARG. */
#define DT_FLAG_POSITIVE_BETA 8u

/* Frozen weights (device pointers, borrowed: they must outlive the context).
 * All bf16, row-major, torch.nn.Linear out-by-in layout.  GRU gate blocks are
 * ordered (r, z, n); the GRU has one input-side bias and no hidden bias. */
typedef struct dt_weights {
  const void* lm_head; /* [V, d]   row v = output vector of token v (L^base = H lm_head^T) */
  const void* emb;     /* [V, d]   token embeddings E (GRU input) */
  const void* w_ih;    /* [3g, d]  GRU input weights */
  const void* b_ih;    /* [3g]     GRU input bias */
  const void* w_hh;    /* [3g, g]  GRU hidden weights */
  const void* w1;      /* [r, d+g] bottleneck over [H_i ; S_{i-1}] */
  const void* w2;      /* [V, r]   up-projection (row c = column c of W2) */
} dt_weights;

typedef struct dt_ctx dt_ctx;

/* --------------------------------------------------------------------------
 * Host-only helpers (no CUDA calls).
 * ------------------------------------------------------------------------ */

/* Validate a configuration: K <= M <= V, M <= 512, 1 <= K <= 32,
 * 1 <= W <= 64, 2 <= block <= 64, d % 8 == 0, g % 8 == 0, r % 8 == 0,
 * r <= 1024, g <= 4096, n_req * block <= 512, 1 <= B <= N, T > 0, beta <= 0
 * (or finite with DT_FLAG_POSITIVE_BETA), flags within DT_FLAG_MARGINAL |
 * DT_FLAG_BEST_FIRST | DT_FLAG_SEPARATE_TOPM | DT_FLAG_POSITIVE_BETA.
 * Returns DT_OK, DT_ERR_INVALID_ARG or DT_ERR_SHAPE. */
dt_status dt_check_config(const dt_config* cfg);

/* N: super-tree nodes of one request without the root (n_1 = K,
 * n_i = min(W, n_{i-1}) K; DARTree page, fixed-width super-tree).  -1 if cfg
 * is NULL. */
int64_t dt_node_count(const dt_config* cfg);

/* Upper bound on the device bytes that dt_create allocates for this
 * configuration (workspace, GRU input table, captured-round buffers); the
 * Top-M scratch depends on the device's SM count, so the bound assumes the
 * largest plan.  0 if the configuration is invalid. */
size_t dt_workspace_bytes(const dt_config* cfg);

/* Static description of a status code. */
const char* dt_status_string(dt_status s);

/* The CUDA call and error text behind the calling thread's last DT_ERR_CUDA /
 * DT_ERR_OOM ("" if none).  Valid until the thread's next libdtree call. */
const char* dt_last_error(void);

/* --------------------------------------------------------------------------
 * Context.
 * ------------------------------------------------------------------------ */

/* Validate cfg, borrow the weights, allocate the workspace on the current
 * device and build the GRU input table X[v] = E[v] W_ih^T + b_ih ([V, 3g]
 * fp32, an exact regrouping of the GRU input projection; Domino page,
 * Codificador Causal) on `stream`.  *out receives the context.  Errors:
 * INVALID_ARG / SHAPE (bad cfg or null weight), OOM, CUDA. */
dt_status dt_create(const dt_config* cfg, const dt_weights* w, void* stream, dt_ctx** out);

/* Synchronise the context's work, free everything it owns.  NULL is a no-op. */
dt_status dt_destroy(dt_ctx* ctx);

/* --------------------------------------------------------------------------
 * Steps of one round (call in this order; each reads what the previous wrote
 * into the context's workspace).
 * ------------------------------------------------------------------------ */

/* Step 1 — base logits (Domino page, Columna Vertebral, Salida; DominoTree
 * page, Hecho Estructural: H is shared by all paths).
 *   H:      [n_req, block, d] bf16 hidden states of the parallel backbone.
 *   logits: [n_req, D, V] fp32 output, logits[q, i-1, v] = H[q, i] . lm_head[v];
 *           NULL keeps them only in the workspace.
 * Also computes H[q, i] W1[:, :d]^T (the H half of the bottleneck) into the
 * workspace for dt_expand_depth.  One tcgen05/TMA kernel. */
dt_status dt_base_logits(dt_ctx* ctx, const void* H, float* logits, void* stream);

/* Step 2 — Top-M candidates and rest log-partition per (request, depth)
 * (DominoTree page, Top-M restriction; the M corrected entries are
 * substituted into the base log-partition).
 *   logits:    [n_req, D, V] fp32 input, or NULL for the workspace copy.
 *   cand_tok:  [n_req, D, M] int32 out (NULL = workspace only), ordered by
 *              logit descending, token id ascending.
 *   cand_base: [n_req, D, M] fp32 out: base logits of those tokens (not / T).
 *   rest_lse:  [n_req, D] fp32 out: log sum_{v not in C} exp(logit_v / T),
 *              -inf when M == V.
 * Up to one row per SM, each row is split into chunks whose sorted lists are
 * merged; with more rows (e.g. 32 requests), two CTAs per SM stream whole rows
 * behind a rising bound (dt_plan_string says which). */
dt_status dt_topm(dt_ctx* ctx, const float* logits, int32_t* cand_tok, float* cand_base,
                  float* rest_lse, void* stream);

/* Steps 1 and 2 as a round runs them: the LM-head GEMM over H ([n_req,
 * block, d] bf16, device, 16-byte aligned) and the Top-M restriction, either
 * in the GEMM's epilogue with a merge of its CTAs' lists (the logits are not
 * written) or as the Top-M kernel over the logits (DT_FLAG_SEPARATE_TOPM, or a
 * shape the epilogue does not take).  The candidates are then read with
 * dt_last_candidates, and dt_expand_prune builds the tree from them. */
dt_status dt_base_topm(dt_ctx* ctx, const void* H, void* stream);

/* The Top-M restriction the context holds now: that of the last round
 * (dt_build_round, dt_build_round_host: with the Top-M in the LM-head GEMM's
 * epilogue or as its own kernel, see DT_FLAG_SEPARATE_TOPM), of the last
 * dt_base_topm or of the last dt_topm, copied on `stream` into the caller's
 * device buffers (any may be NULL), in the layout of dt_topm's outputs.
 * Before any of those the contents are zero. */
dt_status dt_last_candidates(dt_ctx* ctx, int32_t* cand_tok, float* cand_base, float* rest_lse,
                             void* stream);

/* Step 3 — one depth of the batched expansion (DARTree page, Metodología 1;
 * Domino page, Cabeza de Domino).  For every live branch p of depth-1:
 * z = SiLU([H_i ; S(p)] W1^T), lambda_c = (L^base_{i,c} + z . W2[c]) / T on the
 * Top-M candidates c, logp = lambda - log(e^rest_lse + sum_c e^lambda_c); the K
 * best children per branch get score(p) + logp; the W best children of the
 * depth keep a GRU state S = GRU(E[token], S(p)).
 *   depth:     1..D; depths must be called in order 1, 2, ..., D.
 *   root_tok:  [n_req] int32, read at depth 1 (the last verified token).
 *   node_*:    [n_req, N+1] outputs (N = dt_node_count); depth i writes the
 *              entries of its own nodes (depth 1 also writes the root, node 0:
 *              token root_tok, parent -1, logp 0, score 0).
 *              node_tok int32, node_parent int32 (node index), node_logp fp32
 *              (the node's conditional log-prob), node_score fp32 (cumulative).
 *   live:      [n_req, W] int32 out or NULL: node indices of the branches that
 *              live on after this depth, ascending, padded with -1.
 * The same node buffers must be passed at every depth of a round. */
dt_status dt_expand_depth(dt_ctx* ctx, int depth, const int32_t* root_tok, int32_t* node_tok,
                          int32_t* node_parent, float* node_logp, float* node_score,
                          int32_t* live, void* stream);

/* Step 4 — deferred pruning (DARTree page, Poda Diferida: Selección Global,
 * Equivalencia Teórica).
 *   node_score: [n_req, N+1] fp32 (from dt_expand_depth).
 *   sel:        [n_req, B] int32 out: the B non-root nodes with the largest
 *               node_score + beta * depth, ties to the lower index, ascending. */
dt_status dt_prune_topB(dt_ctx* ctx, const float* node_score, int32_t* sel, void* stream);

/* Step 5 — compact tree and ancestor-only attention mask (DominoTree page,
 * Verificación; DARTree page, Verificación).  Tree slot 0 is the root, slots
 * 1..B the selected nodes in ascending node order.
 *   sel, node_tok, node_parent, node_score: inputs from steps 3-4.
 *   tok, parent, depth: [n_req, B+1] int32 out (parent = slot of the parent,
 *   -1 for the root); logp_cum: [n_req, B+1] fp32 out (cumulative score);
 *   mask: [n_req, B+1, B+1] uint8 out, mask[a][b] = 1 iff slot b is slot a or
 *   one of its ancestors.  A parent missing from the selection (impossible for
 *   beta <= 0) is recorded in the device status word. */
dt_status dt_tree_mask(dt_ctx* ctx, const int32_t* sel, const int32_t* node_tok,
                       const int32_t* node_parent, const float* node_score, int32_t* tok,
                       int32_t* parent, int32_t* depth, float* logp_cum, uint8_t* mask,
                       void* stream);

/* Step 6 — greedy verification of the emitted trees: the acceptance walk
 * (DominoTree page, Metodología, 5. Verificación; Resultados Experimentales,
 * Ausencia de Pérdida).  The target model has scored every tree slot in one
 * pass with the ancestor-only mask; its token after slot a is the argmax of its
 * logits at a (equal maxima: the lower token id).  From the root, the walk
 * moves into the child whose draft token equals the target's token at the
 * current slot, while one exists; the target's token at the last slot reached
 * is the bonus token, so accept_len + 1 tokens are committed.
 *   target_logits: [n_req, B+1, V] fp32, finite, 16-byte aligned when V is a
 *                  multiple of 4 (row q, a = the target's logits at slot a).
 *   tok, parent:   [n_req, B+1] int32, a tree in dt_tree_mask's layout
 *                  (parent[0] = -1, parent[c] < c, sibling tokens distinct).
 *   target_tok:    [n_req, B+1] int32 out, or NULL: the target's token per slot.
 *   accepted:      [n_req, D] int32 out: the accepted slots in path order,
 *                  padded with -1.
 *   accept_len:    [n_req] int32 out; bonus: [n_req] int32 out.
 * All device pointers, caller-owned.  One launch; the logits are read once.
 * A parent index outside [0, c) or two siblings carrying the accepted token
 * are recorded in the device status word (DT_DEV_TREE); the lower slot is then
 * taken.  B+1 > 3072 returns DT_ERR_SHAPE. */
dt_status dt_accept_walk(dt_ctx* ctx, const float* target_logits, const int32_t* tok,
                         const int32_t* parent, int32_t* target_tok, int32_t* accepted,
                         int32_t* accept_len, int32_t* bonus, void* stream);

/* Steps 3-5 in as few launches as the shape allows (one for a single request):
 * every depth of the expansion, the global Top-B and the tree/mask, from the
 * Top-M results that the last dt_topm, dt_base_topm or round left in the
 * workspace (or, with
 * DT_FLAG_BEST_FIRST, the best-first builder).  Node arrays and the selection
 * stay in the workspace.
 *   root_tok: [n_req] int32; outputs as dt_tree_mask.
 * A later dt_expand_depth starts a new round at depth 1. */
dt_status dt_expand_prune(dt_ctx* ctx, const int32_t* root_tok, int32_t* tok, int32_t* parent, int32_t* depth,
                          float* logp_cum, uint8_t* mask, void* stream);

/* --------------------------------------------------------------------------
 * Whole round.
 * ------------------------------------------------------------------------ */

/* Steps 1-5 for one round as one CUDA-graph replay on `stream`.  The graph is
 * captured on the first call with a given set of pointer arguments; the
 * context keeps up to 16 captured rounds (least recently used is replaced).
 * H and root_tok as above; outputs as dt_tree_mask.  Intermediate arrays stay
 * in the workspace. */
dt_status dt_build_round(dt_ctx* ctx, const void* H, const int32_t* root_tok, int32_t* tok,
                         int32_t* parent, int32_t* depth, float* logp_cum, uint8_t* mask,
                         void* stream);

/* dt_build_round with HOST buffers: copies H (bf16, [n_req, block, d]) and
 * root_tok to the device, replays the round, copies the outputs back and
 * synchronises `stream`.  Host buffers should be pinned for full speed. */
dt_status dt_build_round_host(dt_ctx* ctx, const void* H_host, const int32_t* root_host,
                              int32_t* tok_host, int32_t* parent_host, int32_t* depth_host,
                              float* logp_cum_host, uint8_t* mask_host, void* stream);

/* --------------------------------------------------------------------------
 * Step 2 without allocation.  The pages have no counterpart of this entry
 * point: it exists for callers that must not allocate device memory — a
 * serving process that fixes its GPU memory budget at start-up, code embedded
 * in another framework whose allocator owns the device, or a loop that cannot
 * afford the implicit synchronisation cudaMalloc/cudaFree bring.
 *
 * dt_topm_noalloc computes what dt_topm computes, with no context:
 *   logits:    [rows, V] fp32 input.
 *   cand_tok:  [rows, M] int32 out, logit descending, token id ascending.
 *   cand_base: [rows, M] fp32 out, the base logits of those tokens.
 *   rest_lse:  [rows] fp32 out, log sum over the non-candidates of exp(logit/T).
 * It allocates nothing: its scratch is one fixed 4 MiB array of device memory
 * inside the library, which every GPU that loads the library keeps until the
 * process exits.  A call needs about rows * S * (8 M + 16) + 4 rows bytes of
 * it, where S, the chunks each row is split into, is
 *   S = min(max(SMs / rows, ceil(V / 16384), 1), max(V / (2 M), 1),
 *           max(8192 / M, 1))          (integer divisions, SMs = the device's)
 * and each chunk must hold at most 16384 logits.  (With at least one row per
 * SM, V a multiple of 4 and 16-byte aligned logits, each row is streamed whole
 * by one CTA instead and the array is not used; the bound above still
 * applies.)  Calls beyond the array, with
 * rows > 65535, M > 512, or a chunk above 16384 logits (V > 8192 * 16384 / M)
 * are rejected with DT_ERR_SHAPE and a message in dt_last_error(), before any
 * work is queued.
 * The first call on each device does a one-time set-up (it looks up the
 * array's device address and sets a kernel attribute), so make that first
 * call before any stream capture.  All calls on a device share that device's
 * array, which keeps the previous call's contents (the call clears what must
 * start at zero): calls that overlap on the GPU, for example on two streams,
 * race and must be ordered by the caller.  Asynchronous on `stream`.
 * Device-side index checks are not reported (there is no status word).
 * Errors: INVALID_ARG (null pointer, M > V, T <= 0), SHAPE, CUDA.
 * ------------------------------------------------------------------------ */
dt_status dt_topm_noalloc(const float* logits, int rows, int V, int M, float T, int32_t* cand_tok,
                          float* cand_base, float* rest_lse, void* stream);

/* Synchronise the context's last stream and read (and clear) its device status
 * word: DT_OK, DT_ERR_TIMEOUT or DT_ERR_DEVICE. */
dt_status dt_get_device_status(dt_ctx* ctx);

/* Self-check of the bounded device-side waits, on the context's status word:
 * which = 0 launches a grid barrier of two CTAs that one CTA never reaches,
 * which = 1 a wait on an mbarrier phase that nothing completes.  The waiting
 * thread gives up after the wait limit (2 s), records the timeout and returns;
 * dt_get_device_status then returns DT_ERR_TIMEOUT and the context stays
 * usable.  Returns DT_ERR_INVALID_ARG for another `which`.
 *
 * Host-side fault injection: with DT_FAULT_INJECT_ALLOC set in the
 * environment, dt_create fails its workspace allocation as an out-of-memory
 * would (DT_ERR_OOM, nothing leaked). */
dt_status dt_check_bounded_waits(dt_ctx* ctx, int which, void* stream);

/* Number of kernel launches one dt_build_round replay performs. */
int dt_round_kernel_count(const dt_ctx* ctx);

/* Which kernels the context's rounds run, chosen at dt_create from the shape,
 * the flags and the device: the Top-M in the LM-head GEMM's epilogue (with the
 * number of CTA lists merged) or the Top-M kernel (with its chunks per row);
 * then, for one request, the clustered depth chain with its cluster size, or
 * the grid-barrier chain and the reason.  Owned by the context; "" for NULL. */
const char* dt_plan_string(const dt_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* DTREE_H_ */

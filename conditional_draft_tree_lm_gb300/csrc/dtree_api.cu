// libdtree C ABI: context, workspace, step launches and the captured round.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "common.cuh"
#include "kernels.h"

using namespace dt;

namespace {

struct Tables {
  int D = 0;
  int N = 0;  // non-root nodes
  int off[kMaxDepth + 2] = {};
  int nn[kMaxDepth + 1] = {};
  int L[kMaxDepth + 1] = {};
};

bool make_tables(const dt_config& c, Tables& t) {
  t.D = c.block - 1;
  if (t.D < 1 || t.D > kMaxDepth) return false;
  t.L[0] = 1;
  t.off[1] = 1;
  long long total = 0;
  for (int i = 1; i <= t.D; ++i) {
    t.nn[i] = t.L[i - 1] * c.K;
    t.L[i] = t.nn[i] < c.W ? t.nn[i] : c.W;
    total += t.nn[i];
    if (total > (1 << 24)) return false;
    t.off[i + 1] = t.off[i] + t.nn[i];
  }
  t.N = static_cast<int>(total);
  return true;
}

dt_status check(const dt_config* c) {
  if (!c) return DT_ERR_INVALID_ARG;
  if ((c->flags & ~(DT_FLAG_MARGINAL | DT_FLAG_BEST_FIRST | DT_FLAG_SEPARATE_TOPM | DT_FLAG_POSITIVE_BETA)) != 0)
    return DT_ERR_INVALID_ARG;
  if ((c->flags & DT_FLAG_BEST_FIRST) && c->n_req != 1) return DT_ERR_SHAPE;
  if (c->d <= 0 || c->V <= 0 || c->g <= 0 || c->r <= 0 || c->M <= 0 || c->K <= 0 || c->W <= 0 ||
      c->B <= 0 || c->n_req <= 0 || c->block < 2)
    return DT_ERR_INVALID_ARG;
  if (!(c->T > 0.0f) || !(c->beta <= 0.0f || ((c->flags & DT_FLAG_POSITIVE_BETA) && c->beta < INFINITY)))
    return DT_ERR_INVALID_ARG;
  if (c->K > c->M || c->M > c->V) return DT_ERR_INVALID_ARG;
  if (c->block > kMaxDepth) return DT_ERR_SHAPE;  // depths 1..63: off[D+1] stays inside the tables
  if (c->M > 512 || c->K > 32 || c->W > 64) return DT_ERR_SHAPE;
  if (c->d % 8 != 0 || c->g % 8 != 0 || c->r % 8 != 0) return DT_ERR_SHAPE;
  if (c->r > 1024 || c->g > 1024) return DT_ERR_SHAPE;
  if (static_cast<long long>(c->n_req) * c->block > 512) return DT_ERR_SHAPE;
  Tables t;
  if (!make_tables(*c, t)) return DT_ERR_SHAPE;
  if (c->B > t.N) return DT_ERR_INVALID_ARG;
  // Top-B in shared memory: N+1 float keys and up to 8192 candidate keys
  if (static_cast<long long>(t.N + 1) * 4 + static_cast<long long>(t.N < 8192 ? t.N : 8192) * 8 > 190 * 1024)
    return DT_ERR_SHAPE;
  if (c->n_req * c->W * 3 * 8 * 4 > 64 * 1024) return DT_ERR_SHAPE;  // chain state projections
  return DT_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Layout {
  size_t fpart_id, fpart_val, fpart_max, fpart_sum, fpart_cnt, fpart_tail;
  size_t logits, h1, part_id, part_val, part_max, part_sum, part_cnt, part_kth, cand_tok, cand_base, rest_lse,
      row_done, S, sfrag, zfrag,
      uW1, live, node_tok, node_parent, node_logp, node_score, sel, bar, status, H_dev, root_dev,
      out_tok, out_parent, out_depth, out_logp, out_mask, acc_key, acc_done, xch, xch_words, total;
  size_t xtab;
};

// fs: the partial lists per row of the fused Top-M (the LM-head GEMM's grid),
// or 0 when the rounds do not fuse it.
void layout(const dt_config& c, const Tables& t, const TopmParams& tp, Layout& L, int fs) {
  const size_t rows = static_cast<size_t>(c.n_req) * t.D;
  const size_t N1 = static_cast<size_t>(t.N) + 1;
  const size_t S1 = static_cast<size_t>(c.B) + 1;
  size_t o = 0;
  auto put = [&](size_t& f, size_t bytes) {
    f = o;
    o = align256(o + bytes);
  };
  put(L.logits, rows * c.V * 4);
  put(L.h1, rows * c.r * 4);
  put(L.part_id, rows * tp.S * c.M * 4);
  put(L.part_val, rows * tp.S * c.M * 4);
  put(L.part_max, rows * tp.S * 4);
  put(L.part_sum, rows * tp.S * 4);
  put(L.part_cnt, rows * tp.S * 4);
  put(L.part_kth, rows * tp.S * 4);
  put(L.cand_tok, rows * c.M * 4);
  put(L.cand_base, rows * c.M * 4);
  put(L.rest_lse, rows * 4);
  put(L.row_done, rows * 4);
  put(L.S, 2ull * c.n_req * c.W * c.g * 4);
  // two parities of the states' hi/lo copy; rows padded to whole tiles of 128
  // for the tcgen05 operand layout
  put(L.sfrag, 2ull * ((static_cast<size_t>(c.n_req) * c.W + 127) / 128 * 128) * c.g * 4);
  put(L.zfrag, static_cast<size_t>(c.n_req) * c.W * c.r * 4);
  put(L.uW1, static_cast<size_t>(c.n_req) * c.W * c.r * 4);
  put(L.live, 2ull * c.n_req * c.W * 4);
  put(L.node_tok, c.n_req * N1 * 4);
  put(L.node_parent, c.n_req * N1 * 4);
  put(L.node_logp, c.n_req * N1 * 4);
  put(L.node_score, c.n_req * N1 * 4);
  put(L.sel, static_cast<size_t>(c.n_req) * c.B * 4);
  put(L.bar, 256);
  put(L.status, 256);
  // clustered chain: [2][g/8][8 rows][4] 16-byte tagged words, then its epoch
  // and abort words
  put(L.xch, 2ull * (c.g / 8) * 8 * 4 * 16);
  put(L.xch_words, 256);
  put(L.H_dev, static_cast<size_t>(c.n_req) * c.block * c.d * 2);
  put(L.root_dev, static_cast<size_t>(c.n_req) * 4);
  put(L.out_tok, c.n_req * S1 * 4);
  put(L.out_parent, c.n_req * S1 * 4);
  put(L.out_depth, c.n_req * S1 * 4);
  put(L.out_logp, c.n_req * S1 * 4);
  put(L.out_mask, c.n_req * S1 * S1);
  put(L.acc_key, c.n_req * S1 * 8);
  put(L.acc_done, static_cast<size_t>(c.n_req) * 8);
  put(L.fpart_id, rows * fs * c.M * 4);
  put(L.fpart_val, rows * fs * c.M * 4);
  put(L.fpart_max, rows * fs * 4);
  put(L.fpart_sum, rows * fs * 4);
  put(L.fpart_cnt, rows * fs * 4);
  put(L.fpart_tail, rows * fs * c.M * 4);
  L.total = o;
  L.xtab = static_cast<size_t>(c.V) * 3 * c.g * 4;
}

// Tile width of the LM-head GEMM over the H rows (the swap-AB N dimension):
// up to 256 rows in one tile; more rows in several 256-wide tiles, which keeps
// four pipeline stages and double-buffered accumulators (the two tiles of a
// vocabulary block run on neighbouring CTAs, so its weights come from HBM once).
int logits_bn(const dt_config& c) {
  const int n = c.n_req * c.block;
  int bn = (n + 15) / 16 * 16;
  if (bn > 256) bn = 256;
  return bn;
}

}  // namespace

struct dt_ctx {
  dt_config cfg;
  dt_weights w;
  Tables t;
  Layout lay;
  int device = 0;
  int num_sms = 0;
  uint8_t* ws = nullptr;
  float* xtab = nullptr;
  CUtensorMap tm_lm, tm_w1h;
  TopmParams topm;
  int fuse_topm = 0;  // rounds keep the Top-M in the LM-head GEMM's epilogue
  TopmParams fmerge;  // the merge of the GEMM CTAs' lists
  AcceptParams acc;
  BestParams best;
  int best_first = 0;
  int chain_grid = 0;
  int use_dchain = 0;  // one request: the clustered depth chain (dchain.cu)
  int dchain_cs = 0;
  int dchain_jc = 0;
  char plan[384] = "";  // which kernels a round runs (dt_plan_string)
  const float* logits_src = nullptr;
  int next_depth = 1;
  cudaStream_t cap_stream = nullptr;
  // captured rounds, keyed by the pointer arguments of dt_build_round
  static constexpr int kGraphCache = 16;
  struct Captured {
    const void* key[8] = {};
    cudaGraphExec_t exec = nullptr;
    unsigned long long used = 0;
  } graphs[kGraphCache];
  unsigned long long graph_clock = 0;
  cudaStream_t last_stream = nullptr;

  template <class T>
  T* at(size_t off) { return reinterpret_cast<T*>(ws + off); }
};

namespace {

thread_local char g_last_error[256] = "";

dt_status cuda_status(cudaError_t e, const char* what = "") {
  if (e == cudaSuccess) return DT_OK;
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%d)", what, cudaGetErrorString(e), static_cast<int>(e));
  if (e == cudaErrorMemoryAllocation) return DT_ERR_OOM;
  return DT_ERR_CUDA;
}

#define DT_TRY(x)                                      \
  do {                                                 \
    cudaError_t _e = (x);                              \
    if (_e != cudaSuccess) return cuda_status(_e, #x); \
  } while (0)

// The launch shape of the LM-head GEMM over one round's H rows (no pointers).
GemmParams logits_gemm_params(const dt_config& k, const Tables& t) {
  const int BN = logits_bn(k);
  GemmParams p = {};
  p.mode = GEMM_LOGITS;
  p.K = k.d;
  p.m_tiles_a = (k.V + 127) / 128;
  p.m_tiles_a2 = (k.r + 127) / 128;
  p.n_tiles = (k.n_req * k.block + BN - 1) / BN;
  p.n_valid = k.n_req * k.block;
  p.a_evict_first = 1;
  p.rows_a = k.V;
  p.rows_a2 = k.r;
  p.block = k.block;
  p.D = t.D;
  gemm_plan(p, BN);
  p.ft_P = t.D;
  p.ft_M = k.M;
  p.ft_invT = 1.0f / k.T;
  return p;
}

// fused: the Top-M runs in the epilogue (dt_ctx::fuse_topm) and the logits
// are not written (logits may be null).
dt_status enqueue_base_logits(dt_ctx* c, const void* H, float* logits, cudaStream_t st, bool fused = false) {
  const dt_config& k = c->cfg;
  const int BN = logits_bn(k);
  CUtensorMap tm_h;
  if (!make_tmap_bf16_2d(&tm_h, H, k.d, static_cast<uint64_t>(k.n_req) * k.block,
                         static_cast<uint64_t>(k.d) * 2, BN > 256 ? 256 : BN))
    return DT_ERR_INVALID_ARG;
  GemmParams p = logits_gemm_params(k, c->t);
  p.logits = fused ? nullptr : logits;
  p.h1 = c->at<float>(c->lay.h1);
  p.status = c->at<int>(c->lay.status);
  if (fused) {
    gemm_ft_plan(p);
    p.part_id = c->fmerge.part_id;
    p.part_val = c->fmerge.part_val;
    p.part_max = c->fmerge.part_max;
    p.part_sum = c->fmerge.part_sum;
    p.part_cnt = c->fmerge.part_cnt;
    p.part_kth = nullptr;
    p.part_tail = c->fmerge.part_tail;
  }
  DT_TRY(launch_gemm_tc(c->tm_lm, c->tm_w1h, tm_h, p, c->num_sms, st));
  return DT_OK;
}

// clear: a word Top-M sets to zero (the following chain's barrier counter),
// or null; pdl: launch as a programmatic dependent of the LM-head GEMM.
dt_status enqueue_topm(dt_ctx* c, const float* logits, cudaStream_t st, unsigned* clear = nullptr, int pdl = 0) {
  TopmParams p = c->topm;
  p.logits = logits;
  p.clear_word = clear;
  p.pdl = pdl;
  DT_TRY(launch_topm(p, st));
  return DT_OK;
}

ChainParams chain_params(dt_ctx* c, const int32_t* root, int32_t* ntok, int32_t* npar, float* nlogp,
                         float* nscore, int32_t* live_out) {
  const dt_config& k = c->cfg;
  ChainParams p = {};
  p.n_req = k.n_req;
  p.D = c->t.D;
  p.g = k.g;
  p.r = k.r;
  p.M = k.M;
  p.K = k.K;
  p.W = k.W;
  p.V = k.V;
  p.d = k.d;
  p.ldw1 = k.d + k.g;
  p.N1 = c->t.N + 1;
  p.T = k.T;
  p.marginal = (k.flags & DT_FLAG_MARGINAL) ? 1 : 0;
  p.w_hh = static_cast<const uint16_t*>(c->w.w_hh);
  p.w1 = static_cast<const uint16_t*>(c->w.w1);
  p.w2 = static_cast<const uint16_t*>(c->w.w2);
  p.xtab = c->xtab;
  p.h1 = c->at<float>(c->lay.h1);
  p.cand_tok = c->at<int>(c->lay.cand_tok);
  p.cand_base = c->at<float>(c->lay.cand_base);
  p.rest_lse = c->at<float>(c->lay.rest_lse);
  p.root_tok = root;
  p.S = c->at<float>(c->lay.S);
  p.sfrag = c->at<uint32_t>(c->lay.sfrag);
  p.zfrag = c->at<uint32_t>(c->lay.zfrag);
  p.uW1 = c->at<float>(c->lay.uW1);
  p.live = c->at<int>(c->lay.live);
  p.node_tok = ntok;
  p.node_parent = npar;
  p.node_logp = nlogp;
  p.node_score = nscore;
  p.live_out = live_out;
  p.bar = c->at<unsigned>(c->lay.bar);
  p.status = c->at<int>(c->lay.status);
  for (int i = 0; i <= kMaxDepth; ++i) {
    p.off[i] = c->t.off[i];
    p.nn[i] = c->t.nn[i];
    p.L[i] = c->t.L[i];
  }
  chain_plan(p, c->chain_grid);
  return p;
}

DchainParams dchain_params(dt_ctx* c, const int32_t* root, int32_t* ntok, int32_t* npar, float* nlogp,
                           float* nscore, int32_t* live_out) {
  const dt_config& k = c->cfg;
  DchainParams p = {};
  p.D = c->t.D;
  p.g = k.g;
  p.r = k.r;
  p.M = k.M;
  p.K = k.K;
  p.W = k.W;
  p.V = k.V;
  p.d = k.d;
  p.ldw1 = k.d + k.g;
  p.N1 = c->t.N + 1;
  p.T = k.T;
  p.w_hh = static_cast<const uint16_t*>(c->w.w_hh);
  p.w1 = static_cast<const uint16_t*>(c->w.w1);
  p.w2 = static_cast<const uint16_t*>(c->w.w2);
  p.xtab = c->xtab;
  p.h1 = c->ws ? c->at<float>(c->lay.h1) : nullptr;
  p.cand_tok = c->ws ? c->at<int>(c->lay.cand_tok) : nullptr;
  p.cand_base = c->ws ? c->at<float>(c->lay.cand_base) : nullptr;
  p.rest_lse = c->ws ? c->at<float>(c->lay.rest_lse) : nullptr;
  p.root_tok = root;
  p.S = c->ws ? c->at<float>(c->lay.S) : nullptr;
  p.live = c->ws ? c->at<int>(c->lay.live) : nullptr;
  p.xch = c->ws ? c->at<void>(c->lay.xch) : nullptr;
  p.epoch = c->ws ? c->at<unsigned>(c->lay.xch_words) : nullptr;
  p.abort_word = p.epoch ? p.epoch + 1 : nullptr;
  p.node_tok = ntok;
  p.node_parent = npar;
  p.node_logp = nlogp;
  p.node_score = nscore;
  p.live_out = live_out;
  p.status = c->ws ? c->at<int>(c->lay.status) : nullptr;
  p.cs = c->dchain_cs;
  p.jc = c->dchain_jc;
  p.B = k.B;
  p.beta = k.beta;
  for (int i = 0; i <= kMaxDepth; ++i) p.L[i] = c->t.L[i];
  for (int i = 0; i <= kMaxDepth + 1; ++i) p.off[i] = c->t.off[i];
  return p;
}

// counter_cleared: the preceding Top-M kernel already zeroed the barrier
// counter (the whole-round path), so no memset is enqueued.
dt_status enqueue_chain(dt_ctx* c, const ChainParams& p, cudaStream_t st, bool counter_cleared = false) {
  if (!counter_cleared) DT_TRY(cudaMemsetAsync(p.bar, 0, sizeof(unsigned), st));
  DT_TRY(launch_chain(p, c->chain_grid, st));
  return DT_OK;
}

PruneParams prune_params(dt_ctx* c, const float* nscore, int32_t* sel) {
  PruneParams p = {};
  p.n_req = c->cfg.n_req;
  p.N1 = c->t.N + 1;
  p.B = c->cfg.B;
  p.D = c->t.D;
  p.beta = c->cfg.beta;
  p.node_score = nscore;
  p.sel = sel;
  p.status = c->at<int>(c->lay.status);
  for (int i = 0; i <= c->t.D + 1 && i < kMaxDepth + 2; ++i) p.off[i] = c->t.off[i];
  return p;
}

// Steps 3-5 of a round from the workspace's Top-M results: the depth-batched
// expansion (or the best-first builder) with the global Top-B and the
// tree/mask.  chained: launched right after Top-M in the same round, as
// programmatic dependents, with the barrier counter already cleared by Top-M;
// otherwise the counter is cleared here and the launches are ordinary.
dt_status enqueue_build(dt_ctx* c, const int32_t* root, int32_t* tok, int32_t* parent, int32_t* depth,
                        float* logp_cum, uint8_t* mask, cudaStream_t st, bool chained) {
  unsigned* bar = c->at<unsigned>(c->lay.bar);
  if (!chained) DT_TRY(cudaMemsetAsync(bar, 0, sizeof(unsigned), st));
  const int pdl = chained ? 1 : 0;
  int32_t* sel = c->at<int32_t>(c->lay.sel);
  if (c->best_first) {
    BestParams bp = c->best;
    bp.w_hh = static_cast<const uint16_t*>(c->w.w_hh);
    bp.w1 = static_cast<const uint16_t*>(c->w.w1);
    bp.w2 = static_cast<const uint16_t*>(c->w.w2);
    bp.xtab = c->xtab;
    bp.h1 = c->at<float>(c->lay.h1);
    bp.cand_tok = c->at<int>(c->lay.cand_tok);
    bp.cand_base = c->at<float>(c->lay.cand_base);
    bp.rest_lse = c->at<float>(c->lay.rest_lse);
    bp.root_tok = root;
    bp.srow = c->at<float>(c->lay.S);
    bp.zrow = c->at<float>(c->lay.uW1);
    bp.bar = bar;
    bp.status = c->at<int>(c->lay.status);
    bp.pdl = pdl;
    bp.sel = sel;
    bp.pops = nullptr;
    bp.tok = tok;
    bp.parent = parent;
    bp.depth = depth;
    bp.logp_cum = logp_cum;
    bp.mask = mask;
    DT_TRY(launch_best(bp, c->chain_grid, st));
    return DT_OK;
  }
  int32_t* ntok = c->at<int32_t>(c->lay.node_tok);
  int32_t* npar = c->at<int32_t>(c->lay.node_parent);
  float* nlogp = c->at<float>(c->lay.node_logp);
  float* nscore = c->at<float>(c->lay.node_score);
  if (c->use_dchain) {
    // one request: all depths, the Top-B and the tree/mask in one clustered launch
    DchainParams dp = dchain_params(c, root, ntok, npar, nlogp, nscore, nullptr);
    dp.depth_first = 1;
    dp.depth_last = c->t.D;
    dp.pdl = pdl;
    dp.fuse_tree = 1;
    dp.sel = sel;
    dp.tok = tok;
    dp.parent = parent;
    dp.depth = depth;
    dp.logp_cum = logp_cum;
    dp.mask = mask;
    DT_TRY(launch_dchain(dp, st));
    return DT_OK;
  }
  ChainParams cp = chain_params(c, root, ntok, npar, nlogp, nscore, nullptr);
  cp.depth_first = 1;
  cp.depth_last = c->t.D;
  cp.pdl = pdl;
  if (chain_can_fuse_tree(cp)) {
    // single request: the chain kernel's CTA 0 also prunes and emits the tree
    cp.fuse_tree = 1;
    cp.B = c->cfg.B;
    cp.beta = c->cfg.beta;
    cp.sel = sel;
    cp.tok = tok;
    cp.parent = parent;
    cp.depth = depth;
    cp.logp_cum = logp_cum;
    cp.mask = mask;
    return enqueue_chain(c, cp, st, true);
  }
  dt_status s = enqueue_chain(c, cp, st, true);
  if (s != DT_OK) return s;
  PruneParams pp = prune_params(c, nscore, sel);
  DT_TRY(launch_prune(pp, st));
  pp.node_tok = ntok;
  pp.node_parent = npar;
  pp.tok = tok;
  pp.parent = parent;
  pp.depth = depth;
  pp.logp_cum = logp_cum;
  pp.mask = mask;
  DT_TRY(launch_tree_mask(pp, st));
  return DT_OK;
}

// The LM-head GEMM and the Top-M of a round: the GEMM with the Top-M in its
// epilogue and the merge of its CTAs' lists, or the GEMM and the Top-M kernel.
// The second kernel launches as a programmatic dependent (it waits for the
// GEMM's end before reading its results) and clears `clear` (the grid-barrier
// chain's counter) when not null.
dt_status enqueue_base_topm(dt_ctx* c, const void* H, cudaStream_t st, unsigned* clear) {
  if (c->fuse_topm) {
    dt_status s = enqueue_base_logits(c, H, nullptr, st, true);
    if (s != DT_OK) return s;
    TopmParams mp = c->fmerge;
    mp.clear_word = clear;
    mp.pdl = 1;
    DT_TRY(launch_topm_merge(mp, st));
    return DT_OK;
  }
  float* logits = c->at<float>(c->lay.logits);
  dt_status s = enqueue_base_logits(c, H, logits, st);
  if (s != DT_OK) return s;
  return enqueue_topm(c, logits, st, clear, 1);
}

dt_status enqueue_round(dt_ctx* c, const void* H, const int32_t* root, int32_t* tok, int32_t* parent,
                        int32_t* depth, float* logp_cum, uint8_t* mask, cudaStream_t st) {
  // the chain launches as a programmatic dependent of the Top-M stage, whose
  // second kernel clears the chain's barrier counter: no memset in a round
  dt_status s = enqueue_base_topm(c, H, st, c->at<unsigned>(c->lay.bar));
  if (s != DT_OK) return s;
  return enqueue_build(c, root, tok, parent, depth, logp_cum, mask, st, true);
}

}  // namespace

extern "C" {

dt_status dt_check_config(const dt_config* cfg) { return check(cfg); }

int64_t dt_node_count(const dt_config* cfg) {
  if (!cfg) return -1;
  Tables t;
  if (cfg->block < 2 || cfg->K <= 0 || cfg->W <= 0 || !make_tables(*cfg, t)) return -1;
  return t.N;
}

size_t dt_workspace_bytes(const dt_config* cfg) {
  if (check(cfg) != DT_OK) return 0;
  Tables t;
  make_tables(*cfg, t);
  TopmParams tp = {};
  tp.V = cfg->V;
  tp.rows = cfg->n_req * t.D;
  tp.M = cfg->M;
  topm_plan(tp, 1 << 20);  // the most chunks any SM count can plan: an upper bound
  Layout L;
  layout(*cfg, t, tp, L, cfg->n_req == 1 ? 1024 : 0);  // fused lists: up to 1024 GEMM CTAs
  return L.total + L.xtab;
}

const char* dt_last_error(void) { return g_last_error; }

}  // extern "C"

namespace dt {
void set_last_error(const char* msg) { snprintf(g_last_error, sizeof(g_last_error), "%s", msg ? msg : ""); }
}  // namespace dt

extern "C" {

const char* dt_status_string(dt_status s) {
  switch (s) {
    case DT_OK: return "ok";
    case DT_ERR_INVALID_ARG: return "invalid argument";
    case DT_ERR_SHAPE: return "unsupported shape";
    case DT_ERR_CUDA: return "CUDA runtime error";
    case DT_ERR_OOM: return "device out of memory";
    case DT_ERR_TIMEOUT: return "device-side wait timed out";
    case DT_ERR_UNIMPLEMENTED: return "not implemented";
    case DT_ERR_DEVICE: return "device-side check failed";
  }
  return "unknown status";
}

dt_status dt_create(const dt_config* cfg, const dt_weights* w, void* stream, dt_ctx** out) {
  if (!out || !w) return DT_ERR_INVALID_ARG;
  *out = nullptr;
  dt_status s = check(cfg);
  if (s != DT_OK) return s;
  if (!w->lm_head || !w->emb || !w->w_ih || !w->b_ih || !w->w_hh || !w->w1 || !w->w2)
    return DT_ERR_INVALID_ARG;
  for (const void* ptr : {w->lm_head, w->emb, w->w_ih, w->b_ih, w->w_hh, w->w1, w->w2})
    if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return DT_ERR_INVALID_ARG;  // 16-byte vector loads / TMA
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dt_ctx* c = new (std::nothrow) dt_ctx();
  if (!c) return DT_ERR_OOM;
  c->cfg = *cfg;
  c->w = *w;
  make_tables(*cfg, c->t);
  cudaError_t e = cudaGetDevice(&c->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, c->device);
  if (e == cudaSuccess) e = gemm_prepare();
  if (e == cudaSuccess) e = topm_prepare();
  if (e == cudaSuccess) e = chain_prepare();
  if (e == cudaSuccess) e = prune_prepare();
  if (e == cudaSuccess) e = best_prepare();
  if (e == cudaSuccess) e = dchain_prepare();
  if (e != cudaSuccess) {
    delete c;
    return cuda_status(e, "dt_create: kernel attributes");
  }
  c->topm = TopmParams{};
  c->topm.V = cfg->V;
  c->topm.rows = cfg->n_req * c->t.D;
  c->topm.M = cfg->M;
  c->topm.T = cfg->T;
  topm_plan(c->topm, c->num_sms);
  if (const char* why = topm_unsupported(c->topm)) {
    set_last_error(why);
    delete c;
    return DT_ERR_SHAPE;
  }
  c->acc = AcceptParams{};
  c->acc.n_req = cfg->n_req;
  c->acc.S = cfg->B + 1;
  c->acc.V = cfg->V;
  c->acc.D = c->t.D;
  accept_plan(c->acc, c->num_sms);
  // the Top-M in the LM-head GEMM's epilogue: one request, and the GEMM and
  // the merge support the shape
  int fs = 0;
  if (cfg->n_req == 1 && !(cfg->flags & DT_FLAG_SEPARATE_TOPM)) {
    const GemmParams gp = logits_gemm_params(*cfg, c->t);
    if (gemm_ft_supported(gp, c->num_sms)) {
      TopmParams mp = c->topm;
      mp.S = gemm_grid(gp, c->num_sms);
      if (!topm_merge_unsupported(mp)) fs = mp.S;
    }
  }
  c->fuse_topm = fs > 0 ? 1 : 0;
  layout(*cfg, c->t, c->topm, c->lay, fs);
  // host-side fault injection: DT_FAULT_INJECT_ALLOC set in the environment
  // makes the workspace allocation fail as an out-of-memory would
  e = getenv("DT_FAULT_INJECT_ALLOC") ? cudaErrorMemoryAllocation : cudaMalloc(&c->ws, c->lay.total);
  if (e == cudaSuccess) e = cudaMalloc(&c->xtab, c->lay.xtab);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->ws, 0, c->lay.total, st);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking);
  if (e != cudaSuccess) {
    dt_destroy(c);
    return cuda_status(e, "dt_create: workspace allocation");
  }
  c->topm.part_id = c->at<int>(c->lay.part_id);
  c->topm.part_val = c->at<float>(c->lay.part_val);
  c->topm.part_max = c->at<float>(c->lay.part_max);
  c->topm.part_sum = c->at<float>(c->lay.part_sum);
  c->topm.part_cnt = c->at<int>(c->lay.part_cnt);
  c->topm.part_kth = c->at<float>(c->lay.part_kth);
  c->topm.cand_tok = c->at<int>(c->lay.cand_tok);
  c->topm.cand_base = c->at<float>(c->lay.cand_base);
  c->topm.rest_lse = c->at<float>(c->lay.rest_lse);
  c->topm.row_done = c->at<unsigned>(c->lay.row_done);
  c->topm.status = c->at<int>(c->lay.status);
  c->fmerge = c->topm;
  c->fmerge.S = fs;
  c->fmerge.part_id = c->at<int>(c->lay.fpart_id);
  c->fmerge.part_val = c->at<float>(c->lay.fpart_val);
  c->fmerge.part_max = c->at<float>(c->lay.fpart_max);
  c->fmerge.part_sum = c->at<float>(c->lay.fpart_sum);
  c->fmerge.part_cnt = c->at<int>(c->lay.fpart_cnt);
  c->fmerge.part_kth = nullptr;
  c->fmerge.part_tail = c->at<float>(c->lay.fpart_tail);
  c->fmerge.row_done = nullptr;
  c->logits_src = c->at<float>(c->lay.logits);
  c->acc.rowkey = c->at<uint64_t>(c->lay.acc_key);
  c->acc.req_done = c->at<uint64_t>(c->lay.acc_done);
  c->acc.status = c->at<int>(c->lay.status);

  ChainParams probe = {};
  probe.g = cfg->g;
  probe.r = cfg->r;
  probe.n_req = cfg->n_req;
  probe.W = cfg->W;
  probe.K = cfg->K;
  probe.M = cfg->M;
  // (the best-first builder always shards the state columns over the CTAs,
  // also under marginal scoring)
  probe.marginal = ((cfg->flags & DT_FLAG_MARGINAL) && !(cfg->flags & DT_FLAG_BEST_FIRST)) ? 1 : 0;
  c->chain_grid = chain_grid(probe, c->num_sms);
  chain_plan(probe, c->chain_grid);
  if (chain_smem_bytes(probe) > 227 * 1024 || probe.cpad > 64) {
    dt_destroy(c);
    return DT_ERR_SHAPE;
  }
  c->best_first = (cfg->flags & DT_FLAG_BEST_FIRST) ? 1 : 0;
  if (c->best_first) {
    BestParams& b = c->best;
    b = BestParams{};
    b.D = c->t.D;
    b.g = cfg->g;
    b.r = cfg->r;
    b.M = cfg->M;
    b.K = cfg->K;
    b.V = cfg->V;
    b.d = cfg->d;
    b.ldw1 = cfg->d + cfg->g;
    b.B = cfg->B;
    b.T = cfg->T;
    b.beta = cfg->beta;
    b.marginal = (cfg->flags & DT_FLAG_MARGINAL) ? 1 : 0;
    if (!best_plan(b, c->chain_grid)) {
      dt_destroy(c);
      return DT_ERR_SHAPE;
    }
  }
  // one request with conditional scoring: the clustered depth chain when the
  // shape fits it and every cluster can be resident at once
  char why[160] = "";
  if (cfg->n_req == 1 && !(cfg->flags & (DT_FLAG_MARGINAL | DT_FLAG_BEST_FIRST))) {
    DchainParams dp = dchain_params(c, nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
    dp.fuse_tree = 1;
    if (dchain_plan(dp, c->num_sms, why, sizeof(why))) {
      c->use_dchain = 1;
      c->dchain_cs = dp.cs;
      c->dchain_jc = dp.jc;
    }
    cudaGetLastError();  // an occupancy query that failed leaves no error behind
  } else {
    snprintf(why, sizeof(why), "%s", cfg->n_req != 1 ? "several requests" : "marginal or best-first mode");
  }
  char tm[96];
  if (c->fuse_topm)
    snprintf(tm, sizeof(tm), "Top-M in the LM-head GEMM's epilogue (%d CTA lists merged); ", c->fmerge.S);
  else if (c->topm.rowwise)
    snprintf(tm, sizeof(tm), "Top-M kernel streaming each row in one CTA; ");
  else
    snprintf(tm, sizeof(tm), "Top-M kernel on %d chunks per row; ", c->topm.S);
  if (c->best_first)
    snprintf(c->plan, sizeof(c->plan), "%sbest-first builder on %d CTAs", tm, c->chain_grid);
  else if (c->use_dchain)
    snprintf(c->plan, sizeof(c->plan), "%sclustered depth chain on %d CTAs: %s", tm, cfg->g / c->dchain_jc, why);
  else
    snprintf(c->plan, sizeof(c->plan), "%sgrid-barrier depth chain on %d CTAs%s (clustered chain not used: %s)", tm,
             c->chain_grid, probe.tc ? ", tcgen05 projection of the states" : "", why);

  // tensor maps of the weights
  const dt_config& k = *cfg;
  bool ok = make_tmap_bf16_2d(&c->tm_lm, w->lm_head, k.d, k.V, static_cast<uint64_t>(k.d) * 2, 128) &&
            make_tmap_bf16_2d(&c->tm_w1h, w->w1, k.d, k.r, static_cast<uint64_t>(k.d + k.g) * 2, 128);
  CUtensorMap tm_emb, tm_wih;
  const int tbn = (3 * k.g >= 256) ? 256 : (3 * k.g + 15) / 16 * 16;
  ok = ok && make_tmap_bf16_2d(&tm_emb, w->emb, k.d, k.V, static_cast<uint64_t>(k.d) * 2, 128) &&
       make_tmap_bf16_2d(&tm_wih, w->w_ih, k.d, 3ull * k.g, static_cast<uint64_t>(k.d) * 2, tbn);
  if (!ok) {
    dt_destroy(c);
    return DT_ERR_INVALID_ARG;
  }
  // GRU input table X = E W_ih^T + b_ih
  GemmParams p = {};
  p.mode = GEMM_TABLE;
  p.K = k.d;
  p.m_tiles_a = (k.V + 127) / 128;
  p.m_tiles_a2 = 0;
  p.n_tiles = (3 * k.g + tbn - 1) / tbn;
  p.n_valid = 3 * k.g;
  p.a_evict_first = 0;
  p.rows_a = k.V;
  p.out = c->xtab;
  p.ldo = 3 * k.g;
  p.bias = static_cast<const uint16_t*>(w->b_ih);
  p.status = c->at<int>(c->lay.status);
  gemm_plan(p, tbn);
  e = launch_gemm_tc(tm_emb, tm_emb, tm_wih, p, c->num_sms, st);
  if (e != cudaSuccess) {
    dt_destroy(c);
    return cuda_status(e, "dt_create: GRU input table GEMM");
  }
  c->last_stream = st;
  *out = c;
  return DT_OK;
}

dt_status dt_destroy(dt_ctx* c) {
  if (!c) return DT_OK;
  cudaDeviceSynchronize();
  for (auto& g : c->graphs)
    if (g.exec) cudaGraphExecDestroy(g.exec);
  if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
  if (c->ws) cudaFree(c->ws);
  if (c->xtab) cudaFree(c->xtab);
  delete c;
  return DT_OK;
}

dt_status dt_base_logits(dt_ctx* c, const void* H, float* logits, void* stream) {
  if (!c || !H) return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  float* dst = logits ? logits : c->at<float>(c->lay.logits);
  dt_status s = enqueue_base_logits(c, H, dst, st);
  if (s == DT_OK) {
    c->logits_src = dst;
    c->last_stream = st;
  }
  return s;
}

dt_status dt_topm(dt_ctx* c, const float* logits, int32_t* cand_tok, float* cand_base, float* rest_lse,
                  void* stream) {
  if (!c) return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dt_status s = enqueue_topm(c, logits ? logits : c->logits_src, st);
  if (s != DT_OK) return s;
  return dt_last_candidates(c, cand_tok, cand_base, rest_lse, stream);
}

dt_status dt_base_topm(dt_ctx* c, const void* H, void* stream) {
  if (!c || !H) return DT_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(H) & 15u) != 0) return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dt_status s = enqueue_base_topm(c, H, st, nullptr);
  if (s == DT_OK) c->last_stream = st;
  return s;
}

dt_status dt_last_candidates(dt_ctx* c, int32_t* cand_tok, float* cand_base, float* rest_lse, void* stream) {
  if (!c) return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(c->cfg.n_req) * c->t.D;
  if (cand_tok)
    DT_TRY(cudaMemcpyAsync(cand_tok, c->topm.cand_tok, rows * c->cfg.M * 4, cudaMemcpyDeviceToDevice, st));
  if (cand_base)
    DT_TRY(cudaMemcpyAsync(cand_base, c->topm.cand_base, rows * c->cfg.M * 4, cudaMemcpyDeviceToDevice, st));
  if (rest_lse)
    DT_TRY(cudaMemcpyAsync(rest_lse, c->topm.rest_lse, rows * 4, cudaMemcpyDeviceToDevice, st));
  c->last_stream = st;
  return DT_OK;
}

dt_status dt_expand_depth(dt_ctx* c, int depth, const int32_t* root_tok, int32_t* node_tok,
                          int32_t* node_parent, float* node_logp, float* node_score, int32_t* live,
                          void* stream) {
  if (!c || !node_tok || !node_parent || !node_logp || !node_score) return DT_ERR_INVALID_ARG;
  if (c->best_first) return DT_ERR_INVALID_ARG;  // not a depth-wise build
  if (depth < 1 || depth > c->t.D) return DT_ERR_INVALID_ARG;
  if (depth == 1 && !root_tok) return DT_ERR_INVALID_ARG;
  if (depth != 1 && depth != c->next_depth) return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (c->use_dchain) {
    DchainParams p = dchain_params(c, root_tok, node_tok, node_parent, node_logp, node_score, live);
    p.depth_first = depth;
    p.depth_last = depth;
    DT_TRY(launch_dchain(p, st));
    c->next_depth = depth + 1;
    c->last_stream = st;
    return DT_OK;
  }
  ChainParams p = chain_params(c, root_tok, node_tok, node_parent, node_logp, node_score, live);
  p.depth_first = depth;
  p.depth_last = depth;
  dt_status s = enqueue_chain(c, p, st);
  if (s != DT_OK) return s;
  c->next_depth = depth + 1;
  c->last_stream = st;
  return DT_OK;
}

dt_status dt_prune_topB(dt_ctx* c, const float* node_score, int32_t* sel, void* stream) {
  if (!c || !node_score || !sel) return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PruneParams p = prune_params(c, node_score, sel);
  DT_TRY(launch_prune(p, st));
  c->last_stream = st;
  return DT_OK;
}

dt_status dt_tree_mask(dt_ctx* c, const int32_t* sel, const int32_t* node_tok, const int32_t* node_parent,
                       const float* node_score, int32_t* tok, int32_t* parent, int32_t* depth,
                       float* logp_cum, uint8_t* mask, void* stream) {
  if (!c || !sel || !node_tok || !node_parent || !node_score || !tok || !parent || !depth || !logp_cum ||
      !mask)
    return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  PruneParams p = prune_params(c, node_score, const_cast<int32_t*>(sel));
  p.node_tok = node_tok;
  p.node_parent = node_parent;
  p.tok = tok;
  p.parent = parent;
  p.depth = depth;
  p.logp_cum = logp_cum;
  p.mask = mask;
  DT_TRY(launch_tree_mask(p, st));
  c->last_stream = st;
  return DT_OK;
}

dt_status dt_expand_prune(dt_ctx* c, const int32_t* root_tok, int32_t* tok, int32_t* parent, int32_t* depth,
                          float* logp_cum, uint8_t* mask, void* stream) {
  if (!c || !root_tok || !tok || !parent || !depth || !logp_cum || !mask) return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  dt_status s = enqueue_build(c, root_tok, tok, parent, depth, logp_cum, mask, st, false);
  if (s != DT_OK) return s;
  c->next_depth = 1;
  c->last_stream = st;
  return DT_OK;
}

dt_status dt_accept_walk(dt_ctx* c, const float* target_logits, const int32_t* tok, const int32_t* parent,
                         int32_t* target_tok, int32_t* accepted, int32_t* accept_len, int32_t* bonus, void* stream) {
  if (!c || !target_logits || !tok || !parent || !accepted || !accept_len || !bonus) return DT_ERR_INVALID_ARG;
  if (c->acc.vec4 && (reinterpret_cast<uintptr_t>(target_logits) & 15u) != 0) return DT_ERR_INVALID_ARG;
  if (c->acc.S > kAcceptMaxSlots) return DT_ERR_SHAPE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  AcceptParams p = c->acc;
  p.Z = target_logits;
  p.tok = tok;
  p.parent = parent;
  p.target_tok = target_tok;
  p.accepted = accepted;
  p.accept_len = accept_len;
  p.bonus = bonus;
  DT_TRY(launch_accept(p, st));
  c->last_stream = st;
  return DT_OK;
}

dt_status dt_build_round(dt_ctx* c, const void* H, const int32_t* root_tok, int32_t* tok, int32_t* parent,
                         int32_t* depth, float* logp_cum, uint8_t* mask, void* stream) {
  if (!c || !H || !root_tok || !tok || !parent || !depth || !logp_cum || !mask) return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* key[8] = {H, root_tok, tok, parent, depth, logp_cum, mask, nullptr};
  dt_ctx::Captured* hit = nullptr;
  for (auto& g : c->graphs) {
    if (!g.exec) continue;
    bool same = true;
    for (int i = 0; i < 8 && same; ++i) same = key[i] == g.key[i];
    if (same) { hit = &g; break; }
  }
  if (!hit) {
    dt_ctx::Captured* victim = &c->graphs[0];
    for (auto& g : c->graphs) {
      if (!g.exec) { victim = &g; break; }
      if (g.used < victim->used) victim = &g;
    }
    if (victim->exec) {
      cudaGraphExecDestroy(victim->exec);
      victim->exec = nullptr;
    }
    DT_TRY(cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
    dt_status s = enqueue_round(c, H, root_tok, tok, parent, depth, logp_cum, mask, c->cap_stream);
    cudaGraph_t graph = nullptr;
    cudaError_t e = cudaStreamEndCapture(c->cap_stream, &graph);
    if (s != DT_OK) {
      if (graph) cudaGraphDestroy(graph);
      return s;
    }
    DT_TRY(e);
    e = cudaGraphInstantiate(&victim->exec, graph, 0);
    cudaGraphDestroy(graph);
    DT_TRY(e);
    for (int i = 0; i < 8; ++i) victim->key[i] = key[i];
    hit = victim;
  }
  hit->used = ++c->graph_clock;
  DT_TRY(cudaGraphLaunch(hit->exec, st));
  c->next_depth = 1;
  c->last_stream = st;
  return DT_OK;
}

dt_status dt_build_round_host(dt_ctx* c, const void* H_host, const int32_t* root_host, int32_t* tok_host,
                              int32_t* parent_host, int32_t* depth_host, float* logp_cum_host,
                              uint8_t* mask_host, void* stream) {
  if (!c || !H_host || !root_host || !tok_host || !parent_host || !depth_host || !logp_cum_host ||
      !mask_host)
    return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const dt_config& k = c->cfg;
  const size_t hb = static_cast<size_t>(k.n_req) * k.block * k.d * 2;
  const size_t S1 = static_cast<size_t>(k.B) + 1;
  void* H = c->at<void>(c->lay.H_dev);
  int32_t* root = c->at<int32_t>(c->lay.root_dev);
  int32_t* tok = c->at<int32_t>(c->lay.out_tok);
  int32_t* parent = c->at<int32_t>(c->lay.out_parent);
  int32_t* depth = c->at<int32_t>(c->lay.out_depth);
  float* logp = c->at<float>(c->lay.out_logp);
  uint8_t* mask = c->at<uint8_t>(c->lay.out_mask);
  DT_TRY(cudaMemcpyAsync(H, H_host, hb, cudaMemcpyHostToDevice, st));
  DT_TRY(cudaMemcpyAsync(root, root_host, k.n_req * 4, cudaMemcpyHostToDevice, st));
  dt_status s = dt_build_round(c, H, root, tok, parent, depth, logp, mask, stream);
  if (s != DT_OK) return s;
  DT_TRY(cudaMemcpyAsync(tok_host, tok, k.n_req * S1 * 4, cudaMemcpyDeviceToHost, st));
  DT_TRY(cudaMemcpyAsync(parent_host, parent, k.n_req * S1 * 4, cudaMemcpyDeviceToHost, st));
  DT_TRY(cudaMemcpyAsync(depth_host, depth, k.n_req * S1 * 4, cudaMemcpyDeviceToHost, st));
  DT_TRY(cudaMemcpyAsync(logp_cum_host, logp, k.n_req * S1 * 4, cudaMemcpyDeviceToHost, st));
  DT_TRY(cudaMemcpyAsync(mask_host, mask, k.n_req * S1 * S1, cudaMemcpyDeviceToHost, st));
  DT_TRY(cudaStreamSynchronize(st));
  return DT_OK;
}

dt_status dt_check_bounded_waits(dt_ctx* c, int which, void* stream) {
  if (!c || (which != 0 && which != 1)) return DT_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned* bar = c->at<unsigned>(c->lay.bar);
  DT_TRY(cudaMemsetAsync(bar, 0, sizeof(unsigned), st));
  DT_TRY(launch_wait_check(bar, c->at<int>(c->lay.status), which, st));
  // leave the barrier counter as the next launch expects it
  DT_TRY(cudaMemsetAsync(bar, 0, sizeof(unsigned), st));
  c->last_stream = st;
  return DT_OK;
}

dt_status dt_get_device_status(dt_ctx* c) {
  if (!c) return DT_ERR_INVALID_ARG;
  DT_TRY(cudaDeviceSynchronize());
  int v = 0;
  int* dev = c->at<int>(c->lay.status);
  DT_TRY(cudaMemcpy(&v, dev, sizeof(int), cudaMemcpyDeviceToHost));
  DT_TRY(cudaMemset(dev, 0, sizeof(int)));
  if (v == DT_DEV_OK) return DT_OK;
  if (v == DT_DEV_TIMEOUT) return DT_ERR_TIMEOUT;
  return DT_ERR_DEVICE;
}

int dt_round_kernel_count(const dt_ctx* c) {
  if (!c) return -1;
  if (c->best_first) return 3;  // LM head GEMM, Top-M, best-first builder (tree and mask in its tail)
  // (the merge of the GEMM's Top-M lists takes the Top-M kernel's place when it is fused)
  if (c->use_dchain) return 3;  // LM head GEMM, Top-M, clustered chain (Top-B and tree/mask in its tail)
  // LM head GEMM, Top-M, depth chain (+ Top-B, tree/mask unless the chain's tail does them)
  ChainParams cp = chain_params(const_cast<dt_ctx*>(c), nullptr, nullptr, nullptr, nullptr, nullptr, nullptr);
  return chain_can_fuse_tree(cp) ? 3 : 5;
}

}  // extern "C"

extern "C" const char* dt_plan_string(const dt_ctx* c) { return c ? c->plan : ""; }

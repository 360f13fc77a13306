// Launch interfaces of the libdtree kernels (host side).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dt {

constexpr int kMaxDepth = 64;

// ---------------------------------------------------------------- tcgen05 GEMM
enum GemmMode { GEMM_LOGITS = 0, GEMM_TABLE = 1 };

struct GemmParams {
  int mode;
  int K;           // inner dimension
  int m_tiles_a;   // 128-row tiles taken from the first A tensor
  int m_tiles_a2;  // 128-row tiles taken from the second A tensor (logits mode: W1[:, :d])
  int n_tiles;     // BN-wide tiles of B
  int BN;          // tile width: 16..256 (multiple of 16) or 512
  int n_valid;     // valid B rows
  int stages;
  uint32_t stage_bytes, b_bytes;
  int tmem_cols;
  int acc_bufs;
  int a_evict_first;
  int rows_a, rows_a2;  // valid rows of the two A tensors
  // logits mode
  int block, D;
  float* logits;  // [n_req*D, rows_a]
  float* h1;      // [n_req*D, rows_a2]
  // table mode
  float* out;
  int ldo;
  const uint16_t* bias;
  int* status;
  // logits mode with the Top-M in the epilogue (topm_fused.cuh): each CTA
  // reports the sorted M best of its vocabulary rows for the ft_P logit rows
  // into the partial lists (S = the grid), and logits may be null
  int ft;
  int ft_P, ft_M;
  float ft_invT;
  int* part_id;     // [ft_P, S, M]
  float* part_val;  // [ft_P, S, M]
  float* part_max;  // [ft_P, S]
  float* part_sum;  // [ft_P, S]
  int* part_cnt;    // [ft_P, S]
  float* part_kth;  // [ft_P, S] or null
  float* part_tail; // [ft_P, S, M]: sum over the list's entries j.. of exp(logit/T - part_max)
};

bool make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_bytes, uint32_t box_rows);
void gemm_plan(GemmParams& p, int BN);
size_t gemm_smem_bytes(const GemmParams& p);
// The grid of a launch (one persistent CTA per SM at most).
int gemm_grid(const GemmParams& p, int num_sms);
// Whether the Top-M can run in the epilogue of this logits launch (one N tile
// of at most 16 columns, ft_P <= 16 rows, M <= 64, and the shared memory for
// it next to at least four pipeline stages); gemm_plan has been applied.
bool gemm_ft_supported(const GemmParams& p, int num_sms);
// Switches the planned launch to the fused Top-M (fewer stages to make room).
void gemm_ft_plan(GemmParams& p);
cudaError_t gemm_prepare();
cudaError_t launch_gemm_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_a2, const CUtensorMap& tm_b,
                           const GemmParams& p, int num_sms, cudaStream_t stream);

// ---------------------------------------------------------------- Top-M
struct TopmParams {
  const float* logits;  // [rows, V]
  int V, rows, M, S, chunk;
  float T;
  int* part_id;     // [rows, S, M]
  float* part_val;  // [rows, S, M]
  float* part_max;  // [rows, S]   max of logit/T over the chunk
  float* part_sum;  // [rows, S]   sum over the chunk's non-candidates of exp(logit/T - max)
  int* part_cnt;    // [rows, S]
  float* part_kth;  // [rows, S]   the chunk's M-th largest logit (-inf if it has <= M)
  // [rows, S, M] or null: part_tail[j] = sum over the list's entries j, j+1,
  // ... of exp(logit/T - part_max); with it a merge reads only the lists' heads
  float* part_tail;
  int* cand_tok;    // [rows, M]
  float* cand_base; // [rows, M]
  float* rest_lse;  // [rows]
  unsigned* row_done;  // [rows] chunk arrival counters (zero between launches)
  int* status;
  unsigned* clear_word;  // or null: a word the kernel sets to zero (the next chain's barrier counter)
  int pdl;               // 1: launched as a programmatic dependent of the previous kernel
  int occ2;              // 1: the two-CTAs-per-SM build (grids of several waves)
  int rowwise;           // 1: one CTA per SM streams whole rows (many rows); no partial lists
  int num_sms;           // the SM count topm_plan planned for
};
void topm_plan(TopmParams& p, int num_sms);
size_t topm_partial_smem(const TopmParams& p);
size_t topm_merge_smem(const TopmParams& p);
cudaError_t topm_prepare();
// Why a planned Top-M launch cannot run (too many rows for the grid, a chunk
// or a merge beyond the kernel's capacity), or null when it can.
const char* topm_unsupported(const TopmParams& p);
cudaError_t launch_topm(const TopmParams& p, cudaStream_t stream);
// The merge of partial lists written by another kernel (S lists of M per row,
// part_* arrays as above), one CTA per row; launch_topm_merge returns
// cudaErrorInvalidValue when topm_merge_unsupported says why not.
size_t topm_merge_only_smem(const TopmParams& p);
const char* topm_merge_unsupported(const TopmParams& p);
cudaError_t launch_topm_merge(const TopmParams& p, cudaStream_t stream);

// Text returned by dt_last_error() on the calling thread.
void set_last_error(const char* msg);

// ---------------------------------------------------------------- depth chain
struct ChainParams {
  int n_req, D, g, r, M, K, W, V, ldw1, d;
  int N1;  // nodes per request including the root
  float T;
  const uint16_t* w_hh;  // [3g, g]
  const uint16_t* w1;    // [r, d+g]
  const uint16_t* w2;    // [V, r]
  const float* xtab;     // [V, 3g]
  const float* h1;       // [n_req*D, r]
  const int* cand_tok;   // [n_req*D, M]
  const float* cand_base;
  const float* rest_lse;  // [n_req*D]
  const int* root_tok;    // [n_req]
  float* S;      // [2, n_req*W, g]
  // the same states split into bf16 high + low parts, laid out as mma.sync
  // A fragments: [2][n_req*W][g/16][4 lane groups][hi pair 0, hi pair 1,
  // lo pair 0, lo pair 1] (used when one request's W rows fit one fragment);
  // with tc, as tcgen05 A-operand chunks: [2][row tile of 128][g/64][hi, lo]
  // chunks of 16 KB (128 rows x 64 bf16, 128-byte swizzled)
  uint32_t* sfrag;
  // z = SiLU(h1_i + u_W1) of the live branches in the same fragment order
  // ([n_req*W][r/16][4][4]), written by the CTAs that own bottleneck rows
  uint32_t* zfrag;
  float* uW1;    // [n_req*W, r]
  int* live;     // [2, n_req, W]
  int* node_tok;
  int* node_parent;
  float* node_logp;
  float* node_score;  // [n_req, N1]
  int* live_out;      // [n_req, W] or null
  unsigned* bar;      // grid-barrier counter, zero at launch
  int* status;
  int depth_first, depth_last;
  int pdl;            // 1: launched as a programmatic dependent of the previous kernel
  int marginal;       // 1: marginal scoring (no correction, no GRU state; one CTA)
  int jper, rper;     // S / r columns owned per CTA
  int cpad;           // padded owned-column count (multiple of 32)
  int stage_w2;       // 1: stage the candidates' W2 rows in shared memory
  int dbuf;           // 1: stage the next depth's candidate data a depth ahead (one request)
  int mma_b;          // 1: corrected logits of all branches as one tensor-core product
  // 1: phase A on tcgen05 (states as the 128-row A operand, streamed from
  // sfrag in the 128-byte swizzled K-major layout, accumulators in tensor
  // memory); tc_ns shared-memory slots of 16 KB for the streamed chunks
  int tc, tc_ns;
  // tail of a whole-round launch of one request: CTA 0 (which wrote every node
  // array itself) runs the global Top-B and the tree/mask, no extra launch
  int fuse_tree;
  int B;
  float beta;
  int* sel;           // [B]
  int* tok;           // [B+1]
  int* parent;
  int* depth;
  float* logp_cum;
  uint8_t* mask;      // [(B+1)^2]
  int off[kMaxDepth + 1];  // first node index of depth i
  int nn[kMaxDepth + 1];   // nodes created at depth i
  int L[kMaxDepth + 1];    // branches that live after depth i (L[0] = 1)
};
int chain_grid(const ChainParams& p, int num_sms);
size_t chain_smem_bytes(const ChainParams& p);
void chain_plan(ChainParams& p, int grid);
bool chain_can_fuse_tree(const ChainParams& p);
cudaError_t chain_prepare();
cudaError_t launch_chain(const ChainParams& p, int grid, cudaStream_t stream);

// ---------------------------------------------------------------- clustered depth chain
// One request, <= 8 live branches, M <= 64: the depth chain on thread-block
// clusters with one tagged state exchange per depth (dchain.cu).
struct DchainParams {
  int D, g, r, M, K, W, V, ldw1, d;
  int N1;  // nodes including the root
  float T;
  const uint16_t* w_hh;   // [3g, g]
  const uint16_t* w1;     // [r, d+g]
  const uint16_t* w2;     // [V, r]
  const float* xtab;      // [V, 3g]
  const float* h1;        // [D, r]
  const int* cand_tok;    // [D, M]
  const float* cand_base; // [D, M]
  const float* rest_lse;  // [D]
  const int* root_tok;    // [1]
  float* S;               // [2][W][g] fp32 states handed from one launch to the next (depth parity)
  int* live;              // [2][W] live node lists handed over the same way
  void* xch;              // [2][g/8][8][4] 16-byte tagged words: the per-depth state exchange
  unsigned* epoch;        // launch counter (part of every tag)
  unsigned* abort_word;   // the epoch of a launch whose wait gave up
  int* node_tok;
  int* node_parent;
  float* node_logp;
  float* node_score;      // [N1]
  int* live_out;          // [W] or null
  int* status;
  int depth_first, depth_last;
  int pdl;
  int cs;                 // cluster size (dchain_plan)
  int jc;                 // state columns per CTA, 8 or 16 (dchain_plan)
  int fuse_tree;          // CTA 0 runs the global Top-B and the tree/mask after depth D
  int B;
  float beta;
  int* sel;
  int* tok;
  int* parent;
  int* depth;
  float* logp_cum;
  uint8_t* mask;
  int off[kMaxDepth + 2];
  int L[kMaxDepth + 1];
};
// Picks the cluster size (16, 8, 4, 2 or 1) for the shape and checks that all
// clusters fit on the device at once; false when the shape is not supported.
// why (optional) receives the choice or the reason for none.
bool dchain_plan(DchainParams& p, int num_sms, char* why = nullptr, size_t why_len = 0);
size_t dchain_smem_bytes(const DchainParams& p);
cudaError_t dchain_prepare();
cudaError_t launch_dchain(const DchainParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- Top-B and tree
struct PruneParams {
  int n_req, N1, B, D;
  float beta;
  const float* node_score;  // [n_req, N1]
  int* sel;                 // [n_req, B]
  const int* node_tok;
  const int* node_parent;
  int* tok;
  int* parent;
  int* depth;
  float* logp_cum;
  uint8_t* mask;
  int* status;
  int off[kMaxDepth + 2];   // off[i] first node of depth i; off[D+1] = N1
};
size_t prune_smem_bytes(const PruneParams& p);
cudaError_t prune_prepare();
cudaError_t launch_prune(const PruneParams& p, cudaStream_t stream);
cudaError_t launch_tree_mask(const PruneParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- best-first builder
struct BestParams {
  int D, g, r, M, K, V, ldw1, d, B;
  float T, beta;
  int marginal;
  const uint16_t* w_hh;    // [3g, g]
  const uint16_t* w1;      // [r, d+g]
  const uint16_t* w2;      // [V, r]
  const float* xtab;       // [V, 3g]
  const float* h1;         // [D, r] of the request
  const int* cand_tok;     // [D, M]
  const float* cand_base;  // [D, M]
  const float* rest_lse;   // [D]
  const int* root_tok;     // [1]
  float* srow;             // [g] state of the node being expanded (exchanged between CTAs)
  float* zrow;             // [r] its bottleneck z (exchanged)
  unsigned* bar;           // grid-barrier counter, zero at launch
  int* status;
  int jper, rper, cpad;    // owned state columns / bottleneck rows per CTA, padded columns
  int nmax;                // node capacity 1 + B*K
  int xpre;                // 1: the children's GRU-input slices are prefetched into shared memory
  int pdl;
  int* sel;                // [B] popped nodes, ascending
  int* pops;               // [B] popped nodes in pop order, or null
  int* tok;                // [B+1]
  int* parent;
  int* depth;
  float* logp_cum;
  uint8_t* mask;           // [(B+1)^2]
};
bool best_plan(BestParams& p, int grid);
size_t best_smem_bytes(const BestParams& p);
cudaError_t best_prepare();
cudaError_t launch_best(const BestParams& p, int grid, cudaStream_t stream);

// ---------------------------------------------------------------- acceptance walk
struct AcceptParams {
  const float* Z;       // [n_req * S, V] target logits, row q*S + a = slot a of request q
  const int* tok;       // [n_req, S]
  const int* parent;    // [n_req, S]
  int n_req, S, V, D;
  long long piece;      // logits per CTA, a multiple of 4 (accept_plan)
  int grid;             // CTAs
  int vec4;             // 1: 16-byte loads (V a multiple of 4)
  uint64_t* rowkey;     // [n_req * S] (value, token) key of each row (zero between launches)
  uint64_t* req_done;   // [n_req] scanned-element counters (zero between launches)
  int* target_tok;      // [n_req, S] or null
  int* accepted;        // [n_req, D]
  int* accept_len;      // [n_req]
  int* bonus;           // [n_req]
  int* status;
};
// Slots per tree the walk handles: its shared memory holds two ints per slot.
constexpr int kAcceptMaxSlots = 3072;
void accept_plan(AcceptParams& p, int num_sms);
size_t accept_smem_bytes(const AcceptParams& p);
cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- bounded-wait self-check
cudaError_t launch_wait_check(unsigned* bar, int* status, int which, cudaStream_t stream);

}  // namespace dt

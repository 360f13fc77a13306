// Stand-alone deferred pruning and tree emission kernels (one CTA per request);
// the arithmetic lives in prune.cuh, shared with the depth-chain kernel's tail.
#include "common.cuh"
#include "kernels.h"
#include "prune.cuh"

namespace dt {

namespace {

constexpr int kThreads = 1024;

DT_HOST_DEVICE_INLINE int topb_cap(int N1) { return N1 - 1 < kTopBCandCap ? N1 - 1 : kTopBCandCap; }

__global__ void __launch_bounds__(kThreads) k_prune_topb(const PruneParams p) {
  extern __shared__ uint64_t cands[];  // [cap] candidate keys, then [N1 - 1] float keys
  __shared__ uint32_t hist[(kThreads / 32) * 256];  // one 256-bin histogram per warp
  __shared__ uint32_t state[4];
  __shared__ float red[64];
  __shared__ int scan_scratch[40];
  __shared__ int off[kMaxDepth + 2];
  const int q = blockIdx.x;
  for (int i = threadIdx.x; i <= p.D + 1; i += blockDim.x) off[i] = p.off[i];
  __syncthreads();
  const int cap = topb_cap(p.N1);
  uint32_t* keys = reinterpret_cast<uint32_t*>(cands + cap);
  topb_select(p.node_score + static_cast<size_t>(q) * p.N1, p.N1, p.B, p.beta, p.D, off, keys, cands, cap, hist,
              static_cast<int>(sizeof(hist) / 4), state, red, scan_scratch, p.sel + static_cast<size_t>(q) * p.B);
}

__global__ void __launch_bounds__(kThreads) k_tree_mask(const PruneParams p) {
  extern __shared__ int sm[];  // nodes[B+1], par[B+1], dep[B+1], ancestor rows
  __shared__ int off[kMaxDepth + 2];
  const int q = blockIdx.x;
  const int S = p.B + 1;
  for (int i = threadIdx.x; i <= p.D + 1; i += blockDim.x) off[i] = p.off[i];
  __syncthreads();
  const size_t nb = static_cast<size_t>(q) * p.N1;
  const size_t ob = static_cast<size_t>(q) * S;
  tree_and_mask(p.sel + static_cast<size_t>(q) * p.B, p.N1, p.B, p.D, off, p.node_tok + nb, p.node_parent + nb,
                p.node_score + nb, nullptr, sm, sm + S, sm + 2 * S, reinterpret_cast<uint32_t*>(sm + 3 * S), p.tok + ob,
                p.parent + ob, p.depth + ob, p.logp_cum + ob, p.mask + ob * S, p.status);
}

}  // namespace

size_t prune_smem_bytes(const PruneParams& p) {
  return static_cast<size_t>(topb_cap(p.N1)) * 8 + static_cast<size_t>(p.N1) * 4;
}

cudaError_t prune_prepare() {
  return dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_prune_topb));
}

cudaError_t launch_prune(const PruneParams& p, cudaStream_t stream) {
  k_prune_topb<<<p.n_req, kThreads, prune_smem_bytes(p), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tree_mask(const PruneParams& p, cudaStream_t stream) {
  const size_t S = static_cast<size_t>(p.B) + 1;
  k_tree_mask<<<p.n_req, kThreads, S * 12 + S * anc_words(static_cast<int>(S)) * 4, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dt

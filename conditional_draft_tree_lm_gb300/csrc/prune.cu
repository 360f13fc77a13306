// Deferred pruning and tree emission.
//
// k_prune_topb: one global Top-B over every materialised non-root node of the
// super-tree with key = score + beta * depth ("DARTree: Speculative Diffusion
// Decoding with Autoregressive Draft Trees", Metodología, 2. Poda Diferida,
// Selección Global; with beta <= 0 the set equals sequential best-first by
// Lemma 1).  Radix select of the B-th key, ties to the lower node index by
// stable compaction, so the output is already in ascending node order.
//
// k_tree_mask: compact tree (root + selected nodes in ascending order) with
// parent slots and the ancestor-only attention mask of tree attention
// ("Resumen Técnico: DominoTree", 5. Verificación).
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace dt {

namespace {

constexpr int kThreads = 1024;

DT_DEVINL int depth_of(const int* off, int D, int v) {
  // off[1] = 1 < off[2] < ... < off[D+1] = N1; node v >= 1 has depth i with off[i] <= v < off[i+1]
  int lo = 1, hi = D;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__global__ void __launch_bounds__(kThreads) k_prune_topb(const PruneParams p) {
  extern __shared__ uint32_t keys[];  // [N1 - 1]
  __shared__ uint32_t hist[(kThreads / 32) * 256];  // one 256-bin histogram per warp
  __shared__ uint32_t state[4];
  __shared__ int scan_scratch[40];
  __shared__ int off[kMaxDepth + 2];
  const int q = blockIdx.x;
  const int n = p.N1 - 1;
  for (int i = threadIdx.x; i <= p.D + 1; i += blockDim.x) off[i] = p.off[i];
  __syncthreads();
  const float* score = p.node_score + static_cast<size_t>(q) * p.N1;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int v = e + 1;
    const float dep = static_cast<float>(depth_of(off, p.D, v));
    keys[e] = f32_key(score[v] + p.beta * dep);
  }
  __syncthreads();
  uint32_t t = 0;
  int need = n;
  if (p.B < n) radix_select_kth_largest(keys, n, p.B, hist, static_cast<int>(sizeof(hist) / 4), state, t, need);
  const int seg = (n + blockDim.x - 1) / blockDim.x;
  const int s0 = min(n, static_cast<int>(threadIdx.x) * seg);
  const int s1 = min(n, s0 + seg);
  int ties = 0;
  for (int e = s0; e < s1; ++e) ties += (keys[e] == t);
  int tot;
  const int tie_base = block_exclusive_scan(ties, scan_scratch, &tot);
  int cnt = 0;
  {
    int tb = tie_base;
    for (int e = s0; e < s1; ++e) {
      const uint32_t k = keys[e];
      if (k > t || (k == t && tb++ < need)) ++cnt;
    }
  }
  const int out_base = block_exclusive_scan(cnt, scan_scratch, &tot);
  int tb = tie_base, o = out_base;
  int* sel = p.sel + static_cast<size_t>(q) * p.B;
  for (int e = s0; e < s1; ++e) {
    const uint32_t k = keys[e];
    if (k > t || (k == t && tb++ < need)) {
      if (o < p.B) sel[o] = e + 1;
      ++o;
    }
  }
}

__global__ void __launch_bounds__(kThreads) k_tree_mask(const PruneParams p) {
  extern __shared__ int sm[];  // nodes[B+1], par[B+1], dep[B+1]
  __shared__ int off[kMaxDepth + 2];
  const int q = blockIdx.x;
  const int S = p.B + 1;
  int* nodes = sm;
  int* par = sm + S;
  int* dep = sm + 2 * S;
  for (int i = threadIdx.x; i <= p.D + 1; i += blockDim.x) off[i] = p.off[i];
  const int* sel = p.sel + static_cast<size_t>(q) * p.B;
  for (int k = threadIdx.x; k < S; k += blockDim.x) {
    int v = 0;
    if (k > 0) {
      v = sel[k - 1];
      if (v < 1 || v >= p.N1) { dt_report(p.status, DT_DEV_BOUNDS); v = 0; }
    }
    nodes[k] = v;
  }
  __syncthreads();
  const size_t nb = static_cast<size_t>(q) * p.N1;
  const size_t ob = static_cast<size_t>(q) * S;
  for (int k = threadIdx.x; k < S; k += blockDim.x) {
    const int v = nodes[k];
    int ps = -1, d = 0;
    if (k > 0) {
      d = depth_of(off, p.D, v);
      const int pv = p.node_parent[nb + v];
      // binary search of pv among nodes[0..S) (ascending)
      int lo = 0, hi = S - 1;
      ps = -2;
      while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int x = nodes[mid];
        if (x == pv) { ps = mid; break; }
        if (x < pv) lo = mid + 1; else hi = mid - 1;
      }
      if (ps < 0 || ps >= k) { dt_report(p.status, DT_DEV_TREE); ps = -2; }
    }
    par[k] = ps;
    dep[k] = d;
    p.tok[ob + k] = p.node_tok[nb + v];
    p.parent[ob + k] = ps;
    p.depth[ob + k] = d;
    p.logp_cum[ob + k] = p.node_score[nb + v];
  }
  __syncthreads();
  uint8_t* mask = p.mask + static_cast<size_t>(q) * S * S;
  for (int idx = threadIdx.x; idx < S * S; idx += blockDim.x) {
    const int a = idx / S, b = idx - a * S;
    uint8_t m = 0;
    if (dep[a] >= dep[b]) {
      int cur = a;
      for (int st = dep[a] - dep[b]; st > 0 && cur >= 0; --st) cur = par[cur];
      m = (cur == b) ? 1 : 0;
    }
    mask[idx] = m;
  }
}

}  // namespace

size_t prune_smem_bytes(const PruneParams& p) { return static_cast<size_t>(p.N1) * 4; }

cudaError_t prune_prepare() {
  return dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_prune_topb));
}

cudaError_t launch_prune(const PruneParams& p, cudaStream_t stream) {
  k_prune_topb<<<p.n_req, kThreads, prune_smem_bytes(p), stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tree_mask(const PruneParams& p, cudaStream_t stream) {
  k_tree_mask<<<p.n_req, kThreads, static_cast<size_t>(p.B + 1) * 12, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dt

// Deferred pruning and tree emission as block-wide device functions, shared by
// the stand-alone kernels (prune.cu) and the tail of the depth-chain kernel.
//
// topb_select: one global Top-B over every materialised non-root node with
// key = score + beta * depth ("DARTree: Speculative Diffusion Decoding with
// Autoregressive Draft Trees", Metodología, 2. Poda Diferida, Selección Global;
// with beta <= 0 the set equals sequential best-first by Lemma 1).  Radix
// select of the B-th key, ties to the lower node index by stable compaction,
// so the output is already in ascending node order.
//
// tree_and_mask: compact tree (root + selected nodes in ascending order) with
// parent slots and the ancestor-only attention mask of tree attention
// ("Resumen Técnico: DominoTree", 5. Verificación).
#pragma once

#include "common.cuh"
#include "select.cuh"

namespace dt {

DT_DEVINL int depth_of(const int* off, int D, int v) {
  // off[1] = 1 < off[2] < ... < off[D+1] = N1; node v >= 1 has depth i with off[i] <= v < off[i+1]
  int lo = 1, hi = D;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (off[mid] <= v) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// score: [N1] node scores of one request (global).  keys: N1-1 uint32 of
// shared memory.  hist: hist_words uint32 of shared memory.  sel: [B] output.
DT_DEVINL void topb_select(const float* score, int N1, int B, float beta, int D, const int* off, uint32_t* keys,
                           uint32_t* hist, int hist_words, uint32_t* state, int* scan, int* sel) {
  const int n = N1 - 1;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const int v = e + 1;
    const float dep = static_cast<float>(depth_of(off, D, v));
    keys[e] = f32_key(score[v] + beta * dep);
  }
  __syncthreads();
  uint32_t t = 0;
  int need = n;
  if (B < n) radix_select_kth_largest(keys, n, B, hist, hist_words, state, t, need);
  const int seg = (n + blockDim.x - 1) / blockDim.x;
  const int s0 = min(n, static_cast<int>(threadIdx.x) * seg);
  const int s1 = min(n, s0 + seg);
  int ties = 0;
  for (int e = s0; e < s1; ++e) ties += (keys[e] == t);
  int tot;
  const int tie_base = block_exclusive_scan(ties, scan, &tot);
  int cnt = 0;
  {
    int tb = tie_base;
    for (int e = s0; e < s1; ++e) {
      const uint32_t k = keys[e];
      if (k > t || (k == t && tb++ < need)) ++cnt;
    }
  }
  const int out_base = block_exclusive_scan(cnt, scan, &tot);
  int tb = tie_base, o = out_base;
  for (int e = s0; e < s1; ++e) {
    const uint32_t k = keys[e];
    if (k > t || (k == t && tb++ < need)) {
      if (o < B) sel[o] = e + 1;
      ++o;
    }
  }
  __syncthreads();
}

// sel: [B] ascending node indices.  nodes/par/dep: B+1 ints of shared memory
// each.  node_*: [N1] arrays of one request.  Outputs: tok/parent/depth/logp_cum
// [B+1], mask [(B+1)^2].
DT_DEVINL void tree_and_mask(const int* sel, int N1, int B, int D, const int* off, const int* node_tok,
                             const int* node_parent, const float* node_score, int* nodes, int* par, int* dep,
                             int* tok, int* parent, int* depth, float* logp_cum, uint8_t* mask, int* status) {
  const int S = B + 1;
  for (int k = threadIdx.x; k < S; k += blockDim.x) {
    int v = 0;
    if (k > 0) {
      v = sel[k - 1];
      if (v < 1 || v >= N1) {
        dt_report(status, DT_DEV_BOUNDS);
        v = 0;
      }
    }
    nodes[k] = v;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < S; k += blockDim.x) {
    const int v = nodes[k];
    int ps = -1, d = 0;
    if (k > 0) {
      d = depth_of(off, D, v);
      const int pv = node_parent[v];
      // binary search of pv among nodes[0..S) (ascending)
      int lo = 0, hi = S - 1;
      ps = -2;
      while (lo <= hi) {
        const int mid = (lo + hi) >> 1;
        const int x = nodes[mid];
        if (x == pv) {
          ps = mid;
          break;
        }
        if (x < pv) lo = mid + 1; else hi = mid - 1;
      }
      if (ps < 0 || ps >= k) {
        dt_report(status, DT_DEV_TREE);
        ps = -2;
      }
    }
    par[k] = ps;
    dep[k] = d;
    tok[k] = node_tok[v];
    parent[k] = ps;
    depth[k] = d;
    logp_cum[k] = node_score[v];
  }
  __syncthreads();
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

}  // namespace dt

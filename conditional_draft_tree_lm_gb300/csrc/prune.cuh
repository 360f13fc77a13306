// Deferred pruning and tree emission as block-wide device functions, shared by
// the stand-alone kernels (prune.cu) and the tail of the depth-chain kernel.
//
// topb_select: one global Top-B over every materialised non-root node with
// key = score + beta * depth ("DARTree: Speculative Diffusion Decoding with
// Autoregressive Draft Trees", Metodología, 2. Poda Diferida, Selección Global;
// with beta <= 0 the set equals sequential best-first by Lemma 1), ties to the
// lower node index, written in ascending node order.
//
// tree_and_mask: compact tree (root + selected nodes in ascending order) with
// parent slots and the ancestor-only attention mask of tree attention
// ("Resumen Técnico: DominoTree", 5. Verificación).
#pragma once

#include "common.cuh"
#include "select.cuh"

// Phase stamps of topb_select / tree_and_mask (a timing build of the file that
// includes this one may define it first).
#ifndef TOPB_STAMP
#define TOPB_STAMP(k) \
  do {                \
  } while (0)
#endif

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

// Top-B entries a caller's candidate buffer holds at most (uint64 each).
constexpr int kTopBCandCap = 8192;

// score: [N1] node scores of one request (global).  keys: N1-1 uint32 of
// shared memory; cands: cap uint64 of shared memory; hist: hist_words uint32
// of shared memory (a multiple of 256); state: 4 uint32; red: 64 floats;
// scan: 40 ints.  sel: [B] output, ascending node indices (also written to
// sel_s, shared memory, when it is not null).
//   1. key_v = score_v + beta * depth_v for every non-root node; min and max;
//   2. a 256-bin histogram of the keys between max and min; the bin holding
//      the B-th largest key bounds the candidates (bins at or above it);
//   3. the candidates, ranked exactly by (key desc, node index asc), keep the
//      B best, which are then ranked by node index into sel.
// When more than cap keys share the bounding bins (flat scores), a radix
// select of the B-th key with index-ordered compaction runs instead.
DT_DEVINL void topb_select(const float* score, int N1, int B, float beta, int D, const int* off, uint32_t* keys,
                           uint64_t* cands, int cap, uint32_t* hist, int hist_words, uint32_t* state, float* red,
                           int* scan, int* sel, int* sel_s = nullptr) {
  const int n = N1 - 1;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarp = blockDim.x >> 5;
  float* kf = reinterpret_cast<float*>(keys);
  float lo = INFINITY, hi = -INFINITY;
  for (int e = tid; e < n; e += blockDim.x) {
    const int v = e + 1;
    const float k = score[v] + beta * static_cast<float>(depth_of(off, D, v));
    kf[e] = k;
    lo = fminf(lo, k);
    hi = fmaxf(hi, k);
  }
  lo = -warp_max(-lo);
  hi = warp_max(hi);
  if (lane == 0) {
    red[warp] = lo;
    red[32 + warp] = hi;
  }
  const int ncopy = min(nwarp, max(1, hist_words / 256));
  for (int b = tid; b < ncopy * 256; b += blockDim.x) hist[b] = 0u;
  if (tid == 0) state[0] = 0u;
  __syncthreads();
  TOPB_STAMP(0);
  if (B >= n) {
    for (int e = tid; e < n; e += blockDim.x) {
      sel[e] = e + 1;
      if (sel_s) sel_s[e] = e + 1;
    }
    __syncthreads();
    return;
  }
  float kmin = INFINITY, kmax = -INFINITY;
  for (int w = 0; w < nwarp; ++w) {
    kmin = fminf(kmin, red[w]);
    kmax = fmaxf(kmax, red[32 + w]);
  }
  const float scale = kmax > kmin ? 256.0f / (kmax - kmin) : 0.0f;
  auto bin_of = [&](float k) { return min(255, max(0, __float2int_rz((kmax - k) * scale))); };
  uint32_t* my = hist + (warp % ncopy) * 256;
  for (int e = tid; e < n; e += blockDim.x) atomicAdd(&my[bin_of(kf[e])], 1u);
  __syncthreads();
  TOPB_STAMP(1);
  for (int b = tid; b < 256; b += blockDim.x) {
    uint32_t c = 0;
    for (int w = 0; w < ncopy; ++w) c += hist[w * 256 + b];
    hist[b] = c;
  }
  __syncthreads();
  if (warp == 0) {
    // lane l totals bins 8l .. 8l+7; the first bin where the running count
    // reaches B bounds the candidates
    uint32_t c8[8], sum = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      c8[j] = hist[8 * lane + j];
      sum += c8[j];
    }
    uint32_t incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl >= static_cast<uint32_t>(B));
    const int first = hit ? __ffs(hit) - 1 : 31;
    if (lane == first) {
      uint32_t cum = incl - sum;
      int bt = 8 * lane + 7;
      for (int j = 0; j < 8; ++j) {
        cum += c8[j];
        if (cum >= static_cast<uint32_t>(B)) {
          bt = 8 * lane + j;
          break;
        }
      }
      state[1] = static_cast<uint32_t>(bt);
    }
  }
  __syncthreads();
  TOPB_STAMP(2);
  const int bt = static_cast<int>(state[1]);
  for (int e = tid; e < n; e += blockDim.x) {
    const float k = kf[e];
    if (bin_of(k) <= bt) {
      const uint32_t at = atomicAdd(&state[0], 1u);
      if (at < static_cast<uint32_t>(cap)) cands[at] = rank_key(k, static_cast<uint32_t>(e + 1));
    }
  }
  __syncthreads();
  TOPB_STAMP(3);
  const int c = static_cast<int>(state[0]);
  if (c > cap) {
    // fallback: radix select of the B-th key over all keys, then the winners
    // (keys above it and the lowest-indexed ties) in index order
    for (int e = tid; e < n; e += blockDim.x) keys[e] = f32_key(kf[e]);
    __syncthreads();
    uint32_t t = 0;
    int need = n;
    radix_select_kth_largest(keys, n, B, hist, hist_words, state, t, need);
    const int seg = (n + blockDim.x - 1) / blockDim.x;
    const int s0 = min(n, tid * seg), s1 = min(n, s0 + seg);
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
        if (o < B) {
          sel[o] = e + 1;
          if (sel_s) sel_s[o] = e + 1;
        }
        ++o;
      }
    }
    __syncthreads();
    return;
  }
  // the B best by key; their node indices in key order into keys[] (reused)
  int* win = reinterpret_cast<int*>(keys);
  block_rank_all(cands, c, [&](int, uint64_t ke, int rk) {
    if (rk < B) win[rk] = static_cast<int>(rank_key_id(ke));
  });
  __syncthreads();
  TOPB_STAMP(4);
  // ascending node order
  for (int a = tid; a < B; a += blockDim.x) {
    const int va = win[a];
    int pos = 0;
    for (int b2 = 0; b2 < B; ++b2) pos += win[b2] < va ? 1 : 0;
    sel[pos] = va;
    if (sel_s) sel_s[pos] = va;
  }
  __syncthreads();
}

// Words of one row of the ancestor bitmask for S tree slots.
DT_HOST_DEVICE_INLINE int anc_words(int S) { return (S + 31) / 32; }

// sel: [B] ascending node indices.  nodes/par/dep: B+1 ints of shared memory
// each; anc: (B+1) * anc_words(B+1) uint32 of shared memory.  node_*: [N1]
// arrays of one request; node_depth may be null, then a node's depth comes
// from the depth offsets off (depth-major numbering).  Outputs:
// tok/parent/depth/logp_cum [B+1], mask [(B+1)^2].
DT_DEVINL void tree_and_mask(const int* sel, int N1, int B, int D, const int* off, const int* node_tok,
                             const int* node_parent, const float* node_score, const int* node_depth, int* nodes,
                             int* par, int* dep,
                             uint32_t* anc, int* tok, int* parent, int* depth, float* logp_cum, uint8_t* mask,
                             int* status) {
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
  TOPB_STAMP(5);
  for (int k = threadIdx.x; k < S; k += blockDim.x) {
    const int v = nodes[k];
    int ps = -1, d = 0;
    if (k > 0) {
      d = node_depth ? node_depth[v] : depth_of(off, D, v);
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
  TOPB_STAMP(6);
  // each slot walks up to the root once and marks itself and its ancestors
  // in its own bitmask row; the mask bytes are then read off the rows
  const int nw = anc_words(S);
  for (int a = threadIdx.x; a < S; a += blockDim.x) {
    uint32_t* row = anc + static_cast<size_t>(a) * nw;
    for (int w = 0; w < nw; ++w) row[w] = 0u;
    for (int cur = a, st = 0; cur >= 0 && st <= D; cur = par[cur], ++st) row[cur >> 5] |= 1u << (cur & 31);
  }
  __syncthreads();
  TOPB_STAMP(7);
  auto bit = [&](int idx) {
    const int a = idx / S, b = idx - a * S;
    return (anc[static_cast<size_t>(a) * nw + (b >> 5)] >> (b & 31)) & 1u;
  };
  // four mask bytes per 32-bit store where the mask is 4-byte aligned (one
  // division per word: the next three bytes step along the row)
  const int n4 = (reinterpret_cast<uintptr_t>(mask) & 3u) == 0 ? S * S / 4 : 0;
  for (int w = threadIdx.x; w < n4; w += blockDim.x) {
    int a = (4 * w) / S, b = 4 * w - a * S;
    uint32_t word = 0u;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      word |= ((anc[static_cast<size_t>(a) * nw + (b >> 5)] >> (b & 31)) & 1u) << (8 * k);
      if (++b == S) {
        b = 0;
        ++a;
      }
    }
    reinterpret_cast<uint32_t*>(mask)[w] = word;
  }
  for (int idx = 4 * n4 + threadIdx.x; idx < S * S; idx += blockDim.x) mask[idx] = static_cast<uint8_t>(bit(idx));
}

}  // namespace dt

// Greedy verification of emitted draft trees: the acceptance walk
// ("Resumen Técnico: DominoTree", Metodología, 5. Verificación; Resultados
// Experimentales, Ausencia de Pérdida).
//
// The target model has scored every tree slot in one pass; its logits at slot
// a give the token it would emit after the path root..a (the row argmax, equal
// maxima to the lower token id).  The walk starts at the root and moves into
// the child whose draft token equals that token, while one exists; the
// target's token at the last slot reached is the bonus token.
//
// One launch streams the logits once, split into equal pieces, one per CTA
// (about eight CTAs per SM, a single wave; a piece may span rows):
//   1. each CTA reduces each row segment of its piece to one (value, token) key
//      (f32 key << 32 | ~token: the largest key is the largest value with the
//      lowest token) and folds it into the row's key with a 64-bit atomic max;
//   2. the last CTA of a request (an arrival counter of scanned elements;
//      nothing waits) takes the
//      row keys of its slots (resetting them, one atomic exchange each) as the
//      target tokens y, marks for each slot the child whose token equals y of
//      its parent, and walks from the root in shared memory.
// The row scan is a plain HBM stream: 16-byte streaming loads, four in flight
// per thread, about eight CTAs per SM.
#include "common.cuh"
#include "kernels.h"

#include <climits>

namespace dt {

namespace {

constexpr int kAThreads = 256;
constexpr int kAUnroll = 4;  // 16-byte loads in flight per thread

// v beats the thread's best when larger; indices only increase within a
// thread, so equal values keep the lower index.
DT_DEVINL void take(float v, int i, float& best, int& bi) {
  const bool gt = v > best;
  best = gt ? v : best;
  bi = gt ? i : bi;
}

// Largest (value, lowest token) key of z[lo, hi) over the block; every thread
// returns it.
DT_DEVINL uint64_t block_row_key(const float* z, int lo, int hi, bool vec4, uint64_t* s_red) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float best = -INFINITY;
  int bi = -1;
  if (vec4) {
    // lo, hi and the row start are multiples of 4 floats (16-byte aligned)
    const float4* z4 = reinterpret_cast<const float4*>(z + lo);
    const int n4 = (hi - lo) >> 2;
    for (int base = 0; base < n4; base += kAThreads * kAUnroll) {
      float4 v[kAUnroll];
#pragma unroll
      for (int u = 0; u < kAUnroll; ++u) {
        const int j = base + u * kAThreads + tid;
        v[u] = j < n4 ? __ldcs(z4 + j) : make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      }
#pragma unroll
      for (int u = 0; u < kAUnroll; ++u) {
        const int j = base + u * kAThreads + tid;
        if (j < n4) {
          const int i = lo + 4 * j;
          take(v[u].x, i, best, bi);
          take(v[u].y, i + 1, best, bi);
          take(v[u].z, i + 2, best, bi);
          take(v[u].w, i + 3, best, bi);
        }
      }
    }
    // a thread whose values are all -inf keeps its first index
    if (bi < 0 && tid < n4) bi = lo + 4 * tid;
  } else {
    for (int i = lo + tid; i < hi; i += kAThreads) take(__ldcs(z + i), i, best, bi);
    if (bi < 0 && lo + tid < hi) bi = lo + tid;
  }
  uint64_t key = bi >= 0 ? rank_key(best, static_cast<uint32_t>(bi)) : 0ull;
  key = warp_max_u64(key);
  __syncthreads();  // s_red is free (a previous segment's readers are done)
  if (lane == 0) s_red[warp] = key;
  __syncthreads();
  uint64_t k = s_red[0];
  for (int w = 1; w < kAThreads / 32; ++w) k = s_red[w] > k ? s_red[w] : k;
  return k;
}

// Request q's target tokens, accepted children and walk (whole CTA).
DT_DEVINL void walk_request(const AcceptParams& p, int q, int* s_dyn) {
  const int tid = threadIdx.x;
  const int S = p.S;
  int* y = s_dyn;
  int* nxt = s_dyn + S;
  const int* tq = p.tok + static_cast<size_t>(q) * S;
  const int* pq = p.parent + static_cast<size_t>(q) * S;
  // the thread's first slot of the tree, loaded while the row keys are exchanged
  const int cs0 = tid + 1;
  int par0 = 0, tok0 = 0;
  if (cs0 < S) {
    par0 = pq[cs0];
    tok0 = tq[cs0];
  }
  for (int a = tid; a < S; a += kAThreads) {
    // read the row's key and leave zero for the next launch
    const uint64_t k = atomicExch(reinterpret_cast<unsigned long long*>(p.rowkey + static_cast<size_t>(q) * S + a),
                                  0ull);
    const int t = static_cast<int>(rank_key_id(k));
    y[a] = t;
    nxt[a] = INT_MAX;
    if (p.target_tok) p.target_tok[static_cast<size_t>(q) * S + a] = t;
  }
  __syncthreads();
  // each slot whose token is the target's token at its parent is that
  // parent's accepted child (siblings carry distinct tokens: at most one)
  for (int cs = cs0; cs < S; cs += kAThreads) {
    const int par = cs == cs0 ? par0 : pq[cs];
    const int tk = cs == cs0 ? tok0 : tq[cs];
    if (par < 0 || par >= cs) {
      dt_report(p.status, DT_DEV_TREE);
      continue;
    }
    if (tk == y[par]) {
      const int old = atomicMin(&nxt[par], cs);
      if (old != INT_MAX) dt_report(p.status, DT_DEV_TREE);  // two siblings share the token
    }
  }
  __syncthreads();
  if (tid == 0) {
    int a = 0, n = 0;
    int* acc = p.accepted + static_cast<size_t>(q) * p.D;
    while (n < p.D) {
      const int cs = nxt[a];
      if (cs == INT_MAX) break;
      a = cs;
      acc[n++] = a;
    }
    p.accept_len[q] = n;
    p.bonus[q] = y[a];
    for (int j = n; j < p.D; ++j) acc[j] = -1;
  }
  __syncthreads();  // the shared arrays are free again
}

// CTA b scans elements [b * piece, (b + 1) * piece) of the logits taken as
// one array of n_req * S rows of V (at most a few row segments).
__global__ void __launch_bounds__(kAThreads, 8) k_accept(const AcceptParams p) {
  extern __shared__ int s_dyn[];  // [S] target tokens, [S] accepted child (walking CTA)
  __shared__ uint64_t s_red[kAThreads / 32];
  __shared__ int s_last;
  const long long V = p.V;
  const long long total = static_cast<long long>(p.n_req) * p.S * V;
  const long long e0 = static_cast<long long>(blockIdx.x) * p.piece;
  const long long e1 = min(total, e0 + p.piece);
  const unsigned long long per_req = static_cast<unsigned long long>(p.S) * static_cast<unsigned long long>(V);
  for (long long r = e0 / V; r * V < e1; ++r) {
    const int lo = static_cast<int>(max(e0, r * V) - r * V);
    const int hi = static_cast<int>(min(e1, (r + 1) * V) - r * V);
    const uint64_t k = block_row_key(p.Z + r * V, lo, hi, p.vec4 != 0, s_red);
    const int q = static_cast<int>(r / p.S);
    if (threadIdx.x == 0) {
      atomicMax(reinterpret_cast<unsigned long long*>(p.rowkey + r), static_cast<unsigned long long>(k));
      // the row-key update is ordered before the arrival (counted in
      // elements); the last arrival's fence orders its reads after all
      __threadfence();
      const unsigned long long n = static_cast<unsigned long long>(hi - lo);
      const unsigned long long old = atomicAdd(reinterpret_cast<unsigned long long*>(p.req_done + q), n);
      s_last = old + n == per_req;
      if (s_last) {
        p.req_done[q] = 0ull;  // ready for the next launch
        __threadfence();
      }
    }
    __syncthreads();
    if (s_last) walk_request(p, q, s_dyn);
  }
}

}  // namespace

size_t accept_smem_bytes(const AcceptParams& p) { return static_cast<size_t>(p.S) * 8; }

void accept_plan(AcceptParams& p, int num_sms) {
  // about eight resident CTAs per SM, one wave, equal pieces (whole float4s)
  const long long total = static_cast<long long>(p.n_req) * p.S * p.V;
  long long g = 8ll * num_sms;
  const long long min_piece = 1024;  // one float4 per thread
  if (total / g < min_piece) g = (total + min_piece - 1) / min_piece;
  if (g < 1) g = 1;
  long long piece = (total + g - 1) / g;
  piece = (piece + 3) / 4 * 4;
  p.piece = piece;
  p.grid = static_cast<int>((total + piece - 1) / piece);
  p.vec4 = (p.V % 4 == 0) ? 1 : 0;
}

cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream) {
  k_accept<<<p.grid, kAThreads, accept_smem_bytes(p), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dt

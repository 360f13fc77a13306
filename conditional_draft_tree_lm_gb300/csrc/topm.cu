// Top-M candidate restriction and the rest log-partition of each (request, depth)
// row of base logits ("Resumen Técnico: DominoTree", Componentes Principales,
// 2. Restricción de Candidatos (Top-M)).
//
// One kernel, grid (S chunks, rows), 512 threads.  Each CTA holds one chunk of
// one row (<= 16384 logits, 32 per thread in registers; padding is -inf) and
// writes the chunk's top-M, sorted by (logit desc, token id asc):
//   1. the chunk's max, and the mean and standard deviation of a sample (the
//      first 4 values of every thread);
//   2. from the sample, a threshold mx - c*sigma (c on a ladder 1 .. 4) that
//      should keep about 2M values;
//   3. the values at or above it are counted exactly (warp scans and one
//      shared-memory atomic per warp) and collected; too few (< M) moves to
//      the next rung and counts again, too many (> 512) or none left falls back
//      to a radix select of the whole chunk;
//   4. the M-th largest candidate is found with a 256-bin histogram of the
//      candidates' values (its bin's few keys ranked exactly); the M best are
//      gathered and ranked among themselves by counting, which gives the
//      sorted list.
// The chunk also reports the max of logit/T and the sum of exp(logit/T - max)
// over its non-selected tokens, each thread adding its own values in a fixed
// order (no result bit depends on the order of atomics).
//
// The last CTA of a row (a per-row arrival counter; nothing waits) merges the
// S sorted lists the same way: the M-th largest of the S*M entries by the
// histogram, the M best ranked among themselves, and
//   rest_lse = log( sum_chunks part_sum e^{part_max} + sum_{losing entries} e^{logit/T} ),
// so every non-candidate token enters the log-partition exactly once.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace dt {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kVPT = 32;              // values per thread: chunk <= kThreads * kVPT
constexpr int kMaxChunk = kThreads * kVPT;
constexpr int kMaxMerge = 8192;       // S * M entries merged per row
constexpr int kSample = 4;            // values per thread in the sample
constexpr int kRungs = 8;             // threshold ladder
constexpr int kCandCap = kThreads;    // candidates ranked in the partial phase
constexpr int kMergeCap = 2048;       // merge candidates ranked among themselves
constexpr int kPre = 4;               // entries of each list a merge thread loads up front

// Phase stamps (built with -DDT_TOPM_TIMING only): %globaltimer at the phase
// boundaries of row 0: [0][split][k] for the chunk CTAs, [1][0][k] for the CTA
// that merges the row; dt_topm_stamps copies them out.
#ifdef DT_TOPM_TIMING
constexpr int kTopmStampSplits = 64;
constexpr int kTopmStamps = 16;
__device__ unsigned long long g_topm_stamps[2][kTopmStampSplits][kTopmStamps];
// which 1 in the merge-only kernel (grid = rows): row 0 is CTA 0
#define TOPM_STAMP(which, k)                                                                      \
  do {                                                                                           \
    if (threadIdx.x == 0 &&                                                                      \
        ((which) ? (gridDim.y == 1 ? blockIdx.x == 0 : blockIdx.y == 0)                          \
                 : (blockIdx.y == 0 && blockIdx.x < kTopmStampSplits)))                          \
      g_topm_stamps[which][(which) ? 0 : blockIdx.x][k] = dt_globaltimer();                       \
  } while (0)
#else
#define TOPM_STAMP(which, k) \
  do {                       \
  } while (0)
#endif

DT_DEVINL float rung_c(int k) {
  return k < 5 ? 1.0f + 0.25f * static_cast<float>(k) : (k == 5 ? 2.5f : (k == 6 ? 3.0f : 4.0f));
}

DT_DEVINL float block_sum(float v, float* red) {
  v = warp_sum(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float s = threadIdx.x < kWarps ? red[threadIdx.x] : 0.0f;
    s = warp_sum(s);
    if (threadIdx.x == 0) red[kWarps] = s;
  }
  __syncthreads();
  return red[kWarps];
}

// Slot of this thread's first flagged value in a block-wide list: a warp scan
// and one atomic per warp on *counter (slot order across warps is arbitrary).
DT_DEVINL int claim_slots(int mine, int* counter) {
  const int lane = threadIdx.x & 31;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  int base = 0;
  if (lane == 31 && incl > 0) base = atomicAdd(counter, incl);
  base = __shfl_sync(0xFFFFFFFFu, base, 31);
  return base + incl - mine;
}

// Exact ranks of keys[0, c) among themselves (the number of larger keys; keys
// are distinct).  Each key is ranked by a group of g consecutive threads (g a
// power of two <= 32, as many as the block allows), whose partial counts are
// added with shuffles; fn(e, key, rank) then runs on the group's first thread.
// Every thread of the block must call.
template <class Fn>
DT_DEVINL void rank_all(const uint64_t* keys, int c, Fn fn) {
  int g = 1;
  while (g < 32 && 2 * g * c <= kThreads) g <<= 1;
  for (int base = 0; base < c * g; base += kThreads) {
    const int idx = base + static_cast<int>(threadIdx.x);
    const int e = idx / g, part = idx - e * g;
    uint64_t ke = 0ull;
    int rk = 0;
    if (e < c) {
      ke = keys[e];
#pragma unroll 4
      for (int f = part; f < c; f += g) rk += keys[f] > ke ? 1 : 0;
    }
    for (int o = 1; o < g; o <<= 1) rk += __shfl_xor_sync(0xFFFFFFFFu, rk, o);
    if (e < c && part == 0) fn(e, ke, rk);
  }
}

// The m-th largest of the nonzero keys among keys[0, n) in shared memory
// (distinct; 1 <= m), or 0 when there are fewer than m of them.  A 256-bin
// histogram over the value range puts the m-th key into one bin (bins are
// monotone in the value, so every key of an earlier bin is larger); that
// bin's keys are gathered into bnd (kMergeCap keys) and ranked among
// themselves, or, when more than that share the bin, each is ranked over the
// whole array.  hist: 256 words; sc: 4 ints; red: 2 kWarps floats; s_key: one
// key.  Every thread of the block calls; all get the key.
template <int kWhich>  // stamp set of the timing build: 0 chunk, 1 merge
DT_DEVINL uint64_t block_kth_key(const uint64_t* keys, int n, int m, uint32_t* hist, int* sc, uint64_t* bnd,
                                 float* red, uint64_t* s_key) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float lo = INFINITY, hi = -INFINITY;
  for (int e = tid; e < n; e += kThreads) {
    const uint64_t k = keys[e];
    if (k != 0ull) {
      const float v = key_f32(static_cast<uint32_t>(k >> 32));
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
  }
  lo = -warp_max(-lo);
  hi = warp_max(hi);
  if (lane == 0) {
    red[warp] = lo;
    red[kWarps + warp] = hi;
  }
  for (int b = tid; b < 256; b += kThreads) hist[b] = 0u;
  if (tid == 0) {
    sc[0] = -1;
    sc[2] = 0;
    *s_key = 0ull;
  }
  __syncthreads();
  TOPM_STAMP(kWhich, 10);
  lo = INFINITY;
  hi = -INFINITY;
  for (int w = 0; w < kWarps; ++w) {
    lo = fminf(lo, red[w]);
    hi = fmaxf(hi, red[kWarps + w]);
  }
  const float scale = hi > lo ? 256.0f / (hi - lo) : 0.0f;
  auto bin_of = [&](uint64_t k) {
    return min(255, max(0, __float2int_rz((hi - key_f32(static_cast<uint32_t>(k >> 32))) * scale)));
  };
  for (int e = tid; e < n; e += kThreads) {
    const uint64_t k = keys[e];
    if (k != 0ull) atomicAdd(&hist[bin_of(k)], 1u);
  }
  __syncthreads();
  TOPM_STAMP(kWhich, 11);
  if (warp == 0) {
    // lane l totals bins 8l .. 8l+7; the first bin where the running count
    // reaches m holds the m-th key
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
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl >= static_cast<uint32_t>(m));
    if (hit && lane == __ffs(hit) - 1) {
      uint32_t cum = incl - sum;
      for (int j = 0; j < 8; ++j) {
        if (cum + c8[j] >= static_cast<uint32_t>(m)) {
          sc[0] = 8 * lane + j;
          sc[1] = static_cast<int>(cum);
          break;
        }
        cum += c8[j];
      }
    }
  }
  __syncthreads();
  TOPM_STAMP(kWhich, 12);
  const int bt = sc[0];
  if (bt < 0) return 0ull;  // fewer than m keys: every one is among the best m (uniform)
  const int need = m - sc[1];  // the need-th largest key of bin bt
  for (int e = tid; e < n; e += kThreads) {
    const uint64_t k = keys[e];
    if (k != 0ull && bin_of(k) == bt) {
      const int at = atomicAdd(&sc[2], 1);
      if (at < kMergeCap) bnd[at] = k;
    }
  }
  __syncthreads();
  TOPM_STAMP(kWhich, 13);
  const int nb = sc[2];
  if (nb <= kMergeCap) {
    rank_all(bnd, nb, [&](int, uint64_t ke, int rk) {
      if (rk == need - 1) *s_key = ke;
    });
  } else {
    for (int e = tid; e < n; e += kThreads) {
      const uint64_t k = keys[e];
      if (k == 0ull || bin_of(k) != bt) continue;
      int rk = 0;
      for (int f = 0; f < n; ++f) {
        const uint64_t kf = keys[f];
        rk += (kf > k && bin_of(kf) == bt) ? 1 : 0;
      }
      if (rk == need - 1) *s_key = k;
    }
  }
  __syncthreads();
  TOPM_STAMP(kWhich, 14);
  return *s_key;
}

// Shared memory a row merge works in.
struct MergeSmem {
  uint32_t* hist;  // 256 words
  int* scan;       // 4 ints
  float* red;      // kWarps + 1 floats
  float* red4;     // 2 kWarps floats
  uint64_t* s_lb;  // one key
  int* s_ncand;
  uint64_t* big;   // S * M entries
  uint64_t* cand;  // kMergeCap keys
};

DT_DEVINL float block_max(float v, float* red) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float s = threadIdx.x < kWarps ? red[threadIdx.x] : -INFINITY;
    s = warp_max(s);
    if (threadIdx.x == 0) red[kWarps] = s;
  }
  __syncthreads();
  return red[kWarps];
}

// The merge when every list carries its suffix sums (part_tail): only the
// lists' heads are read.  The M-th largest of the first t entries of every
// list (S t >= M) bounds the row's M-th from below, so the row's M best are
// among each list's entries at or above it (a prefix of the sorted list);
// those few are selected exactly, and the log-partition takes, per list, its
// rest sum plus the suffix sum after its entries among the M best.  Returns
// false, having written nothing, when more than kMergeCap entries reach the
// bound (or fewer than M exist), for the full merge to run instead.
DT_DEVINL bool merge_row_tails(const TopmParams& p, int row, const MergeSmem& m, float invT, bool arrivals) {
  const int tid = threadIdx.x;
  const size_t rb = static_cast<size_t>(row) * p.S;
  const int S = p.S, M = p.M;
  if (S > 256) return false;  // one thread per list, counts in the 256-word histogram
  auto key_at = [&](int s2, int j) {
    const size_t e = (rb + s2) * M + j;
    return rank_key(p.part_val[e], static_cast<uint32_t>(p.part_id[e]));
  };
  const int t = min(M, max(1, (M + S - 1) / S));
  if (t > kPre) return false;
  // thread s: everything of list s the merge usually needs, loaded at once
  // (its length, max and rest sum, its first kPre keys and suffix sums)
  int cnt = 0;
  float pm = -INFINITY, ps = 0.0f;
  uint64_t k4[kPre];
  float t4[kPre + 1];
  if (tid < S) {
    cnt = p.part_cnt[rb + tid];
    pm = p.part_max[rb + tid];
    ps = p.part_sum[rb + tid];
#pragma unroll
    for (int j = 0; j < kPre; ++j) {
      k4[j] = j < cnt ? key_at(tid, j) : 0ull;
      t4[j] = j < cnt ? p.part_tail[(rb + tid) * M + j] : 0.0f;
    }
    t4[kPre] = kPre < cnt ? p.part_tail[(rb + tid) * M + kPre] : 0.0f;
  }
  const float gmax = block_max(tid < S ? pm : -INFINITY, m.red);
  const int n1 = S * t;
  // the lists' first t entries (t <= kPre: from the registers)
  if (tid < S) {
#pragma unroll
    for (int j = 0; j < kPre; ++j)
      if (j < t) m.big[tid * t + j] = k4[j];
  }
  if (tid == 0) *m.s_lb = 0ull;
  __syncthreads();
  // the M-th largest head: few heads are ranked directly (the key of rank
  // M - 1; zero, i.e. every entry, when fewer than M lists hold any), many
  // through the histogram
  uint64_t lb;
  if (n1 <= kThreads) {
    rank_all(m.big, n1, [&](int, uint64_t ke, int rk) {
      if (rk == M - 1) *m.s_lb = ke;
    });
    __syncthreads();
    lb = *m.s_lb;
  } else {
    lb = block_kth_key<1>(m.big, n1, M, m.hist, m.scan, m.cand, m.red4, m.s_lb);
  }
  TOPM_STAMP(1, 1);
  // thread s: list s's entries at or above the bound (a prefix): the first
  // kPre from the registers, any further ones four at a time from memory;
  // their count, then their place in the candidate list (lists in order, so
  // the list is the same every run)
  int* ncs = reinterpret_cast<int*>(m.hist);  // [S] (the histogram is free again)
  int nmine = 0;
  if (tid < S) {
#pragma unroll
    for (int j = 0; j < kPre; ++j) nmine += (j < cnt && k4[j] >= lb) ? 1 : 0;
    if (nmine == kPre) {
      for (int j0 = kPre; j0 < cnt; j0 += 4) {
        uint64_t q4[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) q4[i] = j0 + i < cnt ? key_at(tid, j0 + i) : 0ull;
        int more = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) more += (j0 + i < cnt && q4[i] >= lb) ? 1 : 0;
        nmine += more;
        if (more < 4) break;
      }
    }
  }
  int total;
  const int base = block_exclusive_scan(nmine, m.scan, &total);
  if (total > kMergeCap || total < M) return false;  // (uniform: every thread has the total)
  int* list_of = reinterpret_cast<int*>(m.big);  // [kMergeCap] list of candidate e (big is free again)
  if (tid < S) {
#pragma unroll
    for (int j = 0; j < kPre; ++j)
      if (j < nmine) {
        m.cand[base + j] = k4[j];
        list_of[base + j] = tid;
      }
    for (int j = kPre; j < nmine; ++j) {
      m.cand[base + j] = key_at(tid, j);
      list_of[base + j] = tid;
    }
  }
  if (tid < S) ncs[tid] = 0;
  __syncthreads();
  TOPM_STAMP(1, 2);
  // ranks among the candidates: the M best are written in order, and each
  // list counts its entries among them
  rank_all(m.cand, total, [&](int e, uint64_t ke, int rk) {
    if (rk < M) {
      p.cand_tok[static_cast<size_t>(row) * M + rk] = static_cast<int>(rank_key_id(ke));
      p.cand_base[static_cast<size_t>(row) * M + rk] = key_f32(static_cast<uint32_t>(ke >> 32));
      atomicAdd(&ncs[list_of[e]], 1);
    }
  });
  __syncthreads();
  TOPM_STAMP(1, 3);
  // per list: its rest sum and the suffix after its entries among the M best
  float rest = 0.0f;
  if (tid < S) {
    const int c = ncs[tid];
    float tail = 0.0f;
    if (c < cnt) {
      tail = t4[kPre];
#pragma unroll
      for (int j = kPre - 1; j >= 0; --j) tail = c == j ? t4[j] : tail;
      if (c > kPre) tail = p.part_tail[(rb + tid) * M + c];
    }
    if (pm > -INFINITY) rest = (ps + tail) * expf(pm - gmax);
  }
  rest = block_sum(rest, m.red);
  if (tid == 0) {
    p.rest_lse[row] = rest > 0.0f ? gmax + logf(rest) : -INFINITY;
    if (arrivals) p.row_done[row] = 0u;  // ready for the next round
  }
  TOPM_STAMP(1, 4);
  return true;
}

// The merge of row `row`'s S sorted partial lists: the M best (cand_tok,
// cand_base, sorted) and rest_lse.  arrivals: the row's arrival counter is
// reset for the next launch (the merge at the end of the Top-M kernel).
DT_DEVINL void merge_row(const TopmParams& p, int row, const MergeSmem& m, float invT, bool arrivals) {
  if (p.part_tail && merge_row_tails(p, row, m, invT, arrivals)) return;
  const int tid = threadIdx.x;
  const size_t rb = static_cast<size_t>(row) * p.S;
  const int S = p.S, M = p.M;
  const int total = S * M;
  float gmax = -INFINITY;
  for (int s2 = tid; s2 < S; s2 += kThreads) gmax = fmaxf(gmax, p.part_max[rb + s2]);
  gmax = block_max(gmax, m.red);
  // entries e = s*M + j; value, id and list length are read together, eight
  // entries per thread at a time (their loads in flight at once); slots past
  // a list's length hold stale data and get key 0
  constexpr int kBatch = 8;
  for (int eb = tid; eb < total; eb += kBatch * kThreads) {
    float v[kBatch];
    int id[kBatch], ok[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int e = min(eb + b * kThreads, total - 1);
      const int s2 = e / M, j = e - s2 * M;
      v[b] = p.part_val[rb * M + e];
      id[b] = p.part_id[rb * M + e];
      ok[b] = j < p.part_cnt[rb + s2];
    }
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int e = eb + b * kThreads;
      if (e < total) m.big[e] = ok[b] ? rank_key(v[b], static_cast<uint32_t>(id[b])) : 0ull;
    }
  }
  if (tid == 0) *m.s_ncand = 0;
  __syncthreads();
  // the row's M-th largest entry; the best M are gathered and ranked among
  // themselves, every other entry feeds the log-partition (each thread over
  // its own fixed range of entries)
  const uint64_t kth = block_kth_key<1>(m.big, total, M, m.hist, m.scan, m.cand, m.red4, m.s_lb);
  TOPM_STAMP(1, 1);
  float rest2 = 0.0f;
  const int per = (total + kThreads - 1) / kThreads;
  const int e0 = min(total, tid * per), e1 = min(total, e0 + per);
  for (int e = e0; e < e1; ++e) {
    const uint64_t k2 = m.big[e];
    const bool lose = k2 != 0ull && k2 < kth;
    rest2 += lose ? expf(key_f32(static_cast<uint32_t>(k2 >> 32)) * invT - gmax) : 0.0f;
    if (k2 != 0ull && k2 >= kth) {
      const int at = atomicAdd(m.s_ncand, 1);
      if (at < kMergeCap) m.cand[at] = k2;
    }
  }
  __syncthreads();
  const int nc = *m.s_ncand;
  TOPM_STAMP(1, 2);
  rank_all(m.cand, min(nc, kMergeCap), [&](int, uint64_t ke, int rk) {
    if (rk < M) {
      p.cand_tok[static_cast<size_t>(row) * M + rk] = static_cast<int>(rank_key_id(ke));
      p.cand_base[static_cast<size_t>(row) * M + rk] = key_f32(static_cast<uint32_t>(ke >> 32));
    }
  });
  for (int s2 = tid; s2 < S; s2 += kThreads) {
    const float ps = p.part_sum[rb + s2];
    if (ps > 0.0f) rest2 += ps * expf(p.part_max[rb + s2] - gmax);
  }
  TOPM_STAMP(1, 3);
  rest2 = block_sum(rest2, m.red);
  if (tid == 0) {
    if (nc < M) dt_report(p.status, DT_DEV_BOUNDS);
    p.rest_lse[row] = rest2 > 0.0f ? gmax + logf(rest2) : -INFINITY;
    if (arrivals) p.row_done[row] = 0u;  // ready for the next round
  }
  TOPM_STAMP(1, 4);
}

// kMinBlocks = 2 caps the registers so that two CTAs share an SM: for grids of
// many waves (many rows), where each CTA's chain of phases is latency-bound.
template <int kMinBlocks>
__global__ void __launch_bounds__(kThreads, kMinBlocks) k_topm(const TopmParams p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ uint32_t hist[kWarps * 256];
  __shared__ uint32_t state[4];
  __shared__ int scan[40];
  __shared__ float red[kWarps + 1];
  __shared__ float red4[4][kWarps + 1];
  __shared__ int rung_cnt[kWarps][kRungs];
  __shared__ int s_rung, s_ncand, s_last;
  __shared__ uint64_t s_lb;

  // dynamic shared memory: a 64 KB area (chunk keys of the fallback, merge
  // entries) followed by the candidate keys
  uint64_t* big = reinterpret_cast<uint64_t*>(dyn);
  uint64_t* cand = big + kMaxMerge;  // [kMergeCap]

  const int row = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int v0 = split * p.chunk;
  const int n = max(0, min(p.V, v0 + p.chunk) - v0);
  const float* x = p.logits + static_cast<size_t>(row) * p.V + v0;
  const float invT = 1.0f / p.T;
  const size_t q = static_cast<size_t>(row) * p.S + split;
  const int mloc = min(p.M, n);
  const int nv = n > tid ? min(kVPT, (n - tid + kThreads - 1) / kThreads) : 0;  // valid values of this thread

  // the logits come from the previous kernel; the next one may then launch
  TOPM_STAMP(0, 0);
  dt_grid_wait();
  TOPM_STAMP(0, 1);
  dt_grid_release();
  if (p.clear_word && blockIdx.x == 0 && blockIdx.y == 0 && tid == 0) *p.clear_word = 0u;

  // ---------------- 1. the chunk in registers; max; sample statistics ----------------
  float vals[kVPT];
#pragma unroll
  for (int j = 0; j < kVPT; ++j) vals[j] = j < nv ? x[tid + j * kThreads] : -INFINITY;
  float mx = -INFINITY;
#pragma unroll
  for (int j = 0; j < kVPT; ++j) mx = fmaxf(mx, vals[j]);
  float sm = 0.0f, sq = 0.0f, ns = 0.0f;
#pragma unroll
  for (int j = 0; j < kSample; ++j)
    if (j < nv) {
      sm += vals[j];
      sq += vals[j] * vals[j];
      ns += 1.0f;
    }
  mx = warp_max(mx);
  sm = warp_sum(sm);
  sq = warp_sum(sq);
  ns = warp_sum(ns);
  if (lane == 0) {
    red4[0][warp] = mx;
    red4[1][warp] = sm;
    red4[2][warp] = sq;
    red4[3][warp] = ns;
  }
  __syncthreads();
  if (tid < 32) {
    float a = tid < kWarps ? red4[0][tid] : -INFINITY;
    float b = tid < kWarps ? red4[1][tid] : 0.0f;
    float c = tid < kWarps ? red4[2][tid] : 0.0f;
    float d = tid < kWarps ? red4[3][tid] : 0.0f;
    a = warp_max(a);
    b = warp_sum(b);
    c = warp_sum(c);
    d = warp_sum(d);
    if (tid == 0) {
      red4[0][kWarps] = a;
      red4[1][kWarps] = b;
      red4[2][kWarps] = c;
      red4[3][kWarps] = d;
    }
  }
  __syncthreads();
  mx = red4[0][kWarps];
  const float nsamp = red4[3][kWarps];
  const float mean = nsamp > 0.0f ? red4[1][kWarps] / nsamp : 0.0f;
  const float sigma = nsamp > 0.0f ? sqrtf(fmaxf(red4[2][kWarps] / nsamp - mean * mean, 0.0f)) : 0.0f;
  const float mxT = mx * invT;

  TOPM_STAMP(0, 2);
  // ---------------- 2. the first rung to try, from the sample ----------------
  if (mloc < n && sigma > 0.0f) {
    int cnt[kRungs];
#pragma unroll
    for (int k = 0; k < kRungs; ++k) cnt[k] = 0;
#pragma unroll
    for (int j = 0; j < kSample; ++j)
#pragma unroll
      for (int k = 0; k < kRungs; ++k) cnt[k] += (j < nv && vals[j] >= mx - rung_c(k) * sigma) ? 1 : 0;
#pragma unroll
    for (int k = 0; k < kRungs; ++k) {
      const int c = __reduce_add_sync(0xFFFFFFFFu, cnt[k]);
      if (lane == 0) rung_cnt[warp][k] = c;
    }
    __syncthreads();
    if (warp == 0) {
      // lane k totals rung k; the first rung expected to keep >= 2M values
      int c = 0;
      if (lane < kRungs)
        for (int w = 0; w < kWarps; ++w) c += rung_cnt[w][lane];
      const float est = static_cast<float>(c) * (static_cast<float>(n) / nsamp);
      const unsigned ok = __ballot_sync(0xFFFFFFFFu, lane < kRungs && est >= 2.0f * mloc);
      if (lane == 0) s_rung = ok ? __ffs(ok) - 1 : kRungs - 1;
    }
  } else if (tid == 0) {
    s_rung = mloc >= n ? kRungs : -1;  // all values are candidates / fall back
  }
  __syncthreads();

  TOPM_STAMP(0, 3);
  // ---------------- 3. exact count and collection above the threshold ----------------
  float rest = 0.0f;
  int k = s_rung;
  int c = 0;
  uint32_t flags = 0u;
  bool fast = k >= 0;
  while (fast) {
    const float th = k >= kRungs ? -INFINITY : mx - rung_c(k) * sigma;
    flags = 0u;
#pragma unroll
    for (int j = 0; j < kVPT; ++j)
      if (j < nv && vals[j] >= th) flags |= 1u << j;
    if (tid == 0) s_ncand = 0;
    __syncthreads();
    const int mine = __popc(flags);
    int pos = claim_slots(mine, &s_ncand);
    if (pos + mine <= kCandCap) {
#pragma unroll
      for (int j = 0; j < kVPT; ++j)
        if ((flags >> j) & 1u) cand[pos++] = rank_key(vals[j], static_cast<uint32_t>(v0 + tid + j * kThreads));
    }
    __syncthreads();
    c = s_ncand;
    __syncthreads();  // every thread has read the count before a retry resets it
    if (c >= mloc && c <= kCandCap) break;      // the candidate set
    if (c < mloc && k + 1 < kRungs) {          // too few: next rung
      ++k;
      continue;
    }
    fast = false;                               // too many, or the ladder is exhausted
  }
  __syncthreads();
  TOPM_STAMP(0, 4);

  if (fast) {
    // ---------------- 4. the M-th candidate; the sorted partial list ----------------
    if (tid == 0) s_ncand = 0;  // (c is held in registers) counts the winners below
    const uint64_t kth = c > mloc ? block_kth_key<0>(cand, c, mloc, hist, scan, big, &red4[0][0], &s_lb) : 0ull;
    __syncthreads();
    TOPM_STAMP(0, 7);
    // each thread's values outside the best M feed the log-partition (in its
    // own fixed order); the best M are gathered and ranked among themselves
#pragma unroll
    for (int j = 0; j < kVPT; ++j) {
      if (!((flags >> j) & 1u)) {
        rest += __expf(vals[j] * invT - mxT);  // padding gives 0
      } else if (rank_key(vals[j], static_cast<uint32_t>(v0 + tid + j * kThreads)) < kth) {
        rest += expf(vals[j] * invT - mxT);
      }
    }
    TOPM_STAMP(0, 8);
    for (int e = tid; e < c; e += kThreads) {
      const uint64_t k2 = cand[e];
      if (k2 >= kth) big[atomicAdd(&s_ncand, 1)] = k2;
    }
    __syncthreads();
    TOPM_STAMP(0, 9);
    rank_all(big, s_ncand, [&](int, uint64_t ke, int rk) {
      const float v = key_f32(static_cast<uint32_t>(ke >> 32));
      p.part_id[q * p.M + rk] = static_cast<int>(rank_key_id(ke));
      p.part_val[q * p.M + rk] = v;
      if (rk == mloc - 1) p.part_kth[q] = (mloc < n) ? v : -INFINITY;
    });
  } else {
    // ---------------- fallback: radix select over the whole chunk ----------------
    uint32_t* keys = reinterpret_cast<uint32_t*>(big);
#pragma unroll
    for (int j = 0; j < kVPT; ++j)
      if (j < nv) keys[tid + j * kThreads] = f32_key(vals[j]);
    __syncthreads();
    uint32_t t = 0;
    int need = n;
    radix_select_kth_largest(keys, n, mloc, hist, kWarps * 256, state, t, need);
    // keys above t win, plus the `need` lowest-indexed keys equal to t
    uint32_t tie_mask = 0u;  // bit j: element tid + j*kThreads equals t
#pragma unroll
    for (int j = 0; j < kVPT; ++j)
      if (j < nv && f32_key(vals[j]) == t) tie_mask |= 1u << j;
    int tot;
    (void)block_exclusive_scan(__popc(tie_mask), scan, &tot);
    uint32_t tie_win = 0u;  // bit j: element tid + j*kThreads is a winning tie
    if (tot <= need) {
      tie_win = tie_mask;
    } else {
      // index order is j-major (e = tid + j * kThreads): one scan per slice
      int before = 0;
      for (int j = 0; j < kVPT; ++j) {
        const int f = static_cast<int>((tie_mask >> j) & 1u);
        int slice;
        const int at = block_exclusive_scan(f, scan, &slice) + before;
        if (f && at < need) tie_win |= 1u << j;
        before += slice;
      }
    }
    uint32_t win = tie_win;
#pragma unroll
    for (int j = 0; j < kVPT; ++j)
      if (j < nv && f32_key(vals[j]) > t) win |= 1u << j;
    int wrote;
    int pos = block_exclusive_scan(__popc(win), scan, &wrote);
#pragma unroll
    for (int j = 0; j < kVPT; ++j) {
      if ((win >> j) & 1u) {
        cand[pos++] = rank_key(vals[j], static_cast<uint32_t>(v0 + tid + j * kThreads));
      } else {
        rest += __expf(vals[j] * invT - mxT);  // padding gives 0
      }
    }
    __syncthreads();
    rank_all(cand, mloc, [&](int, uint64_t ke, int rk) {
      const float v = key_f32(static_cast<uint32_t>(ke >> 32));
      p.part_id[q * p.M + rk] = static_cast<int>(rank_key_id(ke));
      p.part_val[q * p.M + rk] = v;
      if (rk == mloc - 1) p.part_kth[q] = (mloc < n) ? v : -INFINITY;
    });
  }
  TOPM_STAMP(0, 5);
  rest = block_sum(rest, red);
  if (tid == 0) {
    p.part_max[q] = mxT;
    p.part_sum[q] = rest;
    p.part_cnt[q] = mloc;
  }

  // ---------------- last CTA of the row merges ----------------
  // (the barrier orders the CTA's writes before thread 0's fence and arrival;
  // the arriving-last CTA's fence orders its reads after every arrival)
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    s_last = atomicAdd(&p.row_done[row], 1u) == static_cast<unsigned>(p.S - 1);
    __threadfence();
  }
  __syncthreads();
  TOPM_STAMP(0, 6);
  if (!s_last) return;
  TOPM_STAMP(1, 0);

  MergeSmem ms{hist, scan, red, &red4[0][0], &s_lb, &s_ncand, big, cand};
  merge_row(p, row, ms, invT, true);
}

// The merge alone, one CTA per row, over partial lists another kernel wrote
// (the LM-head GEMM's fused Top-M): dynamic shared memory holds S*M entries
// and the candidate keys.
__global__ void __launch_bounds__(kThreads, 1) k_topm_merge(const TopmParams p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ uint32_t hist[256];
  __shared__ int scan[40];
  __shared__ float red[kWarps + 1];
  __shared__ float red4[2 * kWarps];
  __shared__ int s_ncand;
  __shared__ uint64_t s_lb;
  uint64_t* big = reinterpret_cast<uint64_t*>(dyn);
  uint64_t* cand = big + max(static_cast<size_t>(p.S) * p.M, static_cast<size_t>(kMergeCap));
  TOPM_STAMP(1, 0);
  dt_grid_wait();  // the partial lists come from the previous kernel
  dt_grid_release();
  if (p.clear_word && blockIdx.x == 0 && threadIdx.x == 0) *p.clear_word = 0u;
  MergeSmem ms{hist, scan, red, red4, &s_lb, &s_ncand, big, cand};
  merge_row(p, static_cast<int>(blockIdx.x), ms, 1.0f / p.T, false);
}

// Many rows (at least one per SM): two CTAs per SM stream whole rows (rows
// blockIdx.x, + gridDim.x, ...) through kRowStages shared-memory slots filled
// by bulk copies of kRowSub tiles each, tile by tile.  A logit whose
// (value, lowest token) key exceeds the row's running bound tau is appended
// to a candidate buffer; every other one is a loser and feeds the thread's
// running log-partition sum.  When the buffer could overflow with the next
// tile (and after the row's last), it is cut to its M best (block_kth_key):
// the cut entries feed a second running sum and tau becomes the M-th key, so
// later logits enter only when they beat it.  A row starts from a bound taken
// from its first tile's lane maxima (for M up to kRowQuota per warp), so that
// the first tile does not fill the buffer.  The M kept are ranked among
// themselves; the two sums of every thread give rest_lse.  No partial lists
// and no merge.
constexpr int kRowVals = 8;                         // logits per thread and tile
constexpr int kRowTile = kThreads * kRowVals;       // 4096 logits, 16 KB
constexpr int kRowSub = 1;                          // tiles per copy
constexpr int kRowStages = 3;
constexpr int kRowCap = kRowTile + 2 * kCandCap;    // candidate buffer (keys)
constexpr int kRowQuota = 8;                        // first-tile bound: up to M = 8 per warp

// 2^x by the SFU's approximation (flushes subnormal results to zero)
DT_DEVINL float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

DT_DEVINL void row_bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

__global__ void __launch_bounds__(kThreads, 2) k_topm_rows(const TopmParams p) {
  extern __shared__ __align__(16) uint8_t dyn[];
  __shared__ uint32_t hist[256];
  __shared__ int sc[4];
  __shared__ float red[kWarps + 1];
  __shared__ float red4[2 * kWarps];
  __shared__ int s_cnt, s_keep, s_abort;
  __shared__ uint64_t s_key;
  __shared__ __align__(8) uint64_t s_full[kRowStages];
  float* ring = reinterpret_cast<float*>(dyn);  // [kRowStages][kRowSub kRowTile]
  uint64_t* buf = reinterpret_cast<uint64_t*>(ring + kRowStages * kRowSub * kRowTile);  // [kRowCap] candidates
  uint64_t* bnd = buf + kRowCap;  // [kMergeCap] block_kth_key's bin, then the kept keys
  const int tid = threadIdx.x, lane = tid & 31;
  const int V = p.V, M = p.M, G = static_cast<int>(gridDim.x);
  const float invT = 1.0f / p.T;
  const int nt = (V + kRowTile - 1) / kRowTile;  // tiles per row
  const int ncp = (nt + kRowSub - 1) / kRowSub;  // copies per row
  const int my_rows = (p.rows - static_cast<int>(blockIdx.x) + G - 1) / G;
  const int total = my_rows * nt;                // tiles of this CTA, row after row
  const int ncopies = my_rows * ncp;
  if (tid == 0) {
    for (int b = 0; b < kRowStages; ++b) mbar_init(&s_full[b], 1);
    s_abort = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  TOPM_STAMP(0, 0);
  dt_grid_wait();  // the logits come from the previous kernel
  dt_grid_release();
  TOPM_STAMP(0, 1);
  if (p.clear_word && blockIdx.x == 0 && tid == 0) *p.clear_word = 0u;
  __syncthreads();
  // copy c of this CTA: row blockIdx.x + (c / ncp) G, its tiles from
  // kRowSub (c % ncp) on, into slot c % kRowStages
  auto issue = [&](int c) {
    const int row = static_cast<int>(blockIdx.x) + (c / ncp) * G, t0 = (c - (c / ncp) * ncp) * kRowSub;
    const int n = min(kRowSub * kRowTile, V - t0 * kRowTile);
    row_bulk_load(ring + (c % kRowStages) * kRowSub * kRowTile, p.logits + static_cast<size_t>(row) * V + t0 * kRowTile,
                  static_cast<uint32_t>(n) * 4u, &s_full[c % kRowStages]);
  };
  // slot b's copies are issued by lane 0 of warp b
  if (lane == 0 && (tid >> 5) < min(ncopies, kRowStages)) issue(tid >> 5);
  float mt = 0.0f, st = 0.0f, me = 0.0f, se = 0.0f, tauv = 0.0f;
  uint64_t tau = 0ull;
  // the buffer down to its M best: the rest feed (me, se); tau = the M-th key
  auto cut = [&]() {
    const int n = s_cnt;
    const uint64_t kth = block_kth_key<0>(buf, n, M, hist, sc, bnd, red4, &s_key);
    if (kth == 0ull) return;  // at most M candidates: nothing to cut
    if (tid == 0) s_keep = 0;
    __syncthreads();
    for (int e = tid; e < n; e += kThreads) {
      const uint64_t k = buf[e];
      if (k >= kth) {
        bnd[atomicAdd(&s_keep, 1)] = k;
      } else {
        const float l = key_f32(static_cast<uint32_t>(k >> 32)) * invT;
        if (l > me) {
          se = (me > -INFINITY ? se * expf(me - l) : 0.0f) + 1.0f;
          me = l;
        } else {
          se += expf(l - me);
        }
      }
    }
    __syncthreads();
    const int nk = s_keep;
    for (int e = tid; e < nk; e += kThreads) buf[e] = bnd[e];
    if (tid == 0) s_cnt = nk;
    tau = kth;
    tauv = key_f32(static_cast<uint32_t>(kth >> 32));
    __syncthreads();
  };
  for (int q = 0, rn = 0, t = 0; q < total; ++q, t = (t + 1 == nt ? 0 : t + 1), rn += (t == 0 ? 1 : 0)) {
    const int row = static_cast<int>(blockIdx.x) + rn * G;  // the CTA's rn-th row, its tile t
    if (t == 0) {
      // a new row: losers' and cut entries' sums, the bound, the buffer
      mt = -INFINITY;
      st = 0.0f;
      me = -INFINITY;
      se = 0.0f;
      tau = 0ull;
      tauv = -INFINITY;
      if (tid == 0) s_cnt = 0;
    }
    const int c = rn * ncp + t / kRowSub, sub = t % kRowSub;  // the tile's copy, its place in it
    const int slot = c % kRowStages;
    // one thread waits for the copy; the barrier releases the others
#ifdef DT_TOPM_TIMING
    if (tid == 0 && blockIdx.x == 0 && q < kTopmStampSplits) g_topm_stamps[1][q][0] = dt_globaltimer();
#endif
    if (sub == 0 && tid == 0 && !mbar_wait(&s_full[slot], static_cast<uint32_t>(c / kRowStages) & 1u, p.status))
      s_abort = 1;
#ifdef DT_TOPM_TIMING
    if (tid == 0 && blockIdx.x == 0 && q < kTopmStampSplits) g_topm_stamps[1][q][1] = dt_globaltimer();
#endif
    __syncthreads();
    if (s_abort) return;  // a copy that never landed (reported): nothing more is issued or read
    // logits e = t kRowTile + 4 (h kThreads + tid) + {0..3}, h = 0, 1; -inf
    // past the row's end (the slot's bytes there are stale; only the last
    // tile has such places)
    float v[kRowVals];
    const bool full = (t + 1) * kRowTile <= V;
#pragma unroll
    for (int h = 0; h < kRowVals / 4; ++h) {
      const int j = 4 * (h * kThreads + tid);
      const float4 f = *reinterpret_cast<const float4*>(ring + (slot * kRowSub + sub) * kRowTile + j);
      v[4 * h] = f.x;
      v[4 * h + 1] = f.y;
      v[4 * h + 2] = f.z;
      v[4 * h + 3] = f.w;
      if (!full) {
        const int e = t * kRowTile + j;
        if (e >= V) v[4 * h] = -INFINITY;
        if (e + 1 >= V) v[4 * h + 1] = -INFINITY;
        if (e + 2 >= V) v[4 * h + 2] = -INFINITY;
        if (e + 3 >= V) v[4 * h + 3] = -INFINITY;
      }
    }
    float tm = -INFINITY;
#pragma unroll
    for (int u = 0; u < kRowVals; ++u) tm = fmaxf(tm, v[u]);
    if (t == 0 && M <= kWarps * kRowQuota) {
      // a first bound from the row's first tile: in every warp the q-th
      // largest lane maximum (q = ceil(M / warps), counted with repeats), and
      // the smallest of those over the warps.  At least warps x q >= M of the
      // tile's logits (one per lane taken) reach it, so the row's M-th key
      // lies above every key of that value's lowest priority: keys at or
      // below the bound are losers from the start
      const int qw = (M + kWarps - 1) / kWarps;
      uint32_t mk = f32_key(tm), kq = 0u;
      for (int rr = 0; rr < qw; ++rr) {
        kq = __reduce_max_sync(0xFFFFFFFFu, mk);
        const unsigned who = __ballot_sync(0xFFFFFFFFu, mk == kq);
        if (lane == __ffs(who) - 1) mk = 0u;  // (every real key is above 0)
      }
      uint32_t* wq = reinterpret_cast<uint32_t*>(red4);
      if (lane == 0) wq[tid >> 5] = kq;
      __syncthreads();
      uint32_t kmin = wq[0];
#pragma unroll
      for (int w = 1; w < kWarps; ++w) kmin = min(kmin, wq[w]);
      if (kmin > f32_key(-INFINITY)) {
        tau = (static_cast<uint64_t>(kmin) << 32) - 1ull;
        tauv = key_f32(kmin);
      }
      __syncthreads();  // (red4 is the cuts' scratch)
    }
    tm *= invT;
    if (tm > mt) {
      st = mt > -INFINITY ? st * __expf(mt - tm) : 0.0f;
      mt = tm;
    }
    // the losers' exponentials in four independent sums, as 2^(v c - m c)
    // with c = log2(e) / T; a logit at or above tau's value (rare once the
    // bound has risen) is checked by its exact key and appended with one
    // shared atomic, or is a loser after all
    float s4[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const float mref = mt > -INFINITY ? mt : 0.0f;  // (past the row's end: -inf, adds 0)
    const float c2 = invT * 1.4426950408889634f, b2 = -mref * 1.4426950408889634f;
    uint32_t fl = 0u;
#pragma unroll
    for (int u = 0; u < kRowVals; ++u) {
      const bool hi = v[u] >= tauv;
      fl |= hi ? 1u << u : 0u;
      const float y = ex2_approx(fmaf(v[u], c2, b2));
      s4[u & 3] += hi ? 0.0f : y;
    }
    if (__any_sync(0xFFFFFFFFu, fl != 0u)) {
#pragma unroll
      for (int u = 0; u < kRowVals; ++u)
        if ((fl >> u) & 1u) {
          const int e = t * kRowTile + 4 * ((u >> 2) * kThreads + tid) + (u & 3);
          const uint64_t k = rank_key(v[u], static_cast<uint32_t>(e));
          if (e < V && k > tau)
            buf[atomicAdd(&s_cnt, 1)] = k;
          else
            s4[u & 3] += ex2_approx(fmaf(v[u], c2, b2));
        }
    }
    st += (s4[0] + s4[1]) + (s4[2] + s4[3]);
    __syncthreads();  // the copy's last tile is read: refill its slot
    if ((sub == kRowSub - 1 || t + 1 == nt) && tid == 32 * slot && c + kRowStages < ncopies) issue(c + kRowStages);
    if (q == 0) TOPM_STAMP(0, 2);
#ifdef DT_TOPM_TIMING
    if (tid == 0 && blockIdx.x == 0 && q < kTopmStampSplits) g_topm_stamps[1][q][2] = dt_globaltimer();
#endif
    if (s_cnt + kRowTile > kRowCap || t + 1 == nt) cut();
    if (q == 0) TOPM_STAMP(0, 3);
#ifdef DT_TOPM_TIMING
    if (tid == 0 && blockIdx.x == 0 && q < kTopmStampSplits) g_topm_stamps[1][q][3] = dt_globaltimer();
#endif
    if (t + 1 < nt) continue;
    if (q + 1 == nt) TOPM_STAMP(0, 4);
    // the row's M kept, in rank order (value desc, lower token first)
    const int nk = s_cnt;
    rank_all(buf, nk, [&](int, uint64_t ke, int rk) {
      if (rk < M) {
        p.cand_tok[static_cast<size_t>(row) * M + rk] = static_cast<int>(rank_key_id(ke));
        p.cand_base[static_cast<size_t>(row) * M + rk] = key_f32(static_cast<uint32_t>(ke >> 32));
      }
    });
    // log-partition of everything but the M best: the two sums of every thread
    const float gmax = block_max(fmaxf(mt, me), red);
    float rest = (mt > -INFINITY ? st * expf(mt - gmax) : 0.0f) + (me > -INFINITY ? se * expf(me - gmax) : 0.0f);
    rest = block_sum(rest, red);
    if (tid == 0) {
      if (nk < M) dt_report(p.status, DT_DEV_BOUNDS);
      p.rest_lse[row] = rest > 0.0f ? gmax + logf(rest) : -INFINITY;
    }
    if (q + 1 == nt) TOPM_STAMP(0, 5);
    __syncthreads();  // the buffer is reset by the next row
  }
}

}  // namespace

void topm_plan(TopmParams& p, int num_sms) {
  // one CTA per SM over all rows (one wave), chunks of at most kMaxChunk
  // logits and at least 2M, and at most kMaxMerge entries per row to merge
  int S = max(1, num_sms / max(1, p.rows));
  S = max(S, (p.V + kMaxChunk - 1) / kMaxChunk);
  S = min(S, max(1, p.V / (2 * p.M)));
  S = min(S, max(1, kMaxMerge / p.M));
  p.S = S;
  p.chunk = (p.V + S - 1) / S;
  p.occ2 = S * p.rows > num_sms ? 1 : 0;  // more than one wave at one CTA per SM
  // at least one row per SM: one CTA per SM streams whole rows instead
  p.rowwise = (p.rows >= num_sms && p.M <= kCandCap && p.V >= 2 * p.M && p.V % 4 == 0) ? 1 : 0;
  p.num_sms = num_sms;
}

size_t topm_partial_smem(const TopmParams&) {
  return static_cast<size_t>(kMaxMerge) * 8 + static_cast<size_t>(kMergeCap) * 8;
}

size_t topm_merge_smem(const TopmParams& p) { return topm_partial_smem(p); }

size_t topm_rows_smem() {
  return static_cast<size_t>(kRowStages) * kRowSub * kRowTile * 4 + static_cast<size_t>(kRowCap + kMergeCap) * 8;
}

cudaError_t topm_prepare() {
  cudaError_t e = dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_topm<1>));
  if (e == cudaSuccess) e = dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_topm_rows));
  if (e == cudaSuccess) e = dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_topm<2>));
  if (e == cudaSuccess) e = dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_topm_merge));
  return e;
}

const char* topm_unsupported(const TopmParams& p) {
  if (p.rows < 1 || p.rows > 65535) return "rows must be 1..65535 (one grid row per logit row)";
  if (p.M > kCandCap) return "M above 512";
  if (p.chunk > kMaxChunk) return "V too large for M: a chunk would exceed 16384 logits (V <= 8192 * 16384 / M)";
  if (p.S * p.M > kMaxMerge) return "chunks x M above the 8192 merged entries of a row";
  return nullptr;
}

size_t topm_merge_only_smem(const TopmParams& p) {
  return (std::max(static_cast<size_t>(p.S) * p.M, static_cast<size_t>(kMergeCap)) + kMergeCap) * 8;
}

const char* topm_merge_unsupported(const TopmParams& p) {
  if (p.rows < 1 || p.rows > 65535) return "rows must be 1..65535";
  if (p.M < 1 || p.M > kMergeCap) return "M out of range";
  if (topm_merge_only_smem(p) > 227 * 1024) return "too many partial lists to merge in shared memory";
  return nullptr;
}

cudaError_t launch_topm_merge(const TopmParams& p, cudaStream_t stream) {
  if (topm_merge_unsupported(p)) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.rows);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = topm_merge_only_smem(p);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, k_topm_merge, p);
}

cudaError_t launch_topm(const TopmParams& p_in, cudaStream_t stream) {
  if (topm_unsupported(p_in)) return cudaErrorInvalidValue;
  TopmParams p = p_in;
  // the row-streaming kernel bulk-copies whole rows: 16-byte aligned logits
  if (p.rowwise && (reinterpret_cast<uintptr_t>(p.logits) & 15u) != 0) p.rowwise = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.rowwise ? dim3(std::min(p.rows, 2 * p.num_sms)) : dim3(p.S, p.rows);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = p.rowwise ? topm_rows_smem() : topm_partial_smem(p);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 1 : 0;
  if (p.rowwise) return cudaLaunchKernelEx(&cfg, k_topm_rows, p);
  return p.occ2 ? cudaLaunchKernelEx(&cfg, k_topm<2>, p) : cudaLaunchKernelEx(&cfg, k_topm<1>, p);
}

}  // namespace dt

#ifdef DT_TOPM_TIMING
// The Top-M phase stamps of row 0 in the last launch: 2 x 64 x 8 %globaltimer
// values ([chunk CTAs / merging CTA][split][k]; chunk CTA k: start, after the
// wait for the previous kernel, after the chunk's statistics, after the rung
// choice, after the candidate collection, after the ranks, after the arrival;
// merging CTA k: start, after the bound, after the candidates, after the
// ranks, end).  Returns the number of values copied, or -1.
extern "C" int dt_topm_stamps(unsigned long long* out, int n) {
  const int total = 2 * dt::kTopmStampSplits * dt::kTopmStamps;
  if (!out || n < total) return -1;
  return cudaMemcpyFromSymbol(out, dt::g_topm_stamps, sizeof(dt::g_topm_stamps)) == cudaSuccess ? total : -1;
}
#endif


// Top-M candidate restriction and the rest log-partition of each (request, depth)
// row of base logits ("Resumen Técnico: DominoTree", Componentes Principales,
// 2. Restricción de Candidatos (Top-M)).
//
// One kernel, grid (S chunks, rows).  Each CTA holds one chunk of one row
// (<= 16384 logits, 32 per thread in registers) and finds the chunk's top-M:
//   1. max, mean and standard deviation of the chunk;
//   2. a histogram of the values within 4 sigma of the max in quarter-sigma
//      buckets; the tightest bucket edge that keeps >= M values is chosen, so
//      every one of the chunk's top-M lies above it;
//   3. the values above that edge (typically M..2M of them) are collected with
//      an exact count, and an exact radix select of the M largest runs on that
//      small set, ties going to the lower token id.
// When the collected count is outside [M, kCandCap] (flat or degenerate
// chunks) the chunk is radix-selected in full.  The chunk also reports the max
// of logit/T, the sum of exp(logit/T - max) over its non-selected tokens and
// its M-th largest logit.  The last CTA of a row (a per-row arrival counter;
// nothing waits) merges: the largest of the chunks' M-th values is a lower
// bound on the row's M-th value, so only chunk candidates at or above it can
// win; the exact top-M among those is sorted by (logit desc, id asc), and
//   rest_lse = log( sum_chunks part_sum e^{part_max} + sum_{dropped} e^{logit/T} ),
// so every non-candidate enters the log-partition exactly once.
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace dt {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kVPT = 32;            // values per thread: chunk <= kThreads * kVPT
constexpr int kMaxChunk = kThreads * kVPT;
constexpr int kMaxMerge = 8192;
constexpr int kBuckets = 16;
constexpr int kCandCap = 2048;      // candidates kept by the threshold filter

DT_DEVINL float block_max(float v, float* red) {
  v = warp_max(v);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x < 32) {
    float m = threadIdx.x < kWarps ? red[threadIdx.x] : -INFINITY;
    m = warp_max(m);
    if (threadIdx.x == 0) red[kWarps] = m;
  }
  __syncthreads();
  return red[kWarps];
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

// Index-ordered compaction of the keys >= the radix threshold (exactly `need`
// of the keys equal to t, the earliest ones).  Calls emit(e, key, pos) for each
// selected element in index order, and skip(e, key) for the others.
template <class Emit, class Skip>
DT_DEVINL void compact_topk(const uint32_t* keys, int n, uint32_t t, int need, int* scan, Emit emit, Skip skip) {
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
      emit(e, k, o);
      ++o;
    } else {
      skip(e, k);
    }
  }
}

// Exact top-k among c candidates in shared memory (value keys ck, token ids
// cid, any order, ids distinct): radix select on the value key; at the
// threshold the lower ids win.  Sets sel[e] = 1 for the k winners.
DT_DEVINL void small_topk(const uint32_t* ck, const uint32_t* cid, int c, int k, uint8_t* sel, uint32_t* hist,
                          int hist_words, uint32_t* state) {
  if (k >= c) {
    for (int e = threadIdx.x; e < c; e += blockDim.x) sel[e] = 1;
    __syncthreads();
    return;
  }
  uint32_t t;
  int need;
  radix_select_kth_largest(ck, c, k, hist, hist_words, state, t, need);
  for (int e = threadIdx.x; e < c; e += blockDim.x) {
    const uint32_t ke = ck[e];
    uint8_t s = ke > t ? 1 : 0;
    if (ke == t) {
      int rk = 0;
      for (int f = 0; f < c; ++f) rk += (ck[f] == t && cid[f] < cid[e]) ? 1 : 0;
      s = rk < need ? 1 : 0;
    }
    sel[e] = s;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kThreads) k_topm(const TopmParams p) {
  extern __shared__ uint32_t dyn[];
  __shared__ uint32_t hist[kWarps * 256];
  __shared__ uint32_t state[4];
  __shared__ int scan[40];
  __shared__ float red[kWarps + 1];
  __shared__ float red3[3][kWarps + 1];
  __shared__ unsigned cnt[kBuckets];
  __shared__ int s_last, s_ncand;

  const int row = blockIdx.y, split = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31;
  const int v0 = split * p.chunk;
  const int n = max(0, min(p.V, v0 + p.chunk) - v0);
  const float* x = p.logits + static_cast<size_t>(row) * p.V + v0;
  const float invT = 1.0f / p.T;
  const size_t q = static_cast<size_t>(row) * p.S + split;
  const int mloc = min(p.M, n);
  // candidates (keys, ids, flags) live after the chunk-key area
  uint32_t* ck = dyn + kMaxChunk;
  uint32_t* cid = ck + kCandCap;
  uint8_t* csel = reinterpret_cast<uint8_t*>(cid + kCandCap);

  // ---------------- 1. the chunk in registers; max, mean, sigma ----------------
  float vals[kVPT];
  float mx = -INFINITY, sm = 0.0f, sq = 0.0f;
#pragma unroll
  for (int j = 0; j < kVPT; ++j) {
    const int e = tid + j * kThreads;
    vals[j] = e < n ? x[e] : -INFINITY;
  }
#pragma unroll
  for (int j = 0; j < kVPT; ++j) {
    if (tid + j * kThreads < n) {
      mx = fmaxf(mx, vals[j]);
      sm += vals[j];
      sq += vals[j] * vals[j];
    }
  }
  {
    // max, sum and sum of squares in one block reduction
    mx = warp_max(mx);
    sm = warp_sum(sm);
    sq = warp_sum(sq);
    if (lane == 0) {
      red3[0][tid >> 5] = mx;
      red3[1][tid >> 5] = sm;
      red3[2][tid >> 5] = sq;
    }
    __syncthreads();
    if (tid < 32) {
      float a = tid < kWarps ? red3[0][tid] : -INFINITY;
      float b = tid < kWarps ? red3[1][tid] : 0.0f;
      float c = tid < kWarps ? red3[2][tid] : 0.0f;
      a = warp_max(a);
      b = warp_sum(b);
      c = warp_sum(c);
      if (tid == 0) {
        red3[0][kWarps] = a;
        red3[1][kWarps] = b;
        red3[2][kWarps] = c;
      }
    }
    if (tid < kBuckets) cnt[tid] = 0u;
    __syncthreads();
    mx = red3[0][kWarps];
    sm = red3[1][kWarps];
    sq = red3[2][kWarps];
  }
  const float mean = n > 0 ? sm / n : 0.0f;
  const float sigma = n > 0 ? sqrtf(fmaxf(sq / n - mean * mean, 0.0f)) : 0.0f;
  const float mxT = mx * invT;

  // ---------------- 2. histogram of the top 16 quarter-sigma buckets ----------------
  const float step = 0.25f * sigma;
  int chosen = -1;
  const bool try_fast = mloc > 0 && mloc < n && step > 0.0f && step < INFINITY;
  if (try_fast) {
    const float inv_step = 1.0f / step;
#pragma unroll
    for (int j = 0; j < kVPT; ++j) {
      const float dd = (mx - vals[j]) * inv_step;  // padding (-inf) gives +inf: skipped
      if (dd < static_cast<float>(kBuckets)) atomicAdd(&cnt[static_cast<int>(dd)], 1u);
    }
    __syncthreads();
    unsigned cum = 0;
    for (int k = 0; k < kBuckets; ++k) {
      cum += cnt[k];
      if (cum >= static_cast<unsigned>(mloc)) {
        if (cum <= static_cast<unsigned>(kCandCap)) chosen = k;
        break;
      }
    }
  }

  float rest = 0.0f;
  float kth = -INFINITY;  // the chunk's M-th largest logit (when n > M)
  // ---------------- 3. collect above the edge (exact count) ----------------
  int csize = 0;
  float th = INFINITY;
  int pos = 0;
  if (chosen >= 0) {
    th = mx - static_cast<float>(chosen + 1) * step;
    int mine = 0;
#pragma unroll
    for (int j = 0; j < kVPT; ++j) mine += (vals[j] >= th) ? 1 : 0;
    pos = block_exclusive_scan(mine, scan, &csize);
    // the buckets only steer the choice; the exact count decides
    if (csize < mloc || csize > kCandCap) chosen = -1;
  }
  if (chosen >= 0) {
#pragma unroll
    for (int j = 0; j < kVPT; ++j) {
      const int e = tid + j * kThreads;
      if (vals[j] >= th) {
        ck[pos] = f32_key(vals[j]);
        cid[pos] = static_cast<uint32_t>(v0 + e);
        ++pos;
      } else if (e < n) {
        rest += expf(vals[j] * invT - mxT);
      }
    }
    __syncthreads();
    small_topk(ck, cid, csize, mloc, csel, hist, 256, state);
    int mine_sel = 0;
    for (int e = tid; e < csize; e += kThreads) mine_sel += csel[e];
    int wrote;
    int o = block_exclusive_scan(mine_sel, scan, &wrote);
    uint32_t kmin = 0xFFFFFFFFu;
    for (int e = tid; e < csize; e += kThreads) {
      if (csel[e]) {
        p.part_id[q * p.M + o] = static_cast<int>(cid[e]);
        p.part_val[q * p.M + o] = key_f32(ck[e]);
        kmin = min(kmin, ck[e]);
        ++o;
      } else {
        rest += expf(key_f32(ck[e]) * invT - mxT);
      }
    }
    // the M-th largest = the smallest winner
    kth = -block_max(-key_f32(kmin == 0xFFFFFFFFu ? f32_key(INFINITY) : kmin), red);
  } else {
    // ---------------- fallback: full radix select over the chunk ----------------
    uint32_t* keys = dyn;
#pragma unroll
    for (int j = 0; j < kVPT; ++j) {
      const int e = tid + j * kThreads;
      if (e < n) keys[e] = f32_key(vals[j]);
    }
    __syncthreads();
    uint32_t t = 0;
    int need = n;
    if (mloc > 0 && mloc < n) {
      radix_select_kth_largest(keys, n, mloc, hist, static_cast<int>(sizeof(hist) / 4), state, t, need);
      kth = key_f32(t);
    }
    compact_topk(
        keys, n, t, need, scan,
        [&](int e, uint32_t k, int o) {
          p.part_id[q * p.M + o] = v0 + e;
          p.part_val[q * p.M + o] = key_f32(k);
        },
        [&](int, uint32_t k) { rest += expf(key_f32(k) * invT - mxT); });
  }
  rest = block_sum(rest, red);
  if (tid == 0) {
    p.part_max[q] = mxT;
    p.part_sum[q] = rest;
    p.part_cnt[q] = mloc;
    p.part_kth[q] = (mloc < n) ? kth : -INFINITY;
  }

  // ---------------- last CTA of the row merges ----------------
  __threadfence();
  __syncthreads();
  if (tid == 0) s_last = atomicAdd(&p.row_done[row], 1u) == static_cast<unsigned>(p.S - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const size_t rb = static_cast<size_t>(row) * p.S;
  float gmax = -INFINITY, lb = -INFINITY;
  for (int s = tid; s < p.S; s += kThreads) {
    gmax = fmaxf(gmax, p.part_max[rb + s]);
    lb = fmaxf(lb, p.part_kth[rb + s]);
  }
  gmax = block_max(gmax, red);
  lb = block_max(lb, red);
  // candidates at or above the lower bound (slot order, by a block scan); the
  // others feed the log-partition
  float rest2 = 0.0f;
  const int total = p.S * p.M;
  const int per = (total + kThreads - 1) / kThreads;  // contiguous slots per thread
  const int e0 = min(total, tid * per), e1 = min(total, e0 + per);
  int mine_c = 0;
  for (int e = e0; e < e1; ++e) {
    const int s = e / p.M, j = e - s * p.M;
    if (j < p.part_cnt[rb + s] && p.part_val[(rb + s) * p.M + j] >= lb) ++mine_c;
  }
  int ncand;
  int at = block_exclusive_scan(mine_c, scan, &ncand);
  for (int e = e0; e < e1; ++e) {
    const int s = e / p.M, j = e - s * p.M;
    if (j < p.part_cnt[rb + s]) {
      const float v = p.part_val[(rb + s) * p.M + j];
      if (v >= lb) {
        if (at < kCandCap) {
          ck[at] = f32_key(v);
          cid[at] = static_cast<uint32_t>(p.part_id[(rb + s) * p.M + j]);
        }
        ++at;
      } else {
        rest2 += expf(v * invT - gmax);
      }
    }
  }
  if (tid == 0) s_ncand = ncand;
  __syncthreads();
  const int nc = min(s_ncand, kCandCap);
  if (tid == 0 && s_ncand > kCandCap) dt_report(p.status, DT_DEV_BOUNDS);
  small_topk(ck, cid, nc, p.M, csel, hist, 256, state);
  // winners into hist (reused): ids then keys; the rest feeds the log-partition
  uint32_t* win_id = hist;
  uint32_t* win_key = hist + p.M;
  int mine_sel = 0;
  for (int e = tid; e < nc; e += kThreads) mine_sel += csel[e];
  int wrote;
  int o = block_exclusive_scan(mine_sel, scan, &wrote);
  for (int e = tid; e < nc; e += kThreads) {
    if (csel[e]) {
      if (o < p.M) {
        win_id[o] = cid[e];
        win_key[o] = ck[e];
      }
      ++o;
    } else {
      rest2 += expf(key_f32(ck[e]) * invT - gmax);
    }
  }
  for (int s = tid; s < p.S; s += kThreads) {
    const float ps = p.part_sum[rb + s];
    if (ps > 0.0f) rest2 += ps * expf(p.part_max[rb + s] - gmax);
  }
  rest2 = block_sum(rest2, red);
  // order the winners by (logit desc, id asc)
  const int nw = min(wrote, p.M);
  for (int a = tid; a < nw; a += kThreads) {
    const uint64_t ka = (static_cast<uint64_t>(win_key[a]) << 32) | (0xFFFFFFFFu - win_id[a]);
    int pos2 = 0;
    for (int b = 0; b < nw; ++b)
      pos2 += ((static_cast<uint64_t>(win_key[b]) << 32) | (0xFFFFFFFFu - win_id[b])) > ka;
    p.cand_tok[static_cast<size_t>(row) * p.M + pos2] = static_cast<int>(win_id[a]);
    p.cand_base[static_cast<size_t>(row) * p.M + pos2] = key_f32(win_key[a]);
  }
  if (tid == 0) {
    if (nw != p.M) dt_report(p.status, DT_DEV_BOUNDS);
    p.rest_lse[row] = rest2 > 0.0f ? gmax + logf(rest2) : -INFINITY;
    p.row_done[row] = 0u;  // ready for the next round
  }
}

}  // namespace

void topm_plan(TopmParams& p, int num_sms) {
  int S = (p.V + kMaxChunk - 1) / kMaxChunk;
  // 2 CTAs fit per SM (registers); rows * S <= 2 * SMs keeps the grid in one wave
  const int want = max(1, (2 * num_sms) / p.rows);
  const int cap_small = max(1, p.V / (2 * p.M));          // chunks of >= 2M logits
  int S2 = min(want, cap_small);
  if (S2 > S) S = S2;
  const int cap_merge = max(1, kMaxMerge / p.M);
  if (S > cap_merge) S = cap_merge;
  p.S = S;
  p.chunk = (p.V + S - 1) / S;
}

size_t topm_partial_smem(const TopmParams&) {
  return static_cast<size_t>(kMaxChunk) * 4 + static_cast<size_t>(kCandCap) * 9 + 16;
}

size_t topm_merge_smem(const TopmParams& p) { return topm_partial_smem(p); }

cudaError_t topm_prepare() { return dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_topm)); }

cudaError_t launch_topm(const TopmParams& p, cudaStream_t stream) {
  if (p.chunk > kMaxChunk || p.S * p.M > kMaxMerge || 2 * p.M > kWarps * 256) return cudaErrorInvalidValue;
  k_topm<<<dim3(p.S, p.rows), kThreads, topm_partial_smem(p), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dt

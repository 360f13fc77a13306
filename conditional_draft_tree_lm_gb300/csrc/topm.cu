// Top-M candidate restriction and the rest log-partition of each (request, depth)
// row of base logits ("Resumen Técnico: DominoTree", Componentes Principales,
// 2. Restricción de Candidatos (Top-M)).
//
// One kernel, grid (S chunks, rows).  Each CTA stages one chunk of one row
// (<= 16384 logits) in shared memory as order-preserving keys, finds the
// chunk's M-th largest key by an 8-bit radix select, and emits the chunk's
// top-M (ties to the lower token id, by index-ordered compaction) plus the max
// of logit/T and the sum of exp(logit/T - max) over the chunk's OTHER tokens.
// The last CTA of a row to finish (a per-row arrival counter; nothing waits)
// merges the row: radix select of the M largest among the S*M chunk candidates
// (slot order is token order, so ties again go to the lower id), a rank sort of
// the winners by (logit desc, id asc), and
//   rest_lse = log( sum_chunks part_sum e^{part_max} + sum_{dropped} e^{logit/T} ),
// so every non-candidate enters the log-partition exactly once.
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace dt {

namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxChunk = 16384;
constexpr int kMaxMerge = 8192;

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
// of the keys equal to t, the earliest ones).  Calls emit(e, key) for each
// selected element in index order with its output position, and skip(e, key)
// for the others.  Contiguous per-thread segments keep the order.
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

__global__ void __launch_bounds__(kThreads) k_topm(const TopmParams p) {
  extern __shared__ uint32_t dyn[];  // chunk keys, later merge keys + ids
  __shared__ uint32_t hist[kWarps * 256];
  __shared__ uint32_t state[4];
  __shared__ int scan[40];
  __shared__ float red[kWarps + 1];
  __shared__ int s_last;

  const int row = blockIdx.y, split = blockIdx.x;
  const int v0 = split * p.chunk;
  const int n = max(0, min(p.V, v0 + p.chunk) - v0);
  const float* x = p.logits + static_cast<size_t>(row) * p.V + v0;
  const float invT = 1.0f / p.T;
  uint32_t* keys = dyn;

  // ---------------- chunk top-M ----------------
  float mx = -INFINITY;
  for (int e = threadIdx.x; e < n; e += kThreads) {
    const float v = x[e];
    keys[e] = f32_key(v);
    mx = fmaxf(mx, v);
  }
  mx = block_max(mx, red);
  const int mloc = min(p.M, n);
  uint32_t t = 0;
  int need = n;
  if (mloc > 0 && mloc < n)
    radix_select_kth_largest(keys, n, mloc, hist, static_cast<int>(sizeof(hist) / 4), state, t, need);
  const size_t q = static_cast<size_t>(row) * p.S + split;
  const float mxT = mx * invT;
  float rest = 0.0f;
  compact_topk(
      keys, n, t, need, scan,
      [&](int e, uint32_t k, int o) {
        p.part_id[q * p.M + o] = v0 + e;
        p.part_val[q * p.M + o] = key_f32(k);
      },
      [&](int, uint32_t k) { rest += expf(key_f32(k) * invT - mxT); });
  rest = block_sum(rest, red);
  if (threadIdx.x == 0) {
    p.part_max[q] = mxT;
    p.part_sum[q] = rest;
    p.part_cnt[q] = mloc;
  }

  // ---------------- last CTA of the row merges ----------------
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) s_last = atomicAdd(&p.row_done[row], 1u) == static_cast<unsigned>(p.S - 1);
  __syncthreads();
  if (!s_last) return;
  __threadfence();

  const int total = p.S * p.M;
  uint32_t* mk = dyn;              // [total] value keys (0 = empty slot)
  uint32_t* mid = dyn + total;     // [total] token ids
  float gmax = -INFINITY;
  for (int s = threadIdx.x; s < p.S; s += kThreads) gmax = fmaxf(gmax, p.part_max[static_cast<size_t>(row) * p.S + s]);
  gmax = block_max(gmax, red);
  for (int e = threadIdx.x; e < total; e += kThreads) {
    const int s = e / p.M, j = e - s * p.M;
    const size_t qs = static_cast<size_t>(row) * p.S + s;
    uint32_t key = 0, id = 0;
    if (j < p.part_cnt[qs]) {
      key = f32_key(p.part_val[qs * p.M + j]);
      id = static_cast<uint32_t>(p.part_id[qs * p.M + j]);
    }
    mk[e] = key;
    mid[e] = id;
  }
  __syncthreads();
  uint32_t t2 = 0;
  int need2 = total;
  if (p.M < total)
    radix_select_kth_largest(mk, total, p.M, hist, static_cast<int>(sizeof(hist) / 4), state, t2, need2);
  // winners into hist (reused): ids then keys; the rest feeds the log-partition
  uint32_t* win_id = hist;
  uint32_t* win_key = hist + p.M;
  float rest2 = 0.0f;
  compact_topk(
      mk, total, t2, need2, scan,
      [&](int e, uint32_t k, int o) {
        if (o < p.M) {
          win_id[o] = mid[e];
          win_key[o] = k;
        }
      },
      [&](int, uint32_t k) {
        if (k != 0) rest2 += expf(key_f32(k) * invT - gmax);
      });
  for (int s = threadIdx.x; s < p.S; s += kThreads) {
    const size_t qs = static_cast<size_t>(row) * p.S + s;
    const float ps = p.part_sum[qs];
    if (ps > 0.0f) rest2 += ps * expf(p.part_max[qs] - gmax);
  }
  rest2 = block_sum(rest2, red);
  // order the winners by (logit desc, id asc)
  for (int a = threadIdx.x; a < p.M; a += kThreads) {
    const uint64_t ka = (static_cast<uint64_t>(win_key[a]) << 32) | (0xFFFFFFFFu - win_id[a]);
    int pos = 0;
    for (int b = 0; b < p.M; ++b)
      pos += ((static_cast<uint64_t>(win_key[b]) << 32) | (0xFFFFFFFFu - win_id[b])) > ka;
    p.cand_tok[static_cast<size_t>(row) * p.M + pos] = static_cast<int>(win_id[a]);
    p.cand_base[static_cast<size_t>(row) * p.M + pos] = key_f32(win_key[a]);
  }
  if (threadIdx.x == 0) {
    p.rest_lse[row] = rest2 > 0.0f ? gmax + logf(rest2) : -INFINITY;
    p.row_done[row] = 0u;  // ready for the next round
  }
}

}  // namespace

void topm_plan(TopmParams& p, int num_sms) {
  int S = (p.V + kMaxChunk - 1) / kMaxChunk;
  const int want = (2 * num_sms + p.rows - 1) / p.rows;  // ~2 CTAs per SM
  const int cap_small = max(1, p.V / (2 * p.M));          // chunks of >= 2M logits
  int S2 = min(want, cap_small);
  if (S2 > S) S = S2;
  const int cap_merge = max(1, kMaxMerge / p.M);
  if (S > cap_merge) S = cap_merge;
  p.S = S;
  p.chunk = (p.V + S - 1) / S;
}

size_t topm_partial_smem(const TopmParams& p) {
  const size_t a = static_cast<size_t>(p.chunk) * 4;
  const size_t b = static_cast<size_t>(p.S) * p.M * 8;
  return a > b ? a : b;
}

size_t topm_merge_smem(const TopmParams& p) { return static_cast<size_t>(p.S) * p.M * 8; }

cudaError_t topm_prepare() { return dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_topm)); }

cudaError_t launch_topm(const TopmParams& p, cudaStream_t stream) {
  if (p.chunk > kMaxChunk || p.S * p.M > kMaxMerge || 2 * p.M > kWarps * 256) return cudaErrorInvalidValue;
  k_topm<<<dim3(p.S, p.rows), kThreads, topm_partial_smem(p), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dt

// Top-M candidate restriction and the rest log-partition of each (request, depth)
// row of base logits ("Resumen Técnico: DominoTree", Componentes Principales,
// 2. Restricción de Candidatos (Top-M)).
//
// Pass 1 (k_topm_partial): each CTA owns one chunk of one row (<= 16384 logits,
// staged in shared memory as order-preserving keys), finds the chunk's M-th
// largest key by an 8-bit radix select, and emits the chunk's top-M (ties to
// the lower token id, by stable index-order compaction) plus the max of
// logit/T and the sum of exp(logit/T - max) over the chunk's OTHER tokens.
// Pass 2 (k_topm_merge): one CTA per row sorts the S*M chunk candidates
// (bitonic on 64-bit keys value-desc / id-asc), keeps the first M, and forms
// rest_lse = log( sum_chunks part_sum*e^{part_max} + sum_{dropped candidates}
// e^{logit/T} ) — every non-candidate enters exactly once, no cancellation.
#include "common.cuh"
#include "kernels.h"
#include "select.cuh"

namespace dt {

namespace {

constexpr int kPartialThreads = 512;
constexpr int kMergeThreads = 512;
constexpr int kMaxChunk = 16384;
constexpr int kMaxMerge = 8192;

__global__ void __launch_bounds__(kPartialThreads) k_topm_partial(const TopmParams p) {
  extern __shared__ uint32_t sm_keys[];  // [chunk]
  __shared__ uint32_t hist[256];
  __shared__ uint32_t state[4];
  __shared__ int scan_scratch[40];
  __shared__ float red[kPartialThreads / 32];

  const int row = blockIdx.y, split = blockIdx.x;
  const int v0 = split * p.chunk;
  const int v1 = min(p.V, v0 + p.chunk);
  const int n = max(0, v1 - v0);
  const float* x = p.logits + static_cast<size_t>(row) * p.V + v0;
  const float invT = 1.0f / p.T;

  float mx = -INFINITY;
  for (int e = threadIdx.x; e < n; e += blockDim.x) {
    const float v = x[e];
    sm_keys[e] = f32_key(v);
    mx = fmaxf(mx, v);
  }
  mx = warp_max(mx);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = mx;
  __syncthreads();
  if (threadIdx.x < 32) {
    float m = threadIdx.x < (kPartialThreads / 32) ? red[threadIdx.x] : -INFINITY;
    m = warp_max(m);
    if (threadIdx.x == 0) red[0] = m;
  }
  __syncthreads();
  mx = red[0];
  __syncthreads();

  const int mloc = min(p.M, n);
  uint32_t t = 0;
  int need = 0;
  if (mloc > 0 && mloc < n) {
    radix_select_kth_largest(sm_keys, n, mloc, hist, state, t, need);
  } else {
    t = 0;        // every key is >= 0: take all
    need = n;     // ties at t = 0 cannot occur for finite logits; all keys > t
  }
  // stable compaction in index order over contiguous per-thread segments
  const int seg = (n + blockDim.x - 1) / blockDim.x;
  const int s0 = min(n, static_cast<int>(threadIdx.x) * seg);
  const int s1 = min(n, s0 + seg);
  int ties = 0;
  for (int e = s0; e < s1; ++e) ties += (sm_keys[e] == t);
  int tot;
  int tie_base = block_exclusive_scan(ties, scan_scratch, &tot);
  int cnt = 0;
  {
    int tb = tie_base;
    for (int e = s0; e < s1; ++e) {
      const uint32_t k = sm_keys[e];
      if (k > t || (k == t && tb++ < need)) ++cnt;
    }
  }
  int out_base = block_exclusive_scan(cnt, scan_scratch, &tot);
  float rest = 0.0f;
  const float mxT = mx * invT;
  {
    int tb = tie_base, o = out_base;
    const size_t pbase = (static_cast<size_t>(row) * p.S + split) * p.M;
    for (int e = s0; e < s1; ++e) {
      const uint32_t k = sm_keys[e];
      const bool take = k > t || (k == t && tb++ < need);
      if (take) {
        p.part_id[pbase + o] = v0 + e;
        p.part_val[pbase + o] = key_f32(k);
        ++o;
      } else {
        rest += expf(key_f32(k) * invT - mxT);
      }
    }
  }
  rest = warp_sum(rest);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = rest;
  __syncthreads();
  if (threadIdx.x < 32) {
    float s = threadIdx.x < (kPartialThreads / 32) ? red[threadIdx.x] : 0.0f;
    s = warp_sum(s);
    if (threadIdx.x == 0) {
      const size_t q = static_cast<size_t>(row) * p.S + split;
      p.part_max[q] = mxT;
      p.part_sum[q] = s;
      p.part_cnt[q] = tot;
    }
  }
}

__global__ void __launch_bounds__(kMergeThreads) k_topm_merge(const TopmParams p) {
  extern __shared__ uint64_t sm_k64[];  // [npad]
  __shared__ float red[kMergeThreads / 32];
  __shared__ float s_gmax;
  const int row = blockIdx.x;
  const int total = p.S * p.M;
  int npad = 1;
  while (npad < total) npad <<= 1;

  for (int e = threadIdx.x; e < npad; e += blockDim.x) {
    uint64_t key = 0;
    if (e < total) {
      const int s = e / p.M, j = e - s * p.M;
      const size_t q = static_cast<size_t>(row) * p.S + s;
      if (j < p.part_cnt[q]) {
        const int id = p.part_id[q * p.M + j];
        key = rank_key(p.part_val[q * p.M + j], static_cast<uint32_t>(id));
      }
    }
    sm_k64[e] = key;
  }
  // global max of logit/T over all chunks
  float gm = -INFINITY;
  for (int s = threadIdx.x; s < p.S; s += blockDim.x) gm = fmaxf(gm, p.part_max[static_cast<size_t>(row) * p.S + s]);
  gm = warp_max(gm);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = gm;
  __syncthreads();
  if (threadIdx.x < 32) {
    float m = threadIdx.x < (kMergeThreads / 32) ? red[threadIdx.x] : -INFINITY;
    m = warp_max(m);
    if (threadIdx.x == 0) s_gmax = m;
  }
  // bitonic sort, descending
  for (int k = 2; k <= npad; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      __syncthreads();
      for (int i = threadIdx.x; i < npad; i += blockDim.x) {
        const int l = i ^ j;
        if (l > i) {
          const uint64_t a = sm_k64[i], b = sm_k64[l];
          const bool desc = (i & k) == 0;
          if (desc ? (a < b) : (a > b)) {
            sm_k64[i] = b;
            sm_k64[l] = a;
          }
        }
      }
    }
  }
  __syncthreads();
  const float invT = 1.0f / p.T;
  const float gmax = s_gmax;
  for (int j = threadIdx.x; j < p.M; j += blockDim.x) {
    const uint64_t key = sm_k64[j];
    p.cand_tok[static_cast<size_t>(row) * p.M + j] = static_cast<int>(rank_key_id(key));
    p.cand_base[static_cast<size_t>(row) * p.M + j] = key_f32(static_cast<uint32_t>(key >> 32));
  }
  float rest = 0.0f;
  for (int s = threadIdx.x; s < p.S; s += blockDim.x) {
    const size_t q = static_cast<size_t>(row) * p.S + s;
    const float ps = p.part_sum[q];
    if (ps > 0.0f) rest += ps * expf(p.part_max[q] - gmax);
  }
  for (int j = p.M + threadIdx.x; j < total; j += blockDim.x) {
    const uint64_t key = sm_k64[j];
    if (key != 0) rest += expf(key_f32(static_cast<uint32_t>(key >> 32)) * invT - gmax);
  }
  rest = warp_sum(rest);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = rest;
  __syncthreads();
  if (threadIdx.x < 32) {
    float s = threadIdx.x < (kMergeThreads / 32) ? red[threadIdx.x] : 0.0f;
    s = warp_sum(s);
    if (threadIdx.x == 0) p.rest_lse[row] = s > 0.0f ? gmax + logf(s) : -INFINITY;
  }
}

}  // namespace

void topm_plan(TopmParams& p, int num_sms) {
  int S = (p.V + kMaxChunk - 1) / kMaxChunk;
  const int want = (2 * num_sms + p.rows - 1) / p.rows;      // ~2 CTAs per SM
  const int cap_small = max(1, p.V / (2 * p.M));              // chunks of >= 2M logits
  int S2 = min(want, cap_small);
  if (S2 > S) S = S2;
  const int cap_merge = max(1, kMaxMerge / p.M);
  if (S > cap_merge) S = cap_merge;
  p.S = S;
  p.chunk = (p.V + S - 1) / S;
}

size_t topm_partial_smem(const TopmParams& p) { return static_cast<size_t>(p.chunk) * 4; }

size_t topm_merge_smem(const TopmParams& p) {
  int npad = 1;
  while (npad < p.S * p.M) npad <<= 1;
  return static_cast<size_t>(npad) * 8;
}

cudaError_t topm_prepare() {
  cudaError_t e = cudaFuncSetAttribute(k_topm_partial, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kMaxChunk * 4);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_topm_merge, cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxMerge * 8);
}

cudaError_t launch_topm(const TopmParams& p, cudaStream_t stream) {
  if (p.chunk > kMaxChunk || p.S * p.M > kMaxMerge) return cudaErrorInvalidValue;
  k_topm_partial<<<dim3(p.S, p.rows), kPartialThreads, topm_partial_smem(p), stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  k_topm_merge<<<p.rows, kMergeThreads, topm_merge_smem(p), stream>>>(p);
  return cudaGetLastError();
}

}  // namespace dt

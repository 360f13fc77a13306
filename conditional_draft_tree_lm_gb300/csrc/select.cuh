// Block-wide selection primitives: radix select of the k-th largest 32-bit key
// and scans used for stable (index-ordered) compaction.
#pragma once

#include "common.cuh"

namespace dt {

// Exclusive scan of one int per thread over the block (blockDim.x multiple of 32,
// <= 1024).  `scratch` holds >= 33 ints.  Returns the exclusive prefix; *total
// receives the block total.
DT_DEVINL int block_exclusive_scan(int v, int* scratch, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nwarps = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) scratch[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = lane < nwarps ? scratch[lane] : 0;
    int s = w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xFFFFFFFFu, s, o);
      if (lane >= o) s += y;
    }
    if (lane < nwarps) scratch[lane] = s - w;
    if (lane == 31) scratch[32] = s;
  }
  __syncthreads();
  const int res = scratch[warp] + x - v;
  *total = scratch[32];
  __syncthreads();
  return res;
}

// Radix select over keys[0, n) in shared memory: the k-th largest key
// (1 <= k <= n), four passes of 8 bits.  `hist` holds `hist_words` uint32
// (a multiple of 256): up to hist_words/256 warps count into histograms of
// their own, further warps share them, so no access leaves the buffer.
// On return every thread holds `t` (that key) and `need` (how many keys equal
// to t belong to the top k: exactly k - #{key > t}).  `state` holds 4 uint32.
DT_DEVINL void radix_select_kth_largest(const uint32_t* keys, int n, int k, uint32_t* hist, int hist_words,
                                        uint32_t* state, uint32_t& t, int& need) {
  const int nh = max(1, hist_words / 256);
  const int nwarps = min(static_cast<int>(blockDim.x >> 5), nh);
  uint32_t* my = hist + ((threadIdx.x >> 5) % nwarps) * 256;
  uint32_t prefix = 0, pmask = 0;
  uint32_t kk = static_cast<uint32_t>(k);
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < nwarps * 256; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    for (int e = threadIdx.x; e < n; e += blockDim.x) {
      const uint32_t key = keys[e];
      if ((key & pmask) == prefix) atomicAdd(&my[(key >> shift) & 255u], 1u);
    }
    __syncthreads();
    // fold the per-warp histograms into warp 0's
    for (int b = threadIdx.x; b < 256; b += blockDim.x) {
      uint32_t s = 0;
      for (int w = 0; w < nwarps; ++w) s += hist[w * 256 + b];
      hist[b] = s;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      const int lane = threadIdx.x;
      // lane handles digits 255-8*lane down to 248-8*lane
      uint32_t c[8];
      uint32_t s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        c[j] = hist[255 - 8 * lane - j];
        s += c[j];
      }
      uint32_t incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        uint32_t y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
      }
      const uint32_t excl = incl - s;
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl >= kk);
      const int first = hit ? __ffs(hit) - 1 : 0;
      if (lane == first) {
        uint32_t cum = excl;
        int dsel = 0;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (cum + c[j] >= kk) {
            dsel = 255 - 8 * lane - j;
            break;
          }
          cum += c[j];
        }
        state[0] = static_cast<uint32_t>(dsel);
        state[1] = kk - cum;
      }
    }
    __syncthreads();
    prefix |= state[0] << shift;
    pmask |= 255u << shift;
    kk = state[1];
    __syncthreads();
  }
  t = prefix;
  need = static_cast<int>(kk);
}

// Exact ranks of keys[0, c) among themselves (the number of larger keys; keys
// are distinct).  Each key is ranked by a group of g consecutive threads (g a
// power of two <= 32, as many as the block allows), whose partial counts are
// added with shuffles; fn(e, key, rank) then runs on the group's first thread.
// Every thread of the block must call (blockDim.x a multiple of 32).
template <class Fn>
DT_DEVINL void block_rank_all(const uint64_t* keys, int c, Fn fn) {
  const int nt = static_cast<int>(blockDim.x);
  int g = 1;
  while (g < 32 && 2 * g * c <= nt) g <<= 1;
  for (int base = 0; base < c * g; base += nt) {
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

// The m-th largest of the n keys rank_key(v[e], id_e) with id_e = ids[e], or
// e when ids is null (values and ids in shared memory; 1 <= m <= n; the keys
// are distinct, a tie in value going to the lower id).  A 256-bin histogram over the value range [lo, hi] (bin 0
// holds the largest values) locates the bin that holds it; that bin's keys
// are gathered (at most bnd_cap; beyond that every key of the bin is ranked
// against the whole bin instead) and ranked exactly.  `hist` holds 256
// words, `red` 2 x (warps) floats, `sc` 3 ints, `s_key` one key.  Every thread
// of the block calls it and receives the key.
DT_DEVINL uint64_t block_kth_rank_key(const float* v, int n, int m, uint32_t* hist, uint64_t* bnd, int bnd_cap,
                                      float* red, int* sc, uint64_t* s_key, const int* ids = nullptr) {
  auto key_of = [&](int e) { return rank_key(v[e], static_cast<uint32_t>(ids ? ids[e] : e)); };
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nt = blockDim.x, nw = nt >> 5;
  float lo = INFINITY, hi = -INFINITY;
  for (int e = tid; e < n; e += nt) {
    lo = fminf(lo, v[e]);
    hi = fmaxf(hi, v[e]);
  }
  lo = -warp_max(-lo);
  hi = warp_max(hi);
  if (lane == 0) {
    red[warp] = lo;
    red[nw + warp] = hi;
  }
  for (int b = tid; b < 256; b += nt) hist[b] = 0u;
  if (tid == 0) {
    sc[0] = 0;
    sc[1] = 0;
    sc[2] = 0;
  }
  __syncthreads();
  lo = INFINITY;
  hi = -INFINITY;
  for (int w = 0; w < nw; ++w) {
    lo = fminf(lo, red[w]);
    hi = fmaxf(hi, red[nw + w]);
  }
  const float scale = hi > lo ? 256.0f / (hi - lo) : 0.0f;
  auto bin_of = [&](float x) { return min(255, max(0, __float2int_rz((hi - x) * scale))); };
  for (int e = tid; e < n; e += nt) atomicAdd(&hist[bin_of(v[e])], 1u);
  __syncthreads();
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
  const int bt = sc[0];
  const int need = m - sc[1];  // the need-th largest key of bin bt
  for (int e = tid; e < n; e += nt) {
    if (bin_of(v[e]) == bt) {
      const int at = atomicAdd(&sc[2], 1);
      if (at < bnd_cap) bnd[at] = key_of(e);
    }
  }
  __syncthreads();
  const int nb = sc[2];
  if (nb <= bnd_cap) {
    block_rank_all(bnd, nb, [&](int, uint64_t ke, int rk) {
      if (rk == need - 1) *s_key = ke;
    });
  } else {
    for (int e = tid; e < n; e += nt) {
      if (bin_of(v[e]) != bt) continue;
      const uint64_t k = key_of(e);
      int rk = 0;
      for (int f = 0; f < n; ++f) rk += (bin_of(v[f]) == bt && key_of(f) > k) ? 1 : 0;
      if (rk == need - 1) *s_key = k;
    }
  }
  __syncthreads();
  return *s_key;
}

}  // namespace dt

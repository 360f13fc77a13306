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
// (1 <= k <= n).  On return every thread holds `t` (that key) and `need` (how
// many keys equal to t belong to the top k: exactly k - #{key > t}).
// `hist` holds 256 uint32, `state` holds 4 uint32 (shared memory).
DT_DEVINL void radix_select_kth_largest(const uint32_t* keys, int n, int k, uint32_t* hist,
                                        uint32_t* state, uint32_t& t, int& need) {
  uint32_t prefix = 0, pmask = 0;
  uint32_t kk = static_cast<uint32_t>(k);
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int b = threadIdx.x; b < 256; b += blockDim.x) hist[b] = 0;
    __syncthreads();
    // warp-uniform trip count so every lane takes part in __match_any_sync
    for (int base = 0; base < n; base += blockDim.x) {
      const int e = base + threadIdx.x;
      bool in = false;
      uint32_t digit = 0;
      if (e < n) {
        const uint32_t key = keys[e];
        in = (key & pmask) == prefix;
        digit = (key >> shift) & 255u;
      }
      const unsigned grp = __match_any_sync(0xFFFFFFFFu, in ? digit : 0x100u + (threadIdx.x & 31));
      if (in) {
        const int leader = __ffs(grp) - 1;
        if ((threadIdx.x & 31) == leader) atomicAdd(&hist[digit], static_cast<uint32_t>(__popc(grp)));
      }
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
          if (cum + c[j] >= kk) { dsel = 255 - 8 * lane - j; break; }
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

}  // namespace dt

// Top-M inside the LM-head GEMM's epilogue ("Resumen Técnico: DominoTree",
// Componentes Principales, 2. Restricción de Candidatos (Top-M)), for one
// request: every CTA of the persistent GEMM keeps, for each of the P <= 16
// logit rows (block positions 1 .. D), the exact M best (logit desc, token id
// asc) of the vocabulary rows it has produced, and at its end reports them in
// the partial-list format of the Top-M kernel (sorted list, the max of
// logit/T, the sum of exp(logit/T - max) over the rest), which a small merge
// kernel then reduces over the CTAs.
//
// Per tile (128 vocabulary rows), with the sixteen epilogue warps only (named
// barrier 1, 512 threads): warp e (0..15) reads TMEM lane quarter e % 4 (its
// vocabulary rows) and columns 4 h .. 4 h + 3, h = e / 4 (a quarter of the
// logit rows: column c holds row c - 1):
//   1. each thread's logit of each of its rows becomes a key; the keys above
//      the row's held M-th key are appended to the row's new-key list, warp
//      by warp (lane quarter order) in lane order (no atomics: the order is
//      the same every run);
//   2. warp e updates row e: while nothing is held, a bitonic
//      sort of the (at most 128) new keys; otherwise the held list (sorted)
//      and the new keys are ranked against each other (a held key moves down
//      by the new keys above it, a new key counts the held keys above it by
//      bisection and the new keys above it).  The M best go, sorted, into the
//      other copy of the held list; the keys pushed out add exp(logit/T -
//      max) to the row's evicted sum (the warp's lanes in order, so the same
//      bits every run), rescaled when the row's max grows;
//   3. each thread adds exp(logit/T - max) of its own logits that did not
//      enter to its running sums (one per row, rescaled likewise).
// The updates overlap the streaming of the next tiles (the GEMM is bound by
// HBM, about 14 us per tile at the Qwen3-4B shape); after the last tile only
// that tile's update, one reduction of the sums and the lists' writes remain.
#pragma once

#include "common.cuh"

#ifndef FT_STAMP
#define FT_STAMP(t, k) \
  do {                 \
  } while (0)
#endif

namespace dt {

constexpr int kFtMaxRows = 16;   // logit rows P (one request, block <= 17)
constexpr int kFtMaxM = 64;
constexpr int kFtWarps = 16;     // epilogue warps: four per TMEM lane quarter
constexpr int kFtCols = 4;       // accumulator columns (block positions) per epilogue thread

// Shared-memory area of the fused Top-M (byte offsets from a 16-byte aligned base).
struct FtLayout {
  size_t held, ent, misc, total;
};
DT_HOST_DEVICE_INLINE FtLayout ft_layout(int P) {
  FtLayout L;
  size_t o = 0;
  L.held = o;
  o += static_cast<size_t>(2) * P * kFtMaxM * 8;  // [2][row][M] sorted keys
  L.ent = o;
  o += static_cast<size_t>(P) * 128 * 8;          // [row][128] new keys of a tile
  L.misc = o;
  // thr (u64); hn, par, wcnt[4 quarters] (ints); ev_sum, ev_ref, red[4 quarters] (floats)
  o += 8 * kFtMaxRows + 4 * 6 * kFtMaxRows + 4 * 6 * kFtMaxRows;
  L.total = (o + 15) & ~static_cast<size_t>(15);
  return L;
}

struct FtState {
  uint64_t* held;   // [2][P][M]
  uint64_t* ent;    // [P][128]
  uint64_t* thr;    // [P] the held list's M-th key (0 while it holds fewer)
  int* hn;          // [P] keys held
  int* par;         // [P] which copy of the held list is current
  int* wcnt;        // [4][16] new keys of the tile per lane quarter and row
  float* ev_sum;    // [P] sum of exp(logit/T - ev_ref) over the evicted keys
  float* ev_ref;    // [P] the row's max of logit/T
  float* red;       // [4][16]
};

DT_DEVINL FtState ft_state(uint8_t* base, int P) {
  const FtLayout L = ft_layout(P);
  FtState s;
  s.held = reinterpret_cast<uint64_t*>(base + L.held);
  s.ent = reinterpret_cast<uint64_t*>(base + L.ent);
  s.thr = reinterpret_cast<uint64_t*>(base + L.misc);
  s.hn = reinterpret_cast<int*>(base + L.misc + 8 * kFtMaxRows);
  s.par = s.hn + kFtMaxRows;
  s.wcnt = s.par + kFtMaxRows;
  s.ev_sum = reinterpret_cast<float*>(base + L.misc + 8 * kFtMaxRows + 4 * 6 * kFtMaxRows);
  s.ev_ref = s.ev_sum + kFtMaxRows;
  s.red = s.ev_ref + kFtMaxRows;
  return s;
}

DT_DEVINL void ft_bar() { asm volatile("bar.sync 1, 512;" ::: "memory"); }
// The epilogue warps' common verdict (all true), so that they leave the tile
// loop together and no named barrier waits for a warp that has left.
DT_DEVINL bool ft_all(bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, 1, 512, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(static_cast<uint32_t>(v))
      : "memory");
  return r != 0;
}

// The running sums of one epilogue thread (registers): per row of its columns,
// the sum of exp(logit/T - ref) over its logits that never entered, and ref.
struct FtSums {
  float rest[kFtCols];
  float ref[kFtCols];
};

// et: epilogue thread 0..511.
DT_DEVINL void ft_init(FtState& s, FtSums& u, int P, int et) {
  if (et < P) {
    s.thr[et] = 0ull;
    s.hn[et] = 0;
    s.par[et] = 0;
    s.ev_sum[et] = 0.0f;
    s.ev_ref[et] = -INFINITY;
  }
#pragma unroll
  for (int j = 0; j < kFtCols; ++j) {
    u.rest[j] = 0.0f;
    u.ref[j] = -INFINITY;
  }
  ft_bar();
}

// sum * e^(from - to) once the reference has grown from `from` to `to`.
DT_DEVINL float ft_rescale(float sum, float from, float to) { return to > from ? sum * __expf(from - to) : sum; }

// Bitonic sort (descending) of 128 keys held four per lane (element 4 lane + i).
DT_DEVINL void ft_sort128(uint64_t (&a)[4], int lane) {
#pragma unroll
  for (int size = 2; size <= 128; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      uint64_t b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = 4 * lane + i, f = e ^ stride;
        // the pair (min(e,f), max(e,f)) goes in descending order where bit
        // `size` of the index is clear, ascending where it is set
        const uint64_t other = stride >= 4 ? __shfl_xor_sync(0xFFFFFFFFu, a[i], stride >> 2) : a[i ^ stride];
        const bool keep_max = (e < f) == ((e & size) == 0);
        const uint64_t mx = a[i] > other ? a[i] : other, mn = a[i] > other ? other : a[i];
        b[i] = keep_max ? mx : mn;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = b[i];
    }
  }
}

// One logits tile: v[j] is the logit of row 4 h + j - 1 (column 4 h + j;
// rows 0 .. P-1) at vocabulary id `id` (valid: id < V); q: the thread's lane
// quarter, e: its epilogue warp 0..15.
DT_DEVINL void ft_tile(FtState& s, FtSums& u, const uint32_t (&v)[kFtCols], int P, int M, float invT, int id,
                       bool valid, int q, int h, int e, int lt) {
  const int lane = threadIdx.x & 31;
  const unsigned below = (1u << lane) - 1u;
  uint64_t key[kFtCols];
  unsigned bal[kFtCols];
#pragma unroll
  for (int j = 0; j < kFtCols; ++j) {
    const int p = kFtCols * h + j - 1;
    const bool row = p >= 0 && p < P;
    key[j] = valid && row ? rank_key(__uint_as_float(v[j]), static_cast<uint32_t>(id)) : 0ull;
    bal[j] = __ballot_sync(0xFFFFFFFFu, row && key[j] > s.thr[row ? p : 0]);
    if (lane == 0 && row) s.wcnt[q * kFtMaxRows + p] = __popc(bal[j]);
  }
  ft_bar();
#pragma unroll
  for (int j = 0; j < kFtCols; ++j) {
    if ((bal[j] >> lane) & 1u) {
      const int p = kFtCols * h + j - 1;
      int base = 0;
      for (int q2 = 0; q2 < q; ++q2) base += s.wcnt[q2 * kFtMaxRows + p];
      s.ent[p * 128 + base + __popc(bal[j] & below)] = key[j];
    }
  }
  ft_bar();
  FT_STAMP(lt, 4);
  const int w = e;
  // the rows' updates, warp e taking row e
  for (int p = w; p < P; p += kFtWarps) {
    const int en = s.wcnt[p] + s.wcnt[kFtMaxRows + p] + s.wcnt[2 * kFtMaxRows + p] + s.wcnt[3 * kFtMaxRows + p];
    if (en == 0) continue;
    const int hn = s.hn[p];
    const uint64_t* h = s.held + (s.par[p] * P + p) * kFtMaxM;
    const uint64_t* e = s.ent + p * 128;
    uint64_t* out = s.held + ((s.par[p] ^ 1) * P + p) * kFtMaxM;
    float evv[6];  // logits of this lane's keys pushed out of the list (or -inf)
    if (hn == 0) {
      // nothing held yet: sort the new keys (zero keys pad to 128)
      uint64_t a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = 4 * lane + i < en ? e[4 * lane + i] : 0ull;
      ft_sort128(a, lane);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int r = 4 * lane + i;
        if (a[i] != 0ull && r < M) out[r] = a[i];
        evv[i] = (a[i] != 0ull && r >= M) ? key_f32(static_cast<uint32_t>(a[i] >> 32)) : -INFINITY;
      }
      evv[4] = evv[5] = -INFINITY;
    } else {
      // lane l takes keys l, l + 32, ... (held first, then new); a key past
      // the end gets the rank `none`
      constexpr int kQ = (kFtMaxM + 128 + 31) / 32;
      constexpr int none = 1 << 20;
      uint64_t kq[kQ];
      int rq[kQ];
      const int n = hn + en;
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        const int k = lane + 32 * q;
        kq[q] = 0ull;
        rq[q] = none;
        if (32 * q >= n) continue;  // (uniform over the warp)
        if (32 * q + 31 < hn) {     // held keys only: no bisection
          kq[q] = h[k];
          rq[q] = k;
          continue;
        }
        const bool held = k < hn;
        kq[q] = held ? h[min(k, kFtMaxM - 1)] : (k < n ? e[k - hn] : 0ull);
        int lo = 0, hi = hn;
#pragma unroll
        for (int step = 0; step < 7; ++step) {  // hn <= 64
          const int mid = (lo + hi) >> 1;
          const bool go = lo < hi;
          const bool above = h[min(mid, kFtMaxM - 1)] > kq[q];
          lo = (go && above) ? mid + 1 : lo;
          hi = (go && !above) ? mid : hi;
        }
        rq[q] = held ? k : (k < n ? lo : none);
      }
      for (int j = 0; j < en; ++j) {
        const uint64_t ej = e[j];
#pragma unroll
        for (int q = 0; q < kQ; ++q) rq[q] += ej > kq[q] ? 1 : 0;
      }
#pragma unroll
      for (int q = 0; q < kQ; ++q) {
        if (rq[q] < M) out[rq[q]] = kq[q];
        evv[q] = (rq[q] >= M && rq[q] < none) ? key_f32(static_cast<uint32_t>(kq[q] >> 32)) : -INFINITY;
      }
    }
    __syncwarp();
    // the evicted keys' terms against the row's new max, lane by lane
    const float mx = key_f32(static_cast<uint32_t>(out[0] >> 32)) * invT;
    float ev = 0.0f;
#pragma unroll
    for (int i = 0; i < 6; ++i) ev += evv[i] > -INFINITY ? __expf(evv[i] * invT - mx) : 0.0f;
    ev = warp_sum(ev);
    if (lane == 0) {
      s.ev_sum[p] = ft_rescale(s.ev_sum[p], s.ev_ref[p], mx) + ev;
      s.ev_ref[p] = fmaxf(s.ev_ref[p], mx);
      const int hn2 = min(M, hn + en);
      const int np = s.par[p] ^ 1;
      s.hn[p] = hn2;
      s.par[p] = np;
      s.thr[p] = hn2 == M ? out[M - 1] : 0ull;
    }
  }
  ft_bar();
  FT_STAMP(lt, 5);
  // this thread's logits that did not enter, against the rows' new max
#pragma unroll
  for (int j = 0; j < kFtCols; ++j) {
    const int p = kFtCols * h + j - 1;
    if (p >= 0 && p < P) {
      const float mx = s.ev_ref[p];
      u.rest[j] = ft_rescale(u.rest[j], u.ref[j], mx);
      u.ref[j] = fmaxf(u.ref[j], mx);
      const bool skip = valid && !((bal[j] >> lane) & 1u);
      u.rest[j] += skip ? __expf(__uint_as_float(v[j]) * invT - u.ref[j]) : 0.0f;
    }
  }
}

// After the CTA's last tile: the partial lists of CTA `cta` (of S) for the P
// rows.  et: epilogue thread 0..511 (warp e = et / 32); q, h as in ft_tile.
DT_DEVINL void ft_finish(FtState& s, FtSums& u, int P, int M, float invT, int cta, int S, int et, int q, int h,
                         int* part_id, float* part_val, float* part_max, float* part_sum, int* part_cnt,
                         float* part_kth, float* part_tail) {
  const int lane = et & 31, w = et >> 5;
#pragma unroll
  for (int j = 0; j < kFtCols; ++j) {
    const int p = kFtCols * h + j - 1;
    if (p >= 0 && p < P) {
      const float r = warp_sum(u.rest[j]);
      if (lane == 0) s.red[q * kFtMaxRows + p] = r;
    }
  }
  ft_bar();
  FT_STAMP(16, 3);
  // the lists' suffix sums of exp(logit/T - max), warp e taking row e:
  // lane l sums entries 2l, 2l+1, then a suffix scan over the lanes
  if (part_tail) {
    for (int p = w; p < P; p += kFtWarps) {
      const int hn = s.hn[p];
      const uint64_t* h = s.held + (s.par[p] * P + p) * kFtMaxM;
      const float mx = s.ev_ref[p];
      const size_t q = static_cast<size_t>(p) * S + cta;
      float t0 = 2 * lane < hn ? __expf(key_f32(static_cast<uint32_t>(h[2 * lane] >> 32)) * invT - mx) : 0.0f;
      float t1 = 2 * lane + 1 < hn ? __expf(key_f32(static_cast<uint32_t>(h[2 * lane + 1] >> 32)) * invT - mx) : 0.0f;
      float incl = t0 + t1;  // suffix: lanes l .. 31
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_down_sync(0xFFFFFFFFu, incl, o);
        if (lane + o < 32) incl += y;
      }
      float next = __shfl_down_sync(0xFFFFFFFFu, incl, 1);  // lanes l+1 .. 31
      if (lane == 31) next = 0.0f;
      if (2 * lane < hn) part_tail[q * M + 2 * lane] = incl;
      if (2 * lane + 1 < hn) part_tail[q * M + 2 * lane + 1] = t1 + next;
    }
  }
  for (int idx = et; idx < P * M; idx += 32 * kFtWarps) {
    const int p = idx / M, j = idx - p * M;
    const int hn = s.hn[p];
    const size_t q = static_cast<size_t>(p) * S + cta;
    const uint64_t* h = s.held + (s.par[p] * P + p) * kFtMaxM;
    if (j < hn) {
      const uint64_t k = h[j];
      part_id[q * M + j] = static_cast<int>(rank_key_id(k));
      part_val[q * M + j] = key_f32(static_cast<uint32_t>(k >> 32));
    }
    if (j == 0) {
      // every thread's sums and the evicted sum are against the row's max
      part_max[q] = hn > 0 ? s.ev_ref[p] : -INFINITY;
      part_sum[q] = hn > 0 ? ((s.red[0 * kFtMaxRows + p] + s.red[1 * kFtMaxRows + p]) +
                              (s.red[2 * kFtMaxRows + p] + s.red[3 * kFtMaxRows + p])) +
                                 s.ev_sum[p]
                           : 0.0f;
      part_cnt[q] = hn;
      if (part_kth) part_kth[q] = hn == M ? key_f32(static_cast<uint32_t>(h[M - 1] >> 32)) : -INFINITY;
    }
  }
}

}  // namespace dt

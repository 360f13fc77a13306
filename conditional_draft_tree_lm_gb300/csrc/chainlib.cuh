// Device building blocks shared by the depth chain and the best-first builder:
// the hi/lo bf16 split of fp32 operands, mma.sync m16n8k16, cp.async, the
// bounded grid barrier, fast activations, packed candidate keys and the
// one-warp sort of 64 keys.
#pragma once

#include "common.cuh"

namespace dt {
namespace cl {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

// x = hi + lo with hi = bf16(x), lo = bf16(x - hi): the pair carries ~16
// mantissa bits, so two bf16 MMAs reproduce an fp32 operand to ~2^-17.
// For the lanes l < K holding a token each (the others any value): how many of
// lanes 0 .. K-1 hold a smaller token (the rank that puts a branch's children
// in token order).  Eight independent shuffles at a time, so that their
// latencies overlap (a loop of one shuffle per step measured ~290 cycles a
// step at K = 32).
DT_DEVINL int warp_rank_below(int tok, int K) {
  int r = 0;
  for (int m0 = 0; m0 < K; m0 += 8) {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int t2 = __shfl_sync(0xFFFFFFFFu, tok, (m0 + j) & 31);
      r += (m0 + j < K && t2 < tok) ? 1 : 0;
    }
  }
  return r;
}

DT_DEVINL uint32_t split_hi_lo(float a, float b, uint32_t& lo) {
  const __nv_bfloat16 ah = __float2bfloat16_rn(a), bh = __float2bfloat16_rn(b);
  const __nv_bfloat16 al = __float2bfloat16_rn(a - __bfloat162float(ah));
  const __nv_bfloat16 bl = __float2bfloat16_rn(b - __bfloat162float(bh));
  lo = static_cast<uint32_t>(__bfloat16_as_ushort(al)) | (static_cast<uint32_t>(__bfloat16_as_ushort(bl)) << 16);
  return static_cast<uint32_t>(__bfloat16_as_ushort(ah)) | (static_cast<uint32_t>(__bfloat16_as_ushort(bh)) << 16);
}

// D += A B for one m16n8k16 tile, bf16 inputs, fp32 accumulators.
DT_DEVINL void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                              uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

DT_DEVINL unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

DT_DEVINL void cp_async16(void* s, const void* g) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(s)), "l"(g) : "memory");
}
DT_DEVINL void cp_async4(void* s, const void* g) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(s)), "l"(g) : "memory");
}
DT_DEVINL void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
DT_DEVINL void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
DT_DEVINL void cp_async_wait_group1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

DT_DEVINL void red_release_add_u32(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier on a monotonically increasing counter: the CTA's writes are
// ordered before thread 0's release-add by bar.sync, and every CTA's writes are
// visible after the acquire-load that sees the full count.  Returns false on
// timeout (the status word is set).
DT_DEVINL bool grid_barrier(unsigned* bar, unsigned& epoch, int* status, int* s_abort) {
  __syncthreads();
  if (gridDim.x == 1) return true;  // one CTA: bar.sync orders its global writes
  ++epoch;
  if (threadIdx.x == 0) {
    red_release_add_u32(bar, 1u);
    const unsigned target = epoch * gridDim.x;
    int abort = 0;
    if (ld_acquire_u32(bar) < target) {
      const uint64_t t0 = dt_globaltimer();
      uint32_t n = 0;
      while (ld_acquire_u32(bar) < target) {
        if ((++n & 15u) == 0 && dt_globaltimer() - t0 > DT_WAIT_LIMIT_NS) {
          dt_report(status, DT_DEV_TIMEOUT);
          abort = 1;
          break;
        }
      }
    }
    *s_abort = abort;
  }
  __syncthreads();
  return *s_abort == 0;
}

// Store state value v of (row, column j) into the fragment-ordered copy: its
// bf16 high part and the bf16 of the remainder, at the places lane group
// tig = (j mod 8) / 2 of a k16 step reads them as A-fragment registers
// (a0/a2: columns 2tig, 2tig+1 and 2tig+8, 2tig+9 of the step).  Rows form
// blocks of 8 (one MMA tile: rows gid = row mod 8); inside a block the words
// are ordered [k16 step][gid][tig], so that the 32 lanes of a warp read one
// step of a block as 512 contiguous bytes.
DT_DEVINL size_t frag_word(int row, int kt, int tig, int nk16) {
  return (((static_cast<size_t>(row >> 3) * nk16 + kt) * 8 + (row & 7)) * 4 + tig);
}
DT_DEVINL void store_frag(uint32_t* sf, int row, int j, int nk16, float v) {
  const int kt = j >> 4, w = j & 15;
  const int tig = (w & 7) >> 1, half = w & 1, pair = w >> 3;
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
  uint16_t* u = reinterpret_cast<uint16_t*>(sf + frag_word(row, kt, tig, nk16) * 4);
  u[2 * pair + half] = __bfloat16_as_ushort(hi);
  u[2 * (2 + pair) + half] = __bfloat16_as_ushort(lo);
}

// Activations on the fast exponential and division intrinsics (absolute
// error ~1e-7; a large |x| saturates to the right limit: __fdividef returns 0
// for a denominator beyond 2^126).
DT_DEVINL float sigmoidf_(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
DT_DEVINL float tanhf_(float x) { return __fdividef(2.0f, 1.0f + __expf(-2.0f * x)) - 1.0f; }
DT_DEVINL float siluf_(float x) { return __fdividef(x, 1.0f + __expf(-x)); }


// Keys that carry their candidate index: value key (high 32 bits), then the
// token id inverted in 26 bits (ties go to the lower token), then the
// candidate index in 6 bits.  Orders exactly like rank_key(value, token) for
// distinct tokens < 2^26; valid for M <= 64.
DT_DEVINL uint64_t cand_key(float v, int tok, int c) {
  return (static_cast<uint64_t>(f32_key(v)) << 32) |
         (static_cast<uint64_t>((0x3FFFFFFu - static_cast<uint32_t>(tok)) & 0x3FFFFFFu) << 6) |
         static_cast<uint64_t>(c & 63);
}
DT_DEVINL int cand_key_tok(uint64_t k) { return static_cast<int>(0x3FFFFFFu - ((k >> 6) & 0x3FFFFFFu)); }
DT_DEVINL int cand_key_c(uint64_t k) { return static_cast<int>(k & 63u); }

// Bitonic sort of 64 distinct keys held by one warp (elements 2*lane in ka,
// 2*lane + 1 in kb) into descending order, with branch-free min/max steps;
// afterwards the key of rank e sits in lane e/2 (ka when e is even).
DT_DEVINL void warp_sort64_keys_desc(uint64_t& ka, uint64_t& kb) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1) {
    const bool desc = ((2 * lane) & k) == 0;
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j == 1) {
        const uint64_t hi = ka > kb ? ka : kb, lo = ka > kb ? kb : ka;
        ka = desc ? hi : lo;
        kb = desc ? lo : hi;
      } else {
        const int lj = j >> 1;
        const uint64_t oa = __shfl_xor_sync(0xFFFFFFFFu, ka, lj);
        const uint64_t ob = __shfl_xor_sync(0xFFFFFFFFu, kb, lj);
        const bool keep_max = ((lane & lj) == 0) == desc;
        ka = keep_max ? (oa > ka ? oa : ka) : (oa < ka ? oa : ka);
        kb = keep_max ? (ob > kb ? ob : kb) : (ob < kb ? ob : kb);
      }
    }
  }
}

// Row stride (bf16 elements) of the K-major weight columns and of the state
// rows in shared memory: g rounded up to whole k16 steps, plus 8 elements so
// that consecutive rows start 4 banks apart (conflict-free fragment loads).
DT_HOST_DEVICE_INLINE int kstride(int g) { return (g + 15) / 16 * 16 + 8; }

// One contiguous global -> shared copy by the bulk-copy engine, completing on
// the mbarrier (16-byte aligned addresses, a multiple of 16 bytes).
DT_DEVINL void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}

// Orders this thread's generic-proxy view of global memory with its later
// bulk copies (async proxy).
DT_DEVINL void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

}  // namespace cl
}  // namespace dt

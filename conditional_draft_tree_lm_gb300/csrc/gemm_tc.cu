// Skinny "TN" GEMM on the 5th-generation tensor cores: D[m, n] = sum_k A[m, k] B[n, k]
// with A and B bf16 K-major, fp32 accumulation in tensor memory.
//
// Uses:
//  * base logits (Domino page, Columna Vertebral, Salida): A = the frozen LM head
//    [V, d] (tiles 0..ceil(V/128)-1) followed by the H half of W1, W1[:, :d]
//    ([r, d], row stride d+g; the remaining tiles), B = H viewed as
//    [n_req*block, d].  The roles are swapped (A = weights) so that the MMA's
//    M dimension is 128 vocabulary rows and its N dimension the few H rows; the
//    kernel is bound by streaming A from HBM.  The epilogue scatters columns of
//    block position i >= 1 to logits[q, i-1, v] (or h1[q, i-1, j]).
//    With ft set (one request), the epilogue also keeps each CTA's exact
//    Top-M of the logit rows as they stream by (topm_fused.cuh) and the
//    logits need not be written at all.
//  * the GRU input table (create time): A = E [V, d], B = W_ih [3g, d],
//    D + b_ih -> X [V, 3g] fp32.
//
// Structure: one persistent CTA per SM, 18 warps.  Warp 0 issues TMA loads of
// A/B k-blocks (64 bf16 = one 128-byte swizzle row) into a ring of shared-memory
// stages; warp 1 owns the tensor memory and issues tcgen05.mma (M=128, N<=256,
// K=16) from one thread, committing each stage back to the producer and each
// finished tile to the epilogue; warps 2..5 drain the accumulator with
// tcgen05.ld (one TMEM lane quarter each) while the next tile accumulates into
// the other half of tensor memory.  With the fused Top-M, warps 6..17 join
// them (the same lane quarters; each warp takes 4 of the 16 columns), so
// that each warp's share of the Top-M work is a quarter; otherwise they have
// nothing to do.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace dt {
// Tile stamps (built with -DDT_GEMM_TIMING only): clock64() of CTA 0 for its
// first 16 tiles: [tile][0] the MMA warp starts the tile, [1] it commits the
// tile, [2] the epilogue (warp 2, lane 0) has the accumulator, [3] the
// epilogue is done with the tile, [4] / [5] inside the fused Top-M update;
// [16][0] the epilogue's end, [16][3] the fused Top-M's sums reduced.
#ifdef DT_GEMM_TIMING
__device__ unsigned long long g_gemm_stamps[17][8];
#define GEMM_STAMP(t, k)                                                                   \
  do {                                                                                     \
    if (blockIdx.x == 0 && (t) < 17) g_gemm_stamps[t][k] = static_cast<unsigned long long>(clock64()); \
  } while (0)
#else
#define GEMM_STAMP(t, k) \
  do {                   \
  } while (0)
#endif
// (the fused Top-M's inner stamps, by warp 2 lane 0)
#ifdef DT_GEMM_TIMING
#define FT_STAMP(t, k)                    \
  do {                                    \
    if (threadIdx.x == 64) GEMM_STAMP(t, k); \
  } while (0)
#endif
}  // namespace dt

#include "topm_fused.cuh"

namespace dt {

namespace {

constexpr int kThreads = 576;
constexpr uint32_t kABytes = 128 * 128;  // 128 rows x 64 bf16


// Byte offset of the fused Top-M area from the 1024-aligned shared base: after
// the stages, the barriers and the tensor-memory slot.
DT_HOST_DEVICE_INLINE size_t gemm_ft_offset(const GemmParams& p) {
  return (static_cast<size_t>(p.stages) * p.stage_bytes + (2 * p.stages + 4) * 8 + 16 + 15) & ~static_cast<size_t>(15);
}

__global__ void __launch_bounds__(kThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a2,
              const __grid_constant__ CUtensorMap tm_b, const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  // (offset from the shared array itself, so that accesses through smem stay
  // shared-memory instructions rather than generic ones)
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.stages * p.stage_bytes);
  uint64_t* empty = full + p.stages;
  uint64_t* tfull = empty + p.stages;
  uint64_t* tempty = tfull + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int m_tiles = p.m_tiles_a + p.m_tiles_a2;
  const int num_tiles = m_tiles * p.n_tiles;
  const int num_kb = (p.K + 63) / 64;
  dt_grid_release();  // the next kernel may launch; it waits for this one's end

  if (threadIdx.x == 0) {
    for (int s = 0; s < p.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], p.ft ? kFtWarps : 4);  // one arrival per epilogue warp
    }
    fence_mbar_init();
  }
  if (warp == 1) tmem_alloc(tmem_slot, p.tmem_cols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      const uint64_t pol_a = p.a_evict_first ? l2_policy_evict_first() : l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_last();
      uint32_t stage = 0, phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
        const int mt = tile / p.n_tiles, nt = tile % p.n_tiles;
        const bool second = mt >= p.m_tiles_a;
        const void* ta = second ? static_cast<const void*>(&tm_a2) : static_cast<const void*>(&tm_a);
        const int row_a = (second ? mt - p.m_tiles_a : mt) * 128;
        const int row_b = nt * p.BN;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], p.stage_bytes);
          uint8_t* sa = smem + stage * p.stage_bytes;
          uint8_t* sb = sa + kABytes;
          tma_load_2d(sa, ta, &full[stage], kb * 64, row_a, pol_a);
          for (int h = 0; h < p.BN; h += 256)
            tma_load_2d(sb + h * 128, &tm_b, &full[stage], kb * 64, row_b + h, pol_b);
          if (++stage == static_cast<uint32_t>(p.stages)) { stage = 0; phase ^= 1u; }
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      uint32_t stage = 0, phase = 0;
      int local = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x, ++local) {
        const int acc = p.acc_bufs == 2 ? (local & 1) : 0;
        const uint32_t use = p.acc_bufs == 2 ? static_cast<uint32_t>(local >> 1) : static_cast<uint32_t>(local);
        if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, p.status)) break;
        tc_fence_after();
        GEMM_STAMP(local, 0);
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * p.BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * p.stage_bytes);
          const uint32_t sb = sa + kABytes;
          // straight-line issue (a run-time loop over N halves around each
          // MMA slowed the whole stream by a quarter)
          if (p.BN <= 256) {
            const uint32_t idesc = idesc_bf16_f32(128, p.BN);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              tc_mma_bf16(d_tmem, sdesc_k_sw128(sa + k * 32), sdesc_k_sw128(sb + k * 32), idesc, (kb | k) != 0);
          } else {  // BN = 512: two N = 256 halves
            const uint32_t idesc = idesc_bf16_f32(128, 256);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const uint64_t ad = sdesc_k_sw128(sa + k * 32);
              tc_mma_bf16(d_tmem, ad, sdesc_k_sw128(sb + k * 32), idesc, (kb | k) != 0);
              tc_mma_bf16(d_tmem + 256, ad, sdesc_k_sw128(sb + 256 * 128 + k * 32), idesc, (kb | k) != 0);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == static_cast<uint32_t>(p.stages)) { stage = 0; phase ^= 1u; }
        }
        if (ok) tc_commit(&tfull[acc]);
        GEMM_STAMP(local, 1);
      }
    }
  } else if (warp < 6 || p.ft) {
    // epilogue: warps 2..5 (and 6..17 with the fused Top-M); TMEM lanes
    // [32*(warp%4), +32)
    const int quarter = warp & 3;
    const int grp = (warp - 2) >> 2;  // fused Top-M: columns 4 grp .. 4 grp + 3
    const int row_in_tile = quarter * 32 + lane;
    const int et = (warp - 2) * 32 + lane;
    const bool ft = p.ft != 0;
    FtState fs;
    FtSums fsum;
    int ft_tiles = 0;
    if (ft) {
      fs = ft_state(smem + gemm_ft_offset(p), p.ft_P);
      ft_init(fs, fsum, p.ft_P, et);
    }
    int local = 0;
    for (int tile = blockIdx.x; tile < num_tiles; tile += gridDim.x, ++local) {
      const int acc = p.acc_bufs == 2 ? (local & 1) : 0;
      const uint32_t use = p.acc_bufs == 2 ? static_cast<uint32_t>(local >> 1) : static_cast<uint32_t>(local);
      const bool got = mbar_wait(&tfull[acc], use & 1u, p.status);
      if (ft ? !ft_all(got) : !got) break;
      tc_fence_after();
      if (warp == 2 && lane == 0) GEMM_STAMP(local, 2);
      const int mt = tile / p.n_tiles, nt = tile % p.n_tiles;
      const uint32_t tbase =
          tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) + static_cast<uint32_t>(acc * p.BN);
      if (ft && mt < p.m_tiles_a) {
        // one 16-column tile, a quarter of it per warp: read it, give the
        // accumulator back at once, then the logits (if wanted) and the
        // running Top-M
        uint32_t v[kFtCols];
        tmem_ld4(tbase + static_cast<uint32_t>(kFtCols * grp), v);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
        const int row = mt * 128 + row_in_tile;
        const bool valid = row < p.rows_a;
        if (p.logits && valid) {
#pragma unroll
          for (int j = 0; j < kFtCols; ++j) {
            const int c = kFtCols * grp + j;  // column c: logit row c - 1
            if (c >= 1 && c < p.n_valid) p.logits[static_cast<size_t>(c - 1) * p.rows_a + row] = __uint_as_float(v[j]);
          }
        }
        ft_tile(fs, fsum, v, p.ft_P, p.ft_M, p.ft_invT, row, valid, quarter, grp, warp - 2, ft_tiles);
        ++ft_tiles;
        if (warp == 2 && lane == 0) GEMM_STAMP(local, 3);
        continue;
      }
      if (p.mode == GEMM_LOGITS) {
        const bool second = mt >= p.m_tiles_a;
        const int row = (second ? mt - p.m_tiles_a : mt) * 128 + row_in_tile;
        const int nrows = second ? p.rows_a2 : p.rows_a;
        float* dst = second ? p.h1 : p.logits;
        const bool valid = row < nrows;
        for (int c0 = 0; c0 < p.BN; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tbase + c0, v);
          // fully unrolled with predicated stores: v stays in registers
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const int n = nt * p.BN + c0 + j;  // the H row (request q, block position i)
            const int q = n / p.block, i = n - q * p.block;
            if (n < p.n_valid && i > 0 && valid)
              dst[static_cast<size_t>(q * p.D + i - 1) * nrows + row] = __uint_as_float(v[j]);
          }
        }
      } else {
        const int row = mt * 128 + row_in_tile;
        const bool valid = row < p.rows_a;
        for (int c0 = 0; c0 < p.BN; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(tbase + c0, v);
          const int col0 = nt * p.BN + c0;
          if (valid) {
            float* o = p.out + static_cast<size_t>(row) * p.ldo + col0;
            if (col0 + 16 <= p.n_valid) {
#pragma unroll
              for (int j = 0; j < 16; j += 4) {
                float4 f;
                f.x = __uint_as_float(v[j]) + bf16_to_f32(p.bias[col0 + j]);
                f.y = __uint_as_float(v[j + 1]) + bf16_to_f32(p.bias[col0 + j + 1]);
                f.z = __uint_as_float(v[j + 2]) + bf16_to_f32(p.bias[col0 + j + 2]);
                f.w = __uint_as_float(v[j + 3]) + bf16_to_f32(p.bias[col0 + j + 3]);
                *reinterpret_cast<float4*>(o + j) = f;
              }
            } else {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (col0 + j < p.n_valid) o[j] = __uint_as_float(v[j]) + bf16_to_f32(p.bias[col0 + j]);
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
    if (ft) {
      ft_finish(fs, fsum, p.ft_P, p.ft_M, p.ft_invT, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x), et,
                quarter, grp, p.part_id, p.part_val, p.part_max, p.part_sum, p.part_cnt, p.part_kth, p.part_tail);
    }
    if (warp == 2 && lane == 0) GEMM_STAMP(16, 0);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, p.tmem_cols);
  }
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

EncodeFn encode_fn() {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(f);
  }
  return fn;
}

}  // namespace

bool make_tmap_bf16_2d(CUtensorMap* tm, const void* base, uint64_t inner, uint64_t rows,
                       uint64_t row_stride_bytes, uint32_t box_rows) {
  EncodeFn fn = encode_fn();
  if (!fn) return false;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) != 0 || (row_stride_bytes & 15u) != 0) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_stride_bytes};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t es[2] = {1u, 1u};
  return fn(tm, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Fill the launch-shape fields of p for a tile width BN (16..256 or 512).
void gemm_plan(GemmParams& p, int BN) {
  p.BN = BN;
  p.b_bytes = static_cast<uint32_t>(BN) * 128u;
  p.stage_bytes = kABytes + p.b_bytes;
  const uint32_t budget = 200u * 1024u;
  int st = static_cast<int>(budget / p.stage_bytes);
  p.stages = st < 2 ? 2 : (st > 8 ? 8 : st);
  p.acc_bufs = (2 * BN <= 512) ? 2 : 1;
  int cols = 32;
  while (cols < p.acc_bufs * BN) cols <<= 1;
  p.tmem_cols = cols;
}

size_t gemm_smem_bytes(const GemmParams& p) {
  if (p.ft) return 1024 + gemm_ft_offset(p) + ft_layout(p.ft_P).total;
  return 1024 + static_cast<size_t>(p.stages) * p.stage_bytes + (2 * p.stages + 4) * 8 + 16;
}

int gemm_grid(const GemmParams& p, int num_sms) {
  const int tiles = (p.m_tiles_a + p.m_tiles_a2) * p.n_tiles;
  return tiles < num_sms ? tiles : num_sms;
}

bool gemm_ft_supported(const GemmParams& p, int num_sms) {
  if (p.mode != GEMM_LOGITS || p.n_tiles != 1 || p.BN != 16 || p.n_valid > 16) return false;
  if (p.ft_P < 1 || p.ft_P > kFtMaxRows || p.ft_P > p.n_valid - 1) return false;
  if (p.ft_M < 1 || p.ft_M > kFtMaxM) return false;
  GemmParams q = p;
  q.ft = 1;
  gemm_ft_plan(q);
  return q.stages >= 4 && gemm_smem_bytes(q) <= 227 * 1024;
}

void gemm_ft_plan(GemmParams& p) {
  p.ft = 1;
  while (p.stages > 2 && gemm_smem_bytes(p) > 227 * 1024) --p.stages;
}

cudaError_t gemm_prepare() {
  return dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_gemm_tc));
}

cudaError_t launch_gemm_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_a2, const CUtensorMap& tm_b,
                           const GemmParams& p, int num_sms, cudaStream_t stream) {
  const size_t smem = gemm_smem_bytes(p);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  if (p.ft && !gemm_ft_supported(p, num_sms)) return cudaErrorInvalidValue;
  const int grid = gemm_grid(p, num_sms);
  k_gemm_tc<<<grid, kThreads, smem, stream>>>(tm_a, tm_a2, tm_b, p);
  return cudaGetLastError();
}

}  // namespace dt

#ifdef DT_GEMM_TIMING
// The GEMM tile stamps of the last launch (17 x 8 clock64 values, layout as
// above).  Returns the number of values copied, or -1.
extern "C" int dt_gemm_stamps(unsigned long long* out, int n) {
  if (!out || n < 17 * 8) return -1;
  return cudaMemcpyFromSymbol(out, dt::g_gemm_stamps, sizeof(dt::g_gemm_stamps)) == cudaSuccess ? 17 * 8 : -1;
}
#endif

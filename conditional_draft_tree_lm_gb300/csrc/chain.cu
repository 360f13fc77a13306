// Depth-wise batched expansion of the super-tree ("DARTree: Speculative Diffusion
// Decoding with Autoregressive Draft Trees", Metodología, 1. Expansión AR
// Paralela por Profundidad) scored by the Domino head ("Resumen Técnico: Domino",
// Metodología, 2. Cabeza de Domino).
//
// One persistent cooperative kernel runs depths depth_first..depth_last.  Each
// CTA owns a slice J of the g state columns and a slice R of the r bottleneck
// columns, and keeps in shared memory, for the whole launch, the bf16 weight
// columns that produce them: the three GRU gate rows of W_hh for each j in J
// and the S-half of W1 for each row in R.  Per depth:
//   A  u = S(p) [W_hh(J gates) | W1_S(R)]^T for every live branch p (fp32 SIMT
//      from shared-memory weights); the W1_S part goes to global memory.
//   -- grid barrier --
//   B  every CTA (identically): z = SiLU(h1_i + u_W1), lambda_c = (base_c +
//      z . W2[c]) / T on the Top-M candidates, logp = lambda - logsumexp(rest,
//      lambda), per-branch top-K (ties to the lower token id), children sorted
//      by token id, top-W of the depth by cumulative score (ties to the lower
//      node index).  CTA 0 writes the node arrays and the live list.
//   C  GRU update of the survivors' state columns J:
//      r = sigmoid(x_r + u_r), z = sigmoid(x_z + u_z), n = tanh(x_n + r u_n),
//      h' = (1 - z) n + z h, with x = X[token] (the precomputed E W_ih^T + b_ih).
//   -- grid barrier --
// Every wait is bounded; on a timeout the kernel records DT_DEV_TIMEOUT and
// returns.
#include <cooperative_groups.h>

#include "common.cuh"
#include "kernels.h"

namespace dt {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kPC = 8;  // state rows per GEMM chunk

DT_DEVINL unsigned ld_acquire_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Grid-wide barrier on a monotonically increasing counter.  Returns false on
// timeout (the status word is set).
DT_DEVINL bool grid_barrier(unsigned* bar, unsigned& epoch, int* status, int* s_abort) {
  __syncthreads();
  ++epoch;
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(bar, 1u);
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
    __threadfence();
    *s_abort = abort;
  }
  __syncthreads();
  return *s_abort == 0;
}

DT_DEVINL float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

struct Smem {
  uint16_t* w;      // [g][cpad] bf16 owned weight columns
  float* st;        // [g][kPC] transposed state chunk
  float* red;       // [kWarps][kPC][cpad]
  float* uu;        // [n_req*W][3*jper] owned GRU hidden projections
  float* z;         // [kWarps][r]
  float* lam;       // [kWarps][M]
  int* ctok;        // [W*K] children of the current request: token
  float* clogp;     // [W*K]
  float* cscore;    // [W*K]
  int* crank;       // [W*K]
  int* surv;        // [n_req][W] survivor child slot
  float* pscore;    // [W] parent scores of the current request
  int* pnode;       // [W] parent node indices of the current request
};

__global__ void __launch_bounds__(kThreads, 1) k_chain(const ChainParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int s_abort;

  const int g = p.g, r = p.r, M = p.M, K = p.K, W = p.W;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j0 = blockIdx.x * p.jper;
  const int nj = max(0, min(g, j0 + p.jper) - j0);
  const int r0 = blockIdx.x * p.rper;
  const int nr = max(0, min(r, r0 + p.rper) - r0);
  const int ncol = 3 * nj + nr;
  const int cpad = p.cpad;

  Smem s;
  {
    uint8_t* q = smem_raw;
    auto take = [&](size_t bytes) {
      uint8_t* o = q;
      q += (bytes + 15) & ~static_cast<size_t>(15);
      return o;
    };
    s.w = reinterpret_cast<uint16_t*>(take(static_cast<size_t>(g) * cpad * 2));
    s.st = reinterpret_cast<float*>(take(static_cast<size_t>(g) * kPC * 4));
    s.red = reinterpret_cast<float*>(take(static_cast<size_t>(kWarps) * kPC * cpad * 4));
    s.uu = reinterpret_cast<float*>(take(static_cast<size_t>(p.n_req) * W * 3 * p.jper * 4));
    s.z = reinterpret_cast<float*>(take(static_cast<size_t>(kWarps) * r * 4));
    s.lam = reinterpret_cast<float*>(take(static_cast<size_t>(kWarps) * M * 4));
    s.ctok = reinterpret_cast<int*>(take(static_cast<size_t>(W) * K * 4));
    s.clogp = reinterpret_cast<float*>(take(static_cast<size_t>(W) * K * 4));
    s.cscore = reinterpret_cast<float*>(take(static_cast<size_t>(W) * K * 4));
    s.crank = reinterpret_cast<int*>(take(static_cast<size_t>(W) * K * 4));
    s.surv = reinterpret_cast<int*>(take(static_cast<size_t>(p.n_req) * W * 4));
    s.pscore = reinterpret_cast<float*>(take(static_cast<size_t>(W) * 4));
    s.pnode = reinterpret_cast<int*>(take(static_cast<size_t>(W) * 4));
  }

  // ---- load the owned weight columns (transposed: s.w[k][c]) ----
  for (int idx = tid; idx < cpad * g; idx += kThreads) {
    const int c = idx / g, k = idx - c * g;
    uint16_t v = 0;
    if (c < 3 * nj) {
      const int gate = c / nj, jj = c - gate * nj;
      v = p.w_hh[static_cast<size_t>(gate * g + j0 + jj) * g + k];
    } else if (c < ncol) {
      const int rr = r0 + (c - 3 * nj);
      v = p.w1[static_cast<size_t>(rr) * p.ldw1 + p.d + k];
    }
    s.w[k * cpad + c] = v;
  }

  unsigned epoch = 0;

  // ---- depth 0: root state and root node ----
  if (p.depth_first == 1) {
    for (int idx = tid; idx < p.n_req * nj; idx += kThreads) {
      const int q = idx / nj, jj = j0 + (idx - q * nj);
      int tok = p.root_tok[q];
      if (tok < 0 || tok >= p.V) { dt_report(p.status, DT_DEV_BOUNDS); tok = 0; }
      const float* x = p.xtab + static_cast<size_t>(tok) * 3 * g;
      const float zg = sigmoidf_(x[g + jj]);
      const float ng = tanhf(x[2 * g + jj]);
      p.S[static_cast<size_t>(q * W) * g + jj] = (1.0f - zg) * ng;
    }
    if (blockIdx.x == 0) {
      for (int q = tid; q < p.n_req; q += kThreads) {
        const size_t b = static_cast<size_t>(q) * p.N1;
        p.node_tok[b] = p.root_tok[q];
        p.node_parent[b] = -1;
        p.node_logp[b] = 0.0f;
        p.node_score[b] = 0.0f;
        p.live[static_cast<size_t>(q) * W] = 0;
      }
    }
    if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) return;
  }

  for (int i = p.depth_first; i <= p.depth_last; ++i) {
    const int Lp = p.L[i - 1];          // live branches entering this depth
    const int Li = p.L[i];              // branches that live on
    const int P = p.n_req * Lp;
    const float* Sprev = p.S + static_cast<size_t>((i - 1) & 1) * p.n_req * W * g;
    float* Snext = p.S + static_cast<size_t>(i & 1) * p.n_req * W * g;
    const int* live_prev = p.live + static_cast<size_t>((i - 1) & 1) * p.n_req * W;
    int* live_next = p.live + static_cast<size_t>(i & 1) * p.n_req * W;

    // ================= phase A: projections of the live states ==============
    for (int p0 = 0; p0 < P; p0 += kPC) {
      const int pc = min(kPC, P - p0);
      __syncthreads();
      for (int idx = tid; idx < kPC * g; idx += kThreads) {
        const int pp = idx / g, k = idx - pp * g;
        float v = 0.0f;
        if (pp < pc) {
          const int pr = p0 + pp;
          const int q = pr / Lp, b = pr - q * Lp;
          v = Sprev[static_cast<size_t>(q * W + b) * g + k];
        }
        s.st[k * kPC + pp] = v;
      }
      __syncthreads();
      const int kper = (g + kWarps - 1) / kWarps;
      const int k0 = warp * kper, k1 = min(g, k0 + kper);
      for (int cg = 0; cg < cpad; cg += 32) {
        float acc[kPC];
#pragma unroll
        for (int j = 0; j < kPC; ++j) acc[j] = 0.0f;
        const int c = cg + lane;
        for (int k = k0; k < k1; ++k) {
          const float wv = bf16_to_f32(s.w[k * cpad + c]);
          const float4 a = *reinterpret_cast<const float4*>(&s.st[k * kPC]);
          const float4 b = *reinterpret_cast<const float4*>(&s.st[k * kPC + 4]);
          acc[0] = fmaf(wv, a.x, acc[0]);
          acc[1] = fmaf(wv, a.y, acc[1]);
          acc[2] = fmaf(wv, a.z, acc[2]);
          acc[3] = fmaf(wv, a.w, acc[3]);
          acc[4] = fmaf(wv, b.x, acc[4]);
          acc[5] = fmaf(wv, b.y, acc[5]);
          acc[6] = fmaf(wv, b.z, acc[6]);
          acc[7] = fmaf(wv, b.w, acc[7]);
        }
#pragma unroll
        for (int j = 0; j < kPC; ++j) s.red[(warp * kPC + j) * cpad + c] = acc[j];
      }
      __syncthreads();
      for (int idx = tid; idx < pc * ncol; idx += kThreads) {
        const int pp = idx / ncol, c = idx - pp * ncol;
        float sum = 0.0f;
#pragma unroll
        for (int w8 = 0; w8 < kWarps; ++w8) sum += s.red[(w8 * kPC + pp) * cpad + c];
        const int pr = p0 + pp;
        if (c < 3 * nj) {
          s.uu[static_cast<size_t>(pr) * 3 * p.jper + c] = sum;
        } else {
          const int q = pr / Lp, b = pr - q * Lp;
          p.uW1[static_cast<size_t>(q * W + b) * r + r0 + (c - 3 * nj)] = sum;
        }
      }
    }
    if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) return;

    // ================= phase B: corrected log-probs and selections ==========
    const int row_off = p.off[i];
    const int nchild = Lp * K;
    for (int q = 0; q < p.n_req; ++q) {
      const size_t qrow = static_cast<size_t>(q) * p.D + (i - 1);
      const float* h1 = p.h1 + qrow * r;
      const int* ctok_g = p.cand_tok + qrow * M;
      const float* cbase = p.cand_base + qrow * M;
      const float rest = p.rest_lse[qrow];
      __syncthreads();
      for (int b = tid; b < Lp; b += kThreads) {
        const int node = live_prev[static_cast<size_t>(q) * W + b];
        s.pnode[b] = node;
        s.pscore[b] = (node >= 0 && node < p.N1) ? p.node_score[static_cast<size_t>(q) * p.N1 + node] : 0.0f;
      }
      __syncthreads();
      float* zw = s.z + warp * r;
      float* lw = s.lam + warp * M;
      for (int b = warp; b < Lp; b += kWarps) {
        const float* u = p.uW1 + static_cast<size_t>(q * W + b) * r;
        for (int k = lane; k < r; k += 32) {
          const float x = h1[k] + u[k];
          zw[k] = x / (1.0f + expf(-x));
        }
        __syncwarp();
        float lmax = rest;
        for (int c = lane; c < M; c += 32) {
          int tok = ctok_g[c];
          if (tok < 0 || tok >= p.V) { dt_report(p.status, DT_DEV_BOUNDS); tok = 0; }
          const uint4* wrow = reinterpret_cast<const uint4*>(p.w2 + static_cast<size_t>(tok) * r);
          float dot = 0.0f;
          for (int k8 = 0; k8 < r / 8; ++k8) {
            const uint4 w8 = __ldg(wrow + k8);
            const float* zz = zw + k8 * 8;
            dot = fmaf(zz[0], __uint_as_float(w8.x << 16), dot);
            dot = fmaf(zz[1], __uint_as_float(w8.x & 0xFFFF0000u), dot);
            dot = fmaf(zz[2], __uint_as_float(w8.y << 16), dot);
            dot = fmaf(zz[3], __uint_as_float(w8.y & 0xFFFF0000u), dot);
            dot = fmaf(zz[4], __uint_as_float(w8.z << 16), dot);
            dot = fmaf(zz[5], __uint_as_float(w8.z & 0xFFFF0000u), dot);
            dot = fmaf(zz[6], __uint_as_float(w8.w << 16), dot);
            dot = fmaf(zz[7], __uint_as_float(w8.w & 0xFFFF0000u), dot);
          }
          const float lam = (cbase[c] + dot) / p.T;
          lw[c] = lam;
          lmax = fmaxf(lmax, lam);
        }
        lmax = warp_max(lmax);
        float se = 0.0f;
        for (int c = lane; c < M; c += 32) se += expf(lw[c] - lmax);
        se = warp_sum(se);
        if (lane == 0) se += expf(rest - lmax);
        se = __shfl_sync(0xFFFFFFFFu, se, 0);
        const float logZ = lmax + logf(se);
        // top-K by (logp desc, token asc): K rounds of warp argmax
        int my_tok = 0;
        float my_lp = 0.0f;
        for (int kk = 0; kk < K; ++kk) {
          uint64_t best = 0;
          for (int c = lane; c < M; c += 32) {
            const float lam = lw[c];
            if (lam == -INFINITY) continue;  // already taken
            const uint64_t key = rank_key(lam - logZ, static_cast<uint32_t>(ctok_g[c]));
            best = key > best ? key : best;
          }
          best = warp_max_u64(best);
          const uint32_t wtok = rank_key_id(best);
          // the lane holding the winner marks it taken and broadcasts logp
          float wlp = 0.0f;
          int owner = -1;
          for (int c = lane; c < M; c += 32)
            if (static_cast<uint32_t>(ctok_g[c]) == wtok && lw[c] != -INFINITY) {
              wlp = lw[c] - logZ;
              lw[c] = -INFINITY;
              owner = lane;
            }
          const unsigned om = __ballot_sync(0xFFFFFFFFu, owner >= 0);
          const int src = om ? __ffs(om) - 1 : 0;
          wlp = __shfl_sync(0xFFFFFFFFu, wlp, src);
          if (lane == kk) {
            my_tok = static_cast<int>(wtok);
            my_lp = wlp;
          }
        }
        // children of branch b sorted by token id
        int rank = 0;
        for (int m = 0; m < K; ++m) {
          const int t = __shfl_sync(0xFFFFFFFFu, my_tok, m);
          rank += (m < K && t < my_tok) ? 1 : 0;
        }
        if (lane < K) {
          const int slot = b * K + rank;
          s.ctok[slot] = my_tok;
          s.clogp[slot] = my_lp;
          s.cscore[slot] = s.pscore[b] + my_lp;
        }
        __syncwarp();
      }
      __syncthreads();
      // node arrays of this depth (CTA 0)
      if (blockIdx.x == 0) {
        const size_t nb = static_cast<size_t>(q) * p.N1 + row_off;
        for (int e = tid; e < nchild; e += kThreads) {
          p.node_tok[nb + e] = s.ctok[e];
          p.node_parent[nb + e] = s.pnode[e / K];
          p.node_logp[nb + e] = s.clogp[e];
          p.node_score[nb + e] = s.cscore[e];
        }
      }
      if (i < p.D) {
        // top-W of the depth: rank by (score desc, node index asc)
        for (int e = tid; e < nchild; e += kThreads) {
          const uint64_t ke = rank_key(s.cscore[e], static_cast<uint32_t>(e));
          int rk = 0;
          for (int f = 0; f < nchild; ++f) rk += rank_key(s.cscore[f], static_cast<uint32_t>(f)) > ke;
          s.crank[e] = rk;
        }
        __syncthreads();
        // survivors in ascending slot order
        for (int e = tid; e < nchild; e += kThreads) {
          if (s.crank[e] < Li) {
            int pos = 0;
            for (int f = 0; f < e; ++f) pos += s.crank[f] < Li;
            s.surv[q * W + pos] = e;
            if (blockIdx.x == 0) {
              live_next[static_cast<size_t>(q) * W + pos] = row_off + e;
            }
          }
        }
        __syncthreads();
        if (blockIdx.x == 0 && p.live_out) {
          for (int j = tid; j < W; j += kThreads)
            p.live_out[static_cast<size_t>(q) * W + j] = j < Li ? row_off + s.surv[q * W + j] : -1;
        }
        // ================= phase C (this request): GRU of the survivors ======
        for (int idx = tid; idx < Li * nj; idx += kThreads) {
          const int jv = idx / nj, jj = idx - jv * nj;
          const int e = s.surv[q * W + jv];
          const int b = e / K;
          int tok = s.ctok[e];
          if (tok < 0 || tok >= p.V) { dt_report(p.status, DT_DEV_BOUNDS); tok = 0; }
          const float* x = p.xtab + static_cast<size_t>(tok) * 3 * g + j0 + jj;
          const float* uu = s.uu + static_cast<size_t>(q * Lp + b) * 3 * p.jper;
          const float ur = uu[jj], uz = uu[nj + jj], un = uu[2 * nj + jj];
          const float h = Sprev[static_cast<size_t>(q * W + b) * g + j0 + jj];
          const float rg = sigmoidf_(x[0] + ur);
          const float zg = sigmoidf_(x[g] + uz);
          const float ng = tanhf(x[2 * g] + rg * un);
          Snext[static_cast<size_t>(q * W + jv) * g + j0 + jj] = (1.0f - zg) * ng + zg * h;
        }
      } else if (blockIdx.x == 0 && p.live_out) {
        for (int j = tid; j < W; j += kThreads) p.live_out[static_cast<size_t>(q) * W + j] = -1;
      }
    }
    if (i < p.depth_last) {
      if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) return;
    }
  }
}

}  // namespace

int chain_grid(const ChainParams& p, int num_sms) {
  // one CTA per 8 state columns, at most one per SM
  int G = (p.g + 7) / 8;
  if (G > num_sms) G = num_sms;
  if (G < 1) G = 1;
  return G;
}

size_t chain_smem_bytes(const ChainParams& p) {
  auto al = [](size_t b) { return (b + 15) & ~static_cast<size_t>(15); };
  size_t b = 0;
  b += al(static_cast<size_t>(p.g) * p.cpad * 2);
  b += al(static_cast<size_t>(p.g) * kPC * 4);
  b += al(static_cast<size_t>(kWarps) * kPC * p.cpad * 4);
  b += al(static_cast<size_t>(p.n_req) * p.W * 3 * p.jper * 4);
  b += al(static_cast<size_t>(kWarps) * p.r * 4);
  b += al(static_cast<size_t>(kWarps) * p.M * 4);
  b += 4 * al(static_cast<size_t>(p.W) * p.K * 4);
  b += al(static_cast<size_t>(p.n_req) * p.W * 4);
  b += 2 * al(static_cast<size_t>(p.W) * 4);
  return b;
}

void chain_plan(ChainParams& p, int grid) {
  p.jper = (p.g + grid - 1) / grid;
  p.rper = (p.r + grid - 1) / grid;
  const int ncol = 3 * p.jper + p.rper;
  p.cpad = (ncol + 31) / 32 * 32;
}

cudaError_t chain_prepare() {
  return cudaFuncSetAttribute(k_chain, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
}

cudaError_t launch_chain(const ChainParams& p, int grid, cudaStream_t stream) {
  const size_t smem = chain_smem_bytes(p);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_chain, p);
}

}  // namespace dt

// Sequential conditional best-first expansion of one request's draft tree
// ("Resumen Técnico: DominoTree", Metodología, 1. Montículo de Mejor Primera
// Búsqueda con Puntuación Condicional; 2. Restricción de Candidatos): the
// node-by-node builder that the depth-batched chain replaces ("DARTree ...",
// Contribuciones Clave, 1.; Resultados Experimentales, Ablación, Latencia).
//
// One persistent cooperative kernel.  As in the depth chain, each CTA owns a
// slice J of the g state columns and a slice R of the r bottleneck rows, with
// the bf16 weight rows [W_hh(J gates) | W1_S(R)] resident in shared memory.
// Every CTA keeps an identical copy of the frontier: the created nodes (token,
// parent, depth, score) and a 64-bit key per frontier node (f32 key of
// score + beta * depth, then the inverted node index: the largest key is the
// best node, the lower index on equal keys).  Per pop, every CTA takes the same
// node v from its own copy; unless v is the B-th pop or sits at depth D it is
// expanded:
//   1. the candidate data of depth(v)+1 (W2 rows, base logits, rest) is staged
//      with cp.async;
//   2. S(v)[J] = GRU(X[tok v][J gates], u_U(parent)[J], S(parent)[J]) from the
//      CTA's own records of the parent, published to global memory;
//   -- grid barrier
//   3. u(v) = S(v) [W_hh(J gates) | W1_S(R)]^T (mma.sync m16n8k16, the fp32
//      state split into bf16 high and low parts in rows 0 and 8 of the tile);
//      the gate part is kept for v's children, the bottleneck part becomes
//      z(v)[R] = SiLU(h1[R] + u), published;
//   -- grid barrier
//   4. lambda_c = (base_c + z(v) . W2[c]) / T on the M candidates (mma.sync),
//      the log-partition with the rest, the K best in one warp (a register
//      sort of packed keys), the children appended in token order with score
//      s(v) + logp and their keys entered into the frontier.
// After B pops CTA 0 sorts the popped nodes and emits the tree and the
// ancestor mask.  Every wait is bounded; on a timeout the kernel records
// DT_DEV_TIMEOUT and returns.
#include "chainlib.cuh"
#include "common.cuh"
#include "kernels.h"
#include "prune.cuh"

namespace dt {

namespace {

using namespace cl;

constexpr int kBMaxNTiles = 8;  // owned columns per CTA <= 64

struct BestLayout {
  size_t off[21];
  size_t total;
};

DT_HOST_DEVICE_INLINE size_t bal16(size_t b) { return (b + 15) & ~static_cast<size_t>(15); }

// Shared-memory regions: 0 w, 1 sh, 2 sl, 3 red, 4 es_S, 5 es_u, 6 ntok, 7 npar,
// 8 ndep, 9 nscore, 10 nlogp, 11 neslot, 12 fkey, 13 nx, 14 tok_all, 15 w2s,
// 16 cbs+rest, 17 h1own, 18 zh/zl, 19 lamkey, 20 popped.
DT_HOST_DEVICE_INLINE BestLayout best_layout(const BestParams& p) {
  const size_t gp = static_cast<size_t>(kstride(p.g));
  const size_t rp = static_cast<size_t>(p.r) + 8;
  const size_t n = static_cast<size_t>(p.nmax);
  const size_t sz[21] = {
      gp * p.cpad * 2,
      gp * 2,
      gp * 2,
      static_cast<size_t>(kWarps) * p.cpad * 4,
      static_cast<size_t>(p.B) * p.jper * 4,
      static_cast<size_t>(p.B) * 3 * p.jper * 4,
      n * 4,
      n * 4,
      n * 4,
      n * 4,
      n * 4,
      n * 4,
      n * 8,
      p.xpre ? n * 3 * p.jper * 4 : 0,
      static_cast<size_t>(p.D) * p.M * 4,
      static_cast<size_t>(p.M) * rp * 2,
      (static_cast<size_t>(p.M) + 4) * 4,
      static_cast<size_t>(p.D) * p.rper * 4,
      2 * rp * 2,
      64 * 8,
      static_cast<size_t>(p.B) * 4,
  };
  BestLayout L;
  size_t o = 0;
  for (int i = 0; i < 21; ++i) {
    L.off[i] = o;
    o += bal16(sz[i]);
  }
  L.total = o;
  return L;
}

__global__ void __launch_bounds__(kThreads, 1) k_best(const BestParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ int s_pop;
  __shared__ uint64_t s_wmax[kWarps];

  const BestLayout L = best_layout(p);
  uint16_t* w = reinterpret_cast<uint16_t*>(smem_raw + L.off[0]);
  uint16_t* sh = reinterpret_cast<uint16_t*>(smem_raw + L.off[1]);
  uint16_t* sl = reinterpret_cast<uint16_t*>(smem_raw + L.off[2]);
  float* red = reinterpret_cast<float*>(smem_raw + L.off[3]);
  float* es_S = reinterpret_cast<float*>(smem_raw + L.off[4]);
  float* es_u = reinterpret_cast<float*>(smem_raw + L.off[5]);
  int* ntok = reinterpret_cast<int*>(smem_raw + L.off[6]);
  int* npar = reinterpret_cast<int*>(smem_raw + L.off[7]);
  int* ndep = reinterpret_cast<int*>(smem_raw + L.off[8]);
  float* nscore = reinterpret_cast<float*>(smem_raw + L.off[9]);
  float* nlogp = reinterpret_cast<float*>(smem_raw + L.off[10]);
  int* neslot = reinterpret_cast<int*>(smem_raw + L.off[11]);
  uint64_t* fkey = reinterpret_cast<uint64_t*>(smem_raw + L.off[12]);
  float* nx = reinterpret_cast<float*>(smem_raw + L.off[13]);
  int* tok_all = reinterpret_cast<int*>(smem_raw + L.off[14]);
  uint16_t* w2s = reinterpret_cast<uint16_t*>(smem_raw + L.off[15]);
  float* cbs = reinterpret_cast<float*>(smem_raw + L.off[16]);
  float* h1own = reinterpret_cast<float*>(smem_raw + L.off[17]);
  uint16_t* zh = reinterpret_cast<uint16_t*>(smem_raw + L.off[18]);
  uint64_t* lamkey = reinterpret_cast<uint64_t*>(smem_raw + L.off[19]);
  int* popped = reinterpret_cast<int*>(smem_raw + L.off[20]);

  const int g = p.g, r = p.r, M = p.M, K = p.K, D = p.D;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const int j0 = blockIdx.x * p.jper;
  const int nj = max(0, min(g, j0 + p.jper) - j0);
  const int r0 = blockIdx.x * p.rper;
  const int nr = max(0, min(r, r0 + p.rper) - r0);
  const int ncol = 3 * nj + nr;
  const int cpad = p.cpad;
  const int gp = kstride(g);
  const int rp = r + 8;
  uint16_t* zl = zh + rp;
  float* rest = cbs + M;

  // ---- the owned weight rows, K-major (zero padded) ----
  {
    const int g8 = gp / 8;
    for (int idx = tid; idx < cpad * g8; idx += kThreads) {
      const int c = idx / g8, k8 = idx - c * g8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (8 * k8 < g) {
        if (c < 3 * nj) {
          const int gate = c / nj, jj = c - gate * nj;
          v = *reinterpret_cast<const uint4*>(p.w_hh + static_cast<size_t>(gate * g + j0 + jj) * g + 8 * k8);
        } else if (c < ncol) {
          const int rr = r0 + (c - 3 * nj);
          v = *reinterpret_cast<const uint4*>(p.w1 + static_cast<size_t>(rr) * p.ldw1 + p.d + 8 * k8);
        }
      }
      *reinterpret_cast<uint4*>(w + static_cast<size_t>(c) * gp + 8 * k8) = v;
    }
    for (int k = tid; k < gp; k += kThreads) {
      sh[k] = 0;
      sl[k] = 0;
    }
    for (int k = tid; k < 2 * rp; k += kThreads) zh[k] = 0;
  }
  // everything below reads the previous kernels' results
  dt_grid_wait();

  for (int idx = tid; idx < D * M; idx += kThreads) {
    int t = p.cand_tok[idx];
    if (t < 0 || t >= p.V) {
      dt_report(p.status, DT_DEV_BOUNDS);
      t = 0;
    }
    tok_all[idx] = t;
  }
  for (int idx = tid; idx < D * p.rper; idx += kThreads) {
    const int i = idx / p.rper, k = idx - i * p.rper;
    h1own[idx] = k < nr ? p.h1[static_cast<size_t>(i) * r + r0 + k] : 0.0f;
  }
  for (int v = tid; v < p.nmax; v += kThreads) fkey[v] = 0ull;
  if (tid == 0) {
    int t = p.root_tok[0];
    if (t < 0 || t >= p.V) {
      dt_report(p.status, DT_DEV_BOUNDS);
      t = 0;
    }
    ntok[0] = t;
    npar[0] = -1;
    ndep[0] = 0;
    nscore[0] = 0.0f;
    nlogp[0] = 0.0f;
    neslot[0] = -1;
  }
  __syncthreads();

  unsigned epoch = 0;
  int n_nodes = 1;
  int n_exp = 0;
  auto drain = [&]() { cp_async_wait_all(); };

  // Expansion of node v (whole CTA, every CTA): false on a barrier timeout.
  auto expand = [&](int v) -> bool {
    const int i = ndep[v] + 1;  // depth of the children
    const int* ctk = tok_all + static_cast<size_t>(i - 1) * M;
    // the GRU-input slices prefetched at earlier expansions (v's among them)
    // have landed and are visible to the whole CTA
    cp_async_wait_all();
    __syncthreads();
    // 1. stage the candidates of depth i
    {
      const int c8 = r / 8;
      for (int idx = tid; idx < M * c8; idx += kThreads) {
        const int c = idx / c8, k = idx - c * c8;
        cp_async16(w2s + static_cast<size_t>(c) * rp + 8 * k, p.w2 + static_cast<size_t>(ctk[c]) * r + 8 * k);
      }
      for (int c = tid; c < M; c += kThreads) cp_async4(cbs + c, p.cand_base + static_cast<size_t>(i - 1) * M + c);
      if (tid == 0) cp_async4(rest, p.rest_lse + (i - 1));
      cp_async_commit();
    }
    // 2. S(v) on the owned columns
    const int e = n_exp;
    if (tid < nj) {
      const int jj = tid;
      float x[3];
      if (v == 0 || !p.xpre) {
        const float* xr = p.xtab + static_cast<size_t>(ntok[v]) * 3 * g + j0 + jj;
        x[0] = xr[0];
        x[1] = xr[g];
        x[2] = xr[2 * g];
      } else {
        const float* xr = nx + static_cast<size_t>(v) * 3 * p.jper;
        x[0] = xr[jj];
        x[1] = xr[nj + jj];
        x[2] = xr[2 * nj + jj];
      }
      float hn;
      if (v == 0) {
        // the root: GRU over the root token from a zero state
        const float zg = sigmoidf_(x[1]);
        const float ng = tanhf_(x[2]);
        hn = (1.0f - zg) * ng;
      } else {
        const int pe = neslot[npar[v]];
        const float* u = es_u + static_cast<size_t>(pe) * 3 * p.jper;
        const float h = es_S[static_cast<size_t>(pe) * p.jper + jj];
        const float rg = sigmoidf_(x[0] + u[jj]);
        const float zg = sigmoidf_(x[1] + u[nj + jj]);
        const float ng = tanhf_(x[2] + rg * u[2 * nj + jj]);
        hn = (1.0f - zg) * ng + zg * h;
      }
      es_S[static_cast<size_t>(e) * p.jper + jj] = hn;
      p.srow[j0 + jj] = hn;
    }
    if (tid == 0) neslot[v] = e;
    if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) return false;

    // 3. u(v) on the owned columns; z(v) on the owned bottleneck rows
    for (int k = tid; k < g; k += kThreads) {
      const float sv = __ldcg(p.srow + k);
      const __nv_bfloat16 hi = __float2bfloat16_rn(sv);
      sh[k] = __bfloat16_as_ushort(hi);
      sl[k] = __bfloat16_as_ushort(__float2bfloat16_rn(sv - __bfloat162float(hi)));
    }
    __syncthreads();
    {
      float acc[kBMaxNTiles][4];
#pragma unroll
      for (int nt = 0; nt < kBMaxNTiles; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[nt][q] = 0.0f;
      const int ntiles = cpad / 8;
      const int nk16 = (g + 15) / 16;
      for (int kt = warp; kt < nk16; kt += kWarps) {
        const int k0 = kt * 16 + 2 * tig;
        // row 0 of the tile: high parts of S(v); row 8: low parts
        const uint32_t a0 = gid == 0 ? *reinterpret_cast<const uint32_t*>(sh + k0) : 0u;
        const uint32_t a1 = gid == 0 ? *reinterpret_cast<const uint32_t*>(sl + k0) : 0u;
        const uint32_t a2 = gid == 0 ? *reinterpret_cast<const uint32_t*>(sh + k0 + 8) : 0u;
        const uint32_t a3 = gid == 0 ? *reinterpret_cast<const uint32_t*>(sl + k0 + 8) : 0u;
#pragma unroll
        for (int nt = 0; nt < kBMaxNTiles; ++nt) {
          if (nt < ntiles) {
            const uint16_t* wc = w + static_cast<size_t>(nt * 8 + gid) * gp + k0;
            const uint32_t b0 = *reinterpret_cast<const uint32_t*>(wc);
            const uint32_t b1 = *reinterpret_cast<const uint32_t*>(wc + 8);
            mma_bf16_16816(acc[nt], a0, a1, a2, a3, b0, b1);
          }
        }
      }
      if (gid == 0) {
#pragma unroll
        for (int nt = 0; nt < kBMaxNTiles; ++nt) {
          if (nt < ntiles) {
            float* rw = red + warp * cpad + nt * 8 + 2 * tig;
            rw[0] = acc[nt][0] + acc[nt][2];
            rw[1] = acc[nt][1] + acc[nt][3];
          }
        }
      }
    }
    __syncthreads();
    for (int c = tid; c < ncol; c += kThreads) {
      float sum = 0.0f;
#pragma unroll
      for (int w8 = 0; w8 < kWarps; ++w8) sum += red[w8 * cpad + c];
      if (c < 3 * nj) {
        es_u[static_cast<size_t>(e) * 3 * p.jper + c] = sum;
      } else {
        const int k = c - 3 * nj;
        p.zrow[r0 + k] = siluf_(h1own[(i - 1) * p.rper + k] + sum);
      }
    }
    if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) return false;

    // 4. corrected log-probs of the M candidates, the K best, the children
    for (int k = tid; k < r; k += kThreads) {
      const float zv = __ldcg(p.zrow + k);
      const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
      zh[k] = __bfloat16_as_ushort(hi);
      zl[k] = __bfloat16_as_ushort(__float2bfloat16_rn(zv - __bfloat162float(hi)));
    }
    cp_async_wait_all();  // the staged candidates (and earlier X slices) have landed
    __syncthreads();
    for (int nt = warp; nt < M / 8; nt += kWarps) {
      const uint16_t* wr = w2s + static_cast<size_t>(nt * 8 + gid) * rp;
      float a[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      for (int kt = 0; kt < r / 16; ++kt) {
        const int k0 = kt * 16 + 2 * tig;
        const uint32_t a0 = gid == 0 ? *reinterpret_cast<const uint32_t*>(zh + k0) : 0u;
        const uint32_t a1 = gid == 0 ? *reinterpret_cast<const uint32_t*>(zl + k0) : 0u;
        const uint32_t a2 = gid == 0 ? *reinterpret_cast<const uint32_t*>(zh + k0 + 8) : 0u;
        const uint32_t a3 = gid == 0 ? *reinterpret_cast<const uint32_t*>(zl + k0 + 8) : 0u;
        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(wr + k0);
        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(wr + k0 + 8);
        mma_bf16_16816(a, a0, a1, a2, a3, b0, b1);
      }
      if (gid == 0) {
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int c = nt * 8 + 2 * tig + q;
          const float num = p.marginal ? 0.0f : a[q] + a[q + 2];
          const float lam = (cbs[c] + num) / p.T;
          lamkey[c] = cand_key(lam, ctk[c], c);
        }
      }
    }
    for (int c = M + tid; c < 64; c += kThreads) lamkey[c] = 0ull;
    __syncthreads();
    if (warp == 0) {
      uint64_t ka = lamkey[2 * lane], kb = lamkey[2 * lane + 1];
      const bool va = 2 * lane < M, vb = 2 * lane + 1 < M;
      const float la = va ? key_f32(static_cast<uint32_t>(ka >> 32)) : -INFINITY;
      const float lb = vb ? key_f32(static_cast<uint32_t>(kb >> 32)) : -INFINITY;
      const float rs = rest[0];
      const float lmax = warp_max(fmaxf(rs, fmaxf(la, lb)));
      const float se = warp_sum((va ? expf(la - lmax) : 0.0f) + (vb ? expf(lb - lmax) : 0.0f)) + expf(rs - lmax);
      const float logZ = lmax + logf(se);
      warp_sort64_keys_desc(ka, kb);
      const uint64_t xa = __shfl_sync(0xFFFFFFFFu, ka, (lane >> 1) & 31);
      const uint64_t xb = __shfl_sync(0xFFFFFFFFu, kb, (lane >> 1) & 31);
      const uint64_t wk = (lane & 1) ? xb : xa;
      const int tok = lane < K ? cand_key_tok(wk) : 0x7FFFFFFF;
      const int trank = warp_rank_below(tok, K);
      if (lane < K) {
        const float lp = key_f32(static_cast<uint32_t>(wk >> 32)) - logZ;
        const int u = n_nodes + trank;
        const float sc = nscore[v] + lp;
        ntok[u] = tok;
        npar[u] = v;
        ndep[u] = i;
        nlogp[u] = lp;
        nscore[u] = sc;
        neslot[u] = -1;
        fkey[u] = rank_key(sc + p.beta * static_cast<float>(i), static_cast<uint32_t>(u));
      }
    }
    __syncthreads();
    // the children's GRU-input slices, for their own expansion later
    if (p.xpre && i < D) {
      const int per = 3 * nj;
      for (int idx = tid; idx < K * per; idx += kThreads) {
        const int ch = idx / per, rem = idx - ch * per;
        const int gate = rem / nj, jj = rem - gate * nj;
        const int u = n_nodes + ch;
        cp_async4(nx + static_cast<size_t>(u) * 3 * p.jper + gate * nj + jj,
                  p.xtab + static_cast<size_t>(ntok[u]) * 3 * g + gate * g + j0 + jj);
      }
      cp_async_commit();
    }
    n_nodes += K;
    ++n_exp;
    return true;
  };

  if (!expand(0)) {
    drain();
    return;
  }
  for (int np = 0; np < p.B; ++np) {
    // the best frontier node: the largest key (each CTA on its own copy)
    uint64_t best = 0ull;
    for (int u = tid; u < n_nodes; u += kThreads) best = fkey[u] > best ? fkey[u] : best;
    best = warp_max_u64(best);
    if (lane == 0) s_wmax[warp] = best;
    __syncthreads();
    if (tid == 0) {
      uint64_t b = s_wmax[0];
      for (int w8 = 1; w8 < kWarps; ++w8) b = s_wmax[w8] > b ? s_wmax[w8] : b;
      int v = -1;
      if (b != 0ull) {
        v = static_cast<int>(rank_key_id(b));
        fkey[v] = 0ull;
      } else {
        dt_report(p.status, DT_DEV_TREE);  // empty frontier before the budget
      }
      popped[np] = v;
      s_pop = v;
    }
    __syncthreads();
    const int v = s_pop;
    if (v < 0) {
      drain();
      return;
    }
    if (np + 1 < p.B && ndep[v] < D) {
      if (!expand(v)) {
        drain();
        return;
      }
    }
  }
  drain();

  // ---- tail (CTA 0): the popped nodes in ascending order, the tree and mask ----
  if (blockIdx.x != 0) return;
  __syncthreads();
  const int B = p.B, S = B + 1;
  // scratch in the weight area (no longer read)
  int* sel = reinterpret_cast<int*>(w);
  int* tnodes = sel + B;
  int* tpar = tnodes + S;
  int* tdep = tpar + S;
  uint32_t* anc = reinterpret_cast<uint32_t*>(tdep + S);
  for (int a = tid; a < B; a += kThreads) {
    const int va = popped[a];
    int pos = 0;
    for (int b2 = 0; b2 < B; ++b2) pos += popped[b2] < va ? 1 : 0;
    sel[pos] = va;
    if (p.pops) p.pops[a] = va;
  }
  __syncthreads();
  for (int a = tid; a < B; a += kThreads) p.sel[a] = sel[a];
  tree_and_mask(sel, n_nodes, B, D, nullptr, ntok, npar, nscore, ndep, tnodes, tpar, tdep, anc, p.tok, p.parent,
                p.depth, p.logp_cum, p.mask, p.status);
}

}  // namespace

size_t best_smem_bytes(const BestParams& p) { return best_layout(p).total; }

bool best_plan(BestParams& p, int grid) {
  p.jper = (p.g + grid - 1) / grid;
  p.rper = (p.r + grid - 1) / grid;
  p.cpad = (3 * p.jper + p.rper + 31) / 32 * 32;
  p.nmax = 1 + p.B * p.K;
  constexpr size_t kBudget = 224 * 1024;
  p.xpre = 1;
  if (best_smem_bytes(p) > kBudget) p.xpre = 0;
  // the tail reuses the weight area for its scratch
  const size_t S = static_cast<size_t>(p.B) + 1;
  const size_t tail = (static_cast<size_t>(p.B) + 3 * S + S * anc_words(static_cast<int>(S))) * 4;
  const size_t weight_bytes = static_cast<size_t>(kstride(p.g)) * p.cpad * 2;
  return p.cpad <= 8 * kBMaxNTiles && best_smem_bytes(p) <= kBudget && tail <= weight_bytes && p.M <= 64 &&
         p.M % 8 == 0 && p.K <= 32 && p.r % 16 == 0 && p.r % 8 == 0;
}

cudaError_t best_prepare() { return dt_allow_max_dynamic_smem(reinterpret_cast<const void*>(k_best)); }

cudaError_t launch_best(const BestParams& p, int grid, cudaStream_t stream) {
  const size_t smem = best_smem_bytes(p);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, k_best, p);
}

}  // namespace dt

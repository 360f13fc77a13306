// Depth-wise batched expansion of one request's super-tree on thread-block
// clusters ("DARTree: Speculative Diffusion Decoding with Autoregressive Draft
// Trees", Metodología, 1. Expansión AR Paralela por Profundidad), scored by the
// Domino head ("Resumen Técnico: Domino", Metodología, 2. Cabeza de Domino: the
// GRU causal encoder and the rank-r correction, applied to the Top-M candidates
// of "Resumen Técnico: DominoTree", Componentes Principales, 2.).
//
// Work split (G = g/JC CTAs in clusters of CS; every CTA runs every depth):
//   * CTA c owns the state columns J = [JC c, JC c + JC): the three GRU gate
//     rows of W_hh for them stay resident in shared memory (K-major bf16), and
//     so do the fp32 states of those columns for the live branches.
//   * Cluster rank q owns the bottleneck rows R = [q r/CS, (q+1) r/CS): the
//     S-half of W1 for them stays resident as well, so each cluster holds all
//     r rows once.
// Per depth i (P <= 8 live branches):
//   X   the states of depth i-1 arrive through global memory as tagged 8-byte
//       words (a bf16x2 high or low part of two columns, and a tag of launch
//       and depth).  Every CTA polls all of them straight from L2 into its own
//       shared memory, already in mma.sync A-fragment order (a word's tag
//       proves its payload: no fence, no flag, no grid barrier).
//   A1  u_R = S W1_S(R)^T: mma.sync m16n8k16 with the high parts of the states
//       in rows 0-7 and the low parts in rows 8-15 of the tile, so one product
//       gives both (short accumulation chains: a dependent mma.sync is slow);
//       z_R = SiLU(h1_i(R) + u_R) in fp32.
//   A2  the rank's partial correction dL_q = z_R W2(R, C_i): fp32 FMAs over the
//       rank's r/CS rows; its slice s goes to rank s with st.async (16-byte
//       stores into the peer's shared memory that complete on the peer's
//       mbarrier: no fence, no cluster barrier).
//   A3  u_J = S W_hh(J)^T, the hidden projections of the owned columns, while
//       the slices travel.
//   R   rank q adds its slice over the CS ranks in rank order and sends the
//       sum to every rank the same way (reduce-scatter, then all-gather), so
//       every CTA of every cluster holds bit-identical corrections.
//   B   every CTA repeats the same selections: lambda = (base + dL) / T, logp =
//       lambda - log(e^rest + sum e^lambda), per-branch top-K by K rounds of two
//       warp max reductions over packed (lambda, token, candidate) keys (ties to
//       the lower token id), children in token order, cumulative scores, top-W
//       by (score, node index) the same way in each warp that needs it.  CTA 0
//       writes the node arrays once it has published its states.
//   C   GRU update of the survivors' owned columns, r = sigmoid(x_r + u_r),
//       z = sigmoid(x_z + u_z), n = tanh(x_n + r u_n), h' = (1 - z) n + z h with
//       x = X[token] from the GRU-input table; published as the next X.
// The grid exchanges data once per depth and has no grid-wide barrier: a CTA
// waits only for the words it reads, and within a cluster only for the bytes
// its mbarriers count.  Each depth's candidate data (W2 rows of the rank's
// bottleneck rows, GRU-input slices of the owned columns, base logits,
// h1_i(R), the rest log-partition) is copied with cp.async one depth ahead
// into the other of two stage buffers.  Every cluster must be resident at once
// (the CTAs wait on one another); dchain_plan picks JC (8 or 16) and CS (16
// down to 1) so that they are on the device at hand.  The Qwen3-4B shape runs
// an instantiation with every dimension a literal.
//
// A launch covers depths depth_first..depth_last.  Its first depth reads the
// previous depth's states from global fp32 buffers (or, at depth 1, computes
// the root state S_0 = GRU(E[t_0], 0) directly); a launch that stops before
// depth D leaves its states and live list there for the next one.  With
// fuse_tree, CTA 0 then runs the global Top-B and the tree/mask.
//
// Waits are bounded: a poll that sees no word for 2 s records DT_DEV_TIMEOUT,
// marks the launch aborted (other CTAs stop waiting when they see the mark)
// and the kernel runs to its end without further waits or writes, passing
// every cluster barrier, so that no CTA leaves while a peer may still read its
// shared memory.
#include <cstdio>

#include "common.cuh"
#include "kernels.h"
#include "chainlib.cuh"
#ifdef DT_DCHAIN_TIMING
// the Top-B / tree tail's inner phases: slot 0, phases 8.. of CTA 0's stamps
namespace dt {
__device__ unsigned long long g_topb_stamps[8];
}
#define TOPB_STAMP(k)                                                                          \
  do {                                                                                         \
    if (threadIdx.x == 0 && blockIdx.x == 0) dt::g_topb_stamps[k] = static_cast<unsigned long long>(clock64()); \
  } while (0)
#endif
#include "prune.cuh"

namespace dt {

namespace {

using namespace cl;

constexpr int kT = 256;          // threads
constexpr int kNW = kT / 32;     // warps
constexpr int kP = 8;            // live branches (state rows) at most
constexpr int kMP = 64;          // candidate slots (M <= 64)
constexpr int kNS = 2;           // stage buffers
constexpr int kMaxKW = 8;        // k16 steps of the state per warp: g <= 16 * kNW * kMaxKW
constexpr int kMaxT1 = 4;        // W1_S tiles per CTA: r / CS <= 32
constexpr int kMaxCS = 16;
constexpr int kMaxWords = 16;    // tagged state words polled per thread: g <= 1024

// ---------------------------------------------------------------- cluster PTX
DT_DEVINL uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
DT_DEVINL void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
DT_DEVINL void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
DT_DEVINL void cluster_sync() {
  cluster_arrive();
  cluster_wait();
}
// Address of `p` (a shared-memory variable of this CTA) in the shared memory
// of cluster rank `rank`.
DT_DEVINL uint32_t peer_addr(const void* p, uint32_t rank) {
  uint32_t a;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(a) : "r"(smem_u32(p)), "r"(rank));
  return a;
}
// 16 bytes into a peer's shared memory, completing their transaction bytes on
// the peer's mbarrier (both addresses from peer_addr): the writer needs no
// fence, the reader sees the data once that barrier's phase completes.
DT_DEVINL void st_async_f4(uint32_t a, float4 v, uint32_t mbar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];" ::"r"(a),
               "f"(v.x), "f"(v.y), "f"(v.z), "f"(v.w), "r"(mbar)
               : "memory");
}
// Named CTA barrier `id` over n threads: sync waits (and acquires), arrive
// only signals (and releases the caller's shared-memory writes).
DT_DEVINL void named_bar_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
DT_DEVINL void named_bar_arrive(int id, int n) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory"); }
DT_DEVINL bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.b32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// ---------------------------------------------------------------- tagged words
// Two 8-byte words, each (tag << 32 | payload): each word is written and read
// as one single-copy-atomic 64-bit access, so a reader that sees the tag also
// sees the payload stored with it.
DT_DEVINL void st_tagged(uint64_t* p, uint64_t a, uint64_t b) {
  asm volatile("st.relaxed.gpu.global.v2.u64 [%0], {%1, %2};" ::"l"(p), "l"(a), "l"(b) : "memory");
}
DT_DEVINL void ld_tagged(const uint64_t* p, uint64_t& a, uint64_t& b) {
  asm volatile("ld.relaxed.gpu.global.v2.u64 {%0, %1}, [%2];" : "=l"(a), "=l"(b) : "l"(p) : "memory");
}
DT_DEVINL unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
DT_DEVINL void st_relaxed_u32(unsigned* p, unsigned v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
DT_DEVINL uint32_t make_tag(uint32_t epoch, int depth) { return (epoch << 7) | static_cast<uint32_t>(depth); }

// Bounded wait on one of the exchange mbarriers, filled by peers' st.async:
// gives up (and marks the launch aborted) after the wait limit, or at once
// when another CTA has marked it.
DT_DEVINL bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, int* status, unsigned* abort_word, uint32_t epoch) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = dt_globaltimer();
  for (uint32_t n = 1;; ++n) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((n & 63u) == 0) {
      if (ld_relaxed_u32(abort_word) == epoch) return false;
      if (dt_globaltimer() - t0 > DT_WAIT_LIMIT_NS) {
        dt_report(status, DT_DEV_TIMEOUT);
        st_relaxed_u32(abort_word, epoch);
        return false;
      }
    }
  }
}

// Phase stamps (built with -DDT_DCHAIN_TIMING only): thread 0 of CTA 0 and of
// the last CTA records clock64() at the phase boundaries of every depth;
// dt_dchain_stamps copies them out.  Slot layout [CTA 0 / last][depth][phase].
#ifdef DT_DCHAIN_TIMING
constexpr int kStampPhases = 20;
__device__ unsigned long long g_dchain_stamps[2][kMaxDepth + 2][kStampPhases];
#define DCH_STAMP(depth, k)                                                                    \
  do {                                                                                         \
    if (tid == 0 && (cta == 0 || cta == L.G - 1))                                              \
      g_dchain_stamps[cta == 0 ? 0 : 1][depth][k] = static_cast<unsigned long long>(clock64()); \
  } while (0)
// and every CTA's thread 0 records %globaltimer when it has published a
// depth's states ([0][depth][cta]) and when it holds everyone's ([1][depth][cta])
constexpr int kXStampCtas = 128;
__device__ unsigned long long g_dchain_xstamps[2][kMaxDepth + 2][kXStampCtas];
#define DCH_XSTAMP(which, depth)                                                   \
  do {                                                                             \
    if (tid == 0 && cta < kXStampCtas) g_dchain_xstamps[which][depth][cta] = dt_globaltimer(); \
  } while (0)
#else
#define DCH_STAMP(depth, k) \
  do {                      \
  } while (0)
#define DCH_XSTAMP(which, depth) \
  do {                           \
  } while (0)
#endif

// acc += z[0..7] . w[0..7] for eight bf16 weights, in k order.
DT_DEVINL void fma8(float& acc, const float4& za, const float4& zb, const uint4& w8) {
  acc = fmaf(za.x, __uint_as_float(w8.x << 16), acc);
  acc = fmaf(za.y, __uint_as_float(w8.x & 0xFFFF0000u), acc);
  acc = fmaf(za.z, __uint_as_float(w8.y << 16), acc);
  acc = fmaf(za.w, __uint_as_float(w8.y & 0xFFFF0000u), acc);
  acc = fmaf(zb.x, __uint_as_float(w8.z << 16), acc);
  acc = fmaf(zb.y, __uint_as_float(w8.z & 0xFFFF0000u), acc);
  acc = fmaf(zb.z, __uint_as_float(w8.w << 16), acc);
  acc = fmaf(zb.w, __uint_as_float(w8.w & 0xFFFF0000u), acc);
}

// bf16 high and low parts of two values, packed as two bf16x2 words (the first
// value in the low half, as an mma.sync operand register holds its lower k).
DT_DEVINL uint2 hilo_pair(float a, float b) {
  uint32_t lo;
  const uint32_t hi = split_hi_lo(a, b, lo);
  return make_uint2(hi, lo);
}

// ---------------------------------------------------------------- layout
struct Lay {
  int G, RQ, nk16, gp, RQP, NT1, SW;
  size_t w, sfr, red1, red2, zfr, part, dls, recv, dlf, uhh, sown, stage, stage_sz, tok, child, misc, total;
  size_t st_xs, st_cbs, st_h1, st_rest;
};

DT_HOST_DEVICE_INLINE size_t a16(size_t x) { return (x + 15) & ~static_cast<size_t>(15); }

DT_HOST_DEVICE_INLINE Lay make_lay(int jc, int g, int r, int K, int D, int cs) {
  Lay L;
  L.G = g / jc;
  L.RQ = r / cs;
  L.nk16 = g / 16;
  L.gp = kstride(g);
  L.RQP = L.RQ + 8;
  L.NT1 = L.RQ / 8;
  L.SW = kMP / cs;  // candidates of one rank's slice of the correction
  size_t o = 0;
  auto put = [&](size_t& f, size_t b) {
    f = o;
    o += a16(b);
  };
  put(L.w, static_cast<size_t>(L.RQ + 3 * jc) * L.gp * 2);
  put(L.sfr, static_cast<size_t>(L.nk16) * 32 * 16);     // state A fragments [k16][row][tig]
  put(L.red1, static_cast<size_t>(kNW) * kP * L.RQ * 4);
  put(L.red2, static_cast<size_t>(kNW) * kP * 3 * jc * 4);
  put(L.zfr, static_cast<size_t>(kP) * L.RQ * 4);
  put(L.part, static_cast<size_t>(kP) * kMP * 4);        // the rank's partial correction [row][cand]
  put(L.dls, static_cast<size_t>(kP) * L.SW * 4);         // the reduced slice [row][SW]
  put(L.recv, static_cast<size_t>(cs) * kP * L.SW * 4);   // this rank's slice from every rank
  put(L.dlf, static_cast<size_t>(cs) * kP * L.SW * 4);    // every rank's reduced slice
  put(L.uhh, static_cast<size_t>(kP) * 3 * jc * 4);
  put(L.sown, static_cast<size_t>(2) * kP * jc * 4);
  size_t s = a16(static_cast<size_t>(kMP) * L.RQP * 2);  // W2 rows of the candidates
  L.st_xs = s;
  s += a16(static_cast<size_t>(kMP) * 3 * jc * 4);       // GRU-input slices
  L.st_cbs = s;
  s += a16(static_cast<size_t>(kMP) * 4);                // base logits
  L.st_h1 = s;
  s += a16(static_cast<size_t>(L.RQ) * 4);               // h1_i(R)
  L.st_rest = s;
  s += 16;                                               // rest log-partition
  L.stage_sz = s;
  put(L.stage, kNS * s);
  put(L.tok, static_cast<size_t>(D) * kMP * 4);
  put(L.child, static_cast<size_t>(2) * kP * K * 16);  // two depths' children
  put(L.misc, 256);
  L.total = o;
  return L;
}

// Shared memory of the Top-B / tree tail (CTA 0 after the depth loop, when all
// of its shared memory is free).
DT_HOST_DEVICE_INLINE size_t tail_bytes(int N1, int B) {
  const size_t S = static_cast<size_t>(B) + 1;
  return a16((static_cast<size_t>(kMaxDepth) + 2 + 3 * S + S * anc_words(static_cast<int>(S))) * 4) +
         a16(static_cast<size_t>(N1 - 1) * 8) + a16(static_cast<size_t>(N1 - 1) * 4) + kNW * 256 * 4 +
         3 * a16(static_cast<size_t>(N1) * 4) + a16(static_cast<size_t>(B) * 4);  // node scores, parents and
                                                                                   // tokens; the selection
}
// Node scores a tail thread loads into registers before the cluster barrier.
constexpr int kTailScores = 8;

struct Stage {
  uint16_t* w2;  // [kMP][RQP]
  float* xs;     // [kMP][3 JC]
  float* cbs;    // [kMP]
  float* h1;     // [RQ]
  float* rest;   // [1]
};

// The dimensions a launch runs with: read from the parameters, or, for the
// Qwen3-4B shape (g = 1024, r = 256, M = 64, K = W = 8, depth 15, clusters of
// 16), literals, so that index arithmetic folds and guarded loops vanish.
struct DcShape {
  int g, r, M, K, W, D, cs;
};
struct DcRuntime {
  static DT_DEVINL DcShape get(const DchainParams& p) { return DcShape{p.g, p.r, p.M, p.K, p.W, p.D, p.cs}; }
};
struct DcQ4B {
  static constexpr DcShape kShape{1024, 256, 64, 8, 8, 15, 16};
  static DT_DEVINL DcShape get(const DchainParams&) { return kShape; }
};
DT_HOST_DEVICE_INLINE bool is_q4b(const DchainParams& p) {
  return p.jc == 16 && p.g == 1024 && p.r == 256 && p.M == 64 && p.K == 8 && p.W == 8 && p.D == 15 && p.cs == 16;
}

template <int JC, class Dm>
__global__ void __launch_bounds__(kT, 1) k_dchain(const DchainParams p) {
  extern __shared__ __align__(16) uint8_t sm[];
  __shared__ int s_abort;
  __shared__ int s_wcnt[kNW];
  __shared__ uint32_t s_state[4];
  __shared__ float s_tred[64];
  __shared__ int s_tscan[40];
  __shared__ __align__(8) uint64_t s_mbar[2];  // the two rounds of the cluster's correction exchange
  __shared__ __align__(8) uint64_t s_mbar_w;   // the resident weights' bulk copies
  constexpr int kHP = JC / 2;      // column pairs per CTA
  constexpr int kT2 = 3 * JC / 8;  // W_hh tiles per CTA
  constexpr int kWP = kP * kHP;    // 16-byte words one CTA publishes per depth

  const DcShape shp = Dm::get(p);
  const int g = shp.g, r = shp.r, M = shp.M, K = shp.K, W = shp.W, D = shp.D, cs = shp.cs;
  const Lay L = make_lay(JC, g, r, K, D, cs);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t q = cluster_rank();
  const int cta = static_cast<int>(blockIdx.x);
  const int j0 = cta * JC;
  const int r0 = static_cast<int>(q) * L.RQ;
  const int gp = L.gp, RQ = L.RQ, RQP = L.RQP, SW = L.SW;

  uint16_t* w_s = reinterpret_cast<uint16_t*>(sm + L.w);
  uint4* sfr = reinterpret_cast<uint4*>(sm + L.sfr);
  float* red1 = reinterpret_cast<float*>(sm + L.red1);
  float* red2 = reinterpret_cast<float*>(sm + L.red2);
  float* zs = reinterpret_cast<float*>(sm + L.zfr);  // z of the rank's rows [kP][RQ]
  float* part = reinterpret_cast<float*>(sm + L.part);
  float* dls = reinterpret_cast<float*>(sm + L.dls);
  float* recv = reinterpret_cast<float*>(sm + L.recv);
  float* dlf = reinterpret_cast<float*>(sm + L.dlf);
  float* uhh = reinterpret_cast<float*>(sm + L.uhh);
  float* sown = reinterpret_cast<float*>(sm + L.sown);  // [2][kP][JC], by depth parity
  int* tok_all = reinterpret_cast<int*>(sm + L.tok);
  // children of a depth (token, candidate index, log-prob, score), by depth
  // parity: CTA 0 writes a depth's node arrays once it has published the
  // depth's states (every CTA waits for CTA 0's words, so work before that
  // would delay the whole grid)
  int* const child0 = reinterpret_cast<int*>(sm + L.child);
  auto child_tok = [&](int par) { return child0 + par * 4 * kP * K; };
  auto child_slot = [&](int par) { return child0 + par * 4 * kP * K + kP * K; };
  auto child_logp = [&](int par) { return reinterpret_cast<float*>(child0 + par * 4 * kP * K + 2 * kP * K); };
  auto child_score = [&](int par) { return reinterpret_cast<float*>(child0 + par * 4 * kP * K + 3 * kP * K); };
  int* surv = reinterpret_cast<int*>(sm + L.misc);           // [kP]
  int* pnode = surv + kP;                                     // [2][kP] live node indices, by depth parity
  float* pscore = reinterpret_cast<float*>(pnode + 2 * kP);  // [2][kP] their scores
  // node arrays of depth dep from its children (CTA 0)
  auto write_nodes = [&](int dep) {
    const int par = dep & 1, nch = p.L[dep - 1] * K, off = p.off[dep];
    const int* pt = child_tok(par);
    const float* pl = child_logp(par);
    const float* ps = child_score(par);
    const int* pn = pnode + ((dep - 1) & 1) * kP;
    for (int e = tid; e < nch; e += kT) {
      const size_t nidx = static_cast<size_t>(off) + e;
      p.node_tok[nidx] = pt[e];
      p.node_parent[nidx] = pn[e / K];
      p.node_logp[nidx] = pl[e];
      p.node_score[nidx] = ps[e];
    }
  };
  auto stage = [&](int depth) -> Stage {
    uint8_t* b = sm + L.stage + static_cast<size_t>(depth % kNS) * L.stage_sz;
    return Stage{reinterpret_cast<uint16_t*>(b), reinterpret_cast<float*>(b + L.st_xs),
                 reinterpret_cast<float*>(b + L.st_cbs), reinterpret_cast<float*>(b + L.st_h1),
                 reinterpret_cast<float*>(b + L.st_rest)};
  };

  if (tid == 0) {
    s_abort = 0;
    mbar_init(&s_mbar[0], 1);
    mbar_init(&s_mbar[1], 1);
    mbar_init(&s_mbar_w, 1);
    fence_mbar_init();
  }
  uint32_t mb_phase = 0;
  DCH_STAMP(0, 0);

  // ---- resident weights: rows 0..RQ-1 = W1_S(R), rows RQ.. = W_hh gate rows
  // of J, one bulk copy of g bf16 per row (all in flight at once; waited for
  // before the first projection) ----
  {
    const int nrow = RQ + 3 * JC;
    if (tid == 0) {
      mbar_arrive_expect_tx(&s_mbar_w, static_cast<uint32_t>(nrow * g * 2));
      for (int row = 0; row < nrow; ++row) {
        const uint16_t* src;
        if (row < RQ) {
          src = p.w1 + static_cast<size_t>(r0 + row) * p.ldw1 + p.d;
        } else {
          const int rr = row - RQ, gate = rr / JC, jj = rr - gate * JC;
          src = p.w_hh + static_cast<size_t>(gate * g + j0 + jj) * g;
        }
        bulk_g2s(w_s + static_cast<size_t>(row) * gp, src, static_cast<uint32_t>(g * 2), &s_mbar_w);
      }
    }
    // candidate slots beyond M hold zero W2 rows in every stage buffer
    for (int s = 0; s < kNS; ++s) {
      uint16_t* w2 = stage(s).w2;
      for (int idx = tid; idx < (kMP - M) * RQP; idx += kT) w2[static_cast<size_t>(M) * RQP + idx] = 0;
    }
  }

  // ---- the states entering the launch's first depth, in every CTA (none of
  // it is written by the kernels this launch may overlap: the root token and
  // the GRU-input table are inputs; a previous launch of this kernel ended
  // before this one started) ----
  const int f0 = p.depth_first;
  {
    const int pf = (f0 - 1) & 1;
    float* sw = sown + pf * kP * JC;
    if (f0 == 1) {
      // root: S_0 = GRU(E[t_0], 0) = (1 - sigmoid(x_z)) tanh(x_n), x = X[t_0]
      int t0 = p.root_tok[0];
      if (t0 < 0 || t0 >= p.V) {
        dt_report(p.status, DT_DEV_BOUNDS);
        t0 = 0;
      }
      const float* x = p.xtab + static_cast<size_t>(t0) * 3 * g;
      auto root_state = [&](int j) { return (1.0f - sigmoidf_(x[g + j])) * tanhf_(x[2 * g + j]); };
      for (int idx = tid; idx < kP * JC; idx += kT) sw[idx] = idx < JC ? root_state(j0 + idx) : 0.0f;
      for (int idx = tid; idx < L.nk16 * 32; idx += kT) {
        const int kt = idx >> 5, row = (idx >> 2) & 7, tg = idx & 3;
        const int k0 = 16 * kt + 2 * tg;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row == 0) {
          const uint2 a = hilo_pair(root_state(k0), root_state(k0 + 1));
          const uint2 b = hilo_pair(root_state(k0 + 8), root_state(k0 + 9));
          v = make_uint4(a.x, a.y, b.x, b.y);
        }
        sfr[idx] = v;
      }
      if (tid == 0) {
        pnode[0] = 0;
        pscore[0] = 0.0f;
      }
      if (cta == 0 && tid == 0) {
        p.node_tok[0] = t0;
        p.node_parent[0] = -1;
        p.node_logp[0] = 0.0f;
        p.node_score[0] = 0.0f;
      }
    } else {
      // from the previous launch: fp32 states and the live list of depth f0-1
      const int Lp = p.L[f0 - 1];
      const float* Sg = p.S + static_cast<size_t>(pf) * W * g;
      for (int idx = tid; idx < kP * JC; idx += kT) {
        const int w = idx / JC, jj = idx - w * JC;
        sw[idx] = w < Lp ? Sg[static_cast<size_t>(w) * g + j0 + jj] : 0.0f;
      }
      for (int idx = tid; idx < L.nk16 * 32; idx += kT) {
        const int kt = idx >> 5, row = (idx >> 2) & 7, tg = idx & 3;
        const int k0 = 16 * kt + 2 * tg;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < Lp) {
          const float* s = Sg + static_cast<size_t>(row) * g;
          const uint2 a = hilo_pair(s[k0], s[k0 + 1]);
          const uint2 b = hilo_pair(s[k0 + 8], s[k0 + 9]);
          v = make_uint4(a.x, a.y, b.x, b.y);
        }
        sfr[idx] = v;
      }
      for (int w = tid; w < Lp; w += kT) {
        int node = p.live[pf * W + w];
        if (node < 0 || node >= p.N1) {
          dt_report(p.status, DT_DEV_BOUNDS);
          node = 0;
        }
        pnode[pf * kP + w] = node;
        pscore[pf * kP + w] = p.node_score[node];
      }
    }
  }

  // the epoch: the previous launch of this kernel ended before this one started
  const uint32_t E = ld_relaxed_u32(p.epoch) + 1u;
  uint64_t* xch = reinterpret_cast<uint64_t*>(p.xch);
  const int nwords = L.G * kWP;                      // every CTA's words
  bool aborted = false;
  // the peers' barriers are initialised before anyone pushes into them; the
  // resident weights have landed
  cluster_sync();
  if (!mbar_wait(&s_mbar_w, 0, p.status)) {
    st_relaxed_u32(p.abort_word, E);
    aborted = true;
  }

  // everything below reads the previous kernels' results
  DCH_STAMP(0, 4);
  dt_grid_wait();
  DCH_STAMP(0, 5);

  // stage the candidate data of one depth with threads t0 .. t0 + nt - 1 (one
  // cp.async group each, possibly empty); tok(c) gives candidate c's token
  auto stage_with = [&](int i, int t0, int nt, auto tok) {
    const int t = tid - t0;
    if (i <= p.depth_last) {
      const Stage b = stage(i);
      const int r8 = RQ / 8;
      for (int idx = t; idx < M * r8; idx += nt) {
        const int c = idx / r8, k8 = idx - c * r8;
        cp_async16(b.w2 + static_cast<size_t>(c) * RQP + 8 * k8, p.w2 + static_cast<size_t>(tok(c)) * r + r0 + 8 * k8);
      }
      constexpr int kQ4 = JC / 4;  // 16-byte pieces of one gate's owned columns
      for (int idx = t; idx < M * 3 * kQ4; idx += nt) {
        const int c = idx / (3 * kQ4), rem = idx - c * 3 * kQ4, gate = rem / kQ4, h = rem - gate * kQ4;
        cp_async16(b.xs + c * 3 * JC + gate * JC + 4 * h,
                   p.xtab + static_cast<size_t>(tok(c)) * 3 * g + gate * g + j0 + 4 * h);
      }
      for (int c = t; c < M; c += nt) cp_async4(b.cbs + c, p.cand_base + static_cast<size_t>(i - 1) * M + c);
      for (int k4 = t; k4 < RQ / 4; k4 += nt)
        cp_async16(b.h1 + 4 * k4, p.h1 + static_cast<size_t>(i - 1) * r + r0 + 4 * k4);
      if (t == 0) cp_async4(b.rest, p.rest_lse + (i - 1));
    }
    cp_async_commit();
  };
  auto stage_depth = [&](int i, int t0, int nt) {
    const int* tk = tok_all + (i - 1) * kMP;
    stage_with(i, t0, nt, [&](int c) {
      int t = tk[c];
      if (t < 0 || t >= p.V) {
        dt_report(p.status, DT_DEV_BOUNDS);
        t = 0;
      }
      return t;
    });
  };
  auto checked_tok = [&](int idx) {
    int t = p.cand_tok[idx];
    if (t < 0 || t >= p.V) {
      dt_report(p.status, DT_DEV_BOUNDS);
      t = 0;
    }
    return t;
  };
  // the first depth's candidate data straight from its tokens, one round trip
  // sooner: thread c < M holds candidate c's token and copies its rows
  {
    const int tf = tid < M ? checked_tok((f0 - 1) * M + tid) : 0;
    if (tid < M) {
      const Stage b = stage(f0);
      for (int k8 = 0; k8 < RQ / 8; ++k8)
        cp_async16(b.w2 + static_cast<size_t>(tid) * RQP + 8 * k8, p.w2 + static_cast<size_t>(tf) * r + r0 + 8 * k8);
#pragma unroll
      for (int gate = 0; gate < 3; ++gate)
#pragma unroll
        for (int h = 0; h < JC / 4; ++h)
          cp_async16(b.xs + tid * 3 * JC + gate * JC + 4 * h,
                     p.xtab + static_cast<size_t>(tf) * 3 * g + gate * g + j0 + 4 * h);
      cp_async4(b.cbs + tid, p.cand_base + static_cast<size_t>(f0 - 1) * M + tid);
    } else if (tid - M < RQ / 4) {
      const Stage b = stage(f0);
      cp_async16(b.h1 + 4 * (tid - M), p.h1 + static_cast<size_t>(f0 - 1) * r + r0 + 4 * (tid - M));
    } else if (tid == kT - 1) {
      cp_async4(stage(f0).rest, p.rest_lse + (f0 - 1));
    }
    // every depth's tokens into shared memory for the later stagings, copied in
    // the same group (the first depth waits for it; its barriers show the
    // tokens to every thread; the stagings check them)
    for (int idx = tid; idx < D * M; idx += kT) cp_async4(tok_all + (idx / M) * kMP + idx % M, p.cand_tok + idx);
    cp_async_commit();
  }

  const int nkw = (L.nk16 - warp + kNW - 1) / kNW;  // k16 steps of this warp (kt = warp + kNW m)
  // lambda = (base + dL) / T as a product with 1/T (exact at T = 1; within an
  // ulp of the quotient otherwise)
  const float invT = 1.0f / p.T;

  for (int i = f0; i <= p.depth_last; ++i) {
    const int Lp = p.L[i - 1];  // live branches entering this depth
    const int Li = p.L[i];      // branches that live on
    const int ip = (i - 1) & 1, in = i & 1;
    const bool last = i == D;
    int* ctok = child_tok(in);
    int* cslot = child_slot(in);
    float* clogp = child_logp(in);
    float* cscore = child_score(in);

    DCH_STAMP(i, 0);
    if (i > f0) __syncthreads();
    // ================= X: the previous depth's states from every CTA =========
    // the words are laid out as the fragments themselves: word w is uint2 w of
    // the A-fragment array (k16 step, row, lane group, half), so a word that
    // carries its tag is stored as it is
    if (i > f0) {
      if (!aborted) {
        const uint32_t tag = make_tag(E, i - 1);
        const uint64_t* src = xch + static_cast<size_t>(ip) * nwords * 2 + static_cast<size_t>(tid) * 2;
        uint2* dst = reinterpret_cast<uint2*>(sfr) + tid;
        uint64_t e0[kMaxWords], e1[kMaxWords];
        unsigned pending = 0;
#pragma unroll
        for (int j = 0; j < kMaxWords; ++j) {
          if (tid + kT * j < nwords) {
            ld_tagged(src + static_cast<size_t>(kT) * 2 * j, e0[j], e1[j]);
            pending |= 1u << j;
          }
        }
        DCH_STAMP(i, 16);
        uint64_t t0 = 0;
        uint32_t n = 0;
        const uint64_t tag2 = static_cast<uint64_t>(tag) << 32;
        while (pending) {
#pragma unroll
          for (int j = 0; j < kMaxWords; ++j) {
            if ((pending >> j) & 1u) {
              if (((e0[j] & e1[j]) >> 32 << 32) == tag2 && ((e0[j] | e1[j]) >> 32 << 32) == tag2) {
                dst[kT * j] = make_uint2(static_cast<uint32_t>(e0[j]), static_cast<uint32_t>(e1[j]));
                pending &= ~(1u << j);
              }
            }
          }
          if (!pending) break;
          if (t0 == 0) t0 = dt_globaltimer();
          if ((++n & 15u) == 0) {
            if (ld_relaxed_u32(p.abort_word) == E) {
              aborted = true;
              break;
            }
            if (dt_globaltimer() - t0 > DT_WAIT_LIMIT_NS) {
              dt_report(p.status, DT_DEV_TIMEOUT);
              st_relaxed_u32(p.abort_word, E);
              aborted = true;
              break;
            }
          }
#pragma unroll
          for (int j = 0; j < kMaxWords; ++j)
            if (pending & (1u << j)) ld_tagged(src + static_cast<size_t>(kT) * 2 * j, e0[j], e1[j]);
        }
        if (aborted) s_abort = 1;
      }
      DCH_STAMP(i, 17);
      __syncthreads();
      aborted = s_abort != 0;
      DCH_XSTAMP(1, i - 1);
    }
    // this depth's candidate data (issued a depth ago) has landed; the
    // barrier after A1 shows it to every thread
    cp_async_wait_all();
    const Stage st = stage(i);

    DCH_STAMP(i, 1);
    // ================= A1: u_R = S W1_S(R)^T =================================
    uint4 f[kMaxKW];
#pragma unroll
    for (int m = 0; m < kMaxKW; ++m) f[m] = m < nkw ? sfr[(warp + kNW * m) * 32 + lane] : make_uint4(0u, 0u, 0u, 0u);
    {
      // four accumulators per tile (k16 steps m mod 4): a dependent mma.sync
      // costs ~200 cycles, so short chains matter more than the extra adds
      float acc[kMaxT1][4][4];
#pragma unroll
      for (int nt = 0; nt < kMaxT1; ++nt)
#pragma unroll
        for (int a4 = 0; a4 < 4; ++a4)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][a4][e] = 0.0f;
#pragma unroll
      for (int m = 0; m < kMaxKW; ++m) {
        if (m < nkw) {
          const int k0 = (warp + kNW * m) * 16 + 2 * tig;
#pragma unroll
          for (int nt = 0; nt < kMaxT1; ++nt) {
            if (nt < L.NT1) {
              const uint16_t* wc = w_s + static_cast<size_t>(nt * 8 + gid) * gp + k0;
              mma_bf16_16816(acc[nt][m & 3], f[m].x, f[m].y, f[m].z, f[m].w, *reinterpret_cast<const uint32_t*>(wc),
                             *reinterpret_cast<const uint32_t*>(wc + 8));
            }
          }
        }
      }
      DCH_STAMP(i, 11);
#pragma unroll
      for (int nt = 0; nt < kMaxT1; ++nt) {
        if (nt < L.NT1) {
          float s4[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) s4[e] = (acc[nt][0][e] + acc[nt][1][e]) + (acc[nt][2][e] + acc[nt][3][e]);
          float* rw = red1 + (warp * kP + gid) * RQ + nt * 8 + 2 * tig;
          rw[0] = s4[0] + s4[2];
          rw[1] = s4[1] + s4[3];
        }
      }
      DCH_STAMP(i, 12);
    }
    __syncthreads();
    DCH_STAMP(i, 13);
    // z = SiLU(h1_i + u) of every state row (fp32)
    for (int idx = tid; idx < kP * RQ; idx += kT) {
      const int pr = idx / RQ, k = idx - pr * RQ;
      float u = 0.0f;
#pragma unroll
      for (int w8 = 0; w8 < kNW; ++w8) u += red1[(w8 * kP + pr) * RQ + k];
      zs[idx] = siluf_(st.h1[k] + u);
    }
    __syncthreads();
    DCH_STAMP(i, 2);
    // ================= A2: the rank's partial correction =====================
    // dL_q[row][c] = sum_k z[row][k] W2[c][k] over the rank's rows, fp32 FMAs
    // in k order: thread t takes row t/32 and candidates 2 (t mod 32), +1
    {
      const int row = tid >> 5, c = 2 * lane;
      const float* zr = zs + row * RQ;
      const uint16_t* w0 = st.w2 + static_cast<size_t>(c) * RQP;
      const uint16_t* w1r = w0 + RQP;
      float a0 = 0.0f, a1 = 0.0f;
      for (int k8 = 0; k8 < RQ / 8; ++k8) {
        const float4 za = *reinterpret_cast<const float4*>(zr + 8 * k8);
        const float4 zb = *reinterpret_cast<const float4*>(zr + 8 * k8 + 4);
        fma8(a0, za, zb, *reinterpret_cast<const uint4*>(w0 + 8 * k8));
        fma8(a1, za, zb, *reinterpret_cast<const uint4*>(w1r + 8 * k8));
      }
      *reinterpret_cast<float2*>(part + row * kMP + c) = make_float2(a0, a1);
    }
    if (tid == 0) {
      // this depth's phases of the two exchange barriers (the previous ones
      // completed during the previous depth)
      mbar_arrive_expect_tx(&s_mbar[0], static_cast<uint32_t>((cs - 1) * kP * SW * 4));
      mbar_arrive_expect_tx(&s_mbar[1], static_cast<uint32_t>((cs - 1) * kP * SW * 4));
    }
    __syncthreads();
    // ---- reduce-scatter, round 1: slice s of the partial to rank s ----
    // thread t < 128: slice s = t / (2 SW), row, float4 f4 of the slice; the
    // rank's own slice is copied locally
    if (tid < 128) {
      const int nf4 = SW / 4, s = tid / (kP * nf4), rem = tid - s * kP * nf4, row = rem / nf4, f4 = rem - row * nf4;
      const float4 v = *reinterpret_cast<const float4*>(part + row * kMP + s * SW + 4 * f4);
      float* dst = recv + (static_cast<int>(q) * kP + row) * SW + 4 * f4;
      if (s == static_cast<int>(q)) *reinterpret_cast<float4*>(dst) = v;
      else st_async_f4(peer_addr(dst, static_cast<uint32_t>(s)), v, peer_addr(&s_mbar[0], static_cast<uint32_t>(s)));
    }
    DCH_STAMP(i, 3);
    // ================= A3: u_J = S W_hh(J)^T =================================
    {
      // two accumulators per tile (k16 steps m mod 2)
      float acc[kT2][2][4];
#pragma unroll
      for (int nt = 0; nt < kT2; ++nt)
#pragma unroll
        for (int a2 = 0; a2 < 2; ++a2)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][a2][e] = 0.0f;
#pragma unroll
      for (int m = 0; m < kMaxKW; ++m) {
        if (m < nkw) {
          const int k0 = (warp + kNW * m) * 16 + 2 * tig;
#pragma unroll
          for (int nt = 0; nt < kT2; ++nt) {
            const uint16_t* wc = w_s + static_cast<size_t>(RQ + nt * 8 + gid) * gp + k0;
            mma_bf16_16816(acc[nt][m & 1], f[m].x, f[m].y, f[m].z, f[m].w, *reinterpret_cast<const uint32_t*>(wc),
                           *reinterpret_cast<const uint32_t*>(wc + 8));
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < kT2; ++nt) {
        float* rw = red2 + (warp * kP + gid) * 3 * JC + nt * 8 + 2 * tig;
        rw[0] = (acc[nt][0][0] + acc[nt][1][0]) + (acc[nt][0][2] + acc[nt][1][2]);
        rw[1] = (acc[nt][0][1] + acc[nt][1][1]) + (acc[nt][0][3] + acc[nt][1][3]);
      }
    }
    __syncthreads();
    for (int idx = tid; idx < kP * 3 * JC; idx += kT) {
      const int pr = idx / (3 * JC), c = idx - pr * 3 * JC;
      float u = 0.0f;
#pragma unroll
      for (int w8 = 0; w8 < kNW; ++w8) u += red2[(w8 * kP + pr) * 3 * JC + c];
      uhh[idx] = u;
    }
    DCH_STAMP(i, 4);
    // ================= R: the rest of the cluster's reduction ================
    // round 1 landed: this rank's slice from every peer, added in rank order
    if (!mbar_wait_cluster(&s_mbar[0], mb_phase, p.status, p.abort_word, E)) aborted = true;
    __syncthreads();
    for (int idx = tid; idx < kP * SW; idx += kT) {
      float v = 0.0f;
      for (int q2 = 0; q2 < cs; ++q2) v += recv[q2 * kP * SW + idx];
      dls[idx] = v;
    }
    __syncthreads();
    // round 2: the reduced slice to every rank (all-gather), own copy local
    if (tid < cs * kP * (SW / 4)) {
      const int nf4 = SW / 4, s = tid / (kP * nf4), rem = tid - s * kP * nf4;
      const float4 v = *reinterpret_cast<const float4*>(dls + 4 * rem);
      float* dst = dlf + (static_cast<int>(q) * kP * SW) + 4 * rem;
      if (s == static_cast<int>(q)) *reinterpret_cast<float4*>(dst) = v;
      else st_async_f4(peer_addr(dst, static_cast<uint32_t>(s)), v, peer_addr(&s_mbar[1], static_cast<uint32_t>(s)));
    }
    if (!mbar_wait_cluster(&s_mbar[1], mb_phase, p.status, p.abort_word, E)) aborted = true;
    mb_phase ^= 1u;
    __syncthreads();
    DCH_STAMP(i, 5);

    // ================= B: corrected log-probs and selections ================
    const int* tk = tok_all + (i - 1) * kMP;
    const float rest = st.rest[0];
    const int row_off = p.off[i];
    const int nchild = Lp * K;
    if (warp < Lp) {
      const int b = warp;
      // candidates 2 lane, 2 lane + 1: slice (2 lane) / SW, reduced by that rank
      const int c0 = 2 * lane, owner = c0 / SW;
      const float2 dl = *reinterpret_cast<const float2*>(dlf + (owner * kP + b) * SW + (c0 - owner * SW));
      float lam[2];
      uint64_t key[2];
      lam[0] = c0 < M ? (st.cbs[c0] + dl.x) * invT : -INFINITY;
      lam[1] = c0 + 1 < M ? (st.cbs[c0 + 1] + dl.y) * invT : -INFINITY;
      key[0] = c0 < M ? cand_key(lam[0], tk[c0], c0) : 0ull;
      key[1] = c0 + 1 < M ? cand_key(lam[1], tk[c0 + 1], c0 + 1) : 0ull;
      DCH_STAMP(i, 15);
      // the K best keys in descending order: K rounds of two warp max
      // reductions (value part, then the (token, candidate) part among the
      // elements that reach the maximum value; keys are distinct, so exactly
      // one element wins); the winner of round w is kept by lane w.  Round 0
      // gives the largest lambda, and the rounds after it carry the butterfly
      // levels of the log-partition's sum (offsets 16, 8, 4, 2, 1)
      uint32_t ha = static_cast<uint32_t>(key[0] >> 32), la = static_cast<uint32_t>(key[0]);
      uint32_t hb = static_cast<uint32_t>(key[1] >> 32), lb = static_cast<uint32_t>(key[1]);
      uint64_t wk = 0ull;
      float lmax = 0.0f, se = 0.0f;
      int lev = 0;
      for (int w = 0; w < K; ++w) {
        const uint32_t gh = __reduce_max_sync(0xFFFFFFFFu, ha > hb ? ha : hb);
        if (w == 0) {
          lmax = fmaxf(rest, key_f32(gh));
          se = (c0 < M ? expf(lam[0] - lmax) : 0.0f) + (c0 + 1 < M ? expf(lam[1] - lmax) : 0.0f);
        } else if (lev < 5) {
          se += __shfl_xor_sync(0xFFFFFFFFu, se, 16 >> lev);
          ++lev;
        }
        const uint32_t mla = ha == gh ? la : 0u, mlb = hb == gh ? lb : 0u;
        const uint32_t gl = __reduce_max_sync(0xFFFFFFFFu, mla > mlb ? mla : mlb);
        if (ha == gh && la == gl) {
          ha = 0u;
          la = 0u;
        } else if (hb == gh && lb == gl) {
          hb = 0u;
          lb = 0u;
        }
        if (lane == w) wk = (static_cast<uint64_t>(gh) << 32) | gl;
      }
      for (; lev < 5; ++lev) se += __shfl_xor_sync(0xFFFFFFFFu, se, 16 >> lev);
      se += expf(rest - lmax);
      const float logZ = lmax + logf(se);
      DCH_STAMP(i, 6);
      const int tok = lane < K ? cand_key_tok(wk) : 0x7FFFFFFF;
      int trank = 0;
      for (int m0 = 0; m0 < K; m0 += 8) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int t2 = __shfl_sync(0xFFFFFFFFu, tok, (m0 + j) & 31);
          trank += (m0 + j < K && t2 < tok) ? 1 : 0;
        }
      }
      if (lane < K) {
        const float lp = key_f32(static_cast<uint32_t>(wk >> 32)) - logZ;
        const int slot = b * K + trank;
        ctok[slot] = tok;
        cslot[slot] = cand_key_c(wk);
        clogp[slot] = lp;
        cscore[slot] = pscore[ip * kP + b] + lp;
      }
      DCH_STAMP(i, 7);
    }
    __syncthreads();
    DCH_STAMP(i, 8);
    if (last) {
      if (cta == 0 && p.live_out)
        for (int j = tid; j < W; j += kT) p.live_out[j] = -1;
      break;
    }
    // top-W of the depth by (score desc, node index asc); survivors ascending.
    // Up to 64 children: warp 0 takes the Li best by rounds of two warp max
    // reductions over (score key, inverted index) and keeps them in its own
    // scratch (the only warp that reads them); more: ranks counted by the
    // block
    const bool spec = nchild <= 64;
    const int* sv = surv;
    if (spec) {
      if (warp == 0) {
        const int e0 = 2 * lane, e1 = 2 * lane + 1;
        uint32_t ha = e0 < nchild ? f32_key(cscore[e0]) : 0u, la = e0 < nchild ? 0xFFFFFFFFu - e0 : 0u;
        uint32_t hb = e1 < nchild ? f32_key(cscore[e1]) : 0u, lb = e1 < nchild ? 0xFFFFFFFFu - e1 : 0u;
        int mine = 0x7FFFFFFF;
        for (int w = 0; w < Li; ++w) {
          const uint32_t gh = __reduce_max_sync(0xFFFFFFFFu, ha > hb ? ha : hb);
          const uint32_t mla = ha == gh ? la : 0u, mlb = hb == gh ? lb : 0u;
          const uint32_t gl = __reduce_max_sync(0xFFFFFFFFu, mla > mlb ? mla : mlb);
          if (ha == gh && la == gl) {
            ha = 0u;
            la = 0u;
          } else if (hb == gh && lb == gl) {
            hb = 0u;
            lb = 0u;
          }
          if (lane == w) mine = static_cast<int>(0xFFFFFFFFu - gl);
        }
        DCH_STAMP(i, 14);
        int pos = 0;
#pragma unroll
        for (int m = 0; m < kP; ++m) {
          const int t2 = __shfl_sync(0xFFFFFFFFu, mine, m);
          pos += (m < Li && t2 < mine) ? 1 : 0;
        }
        int* ws = reinterpret_cast<int*>(red1);
        if (lane < Li) ws[pos] = mine;
        __syncwarp();
        sv = ws;
      }
    } else {
      // one thread per child (nchild <= kP * 32 = kT)
      const int e = tid;
      int rk = 0;
      if (e < nchild) {
        const float se = cscore[e];
#pragma unroll 4
        for (int f2 = 0; f2 < nchild; ++f2) {
          const float sf = cscore[f2];
          rk += (sf > se || (sf == se && f2 < e)) ? 1 : 0;
        }
      }
      const bool alive = e < nchild && rk < Li;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, alive);
      if (lane == 0) s_wcnt[warp] = __popc(bal);
      __syncthreads();
      if (alive) {
        int pos = __popc(bal & ((1u << lane) - 1u));
        for (int w2 = 0; w2 < warp; ++w2) pos += s_wcnt[w2];
        surv[pos] = e;
      }
      __syncthreads();
    }
    DCH_STAMP(i, 9);
    // ================= C: GRU update of the survivors' owned columns =========
    // Warps 1.. compute the new owned columns of every child (up to 64
    // children: while warp 0 still selects, their rows being ready when it
    // needs them) or of the survivors, into hrow [row][JC] (the A3 partial
    // sums' area, free since uhh); warp 0 then takes the survivors' rows,
    // publishes them and keeps them for the next depth.
    float* hrow = red2;
    if (warp == 0) {
      named_bar_sync(1, kT);  // the rows of warps 1..
      for (int t = lane; t < kWP; t += 32) {
        const int w = t / kHP, pair = t - w * kHP;
        float2 hn = make_float2(0.0f, 0.0f);
        if (w < Li) hn = *reinterpret_cast<const float2*>(hrow + (spec ? sv[w] : w) * JC + 2 * pair);
        *reinterpret_cast<float2*>(sown + (in * kP + w) * JC + 2 * pair) = hn;
        if (i < p.depth_last) {
          if (!aborted) {
            const uint2 hl = hilo_pair(hn.x, hn.y);
            const uint64_t tag = static_cast<uint64_t>(make_tag(E, i)) << 32;
            // word index = the fragment position of columns col, col + 1 of row w
            const int col = j0 + 2 * pair;
            const int wi = (((col >> 4) * 8 + w) * 4 + ((col & 7) >> 1)) * 2 + ((col & 15) >> 3);
            st_tagged(xch + (static_cast<size_t>(in) * nwords + wi) * 2, tag | hl.x, tag | hl.y);
          }
        } else if (w < Li && !aborted) {
          // the launch ends before depth D: fp32 states for the next launch
          float* Sg = p.S + static_cast<size_t>(in) * W * g + static_cast<size_t>(w) * g + j0 + 2 * pair;
          Sg[0] = hn.x;
          Sg[1] = hn.y;
        }
      }
      // the live list (read by the next depth, after its barriers)
      if (lane < kP) {
        const int w = lane;
        if (w < Li) {
          const int e = sv[w];
          pnode[in * kP + w] = row_off + e;
          pscore[in * kP + w] = cscore[e];
          if (cta == 0 && !aborted) {
            if (i == p.depth_last) p.live[in * W + w] = row_off + e;
            if (p.live_out) p.live_out[w] = row_off + e;
          }
        } else if (w < W && cta == 0 && p.live_out) {
          p.live_out[w] = -1;
        }
      }
    } else {
      const int nrows = spec ? nchild : Li;
      // at most kIt rows per thread; unrolled so that their loads and
      // activations overlap
      constexpr int kIt = (kMP * kHP + kT - 33) / (kT - 32);
#pragma unroll
      for (int it = 0; it < kIt; ++it) {
        const int idx = tid - 32 + it * (kT - 32);
        if (idx < nrows * kHP) {
          const int row = idx / kHP, pair = idx - row * kHP;
          const int e = spec ? row : surv[row], b = e / K;
          int c = cslot[e];
          if (c < 0 || c >= M) {
            dt_report(p.status, DT_DEV_BOUNDS);
            c = 0;
          }
          const float* x = st.xs + c * 3 * JC + 2 * pair;
          const float* uu = uhh + b * 3 * JC + 2 * pair;
          const float2 xr = *reinterpret_cast<const float2*>(x), xz = *reinterpret_cast<const float2*>(x + JC),
                       xn = *reinterpret_cast<const float2*>(x + 2 * JC);
          const float2 ur = *reinterpret_cast<const float2*>(uu), uz = *reinterpret_cast<const float2*>(uu + JC),
                       un = *reinterpret_cast<const float2*>(uu + 2 * JC);
          const float2 hp = *reinterpret_cast<const float2*>(sown + (ip * kP + b) * JC + 2 * pair);
          float2 hn;
          {
            const float rg = sigmoidf_(xr.x + ur.x), zg = sigmoidf_(xz.x + uz.x);
            const float ng = tanhf_(xn.x + rg * un.x);
            hn.x = (1.0f - zg) * ng + zg * hp.x;
          }
          {
            const float rg = sigmoidf_(xr.y + ur.y), zg = sigmoidf_(xz.y + uz.y);
            const float ng = tanhf_(xn.y + rg * un.y);
            hn.y = (1.0f - zg) * ng + zg * hp.y;
          }
          *reinterpret_cast<float2*>(hrow + row * JC + 2 * pair) = hn;
        }
      }
      named_bar_arrive(1, kT);
      // the next depth's candidate data, into the buffer depth i-1 used (every
      // thread has passed depth i-1: the barriers of this depth's X and A1)
      stage_depth(i + 1, 32, kT - 32);
    }
    DCH_XSTAMP(0, i);
    if (cta == 0 && !aborted) write_nodes(i);
    DCH_STAMP(i, 10);
    // (the next depth's barriers order these shared-memory writes)
  }

  DCH_STAMP(0, 1);
  // the node arrays of depth D (which ends after its selections)
  if (cta == 0 && !aborted && p.depth_last == D) write_nodes(D);
  // the tail's node scores: loads issued now, their latency hidden by the
  // cluster barrier (the block barrier makes depth D's writes visible)
  const bool tail = p.fuse_tree && cta == 0 && !aborted;
  const bool tail_pre = tail && p.N1 <= kTailScores * kT;
  float scv[kTailScores];
  int pav[kTailScores], tov[kTailScores];
  if (tail_pre) {
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kTailScores; ++k) {
      const int v = tid + k * kT;
      scv[k] = v < p.N1 ? __ldcg(p.node_score + v) : 0.0f;
      pav[k] = v < p.N1 ? __ldcg(p.node_parent + v) : 0;
      tov[k] = v < p.N1 ? __ldcg(p.node_tok + v) : 0;
    }
  }
  cp_async_wait_all();
  cluster_sync();  // no CTA leaves while a peer may read its shared memory
  // the next launch tags its words with a new epoch (also after an abort, so
  // that no word this launch left behind can match a later tag)
  if (cta == 0 && tid == 0) st_relaxed_u32(p.epoch, E);

  // ---- tail: global Top-B and tree/mask (CTA 0, which wrote every node array) ----
  if (tail) {
    __syncthreads();
    const int S = p.B + 1;
    int* offs = reinterpret_cast<int*>(sm);
    int* nodes = offs + (kMaxDepth + 2);
    int* par = nodes + S;
    int* dep = par + S;
    uint32_t* anc = reinterpret_cast<uint32_t*>(dep + S);
    uint8_t* t = sm + a16((static_cast<size_t>(kMaxDepth) + 2 + 3 * S + S * anc_words(S)) * 4);
    uint64_t* tb_cands = reinterpret_cast<uint64_t*>(t);
    uint32_t* tb_keys = reinterpret_cast<uint32_t*>(t + a16(static_cast<size_t>(p.N1 - 1) * 8));
    uint32_t* hist = tb_keys + a16(static_cast<size_t>(p.N1 - 1) * 4) / 4;
    const size_t n1b = a16(static_cast<size_t>(p.N1) * 4);
    float* sc_s = reinterpret_cast<float*>(hist + kNW * 256);                             // [N1]
    int* pa_s = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(sc_s) + n1b);           // [N1]
    int* to_s = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(pa_s) + n1b);           // [N1]
    int* sel_s = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(to_s) + n1b);          // [B]
    for (int k = tid; k <= D + 1; k += kT) offs[k] = p.off[k];
    if (tail_pre) {
#pragma unroll
      for (int k = 0; k < kTailScores; ++k)
        if (tid + k * kT < p.N1) {
          sc_s[tid + k * kT] = scv[k];
          pa_s[tid + k * kT] = pav[k];
          to_s[tid + k * kT] = tov[k];
        }
    }
    __syncthreads();
    DCH_STAMP(0, 6);
    topb_select(tail_pre ? sc_s : p.node_score, p.N1, p.B, p.beta, D, offs, tb_keys, tb_cands, p.N1 - 1, hist,
                kNW * 256, s_state, s_tred, s_tscan, p.sel, sel_s);
    DCH_STAMP(0, 7);
    tree_and_mask(sel_s, p.N1, p.B, D, offs, tail_pre ? to_s : p.node_tok, tail_pre ? pa_s : p.node_parent,
                  tail_pre ? sc_s : p.node_score, nullptr, nodes, par, dep, anc, p.tok, p.parent, p.depth, p.logp_cum,
                  p.mask, p.status);
  }
  DCH_STAMP(0, 2);
}

bool shape_ok(const DchainParams& p, int jc, int cs) {
  if (cs < 1 || cs > kMaxCS || (cs & (cs - 1)) != 0) return false;
  if (p.g % jc != 0 || p.g % 16 != 0) return false;
  const int G = p.g / jc;
  if (G % cs != 0) return false;
  const int nk16 = p.g / 16;
  if (nk16 > kNW * kMaxKW) return false;
  if (G * 4 * jc > kT * kMaxWords) return false;  // tagged words polled per thread
  if (p.r % cs != 0) return false;
  const int RQ = p.r / cs;
  if (RQ % 16 != 0 || RQ / 8 > kMaxT1) return false;
  return true;
}

const void* kernel_of(int jc) {
  return jc == 16 ? reinterpret_cast<const void*>(k_dchain<16, DcRuntime>)
                  : reinterpret_cast<const void*>(k_dchain<8, DcRuntime>);
}

}  // namespace

size_t dchain_smem_bytes(const DchainParams& p) { return make_lay(p.jc, p.g, p.r, p.K, p.D, p.cs).total; }

bool dchain_plan(DchainParams& p, int num_sms, char* why, size_t why_len) {
  auto say = [&](const char* fmt, int a, int b, int c2) {
    if (why && why_len) snprintf(why, why_len, fmt, a, b, c2);
  };
  if (p.W > kP || p.M > kMP || p.K > 32 || p.K > p.M || p.D < 1 || p.D > kMaxDepth - 1) {
    say("shape outside the clustered chain (W=%d, M=%d, K=%d)", p.W, p.M, p.K);
    return false;
  }
  say("no column split and cluster size fit (g=%d, r=%d, D=%d)", p.g, p.r, p.D);
  for (int jc : {8, 16}) {
    for (int cs : {16, 8, 4, 2, 1}) {
      if (!shape_ok(p, jc, cs) || p.g / jc > num_sms) continue;
      p.jc = jc;
      p.cs = cs;
      const Lay L = make_lay(jc, p.g, p.r, p.K, p.D, cs);
      if (L.total > 227 * 1024) continue;
      if (p.fuse_tree && tail_bytes(p.N1, p.B) > L.total) continue;
      // every cluster must be resident at once (the CTAs wait on one another)
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(L.G);
      cfg.blockDim = dim3(kT);
      cfg.dynamicSmemBytes = L.total;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = cs;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, kernel_of(jc), &cfg);
      if (e != cudaSuccess) {
        cudaGetLastError();
        continue;
      }
      if (n * cs >= L.G) {
        say("%d columns per CTA, clusters of %d, %d clusters resident at once", jc, cs, n);
        return true;
      }
    }
  }
  return false;
}

cudaError_t dchain_prepare() {
  for (const void* f : {kernel_of(8), kernel_of(16), reinterpret_cast<const void*>(k_dchain<16, DcQ4B>)}) {
    cudaError_t e = dt_allow_max_dynamic_smem(f);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(f, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_dchain(const DchainParams& p, cudaStream_t stream) {
  const Lay L = make_lay(p.jc, p.g, p.r, p.K, p.D, p.cs);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(L.G);
  cfg.blockDim = dim3(kT);
  cfg.dynamicSmemBytes = L.total;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.pdl ? 2 : 1;
  if (is_q4b(p)) return cudaLaunchKernelEx(&cfg, k_dchain<16, DcQ4B>, p);
  return p.jc == 16 ? cudaLaunchKernelEx(&cfg, k_dchain<16, DcRuntime>, p)
                    : cudaLaunchKernelEx(&cfg, k_dchain<8, DcRuntime>, p);
}

}  // namespace dt

#ifdef DT_DCHAIN_TIMING
// The phase stamps of the last clustered-chain launch: 2 x 66 x 20 clock64()
// values ([CTA 0 / last CTA][slot][phase]; slot 0: kernel start, end of the
// depth loop, end of the tail, before and after the wait for the previous
// kernel, before Top-B and before the tree; slot i: the starts of depth i's
// X, A1, A2, A3, R, B, B's sort, B's writes done, top-W, C, C's end, and the
// finer boundaries 11-17 inside A1, top-W, B and X).
// Returns the number of values copied, or -1.
extern "C" int dt_dchain_stamps(unsigned long long* out, int n) {
  const int total = 2 * (dt::kMaxDepth + 2) * dt::kStampPhases;
  if (!out || n < total) return -1;
  return cudaMemcpyFromSymbol(out, dt::g_dchain_stamps, sizeof(dt::g_dchain_stamps)) == cudaSuccess ? total : -1;
}
// The exchange stamps of the last launch, [published / received][depth][CTA]
// (%globaltimer, ns; CTAs beyond 128 are not recorded).  Returns the number of
// values copied, or -1.
// The tail's inner stamps of the last launch (CTA 0, clock64()): Top-B keys,
// histogram, bound bin, candidates, ranks; tree slots, parents, ancestors.
extern "C" int dt_dchain_topb_stamps(unsigned long long* out, int n) {
  if (!out || n < 8) return -1;
  return cudaMemcpyFromSymbol(out, dt::g_topb_stamps, sizeof(dt::g_topb_stamps)) == cudaSuccess ? 8 : -1;
}
extern "C" int dt_dchain_xstamps(unsigned long long* out, int n) {
  const int total = 2 * (dt::kMaxDepth + 2) * dt::kXStampCtas;
  if (!out || n < total) return -1;
  return cudaMemcpyFromSymbol(out, dt::g_dchain_xstamps, sizeof(dt::g_dchain_xstamps)) == cudaSuccess ? total : -1;
}
#endif

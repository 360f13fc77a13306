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
//   pre  the depth's Top-M candidate tokens (read once per launch), and their
//        base logits, W2 rows, GRU-input slices X[token][gates of J] and the
//        H-half h1_i of the bottleneck are copied to shared memory with
//        cp.async ahead of time, overlapping the barrier and phase A.
//   A    u = S(p) [W_hh(J gates) | W1_S(R)]^T for every live branch p: mma.sync
//        m16n8k16 on the resident K-major bf16 weight columns, with each fp32
//        state split into bf16 high + low parts (two products, fp32
//        accumulation); the W1_S part goes to global memory.
//   --   grid barrier
//   B    every CTA (identically): z = SiLU(h1_i + u_W1); lambda_c = (base_c +
//        z . W2[c]) / T on the Top-M candidates (one tensor-core product over
//        all branches); logp = lambda - logsumexp(rest, lambda); per-branch
//        top-K (ties to the lower token id: a register sort of packed keys for
//        M = 64, else K rounds of a warp argmax); children sorted by token id;
//        top-W of the depth by cumulative score (ties to the lower node index:
//        ranks counted by one warp or by the block, or a sorting network for
//        many children).  CTA 0 writes the node arrays and the live list.
//   C    GRU update of the survivors' state columns J:
//        r = sigmoid(x_r + u_r), z = sigmoid(x_z + u_z), n = tanh(x_n + r u_n),
//        h' = (1 - z) n + z h, with x = X[token] = E[token] W_ih^T + b_ih.
//   --   grid barrier
// Routes through the same kernel (fixed per launch by the shape):
//   one request, <= 8 live branches   phase A reads the states as ready-made
//        mma.sync A fragments from global memory (hi/lo parts in rows 0-7 /
//        8-15 of the tile: one MMA per k16 step), z is published the same way,
//        the next depth's candidate data is staged a depth ahead;
//   several requests                  phase A copies 8-state fragment blocks
//        whole into shared memory (one bulk copy each, two ahead); CTA c
//        selects for requests c, c + G, ... only, and after one more grid
//        barrier every CTA updates its columns of all requests' survivors;
//   one request, > 8 branches, SIMT phase B   CTA c scores branches c, c + G,
//        ... and writes their children into the node arrays; after one more
//        grid barrier every CTA reads them back for the top-W;
//   marginal scoring                  one CTA, no state, no correction.
// The kernel is instantiated twice over the same code: with every dimension
// fixed at compile time for the Qwen3-4B shape (index arithmetic folds to
// constants, loops unroll), and with dimensions read from the parameters.
// Every wait is bounded; on a timeout the kernel records DT_DEV_TIMEOUT and
// returns.
#include "common.cuh"
#include "kernels.h"
#include "chainlib.cuh"
#include "prune.cuh"

namespace dt {

namespace {

using namespace cl;

constexpr int kPC = 8;           // state rows per projection chunk
constexpr int kRankMax = 256;    // top-W by rank counting up to this many children (= kThreads)
constexpr int kMaxNTiles = 8;    // owned columns per CTA <= 64 (8-wide MMA tiles)
constexpr int kSLoads = 9;       // float4 state loads per thread: kPC*(g+24)/4/kThreads for g <= 1024
constexpr int kMaxR32 = 32;      // bottleneck values per lane: r <= 1024
constexpr int kZLoads = 16;      // z values per thread on the tensor-core path: W*r <= 4096
constexpr int kFragMax = 8;      // fragment loads per lane in phase A: g <= 16 * kWarps * kFragMax
constexpr int kZFragMax = 16;    // z fragment loads per lane in phase B: r <= 16 * kZFragMax

// Phase stamps (built with -DDT_CHAIN_TIMING only): thread 0 of CTA 0 and of
// the last CTA records clock64() at the phase boundaries of every depth;
// dt_chain_stamps copies them out.  Slot layout [CTA 0 / last][depth][phase]:
// 0 depth start, 1 phase A done, 2 past the barrier after A, 3 phase B done,
// 4 past the barrier before C (several requests), 5 phase C done, 6 past the
// depth's last barrier, 7 cycles spent waiting for state blocks in phase A;
// branches scored by different CTAs: 8 scoring done, 9 past the barrier after
// it; 10 children ready for the top-W, 11 top-W done; inside the scoring of
// the CTA's first branch: 12 start, 13 z, 14 corrected logits, 15 keys, 16
// the K best; 17 the top-W's threshold key.  g_chain_tcst: the tcgen05 phase
// A of depth 2 in CTA 0, per chunk: copy issued, data landed, slot freed.
#ifdef DT_CHAIN_TIMING
constexpr int kChainStamps = 20;
__device__ unsigned long long g_chain_stamps[2][kMaxDepth + 2][kChainStamps];
#define CH_STAMP(depth, k)                                                                       \
  do {                                                                                           \
    if (tid == 0 && (blockIdx.x == 0 || blockIdx.x == gridDim.x - 1))                            \
      g_chain_stamps[blockIdx.x == 0 ? 0 : 1][depth][k] = static_cast<unsigned long long>(clock64()); \
  } while (0)
__device__ unsigned long long g_chain_tcst[3][128];
#define CH_TCST(which, c, depth)                                                                  \
  do {                                                                                           \
    if (blockIdx.x == 0 && (depth) == 2 && (c) < 128)                                            \
      g_chain_tcst[which][c] = static_cast<unsigned long long>(clock64());                        \
  } while (0)
#define CH_STAMP_SET(depth, k, v)                                                                \
  do {                                                                                           \
    if (tid == 0 && (blockIdx.x == 0 || blockIdx.x == gridDim.x - 1))                            \
      g_chain_stamps[blockIdx.x == 0 ? 0 : 1][depth][k] = (v);                                   \
  } while (0)
#else
#define CH_STAMP(depth, k) \
  do {                     \
  } while (0)
#define CH_STAMP_SET(depth, k, v) \
  do {                            \
  } while (0)
#define CH_TCST(which, c, depth) \
  do {                           \
  } while (0)
#endif

// Dimensions a launch runs with (see chain_plan).
struct Shape {
  int g, r, M, K, W, n_req, D, jper, rper, cpad;
  bool stage_w2, mma_b, prefetch;
  // one request with prefetched tokens: depth i+1's candidate data is staged
  // at the start of depth i into a second buffer
  bool dbuf;
  // one request whose W state rows fit one A fragment: phase A reads the
  // states as ready-made fragments from global memory (sfrag)
  bool frag;
  // with frag and the tensor-core phase B: z is published as fragments by the
  // bottleneck-row owners (zfrag) instead of u_W1
  bool zf;
  // several requests (8-state blocks): phase A copies the states as
  // ready-made fragments block by block into shared memory
  bool mfrag;
  // one request, many branches, SIMT phase B: branches scored by different
  // CTAs; no GRU-input slices are staged (phase C reads the table)
  bool bdist;
  // phase A on tcgen05 (states streamed as 128-row A-operand chunks into ns
  // shared-memory slots, accumulators in tensor memory)
  bool tc;
  int ns;
};

// One shared-memory slot of the tcgen05 phase A: a streamed A-operand chunk
// of 128 (or 64) state rows x 64 bf16 (one part, high or low, of one K
// block), 128-byte swizzled.
constexpr int kTcChunk = 16384;
// Row tile of the tcgen05 phase A: 64 rows when every state row fits one
// (M = 64 products, half the bytes streamed), else 128.
DT_HOST_DEVICE_INLINE int tc_tile_shift(int rows) { return rows <= 64 ? 6 : 7; }

DT_HOST_DEVICE_INLINE bool frag_ok(int n_req, int W, int g) {
  return n_req == 1 && W <= kPC && g % (16 * kWarps) == 0 && g / (16 * kWarps) <= kFragMax;
}

// The candidate tokens of every depth of request 0 are read once, at launch.
DT_HOST_DEVICE_INLINE bool prefetch_tokens(int D, int M) { return D * M <= 4096; }

DT_HOST_DEVICE_INLINE bool mfrag_ok(const ChainParams& p) {
  return !p.marginal && p.n_req > 1 && (p.n_req * p.W) % 8 == 0 && p.g % 16 == 0 &&
         p.g <= 16 * kWarps * kFragMax;
}

// One request with more than 8 live branches on the SIMT phase B: the
// branches are scored by different CTAs (see the kernel).
DT_HOST_DEVICE_INLINE bool bdist_ok(const ChainParams& p) {
  return !p.marginal && p.n_req == 1 && p.mma_b == 0 && p.W > kPC && p.W * p.K >= p.M && p.K <= 32;
}

DT_HOST_DEVICE_INLINE Shape runtime_shape(const ChainParams& p) {
  const bool fr = !p.marginal && frag_ok(p.n_req, p.W, p.g);
  return Shape{p.g, p.r, p.M, p.K, p.W, p.n_req, p.D, p.jper, p.rper, p.cpad, p.stage_w2 != 0, p.mma_b != 0,
               prefetch_tokens(p.D, p.M), p.dbuf != 0, fr,
               fr && p.mma_b != 0 && p.dbuf != 0 && p.r % 16 == 0 && p.r / 16 <= kZFragMax,
               mfrag_ok(p) && p.tc == 0, bdist_ok(p), p.tc != 0, p.tc_ns};
}

// Generic instantiation: every dimension from the launch parameters.
struct DimsRuntime {
  static DT_DEVINL Shape get(const ChainParams& p) { return runtime_shape(p); }
};
// The Qwen3-4B shape (g=1024, r=256, M=64, K=W=8, one request, depth 15, 128
// CTAs): dimensions are literals, so the compiler folds the index arithmetic.
struct DimsQ4B {
  static constexpr Shape kShape{1024, 256, 64, 8, 8, 1, 15, 8, 2, 32, true, true, true, true, true, true, false,
                                false, false, 0};
  static DT_DEVINL Shape get(const ChainParams&) { return kShape; }
};

// Candidate data of one (request, depth) row staged in shared memory.
struct Stage {
  uint16_t* w2s;  // [M][r+8] W2 rows of the candidates
  float* xs;      // [M][3*jper] GRU-input slices of the candidates
  float* cbs;     // [M] candidate base logits
  float* h1s;     // [r]
  float* rest;    // [1]
};

struct Smem {
  uint16_t* w;      // [cpad][gp] bf16 owned weight columns, K-major
  uint16_t* sh;     // [kPC][gp] bf16 high part of the state chunk
  uint16_t* sl;     // [kPC][gp] bf16 low part (S - high)
  float* red;       // [kWarps][kPC][cpad]
  float* uu;        // [n_req*W][3*jper] owned GRU hidden projections
  float* z;         // [kWarps][r] (SIMT phase B)
  uint16_t* w2s;    // [M][r+8] staged W2 rows of the current request's candidates
  float* xs;        // [M][3*jper] staged GRU-input slices of the candidates
  int* ctk;         // [M] candidate tokens of the current row
  float* cbs;       // [M] candidate base logits
  float* h1s;       // [r]
  float* rest;      // [1]
  int* ctok;        // [W*K] children of the current request: token
  int* cslot;       // [W*K] candidate index of each child
  float* clogp;     // [W*K]
  float* cscore;    // [W*K]
  int* crank;       // [W*K] top-K winners / ranks
  uint64_t* wkey;   // [wkey_words] top-W keys (and the spread branches' K-best selection)
  int* surv;        // [n_req][W] survivor child slot
  float* pscore;    // [W] parent scores of the current request
  int* pnode;       // [W] parent node indices of the current request
  int* tok_all;     // [D][M] candidate tokens of the CTA's tok_all request (when prefetched)
  int* ctk_buf;     // the [M] scratch behind ctk when tokens are read per row
  uint16_t* zh;     // [16*ceil(W/16)][r+8] bf16 high part of z (tensor-core phase B)
  uint16_t* zl;     // same, low part
  uint64_t* lamkey; // [W][M] (lambda, token) keys (tensor-core phase B)
  uint4* mf0;       // fragment blocks of the states, two buffers (several requests)
  uint4* mf1;
  uint8_t* ring;    // [ns][kTcChunk] streamed A-operand chunks (tcgen05 phase A)
  Stage st0, st1;   // stage buffers of even and odd depths (the same buffer without dbuf)
};

DT_HOST_DEVICE_INLINE size_t al16(size_t b) { return (b + 15) & ~static_cast<size_t>(15); }

struct SmemSizes {
  size_t off[23];
  size_t total;
};

DT_HOST_DEVICE_INLINE int pow2_at_least(int n) {
  int v = 1;
  while (v < n) v <<= 1;
  return v;
}


// The candidates' GRU-input slices are staged in shared memory only for one
// request whose branches are not spread and whose phase A is not on tcgen05;
// otherwise phase C reads them from the table.
DT_HOST_DEVICE_INLINE bool xs_staged(const Shape& sh) { return !sh.bdist && !sh.tc && sh.n_req == 1; }

// One stage buffer's bytes of each staged array (0 w2s, 1 xs, 2 cbs, 3 h1s,
// 4 rest), and the region that holds both buffers when double-buffered.
DT_HOST_DEVICE_INLINE size_t stage_one(const Shape& sh, int which) {
  switch (which) {
    case 0: return sh.stage_w2 ? static_cast<size_t>(sh.M) * (sh.r + 8) * 2 : 0;
    case 1: return xs_staged(sh) ? static_cast<size_t>(sh.M) * 3 * sh.jper * 4 : 0;
    case 2: return static_cast<size_t>(sh.M) * 4;
    case 3: return static_cast<size_t>(sh.r) * 4;
    default: return 16;
  }
}
DT_HOST_DEVICE_INLINE size_t stage_bytes(const Shape& sh, int which) {
  return sh.dbuf ? 2 * al16(stage_one(sh, which)) : stage_one(sh, which);
}

// Bytes of the tensor-core phase B's z rows (high and low parts) and of its
// (lambda, token) keys.  They share region 1 with the state chunk of phase A
// (sh, sl): phase A is done with it before phase B starts, and phase B before
// the next depth's phase A.
DT_HOST_DEVICE_INLINE size_t zrows_bytes(const Shape& sh) {
  return sh.mma_b ? al16(static_cast<size_t>(2 * 16 * ((sh.W + 15) / 16)) * (sh.r + 8) * 2) : 0;
}
DT_HOST_DEVICE_INLINE size_t lamkey_bytes(const Shape& sh) {
  return sh.mma_b ? static_cast<size_t>(sh.W) * sh.M * 8 : 0;
}

// 64-bit words of the top-W keys' region: >= 64 (the one-warp top-W); with the
// branches spread, also the K-best selection's histogram (128 words) and the
// keys of its bin (up to M).
DT_HOST_DEVICE_INLINE int wkey_words(const Shape& sh) {
  const int a = pow2_at_least(sh.W * sh.K), b = sh.bdist ? 128 + pow2_at_least(sh.M) : 64;
  return a > b ? a : b;
}

DT_HOST_DEVICE_INLINE SmemSizes smem_sizes(const Shape& sh) {
  const size_t WK = static_cast<size_t>(sh.W) * sh.K;
  const size_t gp = static_cast<size_t>(kstride(sh.g));
  const size_t shsl = gp * kPC * 2 * 2, zl = zrows_bytes(sh) + lamkey_bytes(sh);
  const size_t mblk = sh.mfrag ? static_cast<size_t>(32) * sh.g : 0;  // one 8-state fragment block
  // the tcgen05 phase A needs neither the state chunk (region 1) nor the
  // partial sums (region 2); without them the Top-B and tree/mask tail runs
  // in its own launches (chain_can_fuse_tree reads these sizes)
  const bool lean = sh.tc;
  const size_t r1 = (shsl > zl && !lean) ? shsl : zl;
  const size_t sz[23] = {
      gp * sh.cpad * 2,
      r1 > mblk ? r1 : mblk,
      lean ? 0 : static_cast<size_t>(kWarps) * kPC * sh.cpad * 4,
      static_cast<size_t>(sh.n_req) * sh.W * 3 * sh.jper * 4,
      sh.mma_b ? 0 : static_cast<size_t>(kWarps) * sh.r * 4,
      stage_bytes(sh, 0),
      stage_bytes(sh, 1),
      static_cast<size_t>(sh.M) * 4,
      stage_bytes(sh, 2),
      stage_bytes(sh, 3),
      stage_bytes(sh, 4),
      WK * 4,
      WK * 4,
      WK * 4,
      WK * 4,
      WK * 4,
      static_cast<size_t>(wkey_words(sh)) * 8,
      static_cast<size_t>(sh.n_req) * sh.W * 4,
      static_cast<size_t>(sh.W) * 4,
      static_cast<size_t>(sh.W) * 4,
      sh.prefetch ? static_cast<size_t>(sh.D) * sh.M * 4 : 0,
      // the second fragment-block buffer (the first is region 1), or the
      // tcgen05 phase A's chunk slots
      sh.tc ? static_cast<size_t>(sh.ns) * kTcChunk : mblk,
      0,     // (z rows and (lambda, token) keys: in region 1)
  };
  SmemSizes s;
  size_t o = 0;
  for (int i = 0; i < 23; ++i) {
    // tcgen05 operands (the weights, region 0, and the chunk slots, region
    // 21) start on 1024-byte boundaries (the 128-byte swizzle's atoms)
    if (i == 21 && sh.tc) o = (o + 1023) & ~static_cast<size_t>(1023);
    s.off[i] = o;
    o += al16(sz[i]);
  }
  // room to align the base of the dynamic shared memory to 1024 bytes
  s.total = o + (sh.tc ? 1024 : 0);
  return s;
}

// Byte offset of state (row st, column k) in the tcgen05 A-operand chunks of
// one parity (row tiles of 2^ts rows, chunks of 2^ts x 128 bytes): chunk (row
// tile, K block k/64, part), inside it the 128-byte swizzled K-major layout
// (8-row atoms of 1024 bytes, row rr%8 of an atom at 128 rr%8, its 16-byte
// piece k%64/8 at piece (k%64/8) xor (rr%8)).  The low part's chunk follows
// the high part's.
DT_DEVINL size_t tc_off(int st, int k, int KB, int ts) {
  const int mt = st >> ts, rr = st & ((1 << ts) - 1), kb = k >> 6, ch = (k >> 3) & 7;
  return (static_cast<size_t>((mt * KB + kb) * 2) << (ts + 7)) + (rr >> 3) * 1024 + (rr & 7) * 128 +
         ((ch ^ (rr & 7)) << 4) + (k & 7) * 2;
}
// One state value: its bf16 high part and the bf16 of the remainder.
DT_DEVINL void store_tc1(uint8_t* base, int st, int k, int KB, int ts, float v) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(v);
  const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
  uint8_t* a = base + tc_off(st, k, KB, ts);
  *reinterpret_cast<uint16_t*>(a) = __bfloat16_as_ushort(hi);
  *reinterpret_cast<uint16_t*>(a + (1 << (ts + 7))) = __bfloat16_as_ushort(lo);
}
// Eight consecutive values (columns k..k+7, k a multiple of 8): one 16-byte
// piece of each part.
DT_DEVINL void store_tc8(uint8_t* base, int st, int k, int KB, int ts, const float (&v)[8]) {
  uint32_t hi[4], lo[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) hi[e] = split_hi_lo(v[2 * e], v[2 * e + 1], lo[e]);
  uint8_t* a = base + tc_off(st, k, KB, ts);
  *reinterpret_cast<uint4*>(a) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
  *reinterpret_cast<uint4*>(a + (1 << (ts + 7))) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// Bring the W2 rows of one depth's candidates (tokens tok[0, M)) into L2,
// candidate c by CTA c mod G, ahead of the scoring that reads them from L2.
DT_DEVINL void prefetch_w2_rows(const ChainParams& p, const Shape& sh, const int* tok) {
  const int G = static_cast<int>(gridDim.x);
  for (int c = static_cast<int>(blockIdx.x) + G * static_cast<int>(threadIdx.x); c < sh.M; c += G * kThreads)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p.w2 + static_cast<size_t>(tok[c]) * sh.r),
                 "r"(static_cast<uint32_t>(sh.r * 2))
                 : "memory");
}

// Read the candidate tokens of one (request, depth) row into shared memory.
DT_DEVINL void load_cand_tokens(const ChainParams& p, const Shape& sh, const Smem& s, size_t qrow) {
  for (int c = threadIdx.x; c < sh.M; c += kThreads) {
    int t = p.cand_tok[qrow * sh.M + c];
    if (t < 0 || t >= p.V) {
      dt_report(p.status, DT_DEV_BOUNDS);
      t = 0;
    }
    s.ctk[c] = t;
  }
}

// The request whose candidate tokens of every depth a CTA reads once at launch
// (tok_all): request 0, or with several requests the CTA's own first one.
DT_DEVINL int tok_all_request(const Shape& sh) { return sh.n_req > 1 ? static_cast<int>(blockIdx.x) : 0; }

// Point s.ctk at the candidate tokens of (request q, depth i): the launch-time
// prefetch for the CTA's tok_all request, else read into the scratch row.
// Whole CTA; the caller synchronises before the tokens are used.
DT_DEVINL void select_row_tokens(const ChainParams& p, const Shape& sh, Smem& s, int q, int i) {
  if (q == tok_all_request(sh) && sh.prefetch) {
    s.ctk = s.tok_all + static_cast<size_t>(i - 1) * sh.M;
  } else {
    s.ctk = s.ctk_buf;
    load_cand_tokens(p, sh, s, static_cast<size_t>(q) * sh.D + (i - 1));
  }
}

// Asynchronous copies (one cp.async group) of everything phase B/C read for
// one (request, depth) row into buffer b; tok holds the row's M candidate
// tokens.  Whole CTA.
DT_DEVINL void stage_row(const ChainParams& p, const Shape& sh, const Stage& b, const int* tok, size_t qrow, int j0,
                         int nj, bool want_x) {
  const int r = sh.r, M = sh.M, g = sh.g;
  if (sh.stage_w2) {
    const int c8 = r / 8;
    for (int idx = threadIdx.x; idx < M * c8; idx += kThreads) {
      const int c = idx / c8, k = idx - c * c8;
      cp_async16(b.w2s + static_cast<size_t>(c) * (r + 8) + k * 8, p.w2 + static_cast<size_t>(tok[c]) * r + k * 8);
    }
  }
  if (want_x && nj > 0) {
    if (nj == sh.jper && nj % 4 == 0 && g % 4 == 0) {
      // 16-byte pieces: each gate's owned columns are contiguous in X and in xs
      const int q4 = nj / 4, per = 3 * q4;
      for (int idx = threadIdx.x; idx < M * per; idx += kThreads) {
        const int c = idx / per, rem = idx - c * per;
        const int gate = rem / q4, jj = (rem - gate * q4) * 4;
        cp_async16(b.xs + static_cast<size_t>(c) * 3 * sh.jper + gate * nj + jj,
                   p.xtab + static_cast<size_t>(tok[c]) * 3 * g + gate * g + j0 + jj);
      }
    } else {
      const int per = 3 * nj;
      for (int idx = threadIdx.x; idx < M * per; idx += kThreads) {
        const int c = idx / per, rem = idx - c * per;
        const int gate = rem / nj, jj = rem - gate * nj;
        cp_async4(b.xs + static_cast<size_t>(c) * 3 * sh.jper + gate * nj + jj,
                  p.xtab + static_cast<size_t>(tok[c]) * 3 * g + gate * g + j0 + jj);
      }
    }
  }
  if (M % 4 == 0 && r % 4 == 0) {
    for (int c = threadIdx.x; c < M / 4; c += kThreads) cp_async16(b.cbs + 4 * c, p.cand_base + qrow * M + 4 * c);
    for (int k = threadIdx.x; k < r / 4; k += kThreads) cp_async16(b.h1s + 4 * k, p.h1 + qrow * r + 4 * k);
  } else {
    for (int c = threadIdx.x; c < M; c += kThreads) cp_async4(b.cbs + c, p.cand_base + qrow * M + c);
    for (int k = threadIdx.x; k < r; k += kThreads) cp_async4(b.h1s + k, p.h1 + qrow * r + k);
  }
  if (threadIdx.x == 0) cp_async4(b.rest, p.rest_lse + qrow);
  cp_async_commit();
}

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

template <int MPL, class Dm>
__global__ void __launch_bounds__(kThreads, 1) k_chain(const ChainParams p) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  __shared__ int s_abort;
  __shared__ __align__(8) uint64_t s_mbar[2];  // fragment-block copies (several requests)
  __shared__ int s_wcnt[kWarps];
  __shared__ uint32_t s_state[4];
  __shared__ float s_tred[64];  // Top-B min/max partials of the tail
  __shared__ int s_tscan[40];   // Top-B fallback scans; top-W bin search and scan
  __shared__ uint64_t s_kth;    // top-W: the Li-th best key
  // tcgen05 phase A: chunk slots full [0..3] / free [4..7], products done [8]
  __shared__ __align__(8) uint64_t s_tcbar[9];
  __shared__ uint32_t s_tmem;

  const Shape sh = Dm::get(p);
  // candidate keys carry their candidate index (M <= 64, token ids < 2^26)
  const bool packed = sh.M <= 64 && p.V <= (1 << 26);
  const int g = sh.g, r = sh.r, M = sh.M, K = sh.K, W = sh.W, n_req = sh.n_req, D = sh.D;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int j0 = blockIdx.x * sh.jper;
  const int nj = max(0, min(g, j0 + sh.jper) - j0);
  const int r0 = blockIdx.x * sh.rper;
  const int nr = max(0, min(r, r0 + sh.rper) - r0);
  const int ncol = 3 * nj + nr;
  const int cpad = sh.cpad;

  Smem s;
  {
    const SmemSizes L = smem_sizes(sh);
    // (the tcgen05 operands want 1024-byte aligned regions)
    uint8_t* const smem_raw_ = smem_raw;
    uint8_t* const smem_raw =
        sh.tc ? smem_raw_ + ((1024u - (smem_u32(smem_raw_) & 1023u)) & 1023u) : smem_raw_;
    s.w = reinterpret_cast<uint16_t*>(smem_raw + L.off[0]);
    s.sh = reinterpret_cast<uint16_t*>(smem_raw + L.off[1]);
    s.sl = s.sh + static_cast<size_t>(kPC) * kstride(g);
    s.red = reinterpret_cast<float*>(smem_raw + L.off[2]);
    s.uu = reinterpret_cast<float*>(smem_raw + L.off[3]);
    s.z = reinterpret_cast<float*>(smem_raw + L.off[4]);
    const int u = sh.dbuf ? 1 : 0;  // the odd buffer follows the even one
    s.st0.w2s = reinterpret_cast<uint16_t*>(smem_raw + L.off[5]);
    s.st0.xs = reinterpret_cast<float*>(smem_raw + L.off[6]);
    s.st0.cbs = reinterpret_cast<float*>(smem_raw + L.off[8]);
    s.st0.h1s = reinterpret_cast<float*>(smem_raw + L.off[9]);
    s.st0.rest = reinterpret_cast<float*>(smem_raw + L.off[10]);
    s.st1.w2s = reinterpret_cast<uint16_t*>(smem_raw + L.off[5] + u * al16(stage_one(sh, 0)));
    s.st1.xs = reinterpret_cast<float*>(smem_raw + L.off[6] + u * al16(stage_one(sh, 1)));
    s.st1.cbs = reinterpret_cast<float*>(smem_raw + L.off[8] + u * al16(stage_one(sh, 2)));
    s.st1.h1s = reinterpret_cast<float*>(smem_raw + L.off[9] + u * al16(stage_one(sh, 3)));
    s.st1.rest = reinterpret_cast<float*>(smem_raw + L.off[10] + u * al16(stage_one(sh, 4)));
    s.w2s = s.st0.w2s;
    s.xs = s.st0.xs;
    s.ctk = reinterpret_cast<int*>(smem_raw + L.off[7]);
    s.cbs = s.st0.cbs;
    s.h1s = s.st0.h1s;
    s.rest = s.st0.rest;
    s.ctok = reinterpret_cast<int*>(smem_raw + L.off[11]);
    s.cslot = reinterpret_cast<int*>(smem_raw + L.off[12]);
    s.clogp = reinterpret_cast<float*>(smem_raw + L.off[13]);
    s.cscore = reinterpret_cast<float*>(smem_raw + L.off[14]);
    s.crank = reinterpret_cast<int*>(smem_raw + L.off[15]);
    s.wkey = reinterpret_cast<uint64_t*>(smem_raw + L.off[16]);
    s.surv = reinterpret_cast<int*>(smem_raw + L.off[17]);
    s.pscore = reinterpret_cast<float*>(smem_raw + L.off[18]);
    s.pnode = reinterpret_cast<int*>(smem_raw + L.off[19]);
    s.tok_all = reinterpret_cast<int*>(smem_raw + L.off[20]);
    s.ctk_buf = s.ctk;
    s.zh = reinterpret_cast<uint16_t*>(smem_raw + L.off[1]);
    s.zl = s.zh + static_cast<size_t>(16 * ((W + 15) / 16)) * (r + 8);
    s.lamkey = reinterpret_cast<uint64_t*>(smem_raw + L.off[1] + zrows_bytes(sh));
    s.mf0 = reinterpret_cast<uint4*>(smem_raw + L.off[1]);
    s.mf1 = reinterpret_cast<uint4*>(smem_raw + L.off[21]);
    s.ring = smem_raw + L.off[21];
  }

  if (tid == 0) {
    s_abort = 0;
    mbar_init(&s_mbar[0], 1);
    mbar_init(&s_mbar[1], 1);
    if (sh.tc)
      for (int b = 0; b < 9; ++b) mbar_init(&s_tcbar[b], 1);
    fence_mbar_init();
  }
  uint32_t mf_phase = 0;  // completed-phase parity of the two block buffers
  // tcgen05 phase A: tensor-memory columns (one 128-lane tile of cpad fp32
  // columns per 128 state rows), chunks streamed so far, products-done parity
  const int tc_ts = tc_tile_shift(n_req * W), tc_tm = 1 << tc_ts;
  const int tc_nmt = (n_req * W + tc_tm - 1) / tc_tm;
  const uint32_t tc_chunk = static_cast<uint32_t>(tc_tm) * 128u;  // bytes of one streamed chunk
  uint32_t tc_cols = 32;
  while (sh.tc && tc_cols < static_cast<uint32_t>(tc_nmt * cpad)) tc_cols <<= 1;
  uint32_t tc_seq = 0, tc_done_ph = 0;
  if (sh.tc && warp == 0) tmem_alloc(&s_tmem, tc_cols);

  // ---- the owned weight columns, K-major: s.w[c][k] (zero padded) ----
  const int gp = kstride(g);
  if (sh.tc) {
    // tcgen05 B operand: K blocks of 64 (cpad rows x 128 bytes each), the
    // rows 128-byte swizzled in 8-row atoms
    const int g8 = g / 8;
    uint8_t* wb = reinterpret_cast<uint8_t*>(s.w);
    for (int idx = tid; idx < cpad * g8; idx += kThreads) {
      const int c = idx / g8, k8 = idx - c * g8;
      uint4 v = make_uint4(0u, 0u, 0u, 0u);
      if (c < 3 * nj) {
        const int gate = c / nj, jj = c - gate * nj;
        v = *reinterpret_cast<const uint4*>(p.w_hh + static_cast<size_t>(gate * g + j0 + jj) * g + 8 * k8);
      } else if (c < ncol) {
        const int rr = r0 + (c - 3 * nj);
        v = *reinterpret_cast<const uint4*>(p.w1 + static_cast<size_t>(rr) * p.ldw1 + p.d + 8 * k8);
      }
      const int kb = k8 >> 3, ch = k8 & 7;
      *reinterpret_cast<uint4*>(wb + static_cast<size_t>(kb) * cpad * 128 + (c >> 3) * 1024 + (c & 7) * 128 +
                                ((ch ^ (c & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();  // read by tcgen05.mma
    tc_fence_before();
  } else if (!p.marginal) {
    const int g8 = gp / 8;  // 16-byte chunks per padded row
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
      *reinterpret_cast<uint4*>(s.w + static_cast<size_t>(c) * gp + 8 * k8) = v;
    }
  }

  // the resident weights are loaded; everything below reads the previous
  // kernels' results (and the barrier counter Top-M cleared)
  dt_grid_wait();
  uint32_t tmem_base = 0;
  if (sh.tc) {
    __syncthreads();
    tc_fence_after();
    tmem_base = s_tmem;
  }

  // ---- candidate tokens of every depth of the CTA's tok_all request, read once ----
  const int tokq = tok_all_request(sh);
  if (sh.prefetch && tokq < n_req) {
    for (int idx = tid; idx < D * M; idx += kThreads) {
      int t = p.cand_tok[static_cast<size_t>(tokq) * D * M + idx];  // request q owns rows qD .. qD+D-1
      if (t < 0 || t >= p.V) {
        dt_report(p.status, DT_DEV_BOUNDS);
        t = 0;
      }
      s.tok_all[idx] = t;
    }
  }
  __syncthreads();
  // W2 rows read from L2 by the scoring (not staged): the first depth's now,
  // every later depth's one depth ahead
  const bool w2_ahead = !p.marginal && n_req == 1 && !sh.stage_w2 && sh.prefetch && (sh.r * 2) % 16 == 0;
  if (w2_ahead) prefetch_w2_rows(p, sh, s.tok_all + static_cast<size_t>(p.depth_first - 1) * M);
  // Several requests: CTA c selects for requests c, c + G, ... (G CTAs) and
  // every CTA then updates its state columns of all requests after one more
  // grid barrier.  One request: every CTA selects for it (identically) and
  // updates its own columns right away.
  const bool dist = n_req > 1;
  // One request with many live branches and the SIMT phase B: CTA c scores
  // branches c, c + G, ... and writes their children into the node arrays;
  // after a grid barrier every CTA reads all children back for the top-W.
  const bool bdist = sh.bdist;
  const int qfirst = dist ? static_cast<int>(blockIdx.x) : 0;
  const int qstep = dist ? static_cast<int>(gridDim.x) : 1;
  // a CTA that selects for exactly one request keeps that request's next
  // parents in shared memory from one depth to the next
  const bool keep_par = qfirst < n_req && qfirst + qstep >= n_req;
  // stage the first depth's first request of this CTA (overlaps the root
  // step and phase A)
  auto buf = [&](int depth) -> Stage { return (depth & 1) ? s.st1 : s.st0; };
  // on a barrier timeout: let the CTA's own copies land before it returns
  // (and give back the tensor memory)
  auto drain = [&]() {
    cp_async_wait_all();
    if (sh.tc) {
      tc_fence_before();
      __syncthreads();
      if (warp == 0) tmem_dealloc(tmem_base, tc_cols);
    }
  };
  if (qfirst < n_req) {
    select_row_tokens(p, sh, s, qfirst, p.depth_first);
    __syncthreads();
    stage_row(p, sh, buf(p.depth_first), s.ctk,
              static_cast<size_t>(qfirst) * D + (p.depth_first - 1), j0, nj, xs_staged(sh) && p.depth_first != D);
  }

  unsigned epoch = 0;

  // ---- depth 0: root state and root node ----
  if (p.depth_first == 1) {
    for (int idx = tid; idx < n_req * nj; idx += kThreads) {
      const int q = idx / nj, jj = j0 + (idx - q * nj);
      int tok = p.root_tok[q];
      if (tok < 0 || tok >= p.V) {
        dt_report(p.status, DT_DEV_BOUNDS);
        tok = 0;
      }
      const float* x = p.xtab + static_cast<size_t>(tok) * 3 * g;
      const float zg = sigmoidf_(x[g + jj]);
      const float ng = tanhf_(x[2 * g + jj]);
      const float s0 = (1.0f - zg) * ng;
      p.S[static_cast<size_t>(q * W) * g + jj] = s0;
      if (sh.frag || sh.mfrag) store_frag(p.sfrag, q * W, jj, g / 16, s0);  // parity 0 = depth 0
      if (sh.tc) store_tc1(reinterpret_cast<uint8_t*>(p.sfrag), q * W, jj, g / 64, tc_ts, s0);
    }
    if (sh.mfrag || sh.tc) fence_proxy_async_global();
    if (blockIdx.x == 0) {
      for (int q = tid; q < n_req; q += kThreads) {
        const size_t b = static_cast<size_t>(q) * p.N1;
        p.node_tok[b] = p.root_tok[q];
        p.node_parent[b] = -1;
        p.node_logp[b] = 0.0f;
        p.node_score[b] = 0.0f;
        p.live[static_cast<size_t>(q) * W] = 0;
      }
    }
    if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) {
      drain();
      return;
    }
  }

  for (int i = p.depth_first; i <= p.depth_last; ++i) {
    const int Lp = p.L[i - 1];  // live branches entering this depth
    const int Li = p.L[i];      // branches that live on
    const int P = n_req * Lp;
    const bool last = i == D;
    const float* Sprev = p.S + static_cast<size_t>((i - 1) & 1) * n_req * W * g;
    float* Snext = p.S + static_cast<size_t>(i & 1) * n_req * W * g;
    const int* live_prev = p.live + static_cast<size_t>((i - 1) & 1) * n_req * W;
    int* live_next = p.live + static_cast<size_t>(i & 1) * n_req * W;
    CH_STAMP(i, 0);
#ifdef DT_CHAIN_TIMING
    unsigned long long blk_wait = 0;
#endif
    if (w2_ahead && i < p.depth_last) prefetch_w2_rows(p, sh, s.tok_all + static_cast<size_t>(i) * M);
    // one request: the next depth's candidate data is staged now, into the
    // other buffer (its last reader, depth i-1, finished before the barrier);
    // it lands during this depth
    if (sh.dbuf) s.ctk = s.tok_all + static_cast<size_t>(i - 1) * M;  // this depth's candidate tokens

    // ================= phase A: projections of the live states ==============
    if (p.marginal) {
      // marginal scoring: no states to project; only the staging of the next
      // depth's candidate data
      if (sh.dbuf && i < p.depth_last)
        stage_row(p, sh, buf(i + 1), s.tok_all + static_cast<size_t>(i) * M, static_cast<size_t>(i), j0, nj, false);
    } else if (sh.frag) {
      // the live states (one request, P <= 8 rows) as ready-made A fragments:
      // lane (gid, tig) of the warp owning k16 step kt reads one 16-byte word
      // per step, straight into registers (high and low bf16 parts)
      const int gid = lane >> 2, tig = lane & 3;
      const int nk16 = g / 16;
      const uint4* fr = reinterpret_cast<const uint4*>(p.sfrag + static_cast<size_t>((i - 1) & 1) * n_req * W * g);
      uint4 f[kFragMax];
#pragma unroll
      for (int m = 0; m < kFragMax; ++m) {
        const int kt = warp + kWarps * m;
        f[m] = kt < nk16 ? __ldcg(fr + frag_word(gid, kt, tig, nk16)) : make_uint4(0u, 0u, 0u, 0u);
      }
      // one request: the next depth's candidate data is staged now, into the
      // other buffer (its last reader, depth i-1, finished before the
      // barrier), while the state loads are in flight; it lands during this
      // depth
      if (sh.dbuf && i < p.depth_last)
        stage_row(p, sh, buf(i + 1), s.tok_all + static_cast<size_t>(i) * M, static_cast<size_t>(i), j0, nj,
                  xs_staged(sh) && i + 1 != D);
      // rows 0..7 of the tile carry the high parts and rows 8..15 the low
      // parts of the same states: one MMA per k16 step gives both products
      float acc[kMaxNTiles][4];
#pragma unroll
      for (int nt = 0; nt < kMaxNTiles; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
      const int ntiles = cpad / 8;
#pragma unroll
      for (int m = 0; m < kFragMax; ++m) {
        const int kt = warp + kWarps * m;
        if (kt < nk16) {
          const int k0 = kt * 16 + 2 * tig;
#pragma unroll
          for (int nt = 0; nt < kMaxNTiles; ++nt) {
            if (nt < ntiles) {
              const uint16_t* wc = s.w + static_cast<size_t>(nt * 8 + gid) * gp + k0;
              const uint32_t b0 = *reinterpret_cast<const uint32_t*>(wc);
              const uint32_t b1 = *reinterpret_cast<const uint32_t*>(wc + 8);
              mma_bf16_16816(acc[nt], f[m].x, f[m].z, f[m].y, f[m].w, b0, b1);
            }
          }
        }
      }
#pragma unroll
      for (int nt = 0; nt < kMaxNTiles; ++nt) {
        if (nt < ntiles) {
          float* rw = s.red + (warp * kPC + gid) * cpad + nt * 8 + 2 * tig;
          rw[0] = acc[nt][0] + acc[nt][2];
          rw[1] = acc[nt][1] + acc[nt][3];
        }
      }
      // this depth's staged h1_i (copied during the previous depth) is read
      // below: the thread's own copies are complete, the barrier shares them
      if (sh.zf) {
        if (i < p.depth_last) cp_async_wait_group1();  // the next depth's group may still fly
        else cp_async_wait_all();
      }
      __syncthreads();
      const float* h1i = buf(i).h1s;
      for (int idx = tid; idx < P * ncol; idx += kThreads) {
        const int pp = idx / ncol, c = idx - pp * ncol;
        float sum = 0.0f;
#pragma unroll
        for (int w8 = 0; w8 < kWarps; ++w8) sum += s.red[(w8 * kPC + pp) * cpad + c];
        if (c < 3 * nj) {
          s.uu[static_cast<size_t>(pp) * 3 * sh.jper + c] = sum;
        } else {
          const int rho = r0 + (c - 3 * nj);
          if (sh.zf) store_frag(p.zfrag, pp, rho, r / 16, siluf_(h1i[rho] + sum));
          else p.uW1[static_cast<size_t>(pp) * r + rho] = sum;
        }
      }
    }
    if (sh.tc) {
      // the states on tcgen05: u[row][c] = sum_k S[row][k] W[c][k] for every
      // state row (128-row tiles) and owned weight row c (N = cpad), the
      // high and the low parts of the states accumulated into the same fp32
      // accumulator.  Warp 1 streams the A chunks (128 rows x 64 K of one
      // part) from L2 into ns slots with bulk copies; one thread of warp 0
      // issues four K=16 MMAs per chunk against the resident weights and
      // frees the slot through the MMAs' commit.
      if (sh.dbuf && i < p.depth_last)
        stage_row(p, sh, buf(i + 1), s.tok_all + static_cast<size_t>(i) * M, static_cast<size_t>(i), j0, nj,
                  xs_staged(sh) && i + 1 != D);
      const int KB = g / 64;
      const int ns = sh.ns;
      const uint8_t* abase = reinterpret_cast<const uint8_t*>(p.sfrag) +
                             static_cast<size_t>((i - 1) & 1) * tc_nmt * KB * 2 * tc_chunk;
      // every CTA starts at a different K block, so that the CTAs do not all
      // read the same lines at the same time
      const int rot = static_cast<int>(blockIdx.x) % KB;
      // A slot holds both parts of one K block (one copy, eight MMAs, one
      // wait and one commit); a single thread runs each loop, with slots,
      // phases and descriptors stepped, not recomputed, to keep its
      // dependent instructions few.
      const uint32_t pair = 2u * tc_chunk;
      const uint32_t nsl = min(4u, max(1u, static_cast<uint32_t>(ns) * kTcChunk / pair));
      if (warp == 1) {
        if (lane == 0) {
          fence_proxy_async_global();  // the states were written by generic stores
          uint32_t slot = tc_seq % nsl, use = tc_seq / nsl;
          int c = 0;
          for (int mt = 0; mt < tc_nmt && !s_abort; ++mt) {
            for (int kk = 0, kb = rot; kk < KB; ++kk, kb = (kb + 1 == KB ? 0 : kb + 1), ++c) {
              if (use > 0 && !mbar_wait(&s_tcbar[4 + slot], (use - 1) & 1u, p.status)) {
                s_abort = 1;
                break;
              }
              CH_TCST(0, c, i);
              mbar_arrive_expect_tx(&s_tcbar[slot], pair);
              bulk_g2s(s.ring + static_cast<size_t>(slot) * pair, abase + static_cast<size_t>((mt * KB + kb) * 2) * tc_chunk,
                       pair, &s_tcbar[slot]);
              if (++slot == nsl) {
                slot = 0;
                ++use;
              }
            }
          }
        }
        __syncwarp();
      } else if (warp == 0) {
        if (lane == 0) {
          const uint32_t idesc = idesc_bf16_f32(static_cast<uint32_t>(tc_tm), static_cast<uint32_t>(cpad));
          // descriptors of slot 0 and of K block 0 (16-byte units): a slot is
          // pair / 16 further, the low part tc_chunk / 16, a K block
          // cpad * 128 / 16, a K step 32 / 16
          const uint64_t ad0 = sdesc_k_sw128(smem_u32(s.ring)), bd0 = sdesc_k_sw128(smem_u32(s.w));
          const uint64_t lo_off = tc_chunk / 16;
          uint32_t slot = tc_seq % nsl, use = tc_seq / nsl;
          int c = 0;
          for (int mt = 0; mt < tc_nmt && !s_abort; ++mt) {
            const uint32_t d = tmem_base + static_cast<uint32_t>(mt * cpad);
            for (int kk = 0, kb = rot; kk < KB; ++kk, kb = (kb + 1 == KB ? 0 : kb + 1), ++c) {
              if (!mbar_wait(&s_tcbar[slot], use & 1u, p.status)) {
                s_abort = 1;
                break;
              }
              CH_TCST(1, c, i);
              tc_fence_after();
              const uint64_t bd = bd0 + static_cast<uint64_t>(kb * cpad * 8);
              const uint64_t ad = ad0 + static_cast<uint64_t>(slot * (pair / 16));
              tc_mma_bf16(d, ad, bd, idesc, kk != 0 ? 1u : 0u);
              tc_mma_bf16(d, ad + 2, bd + 2, idesc, 1u);
              tc_mma_bf16(d, ad + 4, bd + 4, idesc, 1u);
              tc_mma_bf16(d, ad + 6, bd + 6, idesc, 1u);
              tc_mma_bf16(d, ad + lo_off, bd, idesc, 1u);
              tc_mma_bf16(d, ad + lo_off + 2, bd + 2, idesc, 1u);
              tc_mma_bf16(d, ad + lo_off + 4, bd + 4, idesc, 1u);
              tc_mma_bf16(d, ad + lo_off + 6, bd + 6, idesc, 1u);
              tc_commit(&s_tcbar[4 + slot]);  // the slot is free once these MMAs are done
              if (++slot == nsl) {
                slot = 0;
                ++use;
              }
            }
          }
          tc_commit(&s_tcbar[8]);  // every product of the depth is done
          CH_TCST(2, 0, i);
        }
        __syncwarp();
      }
      tc_seq += static_cast<uint32_t>(tc_nmt * KB);
      if (!mbar_wait(&s_tcbar[8], tc_done_ph, p.status)) s_abort = 1;
      tc_done_ph ^= 1u;
      __syncwarp();
      tc_fence_after();
      // warp w reads lane quarter w%4 of the row tiles w/4, w/4 + 2, ...: of
      // a 128-row tile, rows 32(w%4)..+31 in its 32 lanes; of a 64-row tile,
      // rows 16(w%4)..+15 in its first 16 lanes.  The gate rows go to shared
      // memory (phase C), the W1_S rows to u_W1 (phase B).
      const int q4 = warp & 3;
      for (int mt = warp >> 2; mt < tc_nmt; mt += kWarps / 4) {
        const int st = mt * tc_tm + (tc_tm == 128 ? q4 * 32 + lane : q4 * 16 + lane);
        const int q = st / W, b = st - q * W;
        const bool ok = (tc_tm == 128 || lane < 16) && st < n_req * W && b < Lp;
        const uint32_t ta = tmem_base + (static_cast<uint32_t>(q4 * 32) << 16) + static_cast<uint32_t>(mt * cpad);
        for (int c0 = 0; c0 < ncol; c0 += 16) {
          uint32_t v[16];
          tmem_ld16(ta + static_cast<uint32_t>(c0), v);
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            const int c = c0 + e;
            if (ok && c < ncol) {
              const float u = __uint_as_float(v[e]);
              if (c < 3 * nj) s.uu[static_cast<size_t>(q * Lp + b) * 3 * sh.jper + c] = u;
              else p.uW1[static_cast<size_t>(q * W + b) * r + r0 + (c - 3 * nj)] = u;
            }
          }
        }
      }
      tc_fence_before();
      __syncthreads();
      if (s_abort) {
        // a copy or a product that never completed: stop here (every CTA
        // times out at its next grid barrier)
        drain();
        return;
      }
    }
    if (sh.mfrag) {
      // several requests: the states as ready-made fragments, block by block
      // (8 states: rows 0-7 of the tile carry the high parts, rows 8-15 the
      // low parts), each block copied whole into shared memory with cp.async
      // two blocks ahead; the k16 steps are split over the warps and their
      // partial sums added through s.red
      const int nk16 = g / 16;
      const int nblk = n_req * W / 8;
      const int blk4 = 2 * g;  // 16-byte words of one block: 8 states x g words / 4
      const uint4* fr = reinterpret_cast<const uint4*>(p.sfrag + static_cast<size_t>((i - 1) & 1) * n_req * W * g);
      // every CTA reads every block: each starts at a different block, so
      // that the CTAs do not all read the same lines at the same time
      const int rot = static_cast<int>(blockIdx.x) % nblk;
      // one bulk copy per block (thread 0), completing on the buffer's
      // mbarrier; the fragments were written by generic stores before the
      // grid barrier
      if (tid == 0) fence_proxy_async_global();
      auto load_blk = [&](int rb) {
        if (tid == 0) {
          uint4* dst = (rb & 1) ? s.mf1 : s.mf0;
          const int rbr = rb + rot < nblk ? rb + rot : rb + rot - nblk;
          mbar_arrive_expect_tx(&s_mbar[rb & 1], static_cast<uint32_t>(blk4) * 16u);
          bulk_g2s(dst, fr + static_cast<size_t>(rbr) * blk4, static_cast<uint32_t>(blk4) * 16u, &s_mbar[rb & 1]);
        }
      };
      const int gid = lane >> 2, tig = lane & 3;
      const int ntiles = cpad / 8;
      load_blk(0);
      if (nblk > 1) load_blk(1);
      for (int rb = 0; rb < nblk; ++rb) {
        const int sb = rb & 1;
#ifdef DT_CHAIN_TIMING
        const unsigned long long tw0 = clock64();
#endif
        if (!mbar_wait(&s_mbar[sb], (mf_phase >> sb) & 1u, p.status)) s_abort = 1;
#ifdef DT_CHAIN_TIMING
        blk_wait += clock64() - tw0;
#endif
        mf_phase ^= 1u << sb;
        __syncthreads();
        if (s_abort) {
          // a copy that never completed: stop here (every CTA times out at
          // its next grid barrier)
          drain();
          return;
        }
        const uint4* fb = sb ? s.mf1 : s.mf0;
        float acc[kMaxNTiles][4];
#pragma unroll
        for (int nt = 0; nt < kMaxNTiles; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
        // the warp's fragments first (g <= 16 * kWarps * kFragMax), then the products
        uint4 f[kFragMax];
#pragma unroll
        for (int m = 0; m < kFragMax; ++m) {
          const int kt = warp + kWarps * m;
          f[m] = kt < nk16 ? fb[frag_word(gid, kt, tig, nk16)] : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int m = 0; m < kFragMax; ++m) {
          const int kt = warp + kWarps * m;
          if (kt < nk16) {
            const int k0 = kt * 16 + 2 * tig;
#pragma unroll
            for (int nt = 0; nt < kMaxNTiles; ++nt) {
              if (nt < ntiles) {
                const uint16_t* wc = s.w + static_cast<size_t>(nt * 8 + gid) * gp + k0;
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(wc);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(wc + 8);
                mma_bf16_16816(acc[nt], f[m].x, f[m].z, f[m].y, f[m].w, b0, b1);
              }
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < kMaxNTiles; ++nt) {
          if (nt < ntiles) {
            float* rw = s.red + (warp * kPC + gid) * cpad + nt * 8 + 2 * tig;
            rw[0] = acc[nt][0] + acc[nt][2];
            rw[1] = acc[nt][1] + acc[nt][3];
          }
        }
        __syncthreads();
        if (rb + 2 < nblk) load_blk(rb + 2);  // into the buffer just read
        for (int idx = tid; idx < kPC * ncol; idx += kThreads) {
          const int rr = idx / ncol, c = idx - rr * ncol;
          const int rbr = rb + rot < nblk ? rb + rot : rb + rot - nblk;
          const int st = rbr * 8 + rr, q = st / W, b = st - q * W;
          if (b >= Lp) continue;
          float sum = 0.0f;
#pragma unroll
          for (int w8 = 0; w8 < kWarps; ++w8) sum += s.red[(w8 * kPC + rr) * cpad + c];
          if (c < 3 * nj) s.uu[static_cast<size_t>(q * Lp + b) * 3 * sh.jper + c] = sum;
          else p.uW1[static_cast<size_t>(q * W + b) * r + r0 + (c - 3 * nj)] = sum;
        }
      }
    }
    for (int p0 = 0; p0 < (sh.frag || sh.mfrag || sh.tc || p.marginal ? 0 : P); p0 += kPC) {
      const int pc = min(kPC, P - p0);
      __syncthreads();
      // state rows -> bf16 high + low parts (S = hi + lo to ~16 mantissa bits)
      // (every load of the thread is issued before the first use: one L2 round trip)
      const int gp4 = gp / 4;
      float4 v[kSLoads];
#pragma unroll
      for (int j = 0; j < kSLoads; ++j) {
        const int idx = tid + j * kThreads;
        const int pp = idx / gp4, k4 = idx - pp * gp4;
        v[j] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (idx < kPC * gp4 && pp < pc && 4 * k4 < g) {
          const int pr = p0 + pp;
          const int q = pr / Lp, b = pr - q * Lp;
          v[j] = *reinterpret_cast<const float4*>(Sprev + static_cast<size_t>(q * W + b) * g + 4 * k4);
        }
      }
      // one request: the next depth's candidate data is staged now, into the
      // other buffer (its last reader, depth i-1, finished before the
      // barrier), while the state loads above are in flight; it lands during
      // this depth
      if (sh.dbuf && p0 == 0 && i < p.depth_last)
        stage_row(p, sh, buf(i + 1), s.tok_all + static_cast<size_t>(i) * M, static_cast<size_t>(i), j0, nj,
                  xs_staged(sh) && i + 1 != D);
#pragma unroll
      for (int j = 0; j < kSLoads; ++j) {
        const int idx = tid + j * kThreads;
        if (idx < kPC * gp4) {
          const int pp = idx / gp4, k4 = idx - pp * gp4;
          uint2 hi, lo;
          hi.x = split_hi_lo(v[j].x, v[j].y, lo.x);
          hi.y = split_hi_lo(v[j].z, v[j].w, lo.y);
          *reinterpret_cast<uint2*>(s.sh + static_cast<size_t>(pp) * gp + 4 * k4) = hi;
          *reinterpret_cast<uint2*>(s.sl + static_cast<size_t>(pp) * gp + 4 * k4) = lo;
        }
      }
      __syncthreads();
      // u[pp][c] = sum_k S[pp][k] W[c][k]: mma.sync m16n8k16 (rows 8..15 zero),
      // k16 steps split over the warps, two products (hi, lo) per step
      {
        const int gid = lane >> 2, tig = lane & 3;
        const int nk16 = (g + 15) / 16;
        // high and low parts accumulate in separate chains
        float acc[kMaxNTiles][4], acl[kMaxNTiles][4];
#pragma unroll
        for (int nt = 0; nt < kMaxNTiles; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            acc[nt][e] = 0.0f;
            acl[nt][e] = 0.0f;
          }
        const int ntiles = cpad / 8;
        for (int kt = warp; kt < nk16; kt += kWarps) {
          const int k0 = kt * 16 + 2 * tig;
          const uint32_t ah0 = *reinterpret_cast<const uint32_t*>(s.sh + static_cast<size_t>(gid) * gp + k0);
          const uint32_t ah2 = *reinterpret_cast<const uint32_t*>(s.sh + static_cast<size_t>(gid) * gp + k0 + 8);
          const uint32_t al0 = *reinterpret_cast<const uint32_t*>(s.sl + static_cast<size_t>(gid) * gp + k0);
          const uint32_t al2 = *reinterpret_cast<const uint32_t*>(s.sl + static_cast<size_t>(gid) * gp + k0 + 8);
#pragma unroll
          for (int nt = 0; nt < kMaxNTiles; ++nt) {
            if (nt < ntiles) {
              const uint16_t* wc = s.w + static_cast<size_t>(nt * 8 + gid) * gp + k0;
              const uint32_t b0 = *reinterpret_cast<const uint32_t*>(wc);
              const uint32_t b1 = *reinterpret_cast<const uint32_t*>(wc + 8);
              mma_bf16_16816(acc[nt], ah0, 0u, ah2, 0u, b0, b1);
              mma_bf16_16816(acl[nt], al0, 0u, al2, 0u, b0, b1);
            }
          }
        }
#pragma unroll
        for (int nt = 0; nt < kMaxNTiles; ++nt) {
          if (nt < ntiles) {
            float* rw = s.red + (warp * kPC + gid) * cpad + nt * 8 + 2 * tig;
            rw[0] = acc[nt][0] + acl[nt][0];
            rw[1] = acc[nt][1] + acl[nt][1];
          }
        }
      }
      __syncthreads();
      for (int idx = tid; idx < pc * ncol; idx += kThreads) {
        const int pp = idx / ncol, c = idx - pp * ncol;
        float sum = 0.0f;
#pragma unroll
        for (int w8 = 0; w8 < kWarps; ++w8) sum += s.red[(w8 * kPC + pp) * cpad + c];
        const int pr = p0 + pp;
        if (c < 3 * nj) {
          s.uu[static_cast<size_t>(pr) * 3 * sh.jper + c] = sum;
        } else {
          const int q = pr / Lp, b = pr - q * Lp;
          p.uW1[static_cast<size_t>(q * W + b) * r + r0 + (c - 3 * nj)] = sum;
        }
      }
    }
    CH_STAMP(i, 1);
#ifdef DT_CHAIN_TIMING
    CH_STAMP_SET(i, 7, blk_wait);
#endif
    if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) {
      drain();
      return;
    }
    CH_STAMP(i, 2);

    // ================= phase B: corrected log-probs and selections ==========
    const int row_off = p.off[i];
    const int nchild = Lp * K;
    for (int q = qfirst; q < n_req; q += qstep) {
      const size_t qrow = static_cast<size_t>(q) * D + (i - 1);
      if (q != qfirst) {
        __syncthreads();
        select_row_tokens(p, sh, s, q, i);
        __syncthreads();
        stage_row(p, sh, buf(i), s.ctk, qrow, j0, nj, xs_staged(sh) && !last);
      }
      {
        const Stage cur = buf(i);
        s.w2s = cur.w2s;
        s.xs = cur.xs;
        s.cbs = cur.cbs;
        s.h1s = cur.h1s;
        s.rest = cur.rest;
      }
      // the branches' z fragments (or u_W1 rows) are loaded first, so that
      // their latency overlaps the parent reads and the staging wait
      // z fragments: the CTA reads the 8 x r/16 x 4 words once (two per
      // thread) and keeps them in shared memory as [kt][gid][tig], where a
      // warp's fragment loads of one k16 step are contiguous
      constexpr int kZPer = (kPC * kZFragMax * 4 + kThreads - 1) / kThreads;
      uint4 zq[kZPer];
      if (sh.zf) {
        const int nzw = kPC * (r / 16) * 4;
        const uint4* zr = reinterpret_cast<const uint4*>(p.zfrag);
#pragma unroll
        for (int u = 0; u < kZPer; ++u) {
          const int idx = tid + u * kThreads;
          zq[u] = idx < nzw ? __ldcg(zr + idx) : make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float uv[kZLoads];
      if (sh.mma_b && !sh.zf) {
        const float* ub = p.uW1 + static_cast<size_t>(q * W) * r;  // rows q*W .. q*W+Lp-1
        const int nz = Lp * r;
#pragma unroll
        for (int j = 0; j < kZLoads; ++j) {
          const int idx = tid + j * kThreads;
          uv[j] = idx < nz ? ub[idx] : 0.0f;
        }
      }
      // the parents (this depth's live branches) and their scores: kept from
      // this CTA's own top-W of the previous depth, or read back
      for (int b = tid; b < (keep_par && i > p.depth_first ? 0 : Lp); b += kThreads) {
        const int node = live_prev[static_cast<size_t>(q) * W + b];
        s.pnode[b] = node;
        s.pscore[b] = (node >= 0 && node < p.N1) ? p.node_score[static_cast<size_t>(q) * p.N1 + node] : 0.0f;
      }
      if (sh.zf) {
        // the block's words, [kt][gid][tig] as in global memory
        const int nzw = kPC * (r / 16) * 4;
        uint4* zs4 = reinterpret_cast<uint4*>(s.zh);
#pragma unroll
        for (int u = 0; u < kZPer; ++u) {
          const int idx = tid + u * kThreads;
          if (idx < nzw) zs4[idx] = zq[u];
        }
      }
      if (sh.dbuf && i < p.depth_last)
        cp_async_wait_group1();  // this depth's group; the next depth's may still fly
      else
        cp_async_wait_all();
      __syncthreads();
      const float rest = s.rest[0];
      if (sh.mma_b) {
        // ---- z = SiLU(h1 + u) of every live branch -> bf16 high/low rows ----
        const int zs = r + 8;
        if (!sh.zf) {
          const int nz = Lp * r;
#pragma unroll
          for (int j = 0; j < kZLoads; ++j) {
            const int idx = tid + j * kThreads;
            if (idx < nz) {
              const int b = idx / r, k = idx - b * r;
              const float x = s.h1s[k] + uv[j];
              const float zv = siluf_(x);
              const __nv_bfloat16 hi = __float2bfloat16_rn(zv);
              const __nv_bfloat16 lo = __float2bfloat16_rn(zv - __bfloat162float(hi));
              s.zh[static_cast<size_t>(b) * zs + k] = __bfloat16_as_ushort(hi);
              s.zl[static_cast<size_t>(b) * zs + k] = __bfloat16_as_ushort(lo);
            }
          }
        }
        if (!sh.zf) __syncthreads();
        // ---- lambda[b][c] = (base_c + z_b . W2[c]) / T: mma.sync over (branch, candidate) tiles ----
        if (sh.zf) {
          // z fragments in registers: rows 0..7 high parts, rows 8..15 low
          // parts of the (at most 8) branches; one MMA per k16 step
          const int gid = lane >> 2, tig = lane & 3;
          const int ntiles = M / 8, nk = r / 16;
          const uint4* zs4 = reinterpret_cast<const uint4*>(s.zh);
          for (int nt = warp; nt < ntiles; nt += kWarps) {
            const uint16_t* wr = s.w2s + static_cast<size_t>(nt * 8 + gid) * zs;
            float a0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, a1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
            for (int kt = 0; kt < kZFragMax; ++kt) {
              if (kt < nk) {
                const int k0 = kt * 16 + 2 * tig;
                const uint4 zf = zs4[(kt * kPC + gid) * 4 + tig];
                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(wr + k0);
                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(wr + k0 + 8);
                mma_bf16_16816((kt & 1) ? a1 : a0, zf.x, zf.z, zf.y, zf.w, b0, b1);
              }
            }
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int c = nt * 8 + 2 * tig + e;
              if (gid < Lp) {
                const float lam = (s.cbs[c] + ((a0[e] + a1[e]) + (a0[e + 2] + a1[e + 2]))) / p.T;
                s.lamkey[static_cast<size_t>(gid) * M + c] =
                    packed ? cand_key(lam, s.ctk[c], c) : rank_key(lam, static_cast<uint32_t>(s.ctk[c]));
              }
            }
          }
        } else {
          const int gid = lane >> 2, tig = lane & 3;
          const int mtiles = (Lp + 15) / 16, ntiles = M / 8;
          for (int t = warp; t < mtiles * ntiles; t += kWarps) {
            const int mt = t / ntiles, nt = t - mt * ntiles;
            // four independent accumulation chains (high/low parts x even/odd
            // k16 steps) keep the dependent-MMA latency short
            float a0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, a1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            float a2[4] = {0.0f, 0.0f, 0.0f, 0.0f}, a3[4] = {0.0f, 0.0f, 0.0f, 0.0f};
            const uint16_t* h0 = s.zh + static_cast<size_t>(mt * 16 + gid) * zs;
            const uint16_t* l0 = s.zl + static_cast<size_t>(mt * 16 + gid) * zs;
            const uint16_t* wr = s.w2s + static_cast<size_t>(nt * 8 + gid) * zs;
            // rows 8..15 of the tile hold branches only when Lp > mt*16 + 8;
            // otherwise their fragments are zero and not read
            const bool upper = mt * 16 + 8 < Lp;
            auto kstep = [&](float (&dh)[4], float (&dl)[4], int kt) {
              const int k0 = kt * 16 + 2 * tig;
              const uint32_t b0 = *reinterpret_cast<const uint32_t*>(wr + k0);
              const uint32_t b1 = *reinterpret_cast<const uint32_t*>(wr + k0 + 8);
              mma_bf16_16816(dh, *reinterpret_cast<const uint32_t*>(h0 + k0),
                             upper ? *reinterpret_cast<const uint32_t*>(h0 + 8 * zs + k0) : 0u,
                             *reinterpret_cast<const uint32_t*>(h0 + k0 + 8),
                             upper ? *reinterpret_cast<const uint32_t*>(h0 + 8 * zs + k0 + 8) : 0u, b0, b1);
              mma_bf16_16816(dl, *reinterpret_cast<const uint32_t*>(l0 + k0),
                             upper ? *reinterpret_cast<const uint32_t*>(l0 + 8 * zs + k0) : 0u,
                             *reinterpret_cast<const uint32_t*>(l0 + k0 + 8),
                             upper ? *reinterpret_cast<const uint32_t*>(l0 + 8 * zs + k0 + 8) : 0u, b0, b1);
            };
            const int nk = r / 16;
#pragma unroll 2
            for (int kt = 0; kt < nk; kt += 2) {
              kstep(a0, a1, kt);
              if (kt + 1 < nk) kstep(a2, a3, kt + 1);
            }
            float acc[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[e] = (a0[e] + a2[e]) + (a1[e] + a3[e]);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int b = mt * 16 + gid + (e >= 2 ? 8 : 0);
              const int c = nt * 8 + 2 * tig + (e & 1);
              if (b < Lp) {
                const float lam = (s.cbs[c] + acc[e]) / p.T;
                s.lamkey[static_cast<size_t>(b) * M + c] =
                    packed ? cand_key(lam, s.ctk[c], c) : rank_key(lam, static_cast<uint32_t>(s.ctk[c]));
              }
            }
          }
        }
        __syncthreads();
        // ---- per branch: log-partition, top-K, children by token ----
        if (packed && M == 64 && K <= 32) {
          // the branch's 64 keys (candidate index packed in) sorted in registers,
          // one warp per branch
          for (int b = warp; b < Lp; b += kWarps) {
            const uint64_t* kr = s.lamkey + static_cast<size_t>(b) * 64;
            uint64_t ka = kr[2 * lane], kb2 = kr[2 * lane + 1];
            const float la = key_f32(static_cast<uint32_t>(ka >> 32)), lb = key_f32(static_cast<uint32_t>(kb2 >> 32));
            const float lmax = warp_max(fmaxf(rest, fmaxf(la, lb)));
            const float se = warp_sum(expf(la - lmax) + expf(lb - lmax)) + expf(rest - lmax);
            const float logZ = lmax + logf(se);
            warp_sort64_keys_desc(ka, kb2);
            // lane w < K takes the w-th best (lane w/2, ka or kb)
            const uint64_t xa = __shfl_sync(0xFFFFFFFFu, ka, (lane >> 1) & 31);
            const uint64_t xb = __shfl_sync(0xFFFFFFFFu, kb2, (lane >> 1) & 31);
            const uint64_t wk = (lane & 1) ? xb : xa;
            const int tok = cand_key_tok(wk);
            const int wc = cand_key_c(wk);
            const int trank = warp_rank_below(lane < K ? tok : 0x7FFFFFFF, K);
            if (lane < K) {
              const float lp = key_f32(static_cast<uint32_t>(wk >> 32)) - logZ;
              const int slot = b * K + trank;
              s.ctok[slot] = tok;
              s.cslot[slot] = wc;
              s.clogp[slot] = lp;
              s.cscore[slot] = s.pscore[b] + lp;
            }
          }
        } else
        for (int b = warp; b < Lp; b += kWarps) {
          const uint64_t* kb = s.lamkey + static_cast<size_t>(b) * M;
          float lmax = rest;
          for (int c = lane; c < M; c += 32) lmax = fmaxf(lmax, key_f32(static_cast<uint32_t>(kb[c] >> 32)));
          lmax = warp_max(lmax);
          float se = 0.0f;
          for (int c = lane; c < M; c += 32) se += expf(key_f32(static_cast<uint32_t>(kb[c] >> 32)) - lmax);
          se = warp_sum(se) + expf(rest - lmax);
          const float logZ = lmax + logf(se);
          int* win = s.crank + b * K;
          // the K best by K rounds of a warp argmax over the keys held in
          // registers (candidate c = lane + 32 j; keys are distinct)
          {
            uint64_t kr[MPL];
#pragma unroll
            for (int j = 0; j < MPL; ++j) {
              const int c = lane + 32 * j;
              kr[j] = c < M ? kb[c] : 0ull;
            }
            for (int kk = 0; kk < K; ++kk) {
              uint64_t best = 0ull;
#pragma unroll
              for (int j = 0; j < MPL; ++j) best = kr[j] > best ? kr[j] : best;
              best = warp_max_u64(best);
              int wc = -1;
#pragma unroll
              for (int j = 0; j < MPL; ++j)
                if (best != 0ull && kr[j] == best) {
                  wc = lane + 32 * j;
                  kr[j] = 0ull;
                }
              const unsigned own = __ballot_sync(0xFFFFFFFFu, wc >= 0);
              wc = __shfl_sync(0xFFFFFFFFu, wc, own ? __ffs(own) - 1 : 0);
              if (lane == 0) win[kk] = wc;
            }
          }
          __syncwarp();
          if (lane < K) {
            int c = win[lane];
            if (c < 0 || c >= M) {
              dt_report(p.status, DT_DEV_BOUNDS);
              c = 0;
            }
            const int tok = s.ctk[c];
            int trank = 0;
            for (int m = 0; m < K; ++m) trank += s.ctk[min(max(win[m], 0), M - 1)] < tok ? 1 : 0;
            const float lp = key_f32(static_cast<uint32_t>(kb[c] >> 32)) - logZ;
            const int slot = b * K + trank;
            s.ctok[slot] = tok;
            s.cslot[slot] = c;
            s.clogp[slot] = lp;
            s.cscore[slot] = s.pscore[b] + lp;
          }
          __syncwarp();
        }
      } else if (bdist) {
        float* zv = s.z;           // [r] z of the branch
        float* lamv = s.clogp;     // [M] lambda, then logp
        uint64_t* keys = s.wkey;   // the K best's histogram and bin keys
        int* win = s.crank;        // [K]
        for (int b = blockIdx.x; b < Lp; b += gridDim.x) {
          const float* u = p.uW1 + static_cast<size_t>(b) * r;
          CH_STAMP(i, 12);
          for (int k = tid; k < r; k += kThreads) zv[k] = siluf_(s.h1s[k] + __ldcg(u + k));
          __syncthreads();
          CH_STAMP(i, 13);
          // one candidate per thread: its W2 row from L2, z from shared memory
          float lmax_t = -INFINITY;
          for (int c = tid; c < M; c += kThreads) {
            const uint4* w2r = reinterpret_cast<const uint4*>(p.w2 + static_cast<size_t>(s.ctk[c]) * r);
            float acc = 0.0f;
#pragma unroll 8
            for (int k8 = 0; k8 < r / 8; ++k8) {
              const float4 za = *reinterpret_cast<const float4*>(zv + k8 * 8);
              const float4 zb = *reinterpret_cast<const float4*>(zv + k8 * 8 + 4);
              fma8(acc, za, zb, __ldg(w2r + k8));
            }
            const float lam = (s.cbs[c] + acc) / p.T;
            lamv[c] = lam;
            lmax_t = fmaxf(lmax_t, lam);
          }
          lmax_t = warp_max(lmax_t);
          if (lane == 0) s_tred[warp] = lmax_t;
          __syncthreads();
          CH_STAMP(i, 14);
          float lmax = rest;
          for (int w8 = 0; w8 < kWarps; ++w8) lmax = fmaxf(lmax, s_tred[w8]);
          float se_t = 0.0f;
          for (int c = tid; c < M; c += kThreads) se_t += expf(lamv[c] - lmax);
          se_t = warp_sum(se_t);
          if (lane == 0) s_tred[32 + warp] = se_t;
          __syncthreads();
          float se = expf(rest - lmax);
          for (int w8 = 0; w8 < kWarps; ++w8) se += s_tred[32 + w8];
          const float logZ = lmax + logf(se);
          for (int c = tid; c < M; c += kThreads) lamv[c] -= logZ;
          __syncthreads();
          CH_STAMP(i, 15);
          // the K best (ties to the lower token id) by a value histogram, in
          // any order (the children are ordered by token below)
          {
            uint32_t* hist = reinterpret_cast<uint32_t*>(keys);  // 256 words, then the bin's keys
            const uint64_t kth = block_kth_rank_key(lamv, M, K, hist, keys + 128, wkey_words(sh) - 128, s_tred,
                                                    s_tscan, &s_kth, s.ctk);
            if (tid == 0) s_tscan[0] = 0;
            __syncthreads();
            for (int c = tid; c < M; c += kThreads)
              if (rank_key(lamv[c], static_cast<uint32_t>(s.ctk[c])) >= kth) win[atomicAdd(&s_tscan[0], 1)] = c;
          }
          __syncthreads();
          CH_STAMP(i, 16);
          if (warp == 0) {
            int c = lane < K ? win[lane] : 0;
            if (c < 0 || c >= M) {
              dt_report(p.status, DT_DEV_BOUNDS);
              c = 0;
            }
            const int tok = lane < K ? s.ctk[c] : 0x7FFFFFFF;
            // the children in token order: each counts the winners' smaller
            // tokens (read back from shared memory)
            s_tscan[lane] = tok;
            __syncwarp();
            int trank = 0;
#pragma unroll 8
            for (int m = 0; m < K; ++m) trank += s_tscan[m] < tok ? 1 : 0;
            CH_STAMP(i, 19);
            if (lane < K) {
              const float lp = lamv[c];
              const size_t nidx = static_cast<size_t>(row_off) + b * K + trank;
              p.node_tok[nidx] = tok;
              p.node_parent[nidx] = s.pnode[b];
              p.node_logp[nidx] = lp;
              p.node_score[nidx] = s.pscore[b] + lp;
            }
          }
          CH_STAMP(i, 18);
          __syncthreads();  // z, lambda, keys are free for the next branch
        }
        CH_STAMP(i, 8);
        if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) {
          drain();
          return;
        }
        CH_STAMP(i, 9);
        // every child of the depth, from the node arrays
        for (int e = tid; e < nchild; e += kThreads) {
          const size_t nidx = static_cast<size_t>(row_off) + e;
          s.ctok[e] = __ldcg(p.node_tok + nidx);
          s.clogp[e] = __ldcg(p.node_logp + nidx);
          s.cscore[e] = __ldcg(p.node_score + nidx);
        }
      } else {
        float* zw = s.z + warp * r;
        for (int b = warp; b < Lp; b += kWarps) {
          const float* u = p.uW1 + static_cast<size_t>(q * W + b) * r;
          if (!p.marginal) {
            // all of the lane's loads first (one L2 round trip), then SiLU
            float uv[kMaxR32];
#pragma unroll
            for (int j = 0; j < kMaxR32; ++j) {
              const int k = lane + 32 * j;
              uv[j] = k < r ? u[k] : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < kMaxR32; ++j) {
              const int k = lane + 32 * j;
              if (k < r) {
                const float x = s.h1s[k] + uv[j];
                zw[k] = siluf_(x);
              }
            }
          }
          __syncwarp();
          float acc[MPL];
#pragma unroll
          for (int j = 0; j < MPL; ++j) acc[j] = 0.0f;
          // marginal scoring: no correction, lambda = base / T
          for (int k8 = 0; k8 < (p.marginal ? 0 : r / 8); ++k8) {
            const float4 za = *reinterpret_cast<const float4*>(zw + k8 * 8);
            const float4 zb = *reinterpret_cast<const float4*>(zw + k8 * 8 + 4);
#pragma unroll
            for (int j = 0; j < MPL; ++j) {
              const int c = lane + 32 * j;
              if (c < M) {
                const uint4 w8 =
                    sh.stage_w2
                        ? *reinterpret_cast<const uint4*>(s.w2s + static_cast<size_t>(c) * (r + 8) + k8 * 8)
                        : __ldg(reinterpret_cast<const uint4*>(p.w2 + static_cast<size_t>(s.ctk[c]) * r) + k8);
                fma8(acc[j], za, zb, w8);
              }
            }
          }
          float lam[MPL];
          float lmax = rest;
#pragma unroll
          for (int j = 0; j < MPL; ++j) {
            const int c = lane + 32 * j;
            lam[j] = c < M ? (s.cbs[c] + acc[j]) / p.T : -INFINITY;
            lmax = fmaxf(lmax, lam[j]);
          }
          lmax = warp_max(lmax);
          float se = 0.0f;
#pragma unroll
          for (int j = 0; j < MPL; ++j)
            if (lane + 32 * j < M) se += expf(lam[j] - lmax);
          se = warp_sum(se);
          se += expf(rest - lmax);
          const float logZ = lmax + logf(se);
          // top-K by (logp desc, token asc): K rounds of warp argmax over register keys
          uint64_t key[MPL];
          float lp[MPL];
#pragma unroll
          for (int j = 0; j < MPL; ++j) {
            const int c = lane + 32 * j;
            lp[j] = lam[j] - logZ;
            key[j] = c < M ? rank_key(lp[j], static_cast<uint32_t>(s.ctk[c])) : 0ull;
          }
          int my_c = 0;
          float my_lp = 0.0f;
          int my_tok = 0x7FFFFFFF;
          for (int kk = 0; kk < K; ++kk) {
            uint64_t best = 0;
#pragma unroll
            for (int j = 0; j < MPL; ++j) best = key[j] > best ? key[j] : best;
            best = warp_max_u64(best);
            int wc = -1;
            float wlp = 0.0f;
#pragma unroll
            for (int j = 0; j < MPL; ++j)
              if (best != 0 && key[j] == best) {
                wc = lane + 32 * j;
                wlp = lp[j];
                key[j] = 0;
              }
            const unsigned own = __ballot_sync(0xFFFFFFFFu, wc >= 0);
            const int src = own ? __ffs(own) - 1 : 0;
            wc = __shfl_sync(0xFFFFFFFFu, wc, src);
            wlp = __shfl_sync(0xFFFFFFFFu, wlp, src);
            if (lane == kk) {
              if (wc < 0 || wc >= M) {
                dt_report(p.status, DT_DEV_BOUNDS);
                wc = 0;
              }
              my_c = wc;
              my_lp = wlp;
              my_tok = static_cast<int>(rank_key_id(best));
            }
          }
          // children of branch b, sorted by token id
          const int rank = warp_rank_below(my_tok, K);
          if (lane < K) {
            const int slot = b * K + rank;
            s.ctok[slot] = my_tok;
            s.cslot[slot] = my_c;
            s.clogp[slot] = my_lp;
            s.cscore[slot] = s.pscore[b] + my_lp;
          }
          __syncwarp();
        }
      }
      __syncthreads();
      // node arrays of this depth (CTA 0, or the request's CTA; written by
      // the branches' CTAs when those are spread)
      if (!bdist && (dist || blockIdx.x == 0)) {
        const size_t nb = static_cast<size_t>(q) * p.N1 + row_off;
        for (int e = tid; e < nchild; e += kThreads) {
          p.node_tok[nb + e] = s.ctok[e];
          p.node_parent[nb + e] = s.pnode[e / K];
          p.node_logp[nb + e] = s.clogp[e];
          p.node_score[nb + e] = s.cscore[e];
        }
      }
      CH_STAMP(i, 10);
      if (!last) {
        // top-W of the depth by (score desc, node index asc); survivors ascending
        if (nchild <= 64) {
          // one warp: two children per lane ranked by counting, survivors
          // placed in slot order with two ballots (no CTA barrier)
          if (warp == 0) {
            for (int e = lane; e < 64; e += 32)
              s.wkey[e] = e < nchild ? rank_key(s.cscore[e], static_cast<uint32_t>(e)) : 0ull;
            __syncwarp();
            const uint64_t k0 = s.wkey[lane], k1 = s.wkey[lane + 32];
            int r0 = 0, r1 = 0;
#pragma unroll 8
            for (int f = 0; f < nchild; ++f) {
              const uint64_t kf = s.wkey[f];
              r0 += kf > k0 ? 1 : 0;
              r1 += kf > k1 ? 1 : 0;
            }
            const bool a0 = lane < nchild && r0 < Li, a1 = lane + 32 < nchild && r1 < Li;
            const unsigned b0 = __ballot_sync(0xFFFFFFFFu, a0), b1 = __ballot_sync(0xFFFFFFFFu, a1);
            const unsigned lt = (1u << lane) - 1u;
            if (a0) s.surv[q * W + __popc(b0 & lt)] = lane;
            if (a1) s.surv[q * W + __popc(b0) + __popc(b1 & lt)] = lane + 32;
          }
        } else if (nchild <= kRankMax) {
          // one child per thread: rank over precomputed keys, survivors (rank <
          // Li) placed in slot order with per-warp ballots
          for (int e = tid; e < nchild; e += kThreads) s.wkey[e] = rank_key(s.cscore[e], static_cast<uint32_t>(e));
          __syncthreads();
          bool alive = false;
          if (tid < nchild) {
            const uint64_t ke = s.wkey[tid];
            int rk = 0;
#pragma unroll 8
            for (int f = 0; f < nchild; ++f) rk += s.wkey[f] > ke ? 1 : 0;
            alive = rk < Li;
          }
          const unsigned bal = __ballot_sync(0xFFFFFFFFu, alive);
          if (lane == 0) s_wcnt[warp] = __popc(bal);
          __syncthreads();
          if (alive) {
            int pos = __popc(bal & ((1u << lane) - 1u));
            for (int w2 = 0; w2 < warp; ++w2) pos += s_wcnt[w2];
            s.surv[q * W + pos] = tid;
          }
        } else if ((nchild + kThreads - 1) / kThreads <= 32) {
          // many children: the Li-th best (score, node index) key by a value
          // histogram (block_kth_rank_key); the survivors, the keys at or
          // above it, are placed in slot order by a block scan over
          // consecutive children per thread
          const int npad = pow2_at_least(nchild);
          uint32_t* hist = reinterpret_cast<uint32_t*>(s.wkey);  // 256 words, then the bin's keys
          uint64_t* bnd = s.wkey + 128;
          const uint64_t kth =
              block_kth_rank_key(s.cscore, nchild, Li, hist, bnd, npad - 128, s_tred, s_tscan, &s_kth);
          CH_STAMP(i, 17);
          const int per = (nchild + kThreads - 1) / kThreads, e0 = tid * per;
          int nsv = 0;
          uint32_t msk = 0u;
          for (int j = 0; j < per; ++j) {
            const int e = e0 + j;
            if (e < nchild && rank_key(s.cscore[e], static_cast<uint32_t>(e)) >= kth) {
              msk |= 1u << j;
              ++nsv;
            }
          }
          int tot;
          int pos = block_exclusive_scan(nsv, s_tscan, &tot);
          for (int j = 0; j < per; ++j)
            if ((msk >> j) & 1u) s.surv[q * W + pos++] = e0 + j;
        } else {
          const int npad = pow2_at_least(nchild);
          for (int e = tid; e < npad; e += kThreads)
            s.wkey[e] = e < nchild ? rank_key(s.cscore[e], static_cast<uint32_t>(e)) : 0ull;
          for (int k2 = 2; k2 <= npad; k2 <<= 1) {
            for (int j = k2 >> 1; j > 0; j >>= 1) {
              __syncthreads();
              for (int x = tid; x < npad; x += kThreads) {
                const int l = x ^ j;
                if (l > x) {
                  const uint64_t a = s.wkey[x], bb = s.wkey[l];
                  const bool desc = (x & k2) == 0;
                  if (desc ? (a < bb) : (a > bb)) {
                    s.wkey[x] = bb;
                    s.wkey[l] = a;
                  }
                }
              }
            }
          }
          __syncthreads();
          // the first Li keys are the survivors; order them by slot
          for (int a = tid; a < Li; a += kThreads) {
            const int ea = static_cast<int>(rank_key_id(s.wkey[a]));
            int pos = 0;
            for (int b2 = 0; b2 < Li; ++b2) pos += static_cast<int>(rank_key_id(s.wkey[b2])) < ea;
            s.surv[q * W + pos] = ea;
          }
        }
        __syncthreads();
        CH_STAMP(i, 11);
        if (keep_par) {
          // the next depth's parents: the survivors, their node indices and
          // scores (s.pnode / s.pscore are not read again in this depth)
          for (int j = tid; j < Li; j += kThreads) {
            const int e = s.surv[q * W + j];
            s.pnode[j] = row_off + e;
            s.pscore[j] = s.cscore[e];
          }
        }
        if (dist || blockIdx.x == 0) {
          for (int j = tid; j < W; j += kThreads) {
            const int node = j < Li ? row_off + s.surv[q * W + j] : -1;
            if (j < Li) live_next[static_cast<size_t>(q) * W + j] = node;
            if (p.live_out) p.live_out[static_cast<size_t>(q) * W + j] = node;
          }
        }
        // ================= phase C (this request): GRU of the survivors ======
        for (int idx = tid; idx < (dist ? 0 : Li * nj); idx += kThreads) {
          const int jv = idx / nj, jj = idx - jv * nj;
          const int e = s.surv[q * W + jv];
          const int b = e / K;
          // the GRU-input slice: staged per candidate, or read from the
          // table by token
          const bool xt = !xs_staged(sh);
          const int xst = xt ? g : nj;
          const float* x = xt ? p.xtab + static_cast<size_t>(s.ctok[e]) * 3 * g + j0
                              : s.xs + static_cast<size_t>(s.cslot[e]) * 3 * sh.jper;
          const float* uu = s.uu + static_cast<size_t>(q * Lp + b) * 3 * sh.jper;
          const float h = Sprev[static_cast<size_t>(q * W + b) * g + j0 + jj];
          const float rg = sigmoidf_(x[jj] + uu[jj]);
          const float zg = sigmoidf_(x[xst + jj] + uu[nj + jj]);
          const float ng = tanhf_(x[2 * xst + jj] + rg * uu[2 * nj + jj]);
          const float hn = (1.0f - zg) * ng + zg * h;
          Snext[static_cast<size_t>(q * W + jv) * g + j0 + jj] = hn;
          if (sh.frag || sh.mfrag)
            store_frag(p.sfrag + static_cast<size_t>(i & 1) * n_req * W * g, q * W + jv, j0 + jj, g / 16, hn);
          if (sh.tc)
            store_tc1(reinterpret_cast<uint8_t*>(p.sfrag) + static_cast<size_t>(i & 1) * tc_nmt * (g / 64) * 2 * tc_chunk,
                      q * W + jv, j0 + jj, g / 64, tc_ts, hn);
        }
      } else if ((dist || blockIdx.x == 0) && p.live_out) {
        for (int j = tid; j < W; j += kThreads) p.live_out[static_cast<size_t>(q) * W + j] = -1;
      }
    }
    CH_STAMP(i, 3);
    if (dist && !last) {
      // ================= phase C (all requests): GRU of the survivors =====
      // the survivors (node indices) and their tokens come from the
      // requests' CTAs through global memory
      if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) {
        drain();
        return;
      }
      CH_STAMP(i, 4);
      if (sh.tc) {
        // one survivor row per thread, eight columns at a time: the loads of
        // a group are issued together, and its high and low parts go out as
        // one 16-byte piece each
        uint8_t* sb = reinterpret_cast<uint8_t*>(p.sfrag) + static_cast<size_t>(i & 1) * tc_nmt * (g / 64) * 2 * tc_chunk;
        for (int qv = tid; qv < n_req * Li; qv += kThreads) {
          const int q = qv / Li, jv = qv - q * Li;
          const int node = __ldcg(live_next + static_cast<size_t>(q) * W + jv);
          const int e = node - row_off;
          const int tok = (e >= 0 && e < Lp * K) ? __ldcg(p.node_tok + static_cast<size_t>(q) * p.N1 + node) : -1;
          if (tok < 0 || tok >= p.V) {
            dt_report(p.status, DT_DEV_BOUNDS);
            continue;
          }
          const int b = e / K;
          const float* x = p.xtab + static_cast<size_t>(tok) * 3 * g + j0;
          const float* uu = s.uu + static_cast<size_t>(q * Lp + b) * 3 * sh.jper;
          const float* hp = Sprev + static_cast<size_t>(q * W + b) * g + j0;
          float* ho = Snext + static_cast<size_t>(q * W + jv) * g + j0;
          for (int j8 = 0; j8 < nj; j8 += 8) {
            float xr[8], xz[8], xn[8], h[8], hn[8];
#pragma unroll
            for (int e4 = 0; e4 < 2; ++e4) {
              *reinterpret_cast<float4*>(xr + 4 * e4) = *reinterpret_cast<const float4*>(x + j8 + 4 * e4);
              *reinterpret_cast<float4*>(xz + 4 * e4) = *reinterpret_cast<const float4*>(x + g + j8 + 4 * e4);
              *reinterpret_cast<float4*>(xn + 4 * e4) = *reinterpret_cast<const float4*>(x + 2 * g + j8 + 4 * e4);
              *reinterpret_cast<float4*>(h + 4 * e4) = *reinterpret_cast<const float4*>(hp + j8 + 4 * e4);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
              const float rg = sigmoidf_(xr[jj] + uu[j8 + jj]);
              const float zg = sigmoidf_(xz[jj] + uu[nj + j8 + jj]);
              const float ng = tanhf_(xn[jj] + rg * uu[2 * nj + j8 + jj]);
              hn[jj] = (1.0f - zg) * ng + zg * h[jj];
            }
#pragma unroll
            for (int e4 = 0; e4 < 2; ++e4)
              *reinterpret_cast<float4*>(ho + j8 + 4 * e4) = *reinterpret_cast<const float4*>(hn + 4 * e4);
            store_tc8(sb, q * W + jv, j0 + j8, g / 64, tc_ts, hn);
          }
        }
      }
      for (int idx = tid; idx < (sh.tc ? 0 : n_req * Li * nj); idx += kThreads) {
        const int qv = idx / nj, jj = idx - qv * nj;
        const int q = qv / Li, jv = qv - q * Li;
        const int node = __ldcg(live_next + static_cast<size_t>(q) * W + jv);
        const int e = node - row_off;
        int tok = __ldcg(p.node_tok + static_cast<size_t>(q) * p.N1 + node);
        if (e < 0 || e >= Lp * K || tok < 0 || tok >= p.V) {
          dt_report(p.status, DT_DEV_BOUNDS);
          continue;
        }
        const int b = e / K;
        const float* x = p.xtab + static_cast<size_t>(tok) * 3 * g + j0 + jj;
        const float* uu = s.uu + static_cast<size_t>(q * Lp + b) * 3 * sh.jper;
        const float h = Sprev[static_cast<size_t>(q * W + b) * g + j0 + jj];
        const float rg = sigmoidf_(x[0] + uu[jj]);
        const float zg = sigmoidf_(x[g] + uu[nj + jj]);
        const float ng = tanhf_(x[2 * g] + rg * uu[2 * nj + jj]);
        const float hn = (1.0f - zg) * ng + zg * h;
        Snext[static_cast<size_t>(q * W + jv) * g + j0 + jj] = hn;
        if (sh.mfrag)
          store_frag(p.sfrag + static_cast<size_t>(i & 1) * n_req * W * g, q * W + jv, j0 + jj, g / 16, hn);
      }
    }
    if ((sh.mfrag || sh.tc) && !last) fence_proxy_async_global();  // the next depth bulk-copies these fragments
    CH_STAMP(i, 5);
    if (i < p.depth_last) {
      if (!sh.dbuf && qfirst < n_req) {
        // stage the next depth's first request of this CTA now: the copies
        // overlap the barrier
        __syncthreads();
        select_row_tokens(p, sh, s, qfirst, i + 1);
        if (!(qfirst == tokq && sh.prefetch)) __syncthreads();
        stage_row(p, sh, buf(i + 1), s.ctk, static_cast<size_t>(qfirst) * D + i, j0, nj,
                  xs_staged(sh) && i + 1 != D);
      }
      if (!grid_barrier(p.bar, epoch, p.status, &s_abort)) {
        drain();
        return;
      }
    }
    CH_STAMP(i, 6);
  }

  // ---- tail: global Top-B and tree/mask of the single request (CTA 0) ----
  if (p.fuse_tree && blockIdx.x == 0) {
    __syncthreads();
    // shared memory of the finished depth loop is reused: node keys in the
    // weight area, radix histograms in the reduction area, small arrays in
    // the state area (sizes checked by chain_can_fuse_tree)
    int* offs = reinterpret_cast<int*>(s.sh);
    int* nodes = offs + (kMaxDepth + 2);
    int* par = nodes + (p.B + 1);
    int* dep = par + (p.B + 1);
    uint32_t* anc = reinterpret_cast<uint32_t*>(dep + (p.B + 1));
    for (int k = tid; k <= D + 1; k += kThreads) offs[k] = p.off[k];
    __syncthreads();
    // candidate keys first (8-byte aligned), then the float keys
    uint64_t* tb_cands = reinterpret_cast<uint64_t*>(s.w);
    uint32_t* tb_keys = reinterpret_cast<uint32_t*>(tb_cands + (p.N1 - 1));
    topb_select(p.node_score, p.N1, p.B, p.beta, D, offs, tb_keys, tb_cands, p.N1 - 1,
                reinterpret_cast<uint32_t*>(s.red), kWarps * 256, s_state, s_tred, s_tscan, p.sel);
    tree_and_mask(p.sel, p.N1, p.B, D, offs, p.node_tok, p.node_parent, p.node_score, nullptr, nodes, par, dep, anc,
                  p.tok, p.parent, p.depth, p.logp_cum, p.mask, p.status);
  }
  if (sh.tc) {
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tmem_base, tc_cols);
  }
}

template <int MPL, class Dm>
cudaError_t launch_one(const ChainParams& p, int grid, size_t smem, cudaStream_t stream) {
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
  return cudaLaunchKernelEx(&cfg, k_chain<MPL, Dm>, p);
}

bool is_q4b(const ChainParams& p, int grid) {
  const Shape a = runtime_shape(p);
  const Shape b = DimsQ4B::kShape;
  return grid == 128 && a.g == b.g && a.r == b.r && a.M == b.M && a.K == b.K && a.W == b.W &&
         a.n_req == b.n_req && a.D == b.D && a.jper == b.jper && a.rper == b.rper && a.cpad == b.cpad &&
         a.stage_w2 == b.stage_w2 && a.mma_b == b.mma_b && a.prefetch == b.prefetch && a.dbuf == b.dbuf &&
         a.frag == b.frag && a.zf == b.zf && a.tc == b.tc;
}

}  // namespace

int chain_grid(const ChainParams& p, int num_sms) {
  if (p.marginal) return 1;  // no state: one CTA selects every depth
  // one CTA per 8 state columns, at most one per SM
  int G = (p.g + 7) / 8;
  if (G > num_sms) G = num_sms;
  if (G < 1) G = 1;
  return G;
}

size_t chain_smem_bytes(const ChainParams& p) { return smem_sizes(runtime_shape(p)).total; }

void chain_plan(ChainParams& p, int grid) {
  if (p.marginal) {
    // no GRU columns or bottleneck rows; the weight area (cpad) stays for the
    // Top-B keys of the fused tail
    p.jper = 0;
    p.rper = 0;
    p.cpad = 32;
    p.stage_w2 = 0;
    p.mma_b = 0;
    p.dbuf = (p.n_req == 1 && prefetch_tokens(p.D, p.M)) ? 1 : 0;
    return;
  }
  p.jper = (p.g + grid - 1) / grid;
  p.rper = (p.r + grid - 1) / grid;
  const int ncol = 3 * p.jper + p.rper;
  p.cpad = (ncol + 31) / 32 * 32;
  constexpr size_t kBudget = 224 * 1024;  // dynamic shared memory per CTA
  // tensor-core phase B: staged W2 rows, whole k16 steps, n8 candidate tiles,
  // z of all branches within one pass of kZLoads values per thread
  p.stage_w2 = 1;
  p.mma_b = (p.r % 16 == 0 && p.M % 8 == 0 && p.W * p.r <= kZLoads * kThreads && p.W * p.M <= 4096) ? 1 : 0;
  p.dbuf = (p.n_req == 1 && prefetch_tokens(p.D, p.M)) ? 1 : 0;
  // over the budget: give up, in order, the second stage buffer, the
  // tensor-core phase B and the W2 staging (wide candidate sets read W2 from L2)
  if (p.dbuf && chain_smem_bytes(p) > kBudget) p.dbuf = 0;
  if (p.mma_b && chain_smem_bytes(p) > kBudget) p.mma_b = 0;
  if (!p.mma_b && chain_smem_bytes(p) > kBudget) p.stage_w2 = 0;
  // tcgen05 phase A: more state rows than one A fragment holds, whole K
  // blocks of 64, every CTA owning the same whole groups of 8 state columns,
  // one tile of cpad columns per 128 rows within the 512 tensor-memory
  // columns, and 2 to 4 chunk slots within the budget
  p.tc = 0;
  p.tc_ns = 0;
  const int nmt = (p.n_req * p.W + 127) / 128;
  if (!frag_ok(p.n_req, p.W, p.g) && p.g % 64 == 0 && p.jper % 8 == 0 && p.g % p.jper == 0 &&
      p.g / p.jper == grid && p.cpad % 16 == 0 && p.cpad <= 256 && nmt * p.cpad <= 512) {
    for (int ns = 4; ns >= 2 && !p.tc; --ns) {
      p.tc = 1;
      p.tc_ns = ns;
      if (chain_smem_bytes(p) > kBudget) {
        p.tc = 0;
        p.tc_ns = 0;
      }
    }
  }
}

bool chain_can_fuse_tree(const ChainParams& p) {
  if (p.n_req != 1) return false;
  const SmemSizes L = smem_sizes(runtime_shape(p));
  const size_t weight_bytes = L.off[1] - L.off[0];     // holds the Top-B keys + candidates
  const size_t red_words = (L.off[3] - L.off[2]) / 4;  // holds the histograms
  const size_t state_bytes = L.off[2] - L.off[1];      // holds offsets, slots, ancestor rows
  const size_t S = static_cast<size_t>(p.B) + 1;
  return static_cast<size_t>(p.N1 - 1) * 12 <= weight_bytes && red_words >= static_cast<size_t>(kWarps) * 256 &&
         (static_cast<size_t>(kMaxDepth + 2) + 3 * S + S * anc_words(static_cast<int>(S))) * 4 <= state_bytes;
}

cudaError_t chain_prepare() {
  const void* fns[] = {
      reinterpret_cast<const void*>(k_chain<2, DimsQ4B>),     reinterpret_cast<const void*>(k_chain<2, DimsRuntime>),
      reinterpret_cast<const void*>(k_chain<4, DimsRuntime>), reinterpret_cast<const void*>(k_chain<8, DimsRuntime>),
      reinterpret_cast<const void*>(k_chain<16, DimsRuntime>)};
  for (const void* f : fns) {
    cudaError_t e = dt_allow_max_dynamic_smem(f);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_chain(const ChainParams& p, int grid, cudaStream_t stream) {
  const size_t smem = chain_smem_bytes(p);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  const int mpl = (p.M + 31) / 32;
  if (is_q4b(p, grid)) return launch_one<2, DimsQ4B>(p, grid, smem, stream);
  if (mpl <= 2) return launch_one<2, DimsRuntime>(p, grid, smem, stream);
  if (mpl <= 4) return launch_one<4, DimsRuntime>(p, grid, smem, stream);
  if (mpl <= 8) return launch_one<8, DimsRuntime>(p, grid, smem, stream);
  return launch_one<16, DimsRuntime>(p, grid, smem, stream);
}

}  // namespace dt

#ifdef DT_CHAIN_TIMING
// The phase stamps of the last grid-barrier chain launch: 2 x 66 x 8 values
// ([CTA 0 / last CTA][depth][stamp], clock64(); the stamps are listed where
// g_chain_stamps is defined).  Returns the number of values copied, or -1.
extern "C" int dt_chain_stamps(unsigned long long* out, int n) {
  const int total = 2 * (dt::kMaxDepth + 2) * dt::kChainStamps;
  if (!out || n < total) return -1;
  return cudaMemcpyFromSymbol(out, dt::g_chain_stamps, sizeof(dt::g_chain_stamps)) == cudaSuccess ? total : -1;
}
// The tcgen05 phase A of depth 2 in CTA 0: [copy issued / data landed /
// (slot 0) products of the depth issued][chunk], clock64().
extern "C" int dt_chain_tcstamps(unsigned long long* out, int n) {
  if (!out || n < 3 * 128) return -1;
  return cudaMemcpyFromSymbol(out, dt::g_chain_tcst, sizeof(dt::g_chain_tcst)) == cudaSuccess ? 3 * 128 : -1;
}
#endif

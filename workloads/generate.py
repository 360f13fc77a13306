"""Seeded generators of weights and per-round inputs.

Recipe (the same for the oracle and the CUDA library):

* Every weight is drawn once as N(0, 1/fan_in) in float32 and, for
  ``weight_dtype == "bf16"``, rounded to bfloat16 with round-to-nearest-even.
  Its flattened elements are drawn in chunks of 2**22; chunk c of weight k
  (k = position in ``WEIGHT_NAMES``) comes from ``default_rng([0, k, c])``, so
  the values do not depend on how many threads draw them.
  fan_in is the input width of each projection: d for the LM head, the
  embedding table and the GRU input weights, g for the GRU hidden weights,
  d+g for W1 and r for W2.  The GRU input bias is N(0, 1/g).
* Weights are stored in the out-by-in row-major layout of ``torch.nn.Linear``
  weights: ``lm_head[V, d]`` (row v is the output vector of token v),
  ``emb[V, d]``, ``w_ih[3g, d]``, ``b_ih[3g]``, ``w_hh[3g, g]``,
  ``w1[r, d+g]`` and ``w2[V, r]``.  GRU gate blocks are ordered (r, z, n).
* Round ``s`` draws from ``default_rng([1, s])``: H of shape
  [n_req, block, d] ~ N(0, 1) (times a per-position scale ~ U[0.5, 4] for the
  heavy-tailed workload) rounded to bfloat16 (kept float32 for the fp32
  workload), then one root token per request (id 0 for the tiny workload,
  uniform over the vocabulary otherwise).
* Verification inputs (the acceptance walk): random trees from
  ``default_rng([2, seed])`` and target logits from ``default_rng([3, seed])``
  (``make_tree``, ``make_target_logits``).

bfloat16 arrays are returned as their raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from .configs import WorkloadConfig

WEIGHT_NAMES = ("lm_head", "emb", "w_ih", "b_ih", "w_hh", "w1", "w2")

_CHUNK = 1 << 24  # elements per rounding chunk (bounds temporary memory)


def bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns, round to nearest, ties to even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    flat = x.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint16)
    for s in range(0, flat.size, _CHUNK):
        b = flat[s:s + _CHUNK].view(np.uint32)
        lsb = (b >> np.uint32(16)) & np.uint32(1)
        rounded = b + np.uint32(0x7FFF) + lsb
        out[s:s + _CHUNK] = (rounded >> np.uint32(16)).astype(np.uint16)
    return out.reshape(x.shape)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """bfloat16 bit patterns -> float32 (exact)."""
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def _weight_shapes(cfg: WorkloadConfig):
    d, V, g, r = cfg.d, cfg.V, cfg.g, cfg.r
    return {
        "lm_head": ((V, d), 1.0 / np.sqrt(d)),
        "emb": ((V, d), 1.0 / np.sqrt(d)),
        "w_ih": ((3 * g, d), 1.0 / np.sqrt(d)),
        "b_ih": ((3 * g,), 1.0 / np.sqrt(g)),
        "w_hh": ((3 * g, g), 1.0 / np.sqrt(g)),
        "w1": ((r, d + g), 1.0 / np.sqrt(d + g)),
        "w2": ((V, r), 1.0 / np.sqrt(r)),
    }


_DRAW_CHUNK = 1 << 22


def _draw(shape, std, seed, k, dtype):
    total = int(np.prod(shape))
    out = np.empty(total, dtype=np.uint16 if dtype == "bf16" else np.float32)

    def fill(c):
        s = c * _DRAW_CHUNK
        n = min(_DRAW_CHUNK, total - s)
        x = np.random.default_rng([seed, k, c]).standard_normal(size=n, dtype=np.float32)
        x *= np.float32(std)
        out[s:s + n] = bf16_round_bits(x) if dtype == "bf16" else x

    n_chunks = (total + _DRAW_CHUNK - 1) // _DRAW_CHUNK
    workers = max(1, min(n_chunks, os.cpu_count() or 1))
    if workers == 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(workers) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


def make_weights(cfg: WorkloadConfig, seed: int = 0, only=None) -> dict:
    """All weights of ``cfg`` (bf16 bits as uint16, or float32 arrays)."""
    shapes = _weight_shapes(cfg)
    out = {}
    for k, name in enumerate(WEIGHT_NAMES):
        if only is not None and name not in only:
            continue
        shape, std = shapes[name]
        out[name] = _draw(shape, std, seed, k, cfg.weight_dtype)
    return out


def make_round_inputs(cfg: WorkloadConfig, seed: int):
    """(H, root) for round ``seed``: H bf16 bits [n_req, block, d], root int32 [n_req]."""
    rng = np.random.default_rng([1, seed])
    H = rng.standard_normal(size=(cfg.n_req, cfg.block, cfg.d), dtype=np.float32)
    if cfg.h_scale == "heavy":
        a = rng.uniform(0.5, 4.0, size=(cfg.n_req, cfg.block)).astype(np.float32)
        H *= a[:, :, None]
    elif cfg.h_scale != "unit":
        raise ValueError(f"unknown h_scale {cfg.h_scale!r}")
    if cfg.root == "zero":
        root = np.zeros(cfg.n_req, dtype=np.int32)
    elif cfg.root == "uniform":
        root = rng.integers(0, cfg.V, size=cfg.n_req).astype(np.int32)
    else:
        raise ValueError(f"unknown root rule {cfg.root!r}")
    if cfg.weight_dtype == "fp32":
        return H, root
    return bf16_round_bits(H), root


def make_rounds(cfg: WorkloadConfig, seeds):
    """Stacked inputs of several rounds: H [n, n_req, block, d], root [n, n_req]."""
    Hs, roots = [], []
    for s in seeds:
        H, root = make_round_inputs(cfg, s)
        Hs.append(H)
        roots.append(root)
    return np.stack(Hs), np.stack(roots)


def make_tree(S: int, V: int, D: int, seed: int):
    """A random tree of S slots in the emitted-tree layout, for verification
    inputs: slot 0 is the root (parent -1, depth 0); slot c > 0 takes a parent
    uniformly among the earlier slots of depth < D; sibling tokens are distinct
    and uniform over the vocabulary.  Draws from ``default_rng([2, seed])``.
    Returns (tok, parent, depth) int32 [S]."""
    rng = np.random.default_rng([2, seed])
    tok = np.zeros(S, dtype=np.int32)
    parent = np.full(S, -1, dtype=np.int32)
    depth = np.zeros(S, dtype=np.int32)
    tok[0] = rng.integers(0, V)
    used = [set() for _ in range(S)]
    for c in range(1, S):
        open_slots = np.flatnonzero(depth[:c] < D)
        p = int(open_slots[rng.integers(0, open_slots.size)])
        t = int(rng.integers(0, V))
        while t in used[p]:
            t = int(rng.integers(0, V))
        used[p].add(t)
        tok[c], parent[c], depth[c] = t, p, depth[p] + 1
    return tok, parent, depth


def make_target_logits(tok, parent, V: int, seed: int, follow: float = 0.7, tie: bool = False):
    """Target-model logits [S, V] float32 for one tree, from
    ``default_rng([3, seed])``: N(0, 1) everywhere; at each slot with children,
    with probability ``follow`` the token of one child (uniform among them) is
    raised to the row maximum plus U(0.25, 1), so that the target agrees with
    the draft there.  With ``tie``, the raised value is also written at one
    more token of the row (uniform over the vocabulary): an exact tie at the
    maximum."""
    rng = np.random.default_rng([3, seed])
    tok = np.asarray(tok)
    parent = np.asarray(parent)
    S = tok.size
    Z = rng.standard_normal(size=(S, V), dtype=np.float32)
    kids = [[] for _ in range(S)]
    for c in range(1, S):
        kids[int(parent[c])].append(c)
    for a in range(S):
        if kids[a] and rng.random() < follow:
            c = kids[a][int(rng.integers(0, len(kids[a])))]
            v = np.float32(Z[a].max() + rng.uniform(0.25, 1.0))
            Z[a, int(tok[c])] = v
            if tie:
                Z[a, int(rng.integers(0, V))] = v
    return Z

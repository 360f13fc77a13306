"""fp64 CPU oracle of path-conditioned, depth-batched draft-tree construction.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference arm of ``bench.py`` may import or run this module.
The CUDA library never calls it and shares no code with it; the only thing the
two sides share is the seeded input generator in ``workloads/``.

What it computes, in the order the pages give it:

* Base logits.  The parallel backbone's hidden states H_i go through the frozen
  LM head: L^base_i = H_i W_lm ("Resumen Técnico: Domino", Metodología,
  "Columna Vertebral de Borrador Paralelo", Salida).  Position 0 of the block is
  the last verified token (the root); positions 1..D give depths 1..D.
* Top-M.  At each depth the correction is restricted to the M largest base
  logits ("Resumen Técnico: DominoTree", Componentes Principales, 2.
  "Restricción de Candidatos (Top-M)").  Reading: ties go to the lower token id;
  the other tokens keep their base logits and enter the log-partition through
  rho_i = log sum_{v not in C_i} exp(l_{i,v} / T).
* Domino head ("Resumen Técnico: Domino", Metodología, 2. "Cabeza de Domino"):
  a GRU causal encoder S = GRU(E[token], S_parent) (PyTorch gate order r, z, n,
  one input bias, no hidden bias, zero initial state, root token included), and
  the low-rank correction Delta L = SiLU([H_i ; S_{i-1}] W1) W2 applied to the
  Top-M columns; final logits L_i = L^base_i + Delta L_i, divided by T before
  the log-softmax.
* Depth-wise batched expansion ("DARTree: Speculative Diffusion Decoding with
  Autoregressive Draft Trees", Metodología, 1. "Expansión AR Paralela por
  Profundidad"): every live branch is scored at once, keeps its K best children,
  children carry cumulative corrected log-probabilities, and the W best children
  of the depth live on with their GRU states.  All children are nodes of the
  fixed-width super-tree.
* Marginal scoring (the conditional-versus-marginal ablation, "Resumen
  Técnico: DominoTree", Contribuciones Clave, "Ablación de la
  Condicionalidad"; the position-only scores of factorised tree drafters,
  Planteamiento del Problema): with ``cfg.marginal`` the correction is left out,
  Delta L = 0, over the same super-tree, so a node's log-probability depends
  only on its depth and token.
* Deferred pruning (same page, 2. "Poda Diferida de Mejor Primera Búsqueda"):
  one global Top-B over score + beta * depth (beta <= 0), then the compact tree
  with parent indices and the ancestor-only attention mask used for tree
  attention ("Verificación").

Node numbering: root = 0; the nodes of depth i follow all nodes of depth i-1,
ordered by (parent index, token id).  Every selection breaks ties toward the
lower token id (Top-M, per-branch top-K) or the lower node index (top-W, Top-B).

Parity pins: the functions here are checked by ``tests/test_oracle_pins.py``
against closed forms, library routines (torch GRUCell, log_softmax, SiLU),
brute-force enumeration of all paths, and an independent max-heap (Lemma 1).
"""
from __future__ import annotations

import heapq
from dataclasses import dataclass, field

import numpy as np
from scipy.special import expit, logsumexp

_V_CHUNK = 8192  # LM-head rows widened to fp64 at a time (bounds host memory)


# --------------------------------------------------------------------------
# input widening
# --------------------------------------------------------------------------
def widen(x: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) or float32 -> float64, exactly."""
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return (x.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)
    return x.astype(np.float64)


# --------------------------------------------------------------------------
# elementary functions (definitions)
# --------------------------------------------------------------------------
def sigmoid(x):
    return expit(x)


def silu(x):
    """SiLU(x) = x * sigmoid(x)."""
    return x * expit(x)


# --------------------------------------------------------------------------
# step a1: base logits through the frozen LM head
# --------------------------------------------------------------------------
def base_logits(H_rows: np.ndarray, lm_head: np.ndarray) -> np.ndarray:
    """L^base = H lm_head^T for a stack of hidden-state rows.

    H_rows: [n, d] (bf16 bits or float); lm_head: [V, d] (row v = token v).
    Returns [n, V] float64.  Exact products of the bf16-valued inputs summed in
    fp64 (Domino page, "Columna Vertebral de Borrador Paralelo", Salida).
    """
    Hf = widen(H_rows)
    V = lm_head.shape[0]
    out = np.empty((Hf.shape[0], V), dtype=np.float64)
    for s in range(0, V, _V_CHUNK):
        out[:, s:s + _V_CHUNK] = Hf @ widen(lm_head[s:s + _V_CHUNK]).T
    return out


# --------------------------------------------------------------------------
# step a2: Top-M candidates and the rest log-partition
# --------------------------------------------------------------------------
def top_m(ell: np.ndarray, M: int, T: float, swap=None):
    """Top-M candidate set of one depth (DominoTree page, Top-M restriction).

    ell: [V] base logits.  Order: value descending, then token id ascending.
    Returns (ids [M] int64 in that order, base values [M], rho) with
    rho = log sum over the non-candidates of exp(ell / T) (-inf when M == V).
    ``swap = (a, b)`` replaces candidate a by non-candidate b (near-tie flips).
    """
    V = ell.shape[0]
    order = np.lexsort((np.arange(V), -ell))
    ids = order[:M].copy()
    if swap is not None:
        a, b = swap
        at = np.where(ids == a)[0]
        if at.size != 1 or np.any(ids == b):
            raise ValueError("the flip does not apply to this candidate set")
        ids[at[0]] = b
        ids = ids[np.lexsort((ids, -ell[ids]))]
    mask = np.ones(V, dtype=bool)
    mask[ids] = False
    rest = ell[mask] / T
    rho = logsumexp(rest) if rest.size else -np.inf
    return ids, ell[ids], float(rho)


# --------------------------------------------------------------------------
# the Domino head: GRU causal encoder and low-rank correction
# --------------------------------------------------------------------------
def gru_input(tokens, emb, w_ih, b_ih) -> np.ndarray:
    """a = E[token] W_x + b_x for each token (PyTorch weight_ih layout [3g, d])."""
    E = widen(emb[np.asarray(tokens, dtype=np.int64)])
    return E @ widen(w_ih).T + widen(b_ih)


def gru_step(a: np.ndarray, h: np.ndarray, w_hh: np.ndarray) -> np.ndarray:
    """One GRU step in PyTorch's gate order (r, z, n), no hidden bias.

    r = sigmoid(a_r + u_r), z = sigmoid(a_z + u_z), n = tanh(a_n + r * u_n),
    h' = (1 - z) * n + z * h, with u = h U (Domino page, Codificador Causal).
    a: [..., 3g], h: [..., g].
    """
    g = h.shape[-1]
    u = h @ widen(w_hh).T
    r = sigmoid(a[..., :g] + u[..., :g])
    z = sigmoid(a[..., g:2 * g] + u[..., g:2 * g])
    n = np.tanh(a[..., 2 * g:] + r * u[..., 2 * g:])
    return (1.0 - z) * n + z * h


def correction(H_i: np.ndarray, S: np.ndarray, w1: np.ndarray, w2_rows: np.ndarray):
    """Delta L on the given candidate columns for each state row of S.

    z = SiLU([H_i ; S] W1) (rank r), Delta L_c = z . W2[:, c]
    (Domino page, Cabeza de Corrección de Baja Rango).
    H_i: [d]; S: [P, g]; w1: [r, d+g]; w2_rows: [M, r] (rows c of W2^T).
    Returns [P, M].
    """
    X = np.concatenate([np.broadcast_to(widen(H_i), (S.shape[0], H_i.shape[-1])), S], axis=1)
    z = silu(X @ widen(w1).T)
    return z @ widen(w2_rows).T


def corrected_logprobs(base_c: np.ndarray, dL: np.ndarray, rho: float, T: float):
    """log-softmax over the full vocabulary with the M corrected entries.

    lambda_c = (l_c + Delta L_c) / T on the candidates; the other tokens keep
    l_v / T and enter through rho.  logZ = log(e^rho + sum_c e^lambda_c).
    """
    lam = (base_c[None, :] + dL) / T
    parts = np.concatenate([np.full((lam.shape[0], 1), rho), lam], axis=1)
    logZ = logsumexp(parts, axis=1, keepdims=True)
    return lam - logZ


# --------------------------------------------------------------------------
# selections (deterministic tie rules) with near-tie recording
# --------------------------------------------------------------------------
def _select(keys: np.ndarray, ids: np.ndarray, n: int, tol, rec, tag, swap=None):
    """Indices (into keys) of the n largest keys, ties to the lower id.

    Records boundary pairs (selected, unselected) whose key gap is <= tol.
    ``swap = (id_a, id_b)`` forces id_a out and id_b in.
    """
    order = np.lexsort((ids, -keys))
    sel = list(order[:n])
    rest = list(order[n:])
    if rec is not None and tol is not None and rest and sel:
        k_last = keys[sel[-1]]
        k_first_out = keys[rest[0]]
        a_side = [a for a in reversed(sel) if keys[a] - k_first_out <= tol][:8]
        b_side = [b for b in rest if k_last - keys[b] <= tol][:8]
        for a in a_side:
            for b in b_side:
                gap = keys[a] - keys[b]
                if gap <= tol:
                    rec.append(dict(tag, a=int(ids[a]), b=int(ids[b]), gap=float(gap)))
    if swap is not None:
        pos = {int(ids[j]): j for j in range(ids.shape[0])}
        a, b = swap
        if a not in pos or b not in pos or pos[a] not in sel or pos[b] in sel:
            raise ValueError("the flip does not apply to this selection")
        sel[sel.index(pos[a])] = pos[b]
    return np.array(sel, dtype=np.int64)


# --------------------------------------------------------------------------
# the round
# --------------------------------------------------------------------------
@dataclass
class Tree:
    """One request's result: super-tree nodes and the emitted tree."""
    node_tok: np.ndarray
    node_parent: np.ndarray
    node_depth: np.ndarray
    node_logp: np.ndarray
    node_score: np.ndarray
    sel: np.ndarray
    tok: np.ndarray
    parent: np.ndarray
    depth: np.ndarray
    logp_cum: np.ndarray
    mask: np.ndarray
    cand_tok: np.ndarray = None
    cand_base: np.ndarray = None
    rest_lse: np.ndarray = None
    live: list = field(default_factory=list)


def node_count(K: int, W: int, D: int) -> int:
    """Nodes of the super-tree without the root: n_1 = K, n_i = min(W, n_{i-1}) K."""
    n, total = K, 0
    for _ in range(D):
        total += n
        n = min(W, n) * K
    return total


class Oracle:
    """Holds the weights (bf16 bits or float32) and widens them on demand."""

    def __init__(self, weights: dict, cfg):
        self.cfg = cfg
        self.w = weights
        self.w_ih = widen(weights["w_ih"])
        self.b_ih = widen(weights["b_ih"])
        self.w_hh = widen(weights["w_hh"])
        self.w1 = widen(weights["w1"])

    # -- step a1/a2 for one request ------------------------------------------
    def depth_candidates(self, H_req: np.ndarray, beta=None, T=None, ell=None, swaps=None,
                         rec=None, tol=None):
        cfg = self.cfg
        T = cfg.T if T is None else T
        D = cfg.block - 1
        if ell is None:
            ell = base_logits(H_req[1:], self.w["lm_head"])
        C, base, rho = [], [], []
        for i in range(1, D + 1):
            sw = (swaps or {}).get(("M", i))
            if rec is not None and tol is not None:
                # boundary of the Top-M set on the base logits
                order = np.lexsort((np.arange(ell.shape[1]), -ell[i - 1]))
                _select(ell[i - 1][order[:cfg.M + 8]], order[:cfg.M + 8], cfg.M, tol, rec,
                        {"stage": "M", "depth": i})
            ids, b, r = top_m(ell[i - 1], cfg.M, T, swap=sw)
            C.append(ids)
            base.append(b)
            rho.append(r)
        return ell, C, base, rho

    # -- steps a4..a6 for one request ----------------------------------------
    def build_request(self, H_req: np.ndarray, root_tok: int, beta=None, T=None, ell=None,
                      swaps=None, rec=None, tol=None) -> Tree:
        cfg = self.cfg
        beta = cfg.beta if beta is None else beta
        T = cfg.T if T is None else T
        D, M, K, W, B = cfg.block - 1, cfg.M, cfg.K, cfg.W, cfg.B
        N = node_count(K, W, D)
        if not (1 <= K <= M <= cfg.V and W >= 1 and 1 <= B <= N and T > 0):
            raise ValueError("invalid configuration")
        swaps = swaps or {}
        ell, C, base, rho = self.depth_candidates(H_req, T=T, ell=ell, swaps=swaps, rec=rec, tol=tol)
        Hf = widen(H_req)

        tok, parent, depth, logp, score = [int(root_tok)], [-1], [0], [0.0], [0.0]
        # root state: GRU over the root token from a zero state
        a_root = gru_input([root_tok], self.w["emb"], self.w_ih, self.b_ih)
        state = {0: gru_step(a_root, np.zeros((1, cfg.g)), self.w_hh)[0]}
        live = [0]
        lives = [list(live)]
        marginal = bool(getattr(cfg, "marginal", False))
        for i in range(1, D + 1):
            if marginal:
                dL = np.zeros((len(live), M))
            else:
                S = np.stack([state[p] for p in live])
                w2_rows = self.w["w2"][C[i - 1]]
                dL = correction(Hf[i], S, self.w1, w2_rows)
            lp = corrected_logprobs(base[i - 1], dL, rho[i - 1], T)
            first = len(tok)
            for bi, p in enumerate(live):
                kept = _select(lp[bi], C[i - 1], K, tol, rec,
                               {"stage": "K", "depth": i, "branch": int(p)},
                               swap=swaps.get(("K", i, int(p))))
                for c in sorted(kept, key=lambda j: C[i - 1][j]):
                    tok.append(int(C[i - 1][c]))
                    parent.append(int(p))
                    depth.append(i)
                    logp.append(float(lp[bi, c]))
                    score.append(score[p] + float(lp[bi, c]))
            if i == D:
                break
            idx = np.arange(first, len(tok))
            s_i = np.array(score[first:])
            kept = _select(s_i, idx, min(W, idx.size), tol, rec, {"stage": "W", "depth": i},
                           swap=swaps.get(("W", i)))
            live = sorted(int(idx[j]) for j in kept)
            lives.append(list(live))
            if marginal:
                continue  # no correction, no GRU state
            a = gru_input([tok[q] for q in live], self.w["emb"], self.w_ih, self.b_ih)
            hp = np.stack([state[parent[q]] for q in live])
            hn = gru_step(a, hp, self.w_hh)
            state = {q: hn[j] for j, q in enumerate(live)}

        node_tok = np.array(tok, dtype=np.int64)
        node_parent = np.array(parent, dtype=np.int64)
        node_depth = np.array(depth, dtype=np.int64)
        node_logp = np.array(logp)
        node_score = np.array(score)
        assert node_tok.size == N + 1
        sel = top_b(node_score, node_depth, B, beta, tol=tol, rec=rec, swap=swaps.get(("B",)))
        t = compact_tree(node_tok, node_parent, node_depth, node_score, sel)
        return Tree(node_tok, node_parent, node_depth, node_logp, node_score, sel, *t,
                    cand_tok=np.stack(C), cand_base=np.stack(base), rest_lse=np.array(rho),
                    live=lives)

    def build_round(self, H: np.ndarray, root: np.ndarray, beta=None, T=None, ell=None):
        """All requests of one round. H [n_req, block, d]; root [n_req]."""
        trees = []
        for q in range(H.shape[0]):
            trees.append(self.build_request(H[q], int(root[q]), beta=beta, T=T,
                                            ell=None if ell is None else ell[q]))
        return trees


# --------------------------------------------------------------------------
# step a5: global Top-B; step a6: compaction and ancestor mask
# --------------------------------------------------------------------------
def top_b(score, depth, B, beta, tol=None, rec=None, swap=None):
    """B non-root nodes with the largest score + beta * depth, ties to the lower
    index, returned in ascending index order (DARTree page, Selección Global)."""
    key = score[1:] + beta * depth[1:]
    idx = np.arange(1, score.shape[0])
    kept = _select(key, idx, B, tol, rec, {"stage": "B"}, swap=swap)
    return np.sort(idx[kept])


def compact_tree(node_tok, node_parent, node_depth, node_score, sel):
    """Root plus the selected nodes in index order, parents remapped, and the
    ancestor-only mask: mask[a, b] = 1 iff b is an ancestor of a or a itself
    (DominoTree page, Verificación; DARTree page, Verificación)."""
    nodes = np.concatenate([[0], sel]).astype(np.int64)
    pos = {int(v): k for k, v in enumerate(nodes)}
    n = nodes.size
    tok = node_tok[nodes]
    depth = node_depth[nodes]
    logp_cum = node_score[nodes]
    parent = np.empty(n, dtype=np.int64)
    for k, v in enumerate(nodes):
        p = int(node_parent[v])
        parent[k] = -1 if p < 0 else pos.get(p, -2)
    mask = np.zeros((n, n), dtype=np.uint8)
    for a in range(n):
        b = a
        while b >= 0:
            mask[a, b] = 1
            b = int(parent[b])
            if b == -2:
                raise ValueError("selected set is not ancestor-closed")
    return tok, parent, depth, logp_cum, mask


# --------------------------------------------------------------------------
# Lemma 1 counterpart: sequential max-heap best-first over the same super-tree
# --------------------------------------------------------------------------
def heap_best_first(node_parent, node_score, node_depth, B, beta):
    """DominoTree-style best-first: pop the best key, push its materialised
    children; B pops.  Ties go to the lower node index.  Returns the popped
    node set in ascending order (DominoTree page, Montículo de Mejor Primera
    Búsqueda; DARTree page, Equivalencia Teórica)."""
    n = node_parent.shape[0]
    children = [[] for _ in range(n)]
    for v in range(1, n):
        children[int(node_parent[v])].append(v)
    heap = []
    for c in children[0]:
        heapq.heappush(heap, (-(node_score[c] + beta * node_depth[c]), c))
    out = []
    while heap and len(out) < B:
        _, v = heapq.heappop(heap)
        out.append(v)
        for c in children[v]:
            heapq.heappush(heap, (-(node_score[c] + beta * node_depth[c]), c))
    return np.sort(np.array(out, dtype=np.int64))


# --------------------------------------------------------------------------
# near-tie exclusion rule
# --------------------------------------------------------------------------
def near_tie_report(oracle: Oracle, H_req, root_tok, tol=1e-3, beta=None, T=None, ell=None):
    """Near-ties at selection boundaries and whether flipping one changes the tree.

    Returns dict(literal=bool, relevant=bool, n_ties=int, relevant_ties=[...]).
    A tie is outcome-relevant when swapping that single pair in the oracle and
    re-running the rest of the round changes the emitted tokens, parents or
    depths.
    """
    rec = []
    base = oracle.build_request(H_req, root_tok, beta=beta, T=T, ell=ell, rec=rec, tol=tol)
    ell = ell if ell is not None else base_logits(H_req[1:], oracle.w["lm_head"])
    relevant = []
    for t in rec:
        key = {"M": ("M", t.get("depth")), "K": ("K", t.get("depth"), t.get("branch")),
               "W": ("W", t.get("depth")), "B": ("B",)}[t["stage"]]
        try:
            alt = oracle.build_request(H_req, root_tok, beta=beta, T=T, ell=ell,
                                       swaps={key: (t["a"], t["b"])})
        except ValueError:
            relevant.append(t)
            continue
        if not _same_tree(alt, base):
            relevant.append(t)
    return dict(literal=bool(rec), relevant=bool(relevant), n_ties=len(rec),
                ties=rec, relevant_ties=relevant, tree=base)


def _same_tree(a, b) -> bool:
    """The emitted trees agree: same tokens, parent slots and depths."""
    return (a.tok.shape == b.tok.shape and np.array_equal(a.tok, b.tok)
            and np.array_equal(a.parent, b.parent) and np.array_equal(a.depth, b.depth))

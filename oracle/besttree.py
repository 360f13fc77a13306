"""fp64 CPU oracle of the sequential conditional best-first heap builder.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference arm of ``bench.py`` may import or run this module.
The CUDA library never calls it and shares no code with it.

What it computes ("Resumen Técnico: DominoTree", Metodología, 1. Montículo de
Mejor Primera Búsqueda con Puntuación Condicional; 2. Restricción de
Candidatos; 4. CondAdaptive: a fixed node budget): the node-by-node tree that
the depth-batched builder replaces ("DARTree: Speculative Diffusion Decoding
with Autoregressive Draft Trees", Contribuciones Clave, 1.; Resultados
Experimentales, Ablación, Latencia).  A max-priority queue holds the frontier,
keyed by the cumulative corrected log-probability of the path (plus beta *
depth, beta <= 0, as in the depth-batched builder's selection; beta = 0 is the
plain heap).  Steps, per request:

1. The root's state S = GRU(E[t_0], 0); the root is expanded: its K children
   at depth 1 are the K best corrected log-probabilities over the Top-M
   candidates of depth 1, computed from the root's state (the correction,
   log-partition and tie rules are the depth-batched builder's).
2. Repeat B times: pop the frontier node v with the largest key (equal keys:
   the lower node index).  Unless v is the B-th pop or sits at depth D, its
   state S(v) = GRU(E[tok v], S(parent v)) is computed and v is expanded the
   same way at depth(v) + 1; the children enter the frontier with score
   s(v) + logp.
3. The tree is the root plus the B popped nodes, in ascending node index (a
   child is always created after its parent), with the ancestor-only mask.

Node numbering: root = 0; an expansion appends its K children in ascending
token id.  With cfg.marginal the correction is left out (Delta L = 0).

Pins (``tests/test_oracle_besttree.py``): the popped set equals the B best
keys over the whole K-restricted tree found by breadth-first enumeration with
independent path scoring; with W >= K^(D-1) it equals the depth-batched
builder's tree; popped keys never increase (beta <= 0); planted mistakes.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import dartree as _dartree
from .dartree import (Oracle, _select, compact_tree, correction, corrected_logprobs, gru_input,
                      gru_step, widen)


@dataclass
class HeapTree:
    node_tok: np.ndarray
    node_parent: np.ndarray
    node_depth: np.ndarray
    node_logp: np.ndarray
    node_score: np.ndarray
    pops: list            # popped node indices in pop order
    sel: np.ndarray       # popped nodes, ascending
    tok: np.ndarray
    parent: np.ndarray
    depth: np.ndarray
    logp_cum: np.ndarray
    mask: np.ndarray
    expanded: list = field(default_factory=list)  # expanded nodes in order (root first)


def build_best_first(orc: Oracle, H_req, root_tok: int, B=None, beta=None, T=None, ell=None,
                     swaps=None, rec=None, tol=None) -> HeapTree:
    """One request's tree by sequential conditional best-first expansion."""
    cfg = orc.cfg
    B = cfg.B if B is None else B
    beta = cfg.beta if beta is None else beta
    T = cfg.T if T is None else T
    D, M, K = cfg.block - 1, cfg.M, cfg.K
    full = sum(K ** i for i in range(1, D + 1))
    if not (1 <= K <= M <= cfg.V and 1 <= B <= full and T > 0):
        raise ValueError("invalid configuration")
    swaps = swaps or {}
    marginal = bool(getattr(cfg, "marginal", False))
    _, C, base, rho = orc.depth_candidates(H_req, T=T, ell=ell, swaps=swaps, rec=rec, tol=tol)
    Hf = widen(H_req)

    tok, parent, depth, logp, score = [int(root_tok)], [-1], [0], [0.0], [0.0]
    a_root = gru_input([root_tok], orc.w["emb"], orc.w_ih, orc.b_ih)
    state = {0: gru_step(a_root, np.zeros((1, cfg.g)), orc.w_hh)[0]}
    frontier = []
    expanded = []

    def expand(v):
        d = depth[v] + 1
        if marginal:
            dL = np.zeros((1, M))
        else:
            dL = correction(Hf[d], state[v][None], orc.w1, orc.w["w2"][C[d - 1]])
        lp = corrected_logprobs(base[d - 1], dL, rho[d - 1], T)[0]
        kept = _select(lp, C[d - 1], K, tol, rec, {"stage": "K", "node": int(v)},
                       swap=swaps.get(("K", int(v))))
        for c in sorted(kept, key=lambda j: C[d - 1][j]):
            tok.append(int(C[d - 1][c]))
            parent.append(int(v))
            depth.append(d)
            logp.append(float(lp[c]))
            score.append(score[v] + float(lp[c]))
            frontier.append(len(tok) - 1)
        expanded.append(int(v))

    expand(0)
    pops = []
    while len(pops) < B and frontier:
        ids = np.array(frontier, dtype=np.int64)
        keys = np.array([score[u] + beta * depth[u] for u in frontier])
        j = int(_select(keys, ids, 1, tol, rec, {"stage": "P", "pop": len(pops)},
                        swap=swaps.get(("P", len(pops))))[0])
        v = frontier.pop(j)
        pops.append(v)
        if len(pops) == B or depth[v] == D:
            continue
        a = gru_input([tok[v]], orc.w["emb"], orc.w_ih, orc.b_ih)
        state[v] = gru_step(a, state[parent[v]][None], orc.w_hh)[0]
        expand(v)

    node_tok = np.array(tok, dtype=np.int64)
    node_parent = np.array(parent, dtype=np.int64)
    node_depth = np.array(depth, dtype=np.int64)
    node_score = np.array(score)
    sel = np.sort(np.array(pops, dtype=np.int64))
    t = compact_tree(node_tok, node_parent, node_depth, node_score, sel)
    return HeapTree(node_tok, node_parent, node_depth, np.array(logp), node_score, pops, sel, *t,
                    expanded=expanded)


def best_first_tie_report(orc: Oracle, H_req, root_tok, tol=1e-3, B=None, beta=None, T=None, ell=None):
    """Near-ties of the best-first build within tol at a selection boundary
    (Top-M set, an expansion's top-K, a pop) and whether flipping that single
    decision changes the emitted tokens, parents or depths."""
    rec = []
    base = build_best_first(orc, H_req, root_tok, B=B, beta=beta, T=T, ell=ell, rec=rec, tol=tol)
    relevant = []
    for t in rec:
        key = {"M": ("M", t.get("depth")), "K": ("K", t.get("node")), "P": ("P", t.get("pop"))}[t["stage"]]
        try:
            alt = build_best_first(orc, H_req, root_tok, B=B, beta=beta, T=T, ell=ell,
                                   swaps={key: (t["a"], t["b"])})
        except (ValueError, KeyError):
            relevant.append(t)
            continue
        if not _dartree._same_tree(alt, base):
            relevant.append(t)
    return dict(literal=bool(rec), relevant=bool(relevant), n_ties=len(rec), ties=rec, relevant_ties=relevant,
                tree=base)

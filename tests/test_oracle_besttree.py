"""Pins of the sequential best-first heap builder oracle (``oracle/besttree.py``), no GPU.

The builder ("Resumen Técnico: DominoTree", Metodología, 1. Montículo de
Mejor Primera Búsqueda con Puntuación Condicional) is pinned by:

* enumeration: breadth-first over the whole K-restricted tree, every node's
  children and path score computed independently with torch layers (the
  GRU re-run from the root along the path); the popped set must be the B
  best keys over that whole tree, ties aside, for beta in {0, -0.25, -1};
* the depth-batched builder with W >= K^(D-1) (a complete super-tree) selects
  the same tree (Lemma 1 of "DARTree ...", Equivalencia Teórica);
* keys of successive pops never increase when beta <= 0;
* planted mistakes in the oracle, each caught by one of the pins above.
"""
import numpy as np
import pytest
import torch

import oracle.besttree as ob
import oracle.dartree as od
from tests._bruteforce import PathScorer
from workloads import get_config, make_round_inputs, make_weights


def _small_cfg(**kw):
    # T = 0.3 sharpens the tiny drafter enough that the trees go several levels
    # deep and beta changes the selected set
    base = dict(block=5, K=3, M=6, W=27, B=20, T=0.3)
    base.update(kw)
    return get_config("tiny").with_(**base)


def _paths(t):
    out = set()
    for v in t.sel:
        path, u = [], int(v)
        while u > 0:
            path.append(int(t.node_tok[u]))
            u = int(t.node_parent[u])
        out.add(tuple(reversed(path)))
    return out


def _enumerate(ps, H, root, cfg, beta):
    """Every node of the K-restricted tree: path -> key (score + beta * depth)."""
    D, K = cfg.block - 1, cfg.K
    keys = {}
    level = [()]
    for _ in range(D):
        nxt = []
        for path in level:
            for t in ps.children(H, root, list(path), K):
                p2 = path + (t,)
                keys[p2] = ps.path_score(H, root, list(p2)) + beta * len(p2)
                nxt.append(p2)
        level = nxt
    return keys


def _pin_enumeration(seeds=(0, 1, 2), betas=(0.0, -0.25, -1.0)):
    cfg = _small_cfg()
    w = make_weights(cfg)
    orc = od.Oracle(w, cfg)
    ps = PathScorer(w, cfg)
    for s in seeds:
        H, root = make_round_inputs(cfg, s)
        for beta in betas:
            keys = _enumerate(ps, H[0], int(root[0]), cfg, beta)
            ranked = sorted(keys.items(), key=lambda kv: -kv[1])
            gap = ranked[cfg.B - 1][1] - ranked[cfg.B][1]
            if gap < 1e-9:
                continue  # a tie at the budget boundary: either set is valid
            want = {p for p, _ in ranked[:cfg.B]}
            t = ob.build_best_first(orc, H[0], int(root[0]), beta=beta)
            assert _paths(t) == want, (s, beta)
            # every materialised node's score is its path score
            for v in range(1, t.node_tok.size):
                path, u = [], v
                while u > 0:
                    path.append(int(t.node_tok[u]))
                    u = int(t.node_parent[u])
                p = tuple(reversed(path))
                assert abs(t.node_score[v] + beta * len(p) - keys[p]) < 1e-10


def _pin_lemma1(seeds=(3, 4, 5)):
    cfg = _small_cfg()  # W = 27 = K^(D-1): the depth-batched super-tree is complete
    w = make_weights(cfg)
    orc = od.Oracle(w, cfg)
    for s in seeds:
        H, root = make_round_inputs(cfg, s)
        for beta in (0.0, -0.5):
            a = ob.build_best_first(orc, H[0], int(root[0]), beta=beta)
            b = orc.build_request(H[0], int(root[0]), beta=beta)
            assert _paths(a) == {tuple(int(b.node_tok[u]) for u in _anc(b, v)) for v in b.sel}, (s, beta)


def _anc(t, v):
    out = []
    while v > 0:
        out.append(int(v))
        v = int(t.node_parent[v])
    return list(reversed(out))


def _pin_monotone(seeds=(6, 7)):
    cfg = get_config("tiny").with_(B=40)
    w = make_weights(cfg)
    orc = od.Oracle(w, cfg)
    for s in seeds:
        H, root = make_round_inputs(cfg, s)
        for beta in (0.0, -0.3):
            t = ob.build_best_first(orc, H[0], int(root[0]), beta=beta)
            k = [t.node_score[v] + beta * t.node_depth[v] for v in t.pops]
            assert all(k[i] >= k[i + 1] - 1e-12 for i in range(len(k) - 1))
            assert len(t.pops) == cfg.B and len(set(t.pops)) == cfg.B


def test_popped_set_is_best_over_whole_tree():
    _pin_enumeration()


def test_equals_depth_batched_with_complete_super_tree():
    _pin_lemma1()


def test_pop_keys_never_increase():
    _pin_monotone()


def test_tree_is_ancestor_closed_with_mask():
    cfg = get_config("tiny")
    w = make_weights(cfg)
    orc = od.Oracle(w, cfg)
    H, root = make_round_inputs(cfg, 8)
    t = ob.build_best_first(orc, H[0], int(root[0]))
    n = cfg.B + 1
    assert t.tok.size == n and t.parent[0] == -1
    assert all(0 <= t.parent[k] < k for k in range(1, n))
    assert (t.mask.sum(axis=1) == t.depth + 1).all()


def test_marginal_best_first_children_are_path_independent():
    cfg = get_config("tiny").with_(marginal=True)
    w = make_weights(cfg)
    orc = od.Oracle(w, cfg)
    H, root = make_round_inputs(cfg, 9)
    t = ob.build_best_first(orc, H[0], int(root[0]))
    by_depth = {}
    for v in t.expanded:
        kids = [(int(t.node_tok[c]), round(float(t.node_logp[c]), 12))
                for c in range(1, t.node_tok.size) if t.node_parent[c] == v]
        by_depth.setdefault(int(t.node_depth[v]), []).append(kids)
    for lists in by_depth.values():
        assert all(k == lists[0] for k in lists)


def _planted(name):
    real = ob.build_best_first
    if name == "parent_state":  # expands a popped node with its parent's state
        def f(orc, H_req, root_tok, **kw):
            real_gru = ob.gru_step
            ob.gru_step = lambda a, h, w_hh: h if a.shape[0] == 1 and h.any() else real_gru(a, h, w_hh)
            try:
                return real(orc, H_req, root_tok, **kw)
            finally:
                ob.gru_step = real_gru
        return f
    if name == "min_heap":  # pops the smallest key
        def f(orc, H_req, root_tok, **kw):
            real_sel = ob._select
            def sel(keys, ids, n, tol, rec, tag, swap=None):
                if tag.get("stage") == "P":
                    return real_sel(-keys, ids, n, tol, rec, tag, swap)
                return real_sel(keys, ids, n, tol, rec, tag, swap)
            ob._select = sel
            try:
                return real(orc, H_req, root_tok, **kw)
            finally:
                ob._select = real_sel
        return f
    if name == "beta_ignored":
        def f(orc, H_req, root_tok, **kw):
            kw["beta"] = 0.0
            return real(orc, H_req, root_tok, **kw)
        return f
    raise KeyError(name)


@pytest.mark.parametrize("name", ["parent_state", "min_heap", "beta_ignored"])
def test_planted_mistakes_are_caught(monkeypatch, name):
    monkeypatch.setattr(ob, "build_best_first", _planted(name))
    caught = 0
    for pin in (_pin_enumeration, _pin_lemma1, _pin_monotone):
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught >= 1, name

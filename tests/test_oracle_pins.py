"""Pins of the fp64 oracle against things other than itself.

Each ``check_*`` function raises AssertionError when the oracle disagrees with
a closed form, a library routine, brute-force enumeration or a theorem from
the pages.  ``test_planted_mistakes_are_caught`` plants plausible mistakes in
the oracle (on the CPU) and shows that every one of them trips a check.
"""
from __future__ import annotations

import itertools
import math

import numpy as np
import pytest
import torch

import oracle.dartree as od
from tests._bruteforce import PathScorer, node_path
from workloads import get_config, make_weights, make_round_inputs, bf16_bits_to_f32, bf16_round_bits


def _f64(x):
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_bits_to_f32(x).astype(np.float64)
    return x.astype(np.float64)


def small_cfg(**kw):
    base = dict(d=16, V=12, block=5, g=8, r=8, M=3, K=3, W=27, B=20, beta=0.0, T=1.0,
                root="uniform", weight_dtype="fp32")
    base.update(kw)
    return get_config("tiny").with_(name="small", **base)


# ----------------------------------------------------------------------------
# input conversions
# ----------------------------------------------------------------------------
def test_widen_exact_bf16_values():
    bits = np.array([0x3F80, 0xC000, 0x3F81, 0x0000, 0x8000, 0x4049], dtype=np.uint16)
    got = od.widen(bits)
    want = [1.0, -2.0, 1.0 + 2.0 ** -7, 0.0, -0.0, 3.140625]
    assert got.tolist() == want


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2.0 ** -8,          # exact tie -> even (1.0)
                  1.0 + 3 * 2.0 ** -8,      # exact tie -> even (1.015625)
                  1.0 + 2.0 ** -8 + 2.0 ** -20,  # above tie -> up
                  -2.5, 3.0e-3], dtype=np.float32)
    got = bf16_bits_to_f32(bf16_round_bits(x)).astype(np.float64)
    assert got[0] == 1.0
    assert got[1] == 1.015625
    assert got[2] == 1.0 + 2.0 ** -7
    assert got[3] == -2.5
    assert abs(got[4] - 3.0e-3) <= 3.0e-3 * 2.0 ** -8


# ----------------------------------------------------------------------------
# LM head / Top-M / rest log-partition
# ----------------------------------------------------------------------------
def check_base_logits(mod):
    rng = np.random.default_rng(5)
    H = bf16_round_bits(rng.standard_normal((3, 20)).astype(np.float32))
    W = bf16_round_bits(rng.standard_normal((37, 20)).astype(np.float32))
    got = mod.base_logits(H, W)
    Hf, Wf = _f64(H), _f64(W)
    for i in range(3):
        for v in range(37):
            want = math.fsum(float(Hf[i, k]) * float(Wf[v, k]) for k in range(20))
            assert abs(got[i, v] - want) <= 1e-12 * (1 + abs(want))


def test_base_logits_brute_force():
    check_base_logits(od)


def check_top_m_ties(mod):
    ell = np.array([0.5, 2.0, 1.0, 2.0, -1.0, 1.0, 1.0, 0.0])
    ids, vals, _ = mod.top_m(ell, 4, 1.0)
    assert ids.tolist() == [1, 3, 2, 5]
    assert vals.tolist() == [2.0, 2.0, 1.0, 1.0]
    ids, _, _ = mod.top_m(ell, 5, 1.0)
    assert ids.tolist() == [1, 3, 2, 5, 6]


def test_top_m_tie_rule():
    check_top_m_ties(od)


def check_top_m_brute_and_partition(mod):
    rng = np.random.default_rng(11)
    for T in (1.0, 0.6, 2.5):
        ell = np.round(rng.standard_normal(40) * 3, 1)  # rounding makes ties common
        for M in (1, 5, 17, 39):
            ids, vals, rho = mod.top_m(ell, M, T)
            want = sorted(range(40), key=lambda v: (-ell[v], v))[:M]
            assert ids.tolist() == want
            full = math.log(math.fsum(math.exp(x / T) for x in ell))
            cand = [math.exp(ell[v] / T) for v in want]
            both = math.log(math.exp(rho) + math.fsum(cand))
            assert abs(both - full) <= 1e-12 * max(1.0, abs(full))
        ids, vals, rho = mod.top_m(ell, 40, T)
        assert rho == -np.inf


def test_top_m_brute_force_and_partition():
    check_top_m_brute_and_partition(od)


def check_selection_ties(mod):
    keys = np.array([1.0, 2.0, 2.0, 2.0, 0.0, 2.0])
    ids = np.array([10, 7, 3, 5, 1, 9])
    sel = mod._select(keys, ids, 2, None, None, {})
    assert sorted(ids[sel].tolist()) == [3, 5]
    sel = mod._select(keys, ids, 5, None, None, {})
    assert sorted(ids[sel].tolist()) == [3, 5, 7, 9, 10]
    score = np.array([0.0, -1.0, -1.0, -0.5, -1.0, -1.0])
    depth = np.array([0, 1, 1, 1, 2, 2])
    assert mod.top_b(score, depth, 3, 0.0).tolist() == [1, 2, 3]
    assert mod.top_b(score, depth, 2, -1.0).tolist() == [1, 3]


def test_selection_tie_rule():
    check_selection_ties(od)


# ----------------------------------------------------------------------------
# GRU
# ----------------------------------------------------------------------------
def _gru_case(seed=3, d=6, g=5, n=4):
    rng = np.random.default_rng(seed)
    w_ih = rng.standard_normal((3 * g, d))
    b_ih = rng.standard_normal(3 * g)
    w_hh = rng.standard_normal((3 * g, g))
    x = rng.standard_normal((n, d))
    h = rng.standard_normal((n, g))
    return w_ih, b_ih, w_hh, x, h


def check_gru_torch(mod):
    w_ih, b_ih, w_hh, x, h = _gru_case()
    d, g = x.shape[1], h.shape[1]
    cell = torch.nn.GRUCell(d, g, bias=True, dtype=torch.float64)
    with torch.no_grad():
        cell.weight_ih.copy_(torch.from_numpy(w_ih))
        cell.bias_ih.copy_(torch.from_numpy(b_ih))
        cell.weight_hh.copy_(torch.from_numpy(w_hh))
        cell.bias_hh.zero_()
        want = cell(torch.from_numpy(x), torch.from_numpy(h)).numpy()
    a = x @ w_ih.T + b_ih
    got = mod.gru_step(a, h, w_hh)
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


def test_gru_matches_torch_grucell():
    check_gru_torch(od)


def check_gru_zero_state(mod):
    rng = np.random.default_rng(4)
    g = 7
    a = rng.standard_normal((3, 3 * g))
    w_hh = rng.standard_normal((3 * g, g))
    got = mod.gru_step(a, np.zeros((3, g)), w_hh)
    want = (1.0 - 1.0 / (1.0 + np.exp(-a[:, g:2 * g]))) * np.tanh(a[:, 2 * g:])
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-14)


def test_gru_zero_state_closed_form():
    check_gru_zero_state(od)


def test_gru_scalar_hand_expanded():
    # g = d = 1: a = (0.3, -0.2, 0.5), h = 0.4, U = (0.7, -1.1, 0.9)
    a = np.array([[0.3, -0.2, 0.5]])
    h = np.array([[0.4]])
    U = np.array([[0.7], [-1.1], [0.9]])
    r = 1 / (1 + math.exp(-(0.3 + 0.28)))
    z = 1 / (1 + math.exp(-(-0.2 - 0.44)))
    n = math.tanh(0.5 + r * 0.36)
    want = (1 - z) * n + z * 0.4
    assert abs(od.gru_step(a, h, U)[0, 0] - want) < 1e-15


# ----------------------------------------------------------------------------
# correction head and corrected log-softmax
# ----------------------------------------------------------------------------
def check_correction_torch(mod):
    rng = np.random.default_rng(8)
    d, g, r, V, P = 9, 6, 5, 14, 3
    H_i = rng.standard_normal(d)
    S = rng.standard_normal((P, g))
    w1 = rng.standard_normal((r, d + g))
    w2 = rng.standard_normal((V, r))
    cand = np.array([3, 11, 0, 7])
    got = mod.correction(H_i, S, w1, w2[cand])
    X = torch.cat([torch.from_numpy(H_i)[None].expand(P, d), torch.from_numpy(S)], dim=1)
    z = torch.nn.functional.silu(torch.nn.functional.linear(X, torch.from_numpy(w1)))
    full = torch.nn.functional.linear(z, torch.from_numpy(w2)).numpy()
    np.testing.assert_allclose(got, full[:, cand], rtol=0, atol=1e-12)


def test_correction_matches_torch_layers():
    check_correction_torch(od)


def check_logprob_full_vocab(mod):
    rng = np.random.default_rng(9)
    V = 12
    for T in (1.0, 0.6):
        ell = rng.standard_normal(V) * 2
        dL = rng.standard_normal((3, V))
        ids, base, rho = mod.top_m(ell, V, T)
        got = mod.corrected_logprobs(base, dL[:, ids], rho, T)
        want = torch.log_softmax(torch.from_numpy((ell[None, :] + dL) / T), dim=1).numpy()[:, ids]
        np.testing.assert_allclose(got, want, rtol=0, atol=1e-13)


def test_corrected_logsoftmax_full_vocab_is_log_softmax():
    check_logprob_full_vocab(od)


def check_logprob_partial_vocab(mod):
    rng = np.random.default_rng(10)
    V, M = 30, 7
    for T in (1.0, 0.6, 1.7):
        ell = rng.standard_normal(V) * 2
        ids, base, rho = mod.top_m(ell, M, T)
        dL = rng.standard_normal((4, M))
        got = mod.corrected_logprobs(base, dL, rho, T)
        full = np.tile(ell, (4, 1))
        full[:, ids] += dL
        want = torch.log_softmax(torch.from_numpy(full / T), dim=1).numpy()
        np.testing.assert_allclose(got, want[:, ids], rtol=0, atol=1e-13)
        assert np.all(got <= 0)


def test_corrected_logsoftmax_partial_vocab_normalised():
    check_logprob_partial_vocab(od)


def test_silu_matches_torch():
    x = np.linspace(-30, 30, 121)
    np.testing.assert_allclose(od.silu(x), torch.nn.functional.silu(torch.from_numpy(x)).numpy(),
                               rtol=1e-15, atol=1e-300)


# ----------------------------------------------------------------------------
# expansion: brute force over every path
# ----------------------------------------------------------------------------
def _round(cfg, seed=0, wseed=0):
    w = make_weights(cfg, seed=wseed)
    H, root = make_round_inputs(cfg, seed)
    return w, H[0], int(root[0])


def check_complete_supertree(mod, beta=0.0, T=1.0, seed=0):
    cfg = small_cfg(beta=beta, T=T)
    w, H, root = _round(cfg, seed)
    tree = mod.Oracle(w, cfg).build_request(H, root)
    ps = PathScorer(w, cfg)
    D, K = cfg.block - 1, cfg.K
    cands = []
    h = ps.root_state(root)
    for i in range(1, D + 1):
        _, cand = ps.depth_logprobs(H, i, h)
        cands.append(sorted(int(c) for c in cand))
    all_paths = [p for k in range(1, D + 1) for p in itertools.product(*cands[:k])]
    assert len(all_paths) == tree.node_tok.size - 1
    got = {node_path(tree.node_tok, tree.node_parent, v): tree.node_score[v]
           for v in range(1, tree.node_tok.size)}
    assert set(got) == set(all_paths)
    score = {p: ps.path_score(H, root, p) for p in all_paths}
    for p in all_paths:
        assert abs(got[p] - score[p]) <= 1e-12 * max(1.0, abs(score[p]))
    keyed = sorted(all_paths, key=lambda p: -(score[p] + beta * len(p)))[: cfg.B]
    sel = {node_path(tree.node_tok, tree.node_parent, int(v)) for v in tree.sel}
    assert sel == set(keyed)


def test_complete_supertree_equals_brute_force():
    check_complete_supertree(od)
    check_complete_supertree(od, beta=-0.7, T=0.6, seed=3)


def check_pruned_supertree(mod, cfg, seed=0, T=None):
    w, H, root = _round(cfg, seed)
    tree = mod.Oracle(w, cfg).build_request(H, root, T=T)
    ps = PathScorer(w, cfg, T=T)
    n = tree.node_tok.size
    for v in range(1, n):
        p = node_path(tree.node_tok, tree.node_parent, v)
        want = ps.path_score(H, root, p)
        assert abs(tree.node_score[v] - want) <= 1e-11 * max(1.0, abs(want))
    # every expanded node has exactly the brute-force top-K children
    kids = {}
    for v in range(1, n):
        kids.setdefault(int(tree.node_parent[v]), []).append(int(tree.node_tok[v]))
    for p, toks in kids.items():
        path = node_path(tree.node_tok, tree.node_parent, p) if p else ()
        assert sorted(toks) == ps.children(H, root, path, cfg.K)
    # live sets are the top-W of each depth by score (ties -> lower index)
    for i, live in enumerate(tree.live[1:], start=1):
        idx = np.where(tree.node_depth == i)[0]
        order = sorted(idx, key=lambda v: (-tree.node_score[v], v))[: cfg.W]
        assert sorted(int(v) for v in order) == live


def test_pruned_supertree_scores_match_brute_force():
    check_pruned_supertree(od, small_cfg(W=2, K=2, M=4, B=6))
    check_pruned_supertree(od, get_config("tiny"))


def check_node_order(mod, cfg, seed=1):
    w, H, root = _round(cfg, seed)
    t = mod.Oracle(w, cfg).build_request(H, root)
    n = t.node_tok.size
    for v in range(2, n):
        a = (t.node_depth[v - 1], t.node_parent[v - 1], t.node_tok[v - 1])
        b = (t.node_depth[v], t.node_parent[v], t.node_tok[v])
        assert a < b, (v, a, b)
    assert np.all(t.node_parent[1:] < np.arange(1, n))


def test_node_order_is_parent_then_token():
    check_node_order(od, get_config("tiny"))


def check_mask(mod, cfg, seed=2):
    w, H, root = _round(cfg, seed)
    t = mod.Oracle(w, cfg).build_request(H, root)
    n = cfg.B + 1
    assert t.mask.shape == (n, n)
    assert np.all(np.diag(t.mask) == 1)
    assert np.all(np.triu(t.mask, 1) == 0)
    assert t.parent[0] == -1 and t.depth[0] == 0
    for a in range(1, n):
        assert t.mask[a, t.parent[a]] == 1
        assert t.mask[a].sum() == t.depth[a] + 1
        assert t.depth[a] == t.depth[t.parent[a]] + 1
    assert np.all(np.diff(t.sel) > 0)


def test_tree_mask_invariants():
    check_mask(od, get_config("tiny"))


# ----------------------------------------------------------------------------
# Lemma 1: global Top-B equals sequential best-first when beta <= 0
# ----------------------------------------------------------------------------
def _independent_heap(parent, key, B):
    import heapq
    n = parent.size
    kids = [[] for _ in range(n)]
    for v in range(1, n):
        kids[parent[v]].append(v)
    h = [(-key[c], c) for c in kids[0]]
    heapq.heapify(h)
    out = []
    while h and len(out) < B:
        _, v = heapq.heappop(h)
        out.append(v)
        for c in kids[v]:
            heapq.heappush(h, (-key[c], c))
    return sorted(out)


def check_lemma1(mod, cfg, seeds, betas):
    for s in seeds:
        w, H, root = _round(cfg, s)
        orc = mod.Oracle(w, cfg)
        t = orc.build_request(H, root, beta=0.0)
        for beta in betas:
            key = t.node_score + beta * t.node_depth
            sel = mod.top_b(t.node_score, t.node_depth, cfg.B, beta)
            heap = mod.heap_best_first(t.node_parent, t.node_score, t.node_depth, cfg.B, beta)
            assert sel.tolist() == heap.tolist()
            assert sel.tolist() == _independent_heap(t.node_parent, key, cfg.B)
            chosen = set(sel.tolist()) | {0}
            assert all(int(t.node_parent[v]) in chosen for v in sel)


def test_lemma1_heap_equals_global_top_b():
    check_lemma1(od, get_config("tiny"), seeds=range(6), betas=(0.0, -0.25, -1.0))
    wide_small = small_cfg(d=32, V=600, block=6, g=16, r=16, M=64, K=8, W=16, B=96)
    check_lemma1(od, wide_small, seeds=range(3), betas=(0.0, -0.25, -1.0))


def test_lemma1_negative_control_positive_beta():
    cfg = get_config("tiny")
    found = False
    for s in range(8):
        w, H, root = _round(cfg, s)
        t = od.Oracle(w, cfg).build_request(H, root, beta=0.0)
        sel = od.top_b(t.node_score, t.node_depth, cfg.B, 5.0)
        heap = od.heap_best_first(t.node_parent, t.node_score, t.node_depth, cfg.B, 5.0)
        if sel.tolist() != heap.tolist():
            found = True
            break
    assert found, "beta > 0 never broke the heap equivalence: the Lemma 1 check is vacuous"


# ----------------------------------------------------------------------------
# special cases
# ----------------------------------------------------------------------------
def test_zero_correction_is_path_independent():
    cfg = get_config("tiny")
    w = make_weights(cfg)
    w["w2"] = np.zeros_like(w["w2"])
    H, root = make_round_inputs(cfg, 4)
    t = od.Oracle(w, cfg).build_request(H[0], int(root[0]))
    for i in range(1, cfg.block):
        idx = np.where(t.node_depth == i)[0]
        groups = {}
        for v in idx:
            groups.setdefault(int(t.node_parent[v]), []).append((int(t.node_tok[v]), t.node_logp[v]))
        ref = None
        for p, kids in groups.items():
            toks = [k for k, _ in kids]
            lps = np.array([lp for _, lp in kids])
            if ref is None:
                ref = (toks, lps)
            assert toks == ref[0]
            np.testing.assert_allclose(lps, ref[1], rtol=0, atol=1e-13)
        # marginal scoring: children are the K best base logits of the depth
        ell = od.base_logits(H[0][i:i + 1], w["lm_head"])[0]
        top = sorted(range(cfg.V), key=lambda v: (-ell[v], v))[: cfg.K]
        assert sorted(top) == ref[0]


@pytest.mark.parametrize("seed", [4, 9])
def test_marginal_mode_equals_zeroed_correction(seed):
    """Marginal scoring (Delta L = 0 by flag) builds exactly the tree of the
    conditional build whose W2 is zero, which runs the whole correction and
    GRU path; the two share nothing but the inputs."""
    cfg = get_config("tiny")
    w = make_weights(cfg)
    H, root = make_round_inputs(cfg, seed)
    tm = od.Oracle(w, cfg.with_(marginal=True)).build_request(H[0], int(root[0]))
    w0 = dict(w)
    w0["w2"] = np.zeros_like(w["w2"])
    tz = od.Oracle(w0, cfg).build_request(H[0], int(root[0]))
    for k in ("node_tok", "node_parent", "node_depth", "sel", "tok", "parent", "depth", "mask"):
        assert np.array_equal(getattr(tm, k), getattr(tz, k)), k
    np.testing.assert_allclose(tm.node_score, tz.node_score, rtol=0, atol=1e-12)
    # and it differs from the conditional tree of the real W2 (the ablation is not vacuous)
    tc = od.Oracle(w, cfg).build_request(H[0], int(root[0]))
    assert not np.allclose(tm.node_score, tc.node_score)


def test_single_branch_is_a_chain_of_corrected_argmax():
    cfg = get_config("tiny").with_(K=1, W=1, B=7)
    w = make_weights(cfg)
    H, root = make_round_inputs(cfg, 6)
    t = od.Oracle(w, cfg).build_request(H[0], int(root[0]))
    assert t.node_tok.size == cfg.block
    assert t.parent.tolist() == [-1] + list(range(cfg.block - 1))
    ps = PathScorer(w, cfg)
    h = ps.root_state(int(root[0]))
    for i in range(1, cfg.block):
        lp, _ = ps.depth_logprobs(H[0], i, h)
        best = int(torch.argmax(lp))
        assert best == int(t.tok[i])
        h = ps.gru(ps.emb[best][None], h[None])[0]


def test_node_count():
    assert od.node_count(4, 4, 7) == 100
    assert od.node_count(8, 8, 15) == 904
    assert od.node_count(16, 16, 15) == 3600
    assert od.node_count(32, 64, 15) == 27680


# ----------------------------------------------------------------------------
# planted mistakes: each must trip at least one check above
# ----------------------------------------------------------------------------
def _gru_swapped_gates(a, h, w_hh):
    g = h.shape[-1]
    u = h @ od.widen(w_hh).T
    z = od.sigmoid(a[..., :g] + u[..., :g])
    r = od.sigmoid(a[..., g:2 * g] + u[..., g:2 * g])
    n = np.tanh(a[..., 2 * g:] + r * u[..., 2 * g:])
    return (1 - z) * n + z * h


def _gru_no_reset(a, h, w_hh):
    g = h.shape[-1]
    u = h @ od.widen(w_hh).T
    z = od.sigmoid(a[..., g:2 * g] + u[..., g:2 * g])
    n = np.tanh(a[..., 2 * g:] + u[..., 2 * g:])
    return (1 - z) * n + z * h


def _gru_swapped_mix(a, h, w_hh):
    g = h.shape[-1]
    u = h @ od.widen(w_hh).T
    r = od.sigmoid(a[..., :g] + u[..., :g])
    z = od.sigmoid(a[..., g:2 * g] + u[..., g:2 * g])
    n = np.tanh(a[..., 2 * g:] + r * u[..., 2 * g:])
    return z * n + (1 - z) * h


def _logp_no_rest(base_c, dL, rho, T):
    lam = (base_c[None, :] + dL) / T
    from scipy.special import logsumexp
    return lam - logsumexp(lam, axis=1, keepdims=True)


def _logp_T_on_base_only(base_c, dL, rho, T):
    lam = base_c[None, :] / T + dL
    from scipy.special import logsumexp
    parts = np.concatenate([np.full((lam.shape[0], 1), rho), lam], axis=1)
    return lam - logsumexp(parts, axis=1, keepdims=True)


def _correction_no_state(H_i, S, w1, w2_rows):
    X = np.concatenate([np.broadcast_to(od.widen(H_i), (S.shape[0], H_i.shape[-1])),
                        np.zeros_like(S)], axis=1)
    return od.silu(X @ od.widen(w1).T) @ od.widen(w2_rows).T


def _correction_relu(H_i, S, w1, w2_rows):
    X = np.concatenate([np.broadcast_to(od.widen(H_i), (S.shape[0], H_i.shape[-1])), S], axis=1)
    return np.maximum(X @ od.widen(w1).T, 0) @ od.widen(w2_rows).T


def _top_m_high_id_ties(ell, M, T, swap=None):
    V = ell.shape[0]
    order = np.lexsort((-np.arange(V), -ell))
    ids = order[:M]
    mask = np.ones(V, dtype=bool)
    mask[ids] = False
    from scipy.special import logsumexp
    rest = ell[mask] / T
    return ids, ell[ids], float(logsumexp(rest)) if rest.size else -np.inf


def _top_m_rho_all(ell, M, T, swap=None):
    ids, vals, _ = _REAL["top_m"](ell, M, T, swap)
    from scipy.special import logsumexp
    return ids, vals, float(logsumexp(ell / T))


def _top_m_rho_untempered(ell, M, T, swap=None):
    ids, vals, _ = _REAL["top_m"](ell, M, T, swap)
    mask = np.ones(ell.shape[0], dtype=bool)
    mask[ids] = False
    from scipy.special import logsumexp
    return ids, vals, float(logsumexp(ell[mask])) if mask.any() else -np.inf


def _top_b_no_beta(score, depth, B, beta, tol=None, rec=None, swap=None):
    return _REAL["top_b"](score, depth, B, 0.0, tol=tol, rec=rec, swap=swap)


def _base_logits_shifted(H_rows, lm_head):
    # uses the hidden state of the previous block position (an off-by-one)
    return _REAL["base_logits"](np.roll(H_rows, 1, axis=0), lm_head)


def _select_high_index(keys, ids, n, tol, rec, tag, swap=None):
    order = np.lexsort((-ids, -keys))
    return np.array(order[:n], dtype=np.int64)


_REAL = {"top_m": od.top_m, "top_b": od.top_b, "base_logits": od.base_logits}

_MUTANTS = [
    ("gru_step", _gru_swapped_gates),
    ("gru_step", _gru_no_reset),
    ("gru_step", _gru_swapped_mix),
    ("corrected_logprobs", _logp_no_rest),
    ("corrected_logprobs", _logp_T_on_base_only),
    ("correction", _correction_no_state),
    ("correction", _correction_relu),
    ("top_m", _top_m_high_id_ties),
    ("top_m", _top_m_rho_all),
    ("top_m", _top_m_rho_untempered),
    ("top_b", _top_b_no_beta),
    ("base_logits", _base_logits_shifted),
    ("_select", _select_high_index),
]


def _all_checks():
    yield lambda: check_base_logits(od)
    yield lambda: check_top_m_ties(od)
    yield lambda: check_selection_ties(od)
    yield lambda: check_top_m_brute_and_partition(od)
    yield lambda: check_gru_torch(od)
    yield lambda: check_gru_zero_state(od)
    yield lambda: check_correction_torch(od)
    yield lambda: check_logprob_full_vocab(od)
    yield lambda: check_logprob_partial_vocab(od)
    yield lambda: check_complete_supertree(od)
    yield lambda: check_complete_supertree(od, beta=-0.7, T=0.6, seed=3)
    yield lambda: check_pruned_supertree(od, small_cfg(W=2, K=2, M=4, B=6))
    yield lambda: check_node_order(od, get_config("tiny"))
    yield lambda: check_lemma1(od, small_cfg(d=16, V=40, block=5, M=6, K=3, W=4, B=12),
                               seeds=range(2), betas=(-1.0,))


@pytest.mark.parametrize("name,fn", _MUTANTS, ids=[f"{n}:{f.__name__}" for n, f in _MUTANTS])
def test_planted_mistakes_are_caught(monkeypatch, name, fn):
    monkeypatch.setattr(od, name, fn)
    caught = False
    for check in _all_checks():
        try:
            check()
        except (AssertionError, ValueError, IndexError):
            caught = True
            break
    assert caught, f"planted mistake {fn.__name__} in {name} passed every pin"


@pytest.mark.slow
@pytest.mark.parametrize("name", ["qwen3_4b", "wide"])
def test_lemma1_full_scale(name):
    """Lemma 1 at the benchmarked sizes (DARTree page, Poda Diferida,
    Equivalencia Teórica): over the oracle's own super-tree of seeds 0-2 at the
    Qwen3-4B shape (904 nodes, B = 64) and the wide tree (27 680 nodes,
    B = 512), the global Top-B equals the oracle's heap and an independent heap
    for beta in {0, -0.25, -1}, and the selection is ancestor-closed."""
    cfg = get_config(name)
    w = make_weights(cfg)
    orc = od.Oracle(w, cfg)
    for s in range(3):
        H, root = make_round_inputs(cfg, s)
        t = orc.build_request(H[0], int(root[0]), beta=0.0)
        assert t.node_tok.size == od.node_count(cfg.K, cfg.W, cfg.block - 1) + 1
        for beta in (0.0, -0.25, -1.0):
            key = t.node_score + beta * t.node_depth
            sel = od.top_b(t.node_score, t.node_depth, cfg.B, beta)
            heap = od.heap_best_first(t.node_parent, t.node_score, t.node_depth, cfg.B, beta)
            assert sel.tolist() == heap.tolist(), (name, s, beta)
            assert sel.tolist() == _independent_heap(t.node_parent, key, cfg.B), (name, s, beta)
            chosen = set(sel.tolist()) | {0}
            assert all(int(t.node_parent[v]) in chosen for v in sel), (name, s, beta)

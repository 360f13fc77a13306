"""GPU parity of greedy tree verification (``dt_accept_walk``) against the oracle.

The walk ("Resumen Técnico: DominoTree", Metodología, 5. Verificación;
Resultados Experimentales, Ausencia de Pérdida) is integer work decided by fp32
comparisons that both sides make on the same fp32 logits, so the bar is
bit-exact: target token per slot, accepted slots, accepted length and bonus
token.  Inputs: random trees and target logits with planted agreement (and
planted exact ties at the row maximum) from ``workloads``, and trees the oracle
builds; shapes from the tiny case (with a vocabulary that is not a multiple of
4: the scalar path) to the Qwen3-4B shape, the wide tree and the 32-request
batch.
"""
import numpy as np
import pytest

from tests.parity import upload_weights
from workloads import get_config, make_round_inputs, make_target_logits, make_tree, make_weights

pytestmark = pytest.mark.gpu


def _builder(cfg, w=None):
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    torch.cuda.set_device(0)
    w = make_weights(cfg) if w is None else w
    return DraftTreeBuilder(cfg, upload_weights(w))


def _inputs(cfg, seed, follow, tie):
    S, D = cfg.B + 1, cfg.block - 1
    toks, pars, Zs = [], [], []
    for q in range(cfg.n_req):
        s = seed * 1000 + q
        tok, parent, _ = make_tree(S, cfg.V, D, s)
        toks.append(tok)
        pars.append(parent)
        Zs.append(make_target_logits(tok, parent, cfg.V, s, follow=follow, tie=tie))
    return np.stack(toks), np.stack(pars), np.stack(Zs)


def _run_and_compare(b, cfg, tok, parent, Z):
    import torch
    from oracle.accept import accept_walk
    D = cfg.block - 1
    S = cfg.B + 1
    td = torch.from_numpy(tok.astype(np.int32)).cuda()
    pd = torch.from_numpy(parent.astype(np.int32)).cuda()
    Zd = torch.from_numpy(Z).cuda()
    ttok = torch.empty(cfg.n_req, S, dtype=torch.int32, device="cuda")
    out = b.accept_walk(Zd, td, pd, target_tok=ttok)
    torch.cuda.synchronize()
    acc = out["accepted"].cpu().numpy()
    alen = out["accept_len"].cpu().numpy()
    bon = out["bonus"].cpu().numpy()
    tt = ttok.cpu().numpy()
    lens = []
    for q in range(cfg.n_req):
        v = accept_walk(tok[q], parent[q], Z[q])
        assert tt[q].tolist() == v.target_tok.tolist(), f"request {q}: target tokens"
        assert int(alen[q]) == len(v.accepted), f"request {q}: accepted length"
        assert acc[q].tolist() == v.accepted + [-1] * (D - len(v.accepted)), f"request {q}: path"
        assert int(bon[q]) == v.bonus, f"request {q}: bonus"
        lens.append(len(v.accepted))
    assert b.device_status() == 0
    return lens


@pytest.mark.parametrize("V", [1000, 1002])
def test_tiny_walks(V):
    cfg = get_config("tiny_bf16", V=V)
    b = _builder(cfg)
    try:
        lens = []
        for seed in range(24):
            tok, parent, Z = _inputs(cfg, seed, follow=(0.0, 0.6, 1.0)[seed % 3], tie=seed % 2 == 1)
            lens += _run_and_compare(b, cfg, tok, parent, Z)
        assert max(lens) >= 2 and min(lens) == 0
    finally:
        b.close()


@pytest.fixture(scope="module")
def q4b():
    cfg = get_config("qwen3_4b")
    w = make_weights(cfg)
    b = _builder(cfg, w)
    yield cfg, w, b
    b.close()


def test_qwen4b_walks(q4b):
    cfg, _, b = q4b
    lens = []
    for seed in range(8):
        tok, parent, Z = _inputs(cfg, seed, follow=(0.5, 0.9, 1.0, 0.0)[seed % 4], tie=seed % 2 == 0)
        lens += _run_and_compare(b, cfg, tok, parent, Z)
    assert max(lens) >= 3


def test_qwen4b_walk_over_oracle_trees(q4b):
    """Trees the oracle builds from the same weights and hidden states, target
    logits that follow the draft at most slots."""
    from oracle.dartree import Oracle
    cfg, w, b = q4b
    orc = Oracle(w, cfg)
    for seed in range(2):
        H, root = make_round_inputs(cfg, seed)
        t = orc.build_request(H[0], int(root[0]))
        tok, parent = t.tok[None].astype(np.int32), t.parent[None].astype(np.int32)
        Z = make_target_logits(tok[0], parent[0], cfg.V, 50 + seed, follow=0.9)[None]
        lens = _run_and_compare(b, cfg, tok, parent, Z)
        assert lens[0] >= 1


def test_wide_walks():
    cfg = get_config("wide")
    b = _builder(cfg)
    try:
        for seed in range(3):
            tok, parent, Z = _inputs(cfg, seed, follow=0.95, tie=seed == 1)
            _run_and_compare(b, cfg, tok, parent, Z)
    finally:
        b.close()


def test_serving32_walks():
    cfg = get_config("serving32")
    b = _builder(cfg)
    try:
        tok, parent, Z = _inputs(cfg, 0, follow=0.8, tie=True)
        lens = _run_and_compare(b, cfg, tok, parent, Z)
        assert len(set(lens)) >= 2
    finally:
        b.close()

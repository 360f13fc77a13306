"""GPU parity of marginal scoring (DT_FLAG_MARGINAL) against the fp64 oracle.

Marginal scoring leaves the path correction out ("Resumen Técnico:
DominoTree", Contribuciones Clave, "Ablación de la Condicionalidad"): a
child's log-probability is lambda_c = ell_c / T normalised against the rest
log-partition, the same for every branch of a depth.  Checked here:

* tiny shape, stage by stage: node arrays, live lists, Top-B and the tree
  against the oracle in marginal mode, and the captured round equal to the
  stage-by-stage one (bit for bit but for the log-probs' last bits when the
  round keeps the Top-M in the LM-head GEMM's epilogue);
* Qwen3-4B shape: whole rounds against the oracle;
* at any size: every branch of a depth gets the same children (tokens and
  log-probabilities bit for bit), and the children's log-probabilities are the
  oracle's marginal ones.

Same bar as the other GPU parity tests: tokens, parents, depths and masks
bit-exact and scores within 2e-3, unless the oracle shows an outcome-relevant
near-tie (window 1e-3).
"""
import numpy as np
import pytest

from tests.parity import LOGP_TOL, check_round, to_np, upload_round, upload_weights
from workloads import get_config, make_round_inputs, make_weights

pytestmark = pytest.mark.gpu


def _builder(cfg, w):
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    torch.cuda.set_device(0)
    return DraftTreeBuilder(cfg, upload_weights(w))


def _stepwise_nodes(b, cfg, Hd, rd):
    import torch
    D = cfg.block - 1
    logits = torch.empty(cfg.n_req, D, cfg.V, dtype=torch.float32, device="cuda")
    b.base_logits(Hd, logits)
    ct = torch.empty(cfg.n_req, D, cfg.M, dtype=torch.int32, device="cuda")
    cb = torch.empty(cfg.n_req, D, cfg.M, dtype=torch.float32, device="cuda")
    rl = torch.empty(cfg.n_req, D, dtype=torch.float32, device="cuda")
    b.topm(None, ct, cb, rl)
    nodes = b.new_nodes()
    live = torch.empty(cfg.n_req, cfg.W, dtype=torch.int32, device="cuda")
    lives = []
    for i in range(1, D + 1):
        b.expand_depth(i, rd, nodes["node_tok"], nodes["node_parent"], nodes["node_logp"],
                       nodes["node_score"], live)
        lives.append(live.cpu().numpy()[0].tolist())
    return nodes, lives


def _offsets(K, W, D):
    """off[i]: first node index of depth i (the root is node 0); off[D+1] = N+1."""
    off = [0, 1]
    n = K
    for _ in range(D):
        off.append(off[-1] + n)
        n = min(W, n) * K
    return off


def _children_by_branch(nn, off, i, K):
    """Per parent at depth i: the (token, logp bits) list of its children."""
    toks = nn["node_tok"][0][off[i]:off[i + 1]]
    lps = nn["node_logp"][0][off[i]:off[i + 1]].view(np.uint32)
    par = nn["node_parent"][0][off[i]:off[i + 1]]
    out = {}
    for e in range(toks.size):
        out.setdefault(int(par[e]), []).append((int(toks[e]), int(lps[e])))
    return out


def _check_marginal_property(nn, off, D, K):
    for i in range(2, D + 1):
        groups = list(_children_by_branch(nn, off, i, K).values())
        for gch in groups[1:]:
            assert gch == groups[0], f"depth {i}: branches differ under marginal scoring"


@pytest.mark.parametrize("seed", range(4))
def test_tiny_marginal_stages(seed):
    import torch
    from oracle.dartree import Oracle, base_logits
    cfg = get_config("tiny_bf16", marginal=True)
    w = make_weights(cfg)
    orc = Oracle(w, cfg)
    b = _builder(cfg, w)
    try:
        D = cfg.block - 1
        H, root = make_round_inputs(cfg, seed)
        Hd, rd = upload_round(H, root)
        ell = base_logits(H[0][1:], w["lm_head"])
        nodes, lives = _stepwise_nodes(b, cfg, Hd, rd)
        nn = to_np(nodes)
        t = orc.build_request(H[0], int(root[0]), ell=ell)
        _check_marginal_property(nn, _offsets(cfg.K, cfg.W, D), D, cfg.K)
        sel = torch.empty(cfg.n_req, cfg.B, dtype=torch.int32, device="cuda")
        b.prune_topB(nodes["node_score"], sel)
        tree = b.new_tree()
        b.tree_mask(sel, nodes["node_tok"], nodes["node_parent"], nodes["node_score"], tree["tok"],
                    tree["parent"], tree["depth"], tree["logp_cum"], tree["mask"])
        gt = to_np(tree)
        verdict = check_round(orc, gt, H, root, ells=[ell])
        assert verdict[0][0] != "MISMATCH", verdict
        if verdict[0][0] == "match":
            assert nn["node_tok"][0].tolist() == t.node_tok.tolist()
            assert nn["node_parent"][0].tolist() == t.node_parent.tolist()
            np.testing.assert_allclose(nn["node_logp"][0], t.node_logp, rtol=0, atol=LOGP_TOL)
            np.testing.assert_allclose(nn["node_score"][0], t.node_score, rtol=0, atol=LOGP_TOL)
            assert sel.cpu().numpy()[0].tolist() == t.sel.tolist()
            for i in range(1, D):
                want = list(t.live[i]) + [-1] * (cfg.W - len(t.live[i]))
                assert lives[i - 1] == want, f"live list after depth {i}"
        # (with the Top-M in the GEMM's epilogue the log-partition's terms are
        # added in another order: the same tree, log-probs to fp32 rounding)
        whole = to_np(b.build_round(Hd, rd))
        fused = "epilogue" in b.plan()
        for k in gt:
            if fused and k == "logp_cum":
                np.testing.assert_allclose(whole[k], gt[k], rtol=0, atol=1e-5)
            else:
                assert np.array_equal(whole[k], gt[k]), k
        assert b.device_status() == 0
    finally:
        b.close()


@pytest.fixture(scope="module")
def q4m():
    from oracle.dartree import Oracle
    cfg = get_config("qwen3_4b_marginal")
    w = make_weights(cfg)
    b = _builder(cfg, w)
    yield cfg, w, b, Oracle(w, cfg)
    b.close()


def test_qwen4b_marginal_rounds(q4m):
    from oracle.dartree import base_logits
    cfg, w, b, orc = q4m
    counts = {"match": 0, "excused": 0, "MISMATCH": 0}
    details = []
    for s in range(3):
        H, root = make_round_inputs(cfg, s)
        ells = [base_logits(H[0][1:], w["lm_head"])]
        out = to_np(b.build_round(*upload_round(H, root)))
        for st, why in check_round(orc, out, H, root, ells=ells):
            counts[st] += 1
            details.append((s, st, why))
    assert counts["MISMATCH"] == 0, details
    assert counts["match"] >= 2, details
    assert b.device_status() == 0


def test_qwen4b_marginal_children_shared(q4m):
    """Full size: identical children per depth; their log-probs are the
    oracle's marginal values ell_c / T - logZ of the depth."""
    from oracle.dartree import base_logits
    cfg, w, b, orc = q4m
    D = cfg.block - 1
    H, root = make_round_inputs(cfg, 5)
    Hd, rd = upload_round(H, root)
    nodes, _ = _stepwise_nodes(b, cfg, Hd, rd)
    nn = to_np(nodes)
    ell = base_logits(H[0][1:], w["lm_head"])
    off = _offsets(cfg.K, cfg.W, D)
    _check_marginal_property(nn, off, D, cfg.K)
    # every child's log-prob equals the oracle's marginal log-prob of its token
    for i in range(1, D + 1):
        row = ell[i - 1].astype(np.float64) / cfg.T
        lse = np.logaddexp.reduce(row)
        toks = nn["node_tok"][0][off[i]:off[i + 1]]
        np.testing.assert_allclose(nn["node_logp"][0][off[i]:off[i + 1]], row[toks] - lse,
                                   rtol=0, atol=LOGP_TOL)
    assert b.device_status() == 0

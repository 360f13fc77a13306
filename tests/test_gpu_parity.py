"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Tolerances: base logits within 2e-4 absolute (bf16 products are exact in fp32;
fp32 tensor-core accumulation over d terms of unit-order logits stays ~1e-5),
rest log-partition within 1e-4, node log-probs and cumulative scores within
2e-3 absolute; token ids, parents, depths, selections and masks bit-exact
unless the oracle shows an outcome-relevant near-tie (window 1e-3).
"""
import numpy as np
import pytest

from tests.parity import LOGP_TOL, check_round, report_counts, to_np, upload_round, upload_weights
from workloads import get_config, make_round_inputs, make_weights

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-4
REST_TOL = 1e-4


@pytest.fixture(scope="module")
def torch_cuda():
    import torch
    torch.cuda.set_device(0)
    return torch


def _builder(cfg, w):
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    return DraftTreeBuilder(cfg, upload_weights(w))


# ----------------------------------------------------------------------------
# tiny shape, every stage
# ----------------------------------------------------------------------------
@pytest.fixture(scope="module")
def tiny(torch_cuda):
    from oracle.dartree import Oracle
    cfg = get_config("tiny_bf16")
    w = make_weights(cfg)
    b = _builder(cfg, w)
    yield cfg, w, b, Oracle(w, cfg)
    b.close()


def _topm_boundary_gap(ell_row, M):
    s = np.sort(ell_row)[::-1]
    return s[M - 1] - s[M] if M < s.size else np.inf


@pytest.mark.parametrize("seed", range(6))
def test_tiny_stages(tiny, seed):
    import torch
    from oracle.dartree import base_logits
    cfg, w, b, orc = tiny
    D = cfg.block - 1
    H, root = make_round_inputs(cfg, seed)
    Hd, rd = upload_round(H, root)
    logits = torch.empty(cfg.n_req, D, cfg.V, dtype=torch.float32, device="cuda")
    b.base_logits(Hd, logits)
    ell = base_logits(H[0][1:], w["lm_head"])
    np.testing.assert_allclose(logits[0].cpu().numpy(), ell, rtol=0, atol=LOGIT_TOL)

    ct = torch.empty(cfg.n_req, D, cfg.M, dtype=torch.int32, device="cuda")
    cb = torch.empty(cfg.n_req, D, cfg.M, dtype=torch.float32, device="cuda")
    rl = torch.empty(cfg.n_req, D, dtype=torch.float32, device="cuda")
    b.topm(None, ct, cb, rl)
    t = orc.build_request(H[0], int(root[0]), ell=ell)
    ct_n, cb_n, rl_n = ct.cpu().numpy()[0], cb.cpu().numpy()[0], rl.cpu().numpy()[0]
    for i in range(D):
        if _topm_boundary_gap(ell[i], cfg.M) > 1e-3:
            assert ct_n[i].tolist() == t.cand_tok[i].tolist(), f"depth {i + 1}"
            np.testing.assert_allclose(cb_n[i], t.cand_base[i], rtol=0, atol=LOGIT_TOL)
            assert abs(rl_n[i] - t.rest_lse[i]) <= REST_TOL

    nodes = b.new_nodes()
    live = torch.empty(cfg.n_req, cfg.W, dtype=torch.int32, device="cuda")
    lives = []
    for i in range(1, D + 1):
        b.expand_depth(i, rd, nodes["node_tok"], nodes["node_parent"], nodes["node_logp"],
                       nodes["node_score"], live)
        lives.append(live.cpu().numpy()[0].tolist())
    nn = to_np(nodes)
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
        assert lives[D - 1] == [-1] * cfg.W
    # the captured round reproduces the step-by-step results: bit for bit
    # where both take the Top-M kernel; with the Top-M in the GEMM's epilogue
    # the log-partition adds the same terms in another order, so the tree is
    # the same and its log-probs agree to fp32 rounding
    whole = to_np(b.build_round(Hd, rd))
    fused = "epilogue" in b.plan()
    for k in gt:
        if fused and k == "logp_cum":
            np.testing.assert_allclose(whole[k], gt[k], rtol=0, atol=1e-5)
        else:
            assert np.array_equal(whole[k], gt[k]), k
    assert b.device_status() == 0


def test_tiny_many_rounds_whole(tiny):
    cfg, w, b, orc = tiny
    counts = {"match": 0, "excused": 0, "MISMATCH": 0}
    for seed in range(6, 40):
        H, root = make_round_inputs(cfg, seed)
        Hd, rd = upload_round(H, root)
        out = to_np(b.build_round(Hd, rd))
        for st, _ in check_round(orc, out, H, root):
            counts[st] += 1
    assert counts["MISMATCH"] == 0, counts
    assert counts["match"] >= 30, counts


def test_tiny_host_buffers_round(tiny):
    import torch
    cfg, w, b, orc = tiny
    H, root = make_round_inputs(cfg, 3)
    Hh = torch.from_numpy(H.view(np.int16)).view(torch.bfloat16).pin_memory()
    rh = torch.from_numpy(root.astype(np.int32)).pin_memory()
    out_h = {k: v.cpu().pin_memory() for k, v in b.new_tree().items()}
    b.build_round_host(Hh, rh, out_h)
    Hd, rd = upload_round(H, root)
    dev = to_np(b.build_round(Hd, rd))
    for k in dev:
        assert np.array_equal(out_h[k].numpy(), dev[k]), k


# ----------------------------------------------------------------------------
# Qwen3-4B shape (the benchmarked workload)
# ----------------------------------------------------------------------------
@pytest.fixture(scope="module")
def qwen4b(torch_cuda):
    from oracle.dartree import Oracle
    cfg = get_config("qwen3_4b")
    w = make_weights(cfg)
    b = _builder(cfg, w)
    yield cfg, w, b, Oracle(w, cfg)
    b.close()


def test_qwen4b_logits_and_topm(qwen4b):
    import torch
    from oracle.dartree import base_logits, top_m
    cfg, w, b, orc = qwen4b
    D = cfg.block - 1
    H, root = make_round_inputs(cfg, 0)
    Hd, rd = upload_round(H, root)
    logits = torch.empty(cfg.n_req, D, cfg.V, dtype=torch.float32, device="cuda")
    b.base_logits(Hd, logits)
    ct = torch.empty(cfg.n_req, D, cfg.M, dtype=torch.int32, device="cuda")
    rl = torch.empty(cfg.n_req, D, dtype=torch.float32, device="cuda")
    b.topm(None, ct, None, rl)
    ell = base_logits(H[0][1:], w["lm_head"])
    got = logits[0].cpu().numpy()
    err = np.max(np.abs(got - ell))
    assert err <= LOGIT_TOL, err
    ctn, rln = ct.cpu().numpy()[0], rl.cpu().numpy()[0]
    for i in range(D):
        ids, _, rho = top_m(ell[i], cfg.M, cfg.T)
        if _topm_boundary_gap(ell[i], cfg.M) > 1e-3:
            assert ctn[i].tolist() == ids.tolist(), i
        assert abs(rln[i] - rho) <= REST_TOL
    assert b.device_status() == 0


QWEN4B_ROUNDS = 32


def test_qwen4b_rounds(qwen4b):
    """32 whole rounds (seeds 0..31), every one bit-exact: none excused."""
    from oracle.dartree import base_logits
    cfg, w, b, orc = qwen4b
    counts = {"match": 0, "excused": 0, "MISMATCH": 0}
    details = []
    seeds = list(range(QWEN4B_ROUNDS))
    for c0 in range(0, len(seeds), 8):
        chunk = seeds[c0:c0 + 8]
        Hs = [make_round_inputs(cfg, s) for s in chunk]
        rows = np.concatenate([H[0][1:] for H, _ in Hs])
        ells = base_logits(rows, w["lm_head"]).reshape(len(chunk), cfg.block - 1, cfg.V)
        for k, (H, root) in enumerate(Hs):
            Hd, rd = upload_round(H, root)
            out = to_np(b.build_round(Hd, rd))
            for st, why in check_round(orc, out, H, root, ells=[ells[k]]):
                counts[st] += 1
                details.append((chunk[k], st, why))
    line = report_counts("qwen3_4b rounds", counts, details)
    assert counts["MISMATCH"] == 0 and counts["excused"] == 0, line
    assert counts["match"] == len(seeds), line
    assert b.device_status() == 0

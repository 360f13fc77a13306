"""GPU parity at the degenerate and ragged corners of the method, tiny shapes.

Each case builds whole rounds through the C ABI and compares them with the
fp64 oracle under the usual bar (tokens, parents, depths, masks bit-exact;
scores within 2e-3; a mismatch only excused by an outcome-relevant near-tie):

* W = K = 1: a single chain of corrected argmaxes (the Domino chain);
* B = N: every node of the super-tree is selected;
* block = 2: one depth only;
* M = K: no candidate beyond the children;
* three requests per round (ragged batch);
* T = 0.3 with beta = -1: sharp distributions, deep trees, strong penalty;
* W = 64, K = 32, M = 64, B = 512: wide depths (the sorting-network top-W and
  a large Top-B) at a small vocabulary;
* d = 72: a hidden size that is not a multiple of the GEMM's 64-wide k-block;
* g = 128, 256 or 1024 with many state rows (5 or 20 requests of 8 branches,
  or one request of 64 branches): the chain's tcgen05 projection, one row tile
  or two (the second one ragged), 2 to 16 K blocks;
* the best-first builder with B equal to the whole K-restricted tree (the
  frontier empties exactly at the last pop).
"""
import numpy as np
import pytest

from tests.parity import TIE_TOL, check_round, report_counts, to_np, tree_matches, upload_round, upload_weights
from workloads import get_config, make_round_inputs, make_weights

pytestmark = pytest.mark.gpu

CASES = {
    "chain_w1_k1": dict(W=1, K=1, B=7),
    "all_nodes": dict(B=100),
    "one_depth": dict(block=2, B=3),
    "m_equals_k": dict(M=4, K=4),
    "three_requests": dict(n_req=3),
    "sharp_deep": dict(T=0.3, beta=-1.0),
    "wide_small_vocab": dict(block=4, M=64, K=32, W=64, B=512),
    "ragged_hidden": dict(d=72),
    "tc_requests": dict(g=256, n_req=5, W=8, K=4, B=32),
    "tc_two_tiles": dict(g=128, n_req=20, W=8, K=4, B=32),
    "tc_wide": dict(g=128, block=4, M=64, K=32, W=64, B=512),
    "tc_full_width": dict(g=1024, r=256, n_req=20, W=8, K=4, B=32),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_edge_rounds(case):
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    from oracle.dartree import Oracle, node_count
    torch.cuda.set_device(0)
    cfg = get_config("tiny_bf16", **CASES[case])
    if case == "all_nodes":
        assert cfg.B == node_count(cfg.K, cfg.W, cfg.block - 1)
    w = make_weights(cfg)
    b = DraftTreeBuilder(cfg, upload_weights(w))
    if case.startswith("tc_"):
        assert "tcgen05 projection" in b.plan(), b.plan()
    orc = Oracle(w, cfg)
    counts = {"match": 0, "excused": 0, "MISMATCH": 0}
    details = []
    try:
        for s in range(6):
            H, root = make_round_inputs(cfg, s)
            out = to_np(b.build_round(*upload_round(H, root)))
            for q, (st, why) in enumerate(check_round(orc, out, H, root)):
                counts[st] += 1
                details.append((s, q, st, why))
        status = b.device_status()
    finally:
        b.close()
    line = report_counts(f"edge {case}", counts, details)
    assert counts["MISMATCH"] == 0, line
    assert counts["match"] >= counts["excused"], line
    assert status == 0
    if case == "chain_w1_k1":
        assert all(d[2] == "match" for d in details)


def test_best_first_whole_tree():
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    from oracle.besttree import best_first_tie_report, build_best_first
    from oracle.dartree import Oracle
    torch.cuda.set_device(0)
    # K = 2, depth 3: the whole K-restricted tree has 2 + 4 + 8 = 14 nodes
    cfg = get_config("tiny_bf16", builder="best_first", block=4, M=8, K=2, W=4, B=14)
    w = make_weights(cfg)
    b = DraftTreeBuilder(cfg, upload_weights(w))
    orc = Oracle(w, cfg)
    try:
        for s in range(4):
            H, root = make_round_inputs(cfg, s)
            out = to_np(b.build_round(*upload_round(H, root)))
            t = build_best_first(orc, H[0], int(root[0]))
            assert t.tok.size == 15
            ok, why = tree_matches(out, 0, t)
            if not ok:
                assert best_first_tie_report(orc, H[0], int(root[0]), tol=TIE_TOL)["relevant"], why
        assert b.device_status() == 0
    finally:
        b.close()

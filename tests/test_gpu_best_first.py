"""GPU parity of the sequential best-first builder (DT_FLAG_BEST_FIRST) against its oracle.

The builder ("Resumen Técnico: DominoTree", Metodología, 1. Montículo de
Mejor Primera Búsqueda con Puntuación Condicional) is compared with
``oracle.besttree.build_best_first`` on the same seeded inputs: tokens,
parents, depths and masks bit-exact, cumulative scores within 2e-3, unless
the oracle shows an outcome-relevant near-tie within 1e-3 (a Top-M boundary,
an expansion's top-K or a pop whose single flip changes the emitted tree).
"""
import numpy as np
import pytest

from tests.parity import TIE_TOL, to_np, tree_matches, upload_round, upload_weights
from workloads import get_config, make_round_inputs, make_weights

pytestmark = pytest.mark.gpu


def _rounds(cfg, seeds, w=None):
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    from oracle.besttree import best_first_tie_report, build_best_first
    from oracle.dartree import Oracle, base_logits
    torch.cuda.set_device(0)
    w = make_weights(cfg) if w is None else w
    b = DraftTreeBuilder(cfg, upload_weights(w))
    orc = Oracle(w, cfg)
    counts = {"match": 0, "excused": 0, "MISMATCH": 0}
    details = []
    try:
        for s in seeds:
            H, root = make_round_inputs(cfg, s)
            ell = base_logits(H[0][1:], w["lm_head"])
            out = to_np(b.build_round(*upload_round(H, root)))
            t = build_best_first(orc, H[0], int(root[0]), ell=ell)
            ok, why = tree_matches(out, 0, t)
            if ok:
                counts["match"] += 1
                continue
            rep = best_first_tie_report(orc, H[0], int(root[0]), tol=TIE_TOL, ell=ell)
            st = "excused" if rep["relevant"] else "MISMATCH"
            counts[st] += 1
            details.append((s, st, why))
        status = b.device_status()
    finally:
        b.close()
    return counts, details, status


@pytest.mark.parametrize("beta", [0.0, -0.5])
def test_tiny_best_first(beta):
    cfg = get_config("tiny_bf16", builder="best_first", beta=beta)
    counts, details, status = _rounds(cfg, range(12))
    assert counts["MISMATCH"] == 0, details
    assert counts["match"] >= 10, (counts, details)
    assert status == 0


def test_tiny_best_first_positive_beta():
    """beta = +5 behind DT_FLAG_POSITIVE_BETA: the heap still emits a tree (a
    node is only reached through its parent), the same as the oracle's."""
    cfg = get_config("tiny_bf16", builder="best_first", beta=5.0, positive_beta=True)
    counts, details, status = _rounds(cfg, range(6))
    assert counts["MISMATCH"] == 0, details
    assert counts["match"] >= 5, (counts, details)
    assert status == 0


def test_tiny_best_first_marginal():
    cfg = get_config("tiny_bf16", builder="best_first", marginal=True)
    counts, details, status = _rounds(cfg, range(6))
    assert counts["MISMATCH"] == 0, details
    assert counts["match"] >= 5, (counts, details)
    assert status == 0


def test_qwen4b_best_first():
    cfg = get_config("qwen3_4b_best_first")
    counts, details, status = _rounds(cfg, range(3))
    assert counts["MISMATCH"] == 0, details
    assert counts["match"] >= 2, (counts, details)
    assert status == 0


def test_best_first_rejects_stepwise_and_batches():
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder, DtreeError
    from conditional_draft_tree_lm_gb300.dtree import check_config
    torch.cuda.set_device(0)
    assert check_config(get_config("serving32", builder="best_first")) == 2  # DT_ERR_SHAPE
    cfg = get_config("tiny_bf16", builder="best_first")
    b = DraftTreeBuilder(cfg, upload_weights(make_weights(cfg)))
    try:
        H, root = make_round_inputs(cfg, 0)
        Hd, rd = upload_round(H, root)
        nodes = b.new_nodes()
        with pytest.raises(DtreeError):
            b.expand_depth(1, rd, nodes["node_tok"], nodes["node_parent"], nodes["node_logp"],
                           nodes["node_score"])
        assert b.round_kernel_count() == 3
    finally:
        b.close()

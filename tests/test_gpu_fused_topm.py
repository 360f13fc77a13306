"""GPU: the Top-M kept in the LM-head GEMM's epilogue, against the oracle and
against the separate Top-M kernel on the same inputs, and whole rounds with the
separate kernel.

The two paths take the same fp32 logits from the same tensor-core products, so
their candidate ids and base logits must agree exactly; their log-partitions
add the same terms in another order (per GEMM CTA rather than per chunk), so
they agree to fp32 rounding (1e-5 here).  Against the oracle: ids exact where
the M-th/(M+1)-th gap exceeds 1e-3, base logits within 2e-4, rest within 1e-4.
"""
import numpy as np
import pytest

from tests.parity import check_round, report_counts, to_np, upload_round, upload_weights
from workloads import get_config, make_round_inputs, make_weights

pytestmark = pytest.mark.gpu

LOGIT_TOL = 2e-4
REST_TOL = 1e-4
PATH_REST_TOL = 1e-5


@pytest.fixture(scope="module", params=["tiny_bf16", "qwen3_4b"])
def pair(request):
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    from oracle.dartree import Oracle
    torch.cuda.set_device(0)
    cfg = get_config(request.param)
    w = make_weights(cfg)
    wd = upload_weights(w)
    fused = DraftTreeBuilder(cfg, wd)
    sep = DraftTreeBuilder(cfg.with_(separate_topm=True), wd)
    yield cfg, w, fused, sep, Oracle(w, cfg)
    fused.close()
    sep.close()


def _cands(b, cfg):
    import torch
    D = cfg.block - 1
    ct = torch.zeros(cfg.n_req, D, cfg.M, dtype=torch.int32, device="cuda")
    cb = torch.zeros(cfg.n_req, D, cfg.M, dtype=torch.float32, device="cuda")
    rl = torch.zeros(cfg.n_req, D, dtype=torch.float32, device="cuda")
    b.last_candidates(ct, cb, rl)
    torch.cuda.synchronize()
    return ct.cpu().numpy()[0], cb.cpu().numpy()[0], rl.cpu().numpy()[0]


def test_plans(pair):
    cfg, w, fused, sep, orc = pair
    assert "epilogue" in fused.plan(), fused.plan()
    assert "Top-M kernel" in sep.plan(), sep.plan()


def test_fused_candidates(pair):
    from oracle.dartree import base_logits, top_m
    cfg, w, fused, sep, orc = pair
    D = cfg.block - 1
    checked = 0
    for seed in range(4):
        H, root = make_round_inputs(cfg, seed)
        Hd, rd = upload_round(H, root)
        tf = to_np(fused.build_round(Hd, rd))
        ctf, cbf, rlf = _cands(fused, cfg)
        ts = to_np(sep.build_round(Hd, rd))
        cts, cbs, rls = _cands(sep, cfg)
        # the two paths
        assert np.array_equal(ctf, cts), seed
        assert np.array_equal(cbf, cbs), seed
        np.testing.assert_allclose(rlf, rls, rtol=0, atol=PATH_REST_TOL)
        for k in ("tok", "parent", "depth", "mask"):
            assert np.array_equal(tf[k], ts[k]), (seed, k)
        # the oracle
        ell = base_logits(H[0][1:], w["lm_head"])
        for i in range(D):
            ids, _, rho = top_m(ell[i], cfg.M, cfg.T)
            s = np.sort(ell[i])[::-1]
            if s[cfg.M - 1] - s[cfg.M] > 1e-3:
                assert ctf[i].tolist() == ids.tolist(), (seed, i)
                checked += 1
            np.testing.assert_allclose(cbf[i], ell[i][ctf[i]], rtol=0, atol=LOGIT_TOL)
            assert abs(rlf[i] - rho) <= REST_TOL, (seed, i, rlf[i], rho)
    assert checked >= 2 * D, checked
    assert fused.device_status() == 0 and sep.device_status() == 0


def test_separate_topm_rounds(pair):
    """Whole rounds with the Top-M as its own kernel, against the oracle."""
    cfg, w, fused, sep, orc = pair
    counts = {"match": 0, "excused": 0, "MISMATCH": 0}
    details = []
    for seed in range(100, 108):
        H, root = make_round_inputs(cfg, seed)
        Hd, rd = upload_round(H, root)
        out = to_np(sep.build_round(Hd, rd))
        for st, why in check_round(orc, out, H, root):
            counts[st] += 1
            details.append((seed, st, why))
    line = report_counts(f"{cfg.name} rounds, separate Top-M", counts, details)
    assert counts["MISMATCH"] == 0, line
    if cfg.name == "qwen3_4b":
        assert counts["excused"] == 0, line
    assert sep.device_status() == 0

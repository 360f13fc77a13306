"""Top-M over many rows: the row-streaming kernel against the fp64 oracle and
against the chunked kernel.

With at least one row per SM, dt_topm runs the kernel that streams rows (a
candidate buffer behind a rising bound, cut to its M best whenever it could
overflow) instead of the chunked kernel and its merge; with more rows than
CTAs, some CTAs stream two rows.  The
two must agree: candidate ids and their logits bit-exact, the rest
log-partition within 1e-4 (the two sum in different orders).  Every row is
also checked against the oracle's Top-M ("Resumen Técnico: DominoTree",
Restricción de Candidatos (Top-M)) on rows whose M-th/(M+1)-th gap exceeds
1e-3.  The rows mix Gaussian logits of several scales with two adversarial
kinds: an ascending ramp (every logit beats the bound when it arrives, so the
buffer is cut at every tile) and logits rounded to steps of 0.5 (many equal
values, ties resolved by the lower token id).
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

REST_TOL = 1e-4


def _builder(n_req):
    import torch
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    from tests.parity import upload_weights
    from workloads import get_config, make_weights
    torch.cuda.set_device(0)
    cfg = get_config("tiny_bf16").with_(V=151936, block=16, M=64, K=8, W=8, B=64, n_req=n_req)
    return cfg, DraftTreeBuilder(cfg, upload_weights(make_weights(cfg)))


def _logits(rows, V, seed):
    rng = np.random.default_rng([7, seed])
    x = rng.standard_normal((rows, V)).astype(np.float32)
    x *= rng.uniform(0.5, 6.0, size=(rows, 1)).astype(np.float32)
    x[0] = np.linspace(-8.0, 8.0, V, dtype=np.float32)     # ascending: a cut at every tile
    x[1] = np.round(x[1] * 2.0) / 2.0                       # many equal values
    x[2] = np.linspace(8.0, -8.0, V, dtype=np.float32)     # descending
    return x


def _topm(builder, logits, M):
    import torch
    rows = logits.shape[0]
    tok = torch.full((rows, M), -7, dtype=torch.int32, device="cuda")
    base = torch.full((rows, M), float("nan"), dtype=torch.float32, device="cuda")
    rest = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    builder.topm(logits, tok, base, rest)
    torch.cuda.synchronize()
    return tok.cpu().numpy(), base.cpu().numpy(), rest.cpu().numpy()


def test_row_streaming_topm_matches_oracle_and_chunked_kernel():
    import torch
    from oracle.dartree import top_m
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    D = 15
    n_req = (n_sm + D - 1) // D + 1  # more rows than SMs
    cfg, big = _builder(n_req)
    _, small = _builder(1)
    try:
        assert "streaming each row" in big.plan(), big.plan()
        assert "streaming each row" not in small.plan(), small.plan()
        rows = n_req * D
        x = _logits(rows, cfg.V, 0)
        xd = torch.from_numpy(x).cuda()
        tok, base, rest = _topm(big, xd, cfg.M)
        # the chunked kernel, fifteen rows at a time
        for r0 in range(0, rows, D):
            t2, b2, r2 = _topm(small, xd[r0:r0 + D].contiguous(), cfg.M)
            assert np.array_equal(tok[r0:r0 + D], t2), f"rows {r0}..: ids differ from the chunked kernel"
            assert np.array_equal(base[r0:r0 + D], b2), f"rows {r0}..: logits differ from the chunked kernel"
            err = np.abs(rest[r0:r0 + D] - r2).max()
            assert err <= REST_TOL, f"rows {r0}..: rest differs from the chunked kernel by {err}"
        checked = 0
        for row in range(rows):
            ids, vals, rho = top_m(x[row].astype(np.float64), cfg.M, cfg.T)
            s = np.sort(x[row].astype(np.float64))[::-1]
            if s[cfg.M - 1] - s[cfg.M] > 1e-3 or row == 1:
                # (row 1: equal values share a key only with their token id, so
                # the order is still unique)
                assert tok[row].tolist() == ids.tolist(), f"row {row}: ids differ from the oracle"
                assert np.array_equal(base[row].astype(np.float64), vals), f"row {row}: logits"
                checked += 1
            assert abs(float(rest[row]) - rho) <= REST_TOL, f"row {row}: rest vs the oracle"
        assert checked >= rows // 2
        assert big.device_status() == 0 and small.device_status() == 0
    finally:
        big.close()
        small.close()


@pytest.mark.parametrize("M,extra_rows", [(128, 8), (200, 8), (64, None), (136, None)])
def test_row_streaming_topm_other_m_matches_oracle(M, extra_rows):
    """M = 128 (the first tile's bound taken as the 8th-largest lane maximum
    of every warp) and M = 200 (above what that bound covers: a segment starts
    unbounded), through the context-free entry point, which streams rows the
    same way when there are at least as many rows as SMs.  With more rows than
    two per SM (extra_rows None: 2 SMs + 37 rows) some CTAs stream a second
    row after their first."""
    import torch
    from conditional_draft_tree_lm_gb300.dtree import topm_noalloc
    from oracle.dartree import top_m
    torch.cuda.set_device(0)
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    rows = n_sm + extra_rows if extra_rows is not None else 2 * n_sm + 37
    V, T = 151936, 1.0
    x = _logits(rows, V, 1)
    xd = torch.from_numpy(x).cuda()
    tok = torch.full((rows, M), -7, dtype=torch.int32, device="cuda")
    base = torch.full((rows, M), float("nan"), dtype=torch.float32, device="cuda")
    rest = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
    topm_noalloc(xd, M, T, tok, base, rest)
    torch.cuda.synchronize()
    tok, base, rest = tok.cpu().numpy(), base.cpu().numpy(), rest.cpu().numpy()
    checked = 0
    for row in range(rows):
        ids, vals, rho = top_m(x[row].astype(np.float64), M, T)
        s = np.sort(x[row].astype(np.float64))[::-1]
        if s[M - 1] - s[M] > 1e-3 or row == 1:
            assert tok[row].tolist() == ids.tolist(), f"M={M} row {row}: ids differ from the oracle"
            assert np.array_equal(base[row].astype(np.float64), vals), f"M={M} row {row}: logits"
            checked += 1
        assert abs(float(rest[row]) - rho) <= REST_TOL, f"M={M} row {row}: rest vs the oracle"
    assert checked >= rows // 2

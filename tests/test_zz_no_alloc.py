"""dt_topm_noalloc gives the same Top-M results as dt_topm.

dt_topm_noalloc is for callers that must not allocate device memory — a
serving process whose GPU memory budget is fixed at start-up, or code running
inside another framework that owns the device's allocator.  It keeps its
scratch in one fixed array inside the library instead of a context's
workspace.  Here it runs twice in a row on different logits (so the second
call starts from the first call's leftovers in that array) and each time must
match the regular context-based entry point (and, on the first call, the
fp64 oracle's Top-M).  It must also leave the device's free memory unchanged,
and reject shapes its fixed scratch or the kernel cannot take before any work
is queued.  The file is named so that pytest collects it after every other
test.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

REST_TOL = 1e-4  # the rest log-partition tolerance of the other GPU tests


def _setup():
    import torch
    from conditional_draft_tree_lm_gb300.build import build_library
    build_library()
    from conditional_draft_tree_lm_gb300 import DraftTreeBuilder
    from tests.parity import upload_weights
    from workloads import get_config, make_weights
    torch.cuda.set_device(0)
    # a small model with the full vocabulary, so every row spans many chunks
    cfg = get_config("tiny_bf16").with_(V=151936, block=16, M=64, K=8, W=8, B=64)
    return cfg, DraftTreeBuilder(cfg, upload_weights(make_weights(cfg)))


def test_noalloc_topm_matches_context_topm_on_two_calls():
    import torch
    from conditional_draft_tree_lm_gb300.dtree import topm_noalloc
    cfg, builder = _setup()
    rows = cfg.n_req * (cfg.block - 1)
    for seed in (1, 2):
        gen = torch.Generator(device="cuda").manual_seed(seed)
        logits = torch.randn(rows, cfg.V, generator=gen, device="cuda", dtype=torch.float32) * (1.0 + seed)
        ref_tok = torch.empty(rows, cfg.M, dtype=torch.int32, device="cuda")
        ref_base = torch.empty(rows, cfg.M, dtype=torch.float32, device="cuda")
        ref_rest = torch.empty(rows, dtype=torch.float32, device="cuda")
        builder.topm(logits, ref_tok, ref_base, ref_rest)
        tok = torch.full((rows, cfg.M), -7, dtype=torch.int32, device="cuda")
        base = torch.full((rows, cfg.M), float("nan"), dtype=torch.float32, device="cuda")
        rest = torch.full((rows,), float("nan"), dtype=torch.float32, device="cuda")
        topm_noalloc(logits, cfg.M, cfg.T, tok, base, rest)
        torch.cuda.synchronize()
        assert torch.equal(tok, ref_tok), f"call {seed}: candidate tokens differ"
        assert torch.equal(base, ref_base), f"call {seed}: candidate logits differ"
        err = (rest - ref_rest).abs().max().item()
        assert err <= REST_TOL, f"call {seed}: rest log-partition differs by {err}"
        if seed == 1:
            _check_against_oracle(logits, tok, base, rest, cfg.M, cfg.T)
    assert builder.device_status() == 0
    builder.close()


def _check_against_oracle(logits, tok, base, rest, M, T):
    """The call's own results against the fp64 oracle's Top-M ("Resumen
    Técnico: DominoTree", Restricción de Candidatos (Top-M)): candidate ids
    bit-exact on every row whose M-th/(M+1)-th gap exceeds 1e-3, their logits
    exact, and the rest log-partition within 1e-4."""
    from oracle.dartree import top_m
    ell = logits.double().cpu().numpy()
    tok, base, rest = tok.cpu().numpy(), base.cpu().numpy(), rest.cpu().numpy()
    checked = 0
    for row in range(ell.shape[0]):
        ids, vals, rho = top_m(ell[row], M, T)
        s = np.sort(ell[row])[::-1]
        if s[M - 1] - s[M] > 1e-3:
            assert tok[row].tolist() == ids.tolist(), f"row {row}: candidate ids differ from the oracle"
            assert np.array_equal(base[row].astype(np.float64), vals), f"row {row}: candidate logits"
            checked += 1
        assert abs(float(rest[row]) - rho) <= REST_TOL, f"row {row}: rest log-partition vs the oracle"
    assert checked >= ell.shape[0] // 2


def test_noalloc_topm_allocates_nothing():
    """After its first call on the device (the one-time set-up), a call leaves
    the device's free memory unchanged."""
    import torch
    from conditional_draft_tree_lm_gb300.dtree import topm_noalloc
    cfg, builder = _setup()
    builder.close()
    rows = cfg.block - 1
    logits = torch.randn(rows, cfg.V, device="cuda", dtype=torch.float32)
    tok = torch.empty(rows, cfg.M, dtype=torch.int32, device="cuda")
    base = torch.empty(rows, cfg.M, dtype=torch.float32, device="cuda")
    rest = torch.empty(rows, dtype=torch.float32, device="cuda")
    topm_noalloc(logits, cfg.M, cfg.T, tok, base, rest)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(3):
        topm_noalloc(logits, cfg.M, cfg.T, tok, base, rest)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, f"free device memory changed by {free0 - free1} bytes"


def test_noalloc_topm_rejects_sizes_beyond_its_scratch():
    import torch
    from conditional_draft_tree_lm_gb300 import load_library
    _setup()
    lib = load_library()
    x = torch.zeros(4, dtype=torch.float32, device="cuda")
    out_i = torch.zeros(4, dtype=torch.int32, device="cuda")
    # 5000 rows of a 151936-token vocabulary need ~26 MB of scratch: rejected
    # on the host before any kernel runs
    st = lib.dt_topm_noalloc(ctypes.c_void_p(x.data_ptr()), 5000, 151936, 64, 1.0,
                             ctypes.c_void_p(out_i.data_ptr()), ctypes.c_void_p(x.data_ptr()),
                             ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 2  # DT_ERR_SHAPE
    assert "maximum" in lib.dt_last_error().decode()

    def call(rows, V, M):
        # buffers of the full size: nothing would be read out of bounds even
        # if a shape were not rejected
        lg = torch.zeros(rows, V, dtype=torch.float32, device="cuda")
        ti = torch.zeros(rows, M, dtype=torch.int32, device="cuda")
        tb = torch.zeros(rows, M, dtype=torch.float32, device="cuda")
        rl = torch.zeros(rows, dtype=torch.float32, device="cuda")
        st = lib.dt_topm_noalloc(ctypes.c_void_p(lg.data_ptr()), rows, V, M, 1.0,
                                 ctypes.c_void_p(ti.data_ptr()), ctypes.c_void_p(tb.data_ptr()),
                                 ctypes.c_void_p(rl.data_ptr()),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        torch.cuda.synchronize()
        return st, lib.dt_last_error().decode()

    # more rows than one grid dimension holds, with little scratch
    st, msg = call(70000, 16, 1)
    assert st == 2 and "rows" in msg, msg
    # M = 512 over a vocabulary whose chunks would exceed 16384 logits
    st, msg = call(1, 300000, 512)
    assert st == 2 and "chunk" in msg, msg

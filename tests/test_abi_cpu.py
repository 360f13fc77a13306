"""The C-ABI library builds, loads without a GPU and exports every declared
symbol; its host-only helpers validate configurations (no compute calls)."""
import os
import re

import pytest

from conditional_draft_tree_lm_gb300 import build as dtbuild
from workloads import CONFIGS, get_config

HEADER = os.path.join(dtbuild.ROOT, "include", "dtree.h")


@pytest.fixture(scope="module")
def lib():
    dtbuild.build_library()
    from conditional_draft_tree_lm_gb300 import load_library
    return load_library()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dt_[a-zA-Z0-9_]+)\s*\(", src)))


def test_header_declares_the_steps():
    names = declared_functions()
    for n in ("dt_base_logits", "dt_topm", "dt_expand_depth", "dt_prune_topB", "dt_tree_mask",
              "dt_build_round", "dt_create", "dt_destroy"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_exports_are_c_symbols():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", dtbuild.LIB_PATH], capture_output=True, text=True).stdout
    syms = set(re.findall(r"\sT\s(dt_\w+)", out))
    assert set(declared_functions()) <= syms


def test_check_config_accepts_named_workloads(lib):
    from conditional_draft_tree_lm_gb300 import check_config, node_count
    from oracle.dartree import node_count as oracle_nodes
    for name, cfg in CONFIGS.items():
        assert check_config(cfg) == 0, name
        assert node_count(cfg) == oracle_nodes(cfg.K, cfg.W, cfg.block - 1)


@pytest.mark.parametrize("bad,code", [
    (dict(K=20, M=16), 1),          # K > M
    (dict(beta=0.5), 1),            # positive depth bonus without DT_FLAG_POSITIVE_BETA
    (dict(beta=float("inf"), positive_beta=True), 1),  # with the flag, still finite
    (dict(T=0.0), 1),               # temperature must be positive
    (dict(B=10 ** 6), 1),           # budget above the super-tree size
    (dict(M=2000), 1),              # M > V
    (dict(d=60), 2),                # hidden size not a multiple of 8
    (dict(n_req=100), 2),           # n_req * block > 512
    (dict(K=40, M=64), 2),          # K above 32
    (dict(block=1), 1),
    (dict(builder="best_first", n_req=2), 2),   # the best-first builder takes one request
])
def test_check_config_rejects(lib, bad, code):
    from conditional_draft_tree_lm_gb300 import check_config
    cfg = get_config("tiny_bf16", **bad)
    assert check_config(cfg) == code


def test_status_strings(lib):
    from conditional_draft_tree_lm_gb300 import status_string
    assert status_string(0) == "ok"
    assert "timed out" in status_string(5)
    assert status_string(99) == "unknown status"


def test_workspace_bytes(lib):
    from conditional_draft_tree_lm_gb300 import workspace_bytes
    cfg = get_config("qwen3_4b")
    n = workspace_bytes(cfg)
    xtab = cfg.V * 3 * cfg.g * 4
    logits = (cfg.block - 1) * cfg.V * 4
    assert xtab + logits < n < xtab + logits + 64 * 2 ** 20
    assert workspace_bytes(get_config("tiny_bf16", K=20, M=16)) == 0


def test_check_config_flags(lib):
    """Unknown flag bits are rejected; the four defined flags combine; beta > 0
    passes only with DT_FLAG_POSITIVE_BETA."""
    import ctypes
    from conditional_draft_tree_lm_gb300.dtree import load_library, make_config
    cfg = make_config(get_config("tiny_bf16", builder="best_first", marginal=True, separate_topm=True,
                                 positive_beta=True, beta=5.0))
    assert cfg.flags == 15
    L = load_library()
    assert L.dt_check_config(ctypes.byref(cfg)) == 0
    cfg.flags = 7  # the same beta = 5 without the flag
    assert L.dt_check_config(ctypes.byref(cfg)) == 1
    for bad in (16, 31, 1 << 31):
        cfg.flags = bad
        assert L.dt_check_config(ctypes.byref(cfg)) == 1

"""Thin Python binding of libdtree (argument marshalling only).

Every step runs in the CUDA kernels of ``libdtree.so``; this module only turns
torch tensors into device pointers and streams, calls the C ABI declared in
``include/dtree.h`` and raises on a non-zero status.  There is no fallback: if
the library is missing, importing the binding's loader raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_float, c_int, c_int64, c_size_t, c_uint, c_void_p, c_char_p

from .build import LIB_PATH

_lib = None

STATUS = {
    0: "DT_OK", 1: "DT_ERR_INVALID_ARG", 2: "DT_ERR_SHAPE", 3: "DT_ERR_CUDA", 4: "DT_ERR_OOM",
    5: "DT_ERR_TIMEOUT", 6: "DT_ERR_UNIMPLEMENTED", 7: "DT_ERR_DEVICE",
}


class DtreeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        detail = ""
        if status in (3, 4):
            detail = " — " + load_library().dt_last_error().decode(errors="replace")
        super().__init__(f"{where}: {STATUS.get(status, status)} ({status_string(status)}){detail}")


class DtConfig(ctypes.Structure):
    _fields_ = [("d", c_int), ("V", c_int), ("block", c_int), ("g", c_int), ("r", c_int), ("M", c_int),
                ("K", c_int), ("W", c_int), ("B", c_int), ("n_req", c_int), ("beta", c_float),
                ("T", c_float), ("flags", c_uint)]


WEIGHT_FIELDS = ("lm_head", "emb", "w_ih", "b_ih", "w_hh", "w1", "w2")
FLAG_MARGINAL = 1  # DT_FLAG_MARGINAL: marginal scoring (no correction)
FLAG_BEST_FIRST = 2  # DT_FLAG_BEST_FIRST: sequential conditional best-first builder
FLAG_SEPARATE_TOPM = 4  # DT_FLAG_SEPARATE_TOPM: the Top-M as its own kernel in rounds
FLAG_POSITIVE_BETA = 8  # DT_FLAG_POSITIVE_BETA: beta > 0 accepted (Lemma 1 not guaranteed)


class DtWeights(ctypes.Structure):
    _fields_ = [(n, c_void_p) for n in WEIGHT_FIELDS]


def load_library(path: str | None = None) -> ctypes.CDLL:
    """Load libdtree.so (built by ``build.build_library``); raise if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libdtree.so not built ({p}); run __graft_entry__.build()")
    lib = ctypes.CDLL(p, mode=ctypes.RTLD_GLOBAL)
    vp, i32p = c_void_p, c_void_p
    sig = {
        "dt_check_config": (c_int, [POINTER(DtConfig)]),
        "dt_node_count": (c_int64, [POINTER(DtConfig)]),
        "dt_workspace_bytes": (c_size_t, [POINTER(DtConfig)]),
        "dt_status_string": (c_char_p, [c_int]),
        "dt_last_error": (c_char_p, []),
        "dt_create": (c_int, [POINTER(DtConfig), POINTER(DtWeights), vp, POINTER(c_void_p)]),
        "dt_destroy": (c_int, [vp]),
        "dt_base_logits": (c_int, [vp, vp, vp, vp]),
        "dt_topm": (c_int, [vp, vp, vp, vp, vp, vp]),
        "dt_last_candidates": (c_int, [vp, vp, vp, vp, vp]),
        "dt_base_topm": (c_int, [vp, vp, vp]),
        "dt_expand_depth": (c_int, [vp, c_int, i32p, vp, vp, vp, vp, vp, vp]),
        "dt_prune_topB": (c_int, [vp, vp, vp, vp]),
        "dt_tree_mask": (c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "dt_expand_prune": (c_int, [vp, vp, vp, vp, vp, vp, vp, vp]),
        "dt_accept_walk": (c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "dt_build_round": (c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "dt_build_round_host": (c_int, [vp, vp, vp, vp, vp, vp, vp, vp, vp]),
        "dt_get_device_status": (c_int, [vp]),
        "dt_check_bounded_waits": (c_int, [vp, c_int, vp]),
        "dt_round_kernel_count": (c_int, [vp]),
        "dt_plan_string": (c_char_p, [vp]),
        "dt_topm_noalloc": (c_int, [vp, c_int, c_int, c_int, c_float, vp, vp, vp, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


def status_string(s: int) -> str:
    return load_library().dt_status_string(int(s)).decode()


def make_config(cfg) -> DtConfig:
    """DtConfig from any object with the workload fields (d, V, block, g, r, M, K, W, B, n_req, beta, T,
    and optionally marginal, builder, separate_topm and positive_beta)."""
    flags = FLAG_MARGINAL if getattr(cfg, "marginal", False) else 0
    if getattr(cfg, "builder", "dartree") == "best_first":
        flags |= FLAG_BEST_FIRST
    if getattr(cfg, "separate_topm", False):
        flags |= FLAG_SEPARATE_TOPM
    if getattr(cfg, "positive_beta", False):
        flags |= FLAG_POSITIVE_BETA
    return DtConfig(cfg.d, cfg.V, cfg.block, cfg.g, cfg.r, cfg.M, cfg.K, cfg.W, cfg.B,
                    getattr(cfg, "n_req", 1), float(cfg.beta), float(cfg.T), flags)


def check_config(cfg) -> int:
    c = make_config(cfg)
    return load_library().dt_check_config(ctypes.byref(c))


def node_count(cfg) -> int:
    c = make_config(cfg)
    return int(load_library().dt_node_count(ctypes.byref(c)))


def workspace_bytes(cfg) -> int:
    c = make_config(cfg)
    return int(load_library().dt_workspace_bytes(ctypes.byref(c)))


def _ptr(t, dtype=None, numel=None, name="tensor"):
    if t is None:
        return None
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name}: expected {numel} elements, got {t.numel()}")
    return c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return c_void_p(stream.cuda_stream)


def _check(status, where):
    if status != 0:
        raise DtreeError(status, where)


class DraftTreeBuilder:
    """Owns one libdtree context (workspace, GRU input table, captured round).

    ``weights`` maps the names of ``WEIGHT_FIELDS`` to contiguous bf16 CUDA
    tensors in torch.nn.Linear layout; they are borrowed and kept alive here.
    """

    def __init__(self, cfg, weights: dict, stream=None):
        import torch
        self.lib = load_library()
        self.cfg = cfg
        self.c = make_config(cfg)
        self.D = cfg.block - 1
        self.N = node_count(cfg)
        self.N1 = self.N + 1
        shapes = {
            "lm_head": cfg.V * cfg.d, "emb": cfg.V * cfg.d, "w_ih": 3 * cfg.g * cfg.d, "b_ih": 3 * cfg.g,
            "w_hh": 3 * cfg.g * cfg.g, "w1": cfg.r * (cfg.d + cfg.g), "w2": cfg.V * cfg.r,
        }
        self._weights = {k: weights[k] for k in WEIGHT_FIELDS}
        w = DtWeights(*[_ptr(self._weights[k], torch.bfloat16, shapes[k], k) for k in WEIGHT_FIELDS])
        out = c_void_p()
        _check(self.lib.dt_create(ctypes.byref(self.c), ctypes.byref(w), _stream(stream), ctypes.byref(out)),
               "dt_create")
        self.ctx = out

    # -- lifetime -----------------------------------------------------------
    def close(self):
        if getattr(self, "ctx", None):
            self.lib.dt_destroy(self.ctx)
            self.ctx = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    # -- steps --------------------------------------------------------------
    def base_logits(self, H, logits=None, stream=None):
        import torch
        cfg = self.cfg
        _check(self.lib.dt_base_logits(self.ctx, _ptr(H, torch.bfloat16, cfg.n_req * cfg.block * cfg.d, "H"),
                                       _ptr(logits, torch.float32, cfg.n_req * self.D * cfg.V, "logits"),
                                       _stream(stream)), "dt_base_logits")

    def topm(self, logits=None, cand_tok=None, cand_base=None, rest_lse=None, stream=None):
        import torch
        cfg = self.cfg
        rows = cfg.n_req * self.D
        _check(self.lib.dt_topm(self.ctx, _ptr(logits, torch.float32, rows * cfg.V, "logits"),
                                _ptr(cand_tok, torch.int32, rows * cfg.M, "cand_tok"),
                                _ptr(cand_base, torch.float32, rows * cfg.M, "cand_base"),
                                _ptr(rest_lse, torch.float32, rows, "rest_lse"), _stream(stream)), "dt_topm")

    def base_topm(self, H, stream=None):
        """The LM-head GEMM and the Top-M of a round (dt_base_topm)."""
        import torch
        cfg = self.cfg
        _check(self.lib.dt_base_topm(self.ctx, _ptr(H, torch.bfloat16, cfg.n_req * cfg.block * cfg.d, "H"),
                                     _stream(stream)), "dt_base_topm")

    def last_candidates(self, cand_tok=None, cand_base=None, rest_lse=None, stream=None):
        """The Top-M restriction of the last round (or dt_topm) into these buffers (dt_last_candidates)."""
        import torch
        cfg = self.cfg
        rows = cfg.n_req * (cfg.block - 1)
        _check(self.lib.dt_last_candidates(self.ctx, _ptr(cand_tok, torch.int32, rows * cfg.M, "cand_tok"),
                                           _ptr(cand_base, torch.float32, rows * cfg.M, "cand_base"),
                                           _ptr(rest_lse, torch.float32, rows, "rest_lse"), _stream(stream)),
               "dt_last_candidates")

    def expand_depth(self, depth, root_tok, node_tok, node_parent, node_logp, node_score, live=None,
                     stream=None):
        import torch
        cfg = self.cfg
        n = cfg.n_req * self.N1
        _check(self.lib.dt_expand_depth(self.ctx, int(depth), _ptr(root_tok, torch.int32, cfg.n_req, "root_tok"),
                                        _ptr(node_tok, torch.int32, n, "node_tok"),
                                        _ptr(node_parent, torch.int32, n, "node_parent"),
                                        _ptr(node_logp, torch.float32, n, "node_logp"),
                                        _ptr(node_score, torch.float32, n, "node_score"),
                                        _ptr(live, torch.int32, cfg.n_req * cfg.W, "live"), _stream(stream)),
               "dt_expand_depth")

    def prune_topB(self, node_score, sel, stream=None):
        import torch
        cfg = self.cfg
        _check(self.lib.dt_prune_topB(self.ctx, _ptr(node_score, torch.float32, cfg.n_req * self.N1, "node_score"),
                                      _ptr(sel, torch.int32, cfg.n_req * cfg.B, "sel"), _stream(stream)),
               "dt_prune_topB")

    def tree_mask(self, sel, node_tok, node_parent, node_score, tok, parent, depth, logp_cum, mask, stream=None):
        import torch
        cfg = self.cfg
        n = cfg.n_req * self.N1
        s1 = cfg.B + 1
        _check(self.lib.dt_tree_mask(self.ctx, _ptr(sel, torch.int32, cfg.n_req * cfg.B, "sel"),
                                     _ptr(node_tok, torch.int32, n, "node_tok"),
                                     _ptr(node_parent, torch.int32, n, "node_parent"),
                                     _ptr(node_score, torch.float32, n, "node_score"),
                                     _ptr(tok, torch.int32, cfg.n_req * s1, "tok"),
                                     _ptr(parent, torch.int32, cfg.n_req * s1, "parent"),
                                     _ptr(depth, torch.int32, cfg.n_req * s1, "depth"),
                                     _ptr(logp_cum, torch.float32, cfg.n_req * s1, "logp_cum"),
                                     _ptr(mask, torch.uint8, cfg.n_req * s1 * s1, "mask"), _stream(stream)),
               "dt_tree_mask")

    def expand_prune(self, root_tok, out=None, stream=None):
        """Steps 3-5 (all depths, Top-B, tree/mask) from the last topm()'s
        candidates, in one launch for a single request (``dt_expand_prune``)."""
        import torch
        cfg = self.cfg
        out = out if out is not None else self.new_tree(root_tok.device)
        s1 = cfg.B + 1
        _check(self.lib.dt_expand_prune(self.ctx, _ptr(root_tok, torch.int32, cfg.n_req, "root_tok"),
                                        _ptr(out["tok"], torch.int32, cfg.n_req * s1, "tok"),
                                        _ptr(out["parent"], torch.int32, cfg.n_req * s1, "parent"),
                                        _ptr(out["depth"], torch.int32, cfg.n_req * s1, "depth"),
                                        _ptr(out["logp_cum"], torch.float32, cfg.n_req * s1, "logp_cum"),
                                        _ptr(out["mask"], torch.uint8, cfg.n_req * s1 * s1, "mask"),
                                        _stream(stream)), "dt_expand_prune")
        return out

    def accept_walk(self, target_logits, tok, parent, accepted=None, accept_len=None, bonus=None,
                    target_tok=None, stream=None):
        """Greedy verification of the emitted trees (``dt_accept_walk``).
        target_logits [n_req, B+1, V] fp32; tok, parent [n_req, B+1] int32.
        Returns dict(accepted [n_req, D], accept_len [n_req], bonus [n_req],
        target_tok [n_req, B+1] or None)."""
        import torch
        cfg = self.cfg
        s1 = cfg.B + 1
        D = cfg.block - 1
        dev = target_logits.device
        accepted = accepted if accepted is not None else torch.empty(cfg.n_req, D, dtype=torch.int32, device=dev)
        accept_len = accept_len if accept_len is not None else torch.empty(cfg.n_req, dtype=torch.int32, device=dev)
        bonus = bonus if bonus is not None else torch.empty(cfg.n_req, dtype=torch.int32, device=dev)
        _check(self.lib.dt_accept_walk(self.ctx, _ptr(target_logits, torch.float32, cfg.n_req * s1 * cfg.V,
                                                      "target_logits"),
                                       _ptr(tok, torch.int32, cfg.n_req * s1, "tok"),
                                       _ptr(parent, torch.int32, cfg.n_req * s1, "parent"),
                                       _ptr(target_tok, torch.int32, cfg.n_req * s1, "target_tok"),
                                       _ptr(accepted, torch.int32, cfg.n_req * D, "accepted"),
                                       _ptr(accept_len, torch.int32, cfg.n_req, "accept_len"),
                                       _ptr(bonus, torch.int32, cfg.n_req, "bonus"), _stream(stream)),
               "dt_accept_walk")
        return {"accepted": accepted, "accept_len": accept_len, "bonus": bonus, "target_tok": target_tok}

    def new_tree(self, device="cuda"):
        """Output tensors of one round: tok, parent, depth [n_req, B+1], logp_cum, mask."""
        import torch
        cfg = self.cfg
        s1 = cfg.B + 1
        return {
            "tok": torch.empty(cfg.n_req, s1, dtype=torch.int32, device=device),
            "parent": torch.empty(cfg.n_req, s1, dtype=torch.int32, device=device),
            "depth": torch.empty(cfg.n_req, s1, dtype=torch.int32, device=device),
            "logp_cum": torch.empty(cfg.n_req, s1, dtype=torch.float32, device=device),
            "mask": torch.empty(cfg.n_req, s1, s1, dtype=torch.uint8, device=device),
        }

    def new_nodes(self, device="cuda"):
        import torch
        cfg = self.cfg
        return {
            "node_tok": torch.empty(cfg.n_req, self.N1, dtype=torch.int32, device=device),
            "node_parent": torch.empty(cfg.n_req, self.N1, dtype=torch.int32, device=device),
            "node_logp": torch.empty(cfg.n_req, self.N1, dtype=torch.float32, device=device),
            "node_score": torch.empty(cfg.n_req, self.N1, dtype=torch.float32, device=device),
        }

    def build_round(self, H, root_tok, out=None, stream=None):
        import torch
        cfg = self.cfg
        out = out if out is not None else self.new_tree(H.device)
        s1 = cfg.B + 1
        _check(self.lib.dt_build_round(self.ctx, _ptr(H, torch.bfloat16, cfg.n_req * cfg.block * cfg.d, "H"),
                                       _ptr(root_tok, torch.int32, cfg.n_req, "root_tok"),
                                       _ptr(out["tok"], torch.int32, cfg.n_req * s1, "tok"),
                                       _ptr(out["parent"], torch.int32, cfg.n_req * s1, "parent"),
                                       _ptr(out["depth"], torch.int32, cfg.n_req * s1, "depth"),
                                       _ptr(out["logp_cum"], torch.float32, cfg.n_req * s1, "logp_cum"),
                                       _ptr(out["mask"], torch.uint8, cfg.n_req * s1 * s1, "mask"),
                                       _stream(stream)), "dt_build_round")
        return out

    def build_round_host(self, H_host, root_host, out_host, stream=None):
        """Round from host (ideally pinned) CPU tensors; synchronises the stream."""
        import torch
        cfg = self.cfg
        s1 = cfg.B + 1

        def hp(t, dtype, n, name):
            if t.is_cuda or not t.is_contiguous() or t.dtype != dtype or t.numel() != n:
                raise ValueError(f"{name}: expected a contiguous host {dtype} tensor of {n} elements")
            return c_void_p(t.data_ptr())

        _check(self.lib.dt_build_round_host(
            self.ctx, hp(H_host, torch.bfloat16, cfg.n_req * cfg.block * cfg.d, "H"),
            hp(root_host, torch.int32, cfg.n_req, "root_tok"),
            hp(out_host["tok"], torch.int32, cfg.n_req * s1, "tok"),
            hp(out_host["parent"], torch.int32, cfg.n_req * s1, "parent"),
            hp(out_host["depth"], torch.int32, cfg.n_req * s1, "depth"),
            hp(out_host["logp_cum"], torch.float32, cfg.n_req * s1, "logp_cum"),
            hp(out_host["mask"], torch.uint8, cfg.n_req * s1 * s1, "mask"), _stream(stream)),
            "dt_build_round_host")
        return out_host

    def check_bounded_waits(self, which: int, stream=None):
        """Launch the bounded-wait self-check (0: grid barrier with a missing
        participant, 1: an mbarrier nothing arrives on); read the outcome with
        device_status()."""
        _check(self.lib.dt_check_bounded_waits(self.ctx, int(which), _stream(stream)), "dt_check_bounded_waits")

    def device_status(self) -> int:
        return int(self.lib.dt_get_device_status(self.ctx))

    def round_kernel_count(self) -> int:
        return int(self.lib.dt_round_kernel_count(self.ctx))

    def plan(self) -> str:
        """Which kernels this context's rounds run (``dt_plan_string``)."""
        return self.lib.dt_plan_string(self.ctx).decode(errors="replace")


def topm_noalloc(logits, M, T, cand_tok, cand_base, rest_lse, stream=None):
    """Top-M and rest log-partition of each row of ``logits`` ([rows, V] fp32)
    without a context and without allocating device memory (dt_topm_noalloc):
    for callers that must not allocate.  Outputs are caller tensors:
    cand_tok [rows, M] int32, cand_base [rows, M] fp32, rest_lse [rows] fp32."""
    import torch
    if logits.dim() != 2:
        raise ValueError("logits: expected [rows, V]")
    rows, V = logits.shape
    lib = load_library()
    st = lib.dt_topm_noalloc(_ptr(logits, torch.float32, rows * V, "logits"), int(rows), int(V), int(M), float(T),
                             _ptr(cand_tok, torch.int32, rows * M, "cand_tok"),
                             _ptr(cand_base, torch.float32, rows * M, "cand_base"),
                             _ptr(rest_lse, torch.float32, rows, "rest_lse"), _stream(stream))
    if st != 0:
        raise DtreeError(st, "dt_topm_noalloc: " + lib.dt_last_error().decode(errors="replace"))


def bf16_tensor(bits, device="cuda"):
    """torch.bfloat16 tensor from a numpy uint16 array of bf16 bit patterns."""
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)

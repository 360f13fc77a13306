"""Named workload shapes.

The shapes follow the drafter the pages evaluate: a Qwen3-4B / Qwen3-8B
target's hidden size and vocabulary, a block of 16 positions (the last
verified token plus 15 masked positions, so depth 15), a GRU causal encoder
and a rank-256 correction bottleneck (Domino page, "Cabeza de Domino"), and
the DARTree hyper-parameters W (live branches kept per depth), K (children
per branch), B (verification budget) and beta (depth bonus, DARTree page,
"Poda Diferida", Lemma 1).  M is the Top-M candidate restriction of the
DominoTree page ("Restricción de Candidatos (Top-M)").
"""
from __future__ import annotations

from dataclasses import dataclass, replace, asdict


@dataclass(frozen=True)
class WorkloadConfig:
    name: str
    d: int          # backbone hidden size (rows of H, inner dim of the LM head)
    V: int          # vocabulary size
    block: int      # block length; depths are 1..block-1
    g: int          # GRU hidden size
    r: int          # correction bottleneck rank
    M: int          # Top-M candidates per depth
    K: int          # children kept per branch
    W: int          # live branches kept per depth
    B: int          # node budget of the emitted tree (root excluded)
    n_req: int = 1  # independent requests per round
    beta: float = 0.0   # depth bonus, <= 0 (> 0 only with positive_beta)
    T: float = 1.0      # temperature dividing the corrected logits
    root: str = "uniform"   # "zero": root token id 0; "uniform": uniform over V
    h_scale: str = "unit"   # "unit": H ~ N(0,1); "heavy": per-position scale ~ U[0.5, 4]
    weight_dtype: str = "bf16"  # "bf16" (rounded, RNE) or "fp32"
    marginal: bool = False      # marginal scoring: Delta L = 0 (path-independent children)
    builder: str = "dartree"    # "dartree" (depth-batched) or "best_first" (sequential heap)
    separate_topm: bool = False  # run the Top-M as its own kernel, not in the LM-head GEMM
    positive_beta: bool = False  # accept beta > 0 (DT_FLAG_POSITIVE_BETA; Lemma 1 not guaranteed)

    @property
    def D(self) -> int:
        return self.block - 1

    def with_(self, **kw) -> "WorkloadConfig":
        return replace(self, **kw)

    def as_dict(self) -> dict:
        return asdict(self)


CONFIGS = {
    # Tiny case the oracle finishes instantly; fp32 weights as stated for it,
    # root token id 0.
    "tiny": WorkloadConfig("tiny", d=64, V=1000, block=8, g=32, r=32, M=16, K=4,
                           W=4, B=16, beta=0.0, T=1.0, root="zero",
                           weight_dtype="fp32"),
    # The same shape with bf16 weights: what the CUDA path computes on.
    "tiny_bf16": WorkloadConfig("tiny_bf16", d=64, V=1000, block=8, g=32, r=32,
                                M=16, K=4, W=4, B=16, beta=0.0, T=1.0,
                                root="zero"),
    # Qwen3-4B shape, one request per round.
    "qwen3_4b": WorkloadConfig("qwen3_4b", d=2560, V=151936, block=16, g=1024,
                               r=256, M=64, K=8, W=8, B=64, beta=0.0, T=1.0),
    # Qwen3-8B shape (two temperatures are run: 0.6 and 1.0).
    "qwen3_8b": WorkloadConfig("qwen3_8b", d=4096, V=151936, block=16, g=1024,
                               r=256, M=128, K=16, W=16, B=128, beta=-0.5,
                               T=1.0),
    # Serving batch: 32 independent requests at the Qwen3-4B shape.
    "serving32": WorkloadConfig("serving32", d=2560, V=151936, block=16,
                                g=1024, r=256, M=64, K=8, W=8, B=64, n_req=32,
                                beta=0.0, T=1.0),
    # The Qwen3-4B shape with marginal scoring (the correction left out): the
    # conditional-versus-marginal ablation over the same super-tree.
    "qwen3_4b_marginal": WorkloadConfig("qwen3_4b_marginal", d=2560, V=151936, block=16, g=1024,
                                        r=256, M=64, K=8, W=8, B=64, beta=0.0, T=1.0, marginal=True),
    # Wide tree with heavy-tailed H (betas 0, -0.25, -1 are run).
    # The Qwen3-4B shape built node by node by the sequential conditional
    # best-first heap (the builder that depth batching replaces).
    "qwen3_4b_best_first": WorkloadConfig("qwen3_4b_best_first", d=2560, V=151936, block=16, g=1024,
                                          r=256, M=64, K=8, W=8, B=64, beta=0.0, T=1.0,
                                          builder="best_first"),
    "wide": WorkloadConfig("wide", d=2560, V=151936, block=16, g=1024, r=256,
                           M=256, K=32, W=64, B=512, beta=0.0, T=1.0,
                           h_scale="heavy"),
}


def get_config(name: str, **overrides) -> WorkloadConfig:
    cfg = CONFIGS[name]
    return cfg.with_(**overrides) if overrides else cfg

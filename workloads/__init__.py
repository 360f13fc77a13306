"""Seeded synthetic workloads for conditional draft-tree construction.

This package holds the named workload shapes and the seeded generators of
weights and per-round inputs.  It holds none of the method's arithmetic:
both the fp64 oracle (``oracle/``) and the CUDA library read what it makes.
"""
from .configs import WorkloadConfig, CONFIGS, get_config
from .generate import (
    bf16_round_bits,
    bf16_bits_to_f32,
    make_weights,
    make_round_inputs,
    make_rounds,
    make_target_logits,
    make_tree,
    WEIGHT_NAMES,
)

__all__ = [
    "WorkloadConfig",
    "CONFIGS",
    "get_config",
    "bf16_round_bits",
    "bf16_bits_to_f32",
    "make_weights",
    "make_round_inputs",
    "make_rounds",
    "make_target_logits",
    "make_tree",
    "WEIGHT_NAMES",
]

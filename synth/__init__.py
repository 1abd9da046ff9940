"""Seeded synthetic inputs for the routed bit-plane MoE expert layer.

This package only draws random tensors with the shapes and value
distributions of the workloads (and the per-expert bitwidth plans that the
workloads prescribe).  It holds none of the layer's arithmetic: no routing,
no permutation, no dequantisation, no FFN.  Both the fp64 oracle tests and the
GPU tests/bench take their inputs from here.
"""
from .workloads import (CONFIGS, LayerConfig, get_config, make_router, make_expert,
                        make_sensitivity, make_shared, make_tokens, bits_plan, zipf_bias)

__all__ = ["CONFIGS", "LayerConfig", "get_config", "make_router", "make_expert", "make_sensitivity",
           "make_shared", "make_tokens", "bits_plan", "zipf_bias"]

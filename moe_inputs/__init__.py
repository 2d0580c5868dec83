"""Seeded synthetic inputs for the DeepSeekMoE layer.

This package is the only code shared by the CUDA path's tests/bench and the CPU
oracle.  It holds layer shapes and random-number recipes, and none of the
method's arithmetic (no routing, no gating, no expert math).
"""
from .configs import LayerCfg, CONFIGS, get_config, small_cases  # noqa: F401
from .gen import make_inputs, make_tokens, make_norm_weight, make_dout  # noqa: F401

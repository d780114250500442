"""Seeded synthetic inputs for the W4A16 MoE expert layer.

This module is shared by the CUDA path's tests/bench and by the oracle's
tests. It holds no arithmetic of the method itself (no routing, no dequant,
no GEMM): only the random draws, their bf16 encoding as raw bits, and the
named workload shapes.
"""
from .configs import CONFIGS, LayerShape, Workload, workload  # noqa: F401
from .gen import (  # noqa: F401
    LayerInputs,
    bf16_bits,
    bf16_bits_to_f32,
    gen_attn,
    gen_embed,
    gen_gdn,
    gen_gain,
    gen_layer,
    gen_tokens,
    zipf_router_bias,
)

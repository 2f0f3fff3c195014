"""Seeded synthetic inputs for the fused mixed-precision MoE layer.

This package draws random numbers and lays them out; it holds none of the
layer's arithmetic (no bitplane packing, no dequantisation, no routing, no
matmul).  Both the CPU oracle and the CUDA library consume what it produces.
"""
from .configs import CONFIGS, LayerConfig, config_by_name  # noqa: F401
from .gen import Layer, make_layer, make_tokens, make_recommit  # noqa: F401

"""Seeded synthetic inputs for the int4 routed-expert MoE layer.

This package generates weights and activations only; it holds none of the
layer's arithmetic (no routing, no dequantisation, no matmul).  Both the CUDA
library's tests/benchmark and the CPU oracle take their inputs from here.
"""
from .configs import CONFIGS, LayerShape, config_by_name  # noqa: F401
from .gen import (  # noqa: F401
    LayerInputs,
    gen_activations,
    gen_expert_matrix,
    gen_layer,
    gen_router,
    scale_table,
)

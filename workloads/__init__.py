"""Seeded synthetic inputs for the routed MoE FFN forward.

This package draws inputs only, already in their storage formats (bf16 and
fp16 bit patterns, packed int4 bytes, fp32).  It holds none of the layer's
arithmetic: no routing, no dequantisation, no normalisation, no FFN.  Both the
CUDA library's tests/bench and the CPU oracle take their inputs from here.
"""
from .gen import (  # noqa: F401
    CONFIGS,
    LayerDims,
    WorkloadConfig,
    draw_layer,
    draw_tokens,
    draw_ids,
    ZIPF_S,
)

"""Seeded synthetic inputs for the MXFP4 mixture-of-experts layer.

This module only draws random numbers and packs them into the storage types of
the layer's inputs (bf16 bit patterns, MXFP4 code bytes, E8M0 scale bytes).  It
holds none of the layer's arithmetic, so both the CPU oracle and the CUDA path
can be fed from it without sharing any computation.
"""

from .gen import (  # noqa: F401
    CONFIGS,
    DENSE_CONFIGS,
    DenseLayerInputs,
    LayerInputs,
    bf16_bits_from_f32,
    bf16_bits_to_f32,
    make_layer,
    make_config,
    make_dense_config,
    make_dense_layer,
    make_norm_inputs,
    random_logits,
    random_topk_idx,
    zipf_router_bias,
)

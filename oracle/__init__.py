"""CPU oracle for the MXFP4 mixture-of-experts layer -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and its
Python binding) never imports, calls or links anything here, and nothing here
imports the product path.
"""

from .moe_oracle import (  # noqa: F401
    E2M1_VALUES,
    GATING_SIGMOID,
    GATING_SOFTMAX_ALL,
    GATING_SOFTMAX_TOPK,
    bf16_bits,
    bf16_round,
    bf16_to_f32,
    decode_e8m0,
    decode_mxfp4,
    expert_hidden,
    expert_hidden_dense,
    expert_output,
    expert_output_dense,
    moe_layer,
    moe_layer_dense,
    moe_layer_norm,
    rmsnorm_residual,
    router_logits,
    tile_rows_policy,
    tile_table,
    topk_gating,
    topk_margin,
    topk_softmax,
    max_tiles_bound,
)

"""CPU fp64 oracle of the sparse MoE FFN layer (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU baseline may
import this package; the product path never does.
"""
from .moe_oracle import (  # noqa: F401
    ACT_GEGLU_TANH,
    ACT_QUANT_E4M3_ROW,
    ACT_SWIGLU,
    E4M3_MAX,
    bf16_round,
    dequantize_rows,
    e4m3_round,
    quantize_rows_e4m3,
    activation,
    expert_ffn,
    finalize,
    grouped_ffn,
    init_routing,
    moe_layer,
    moe_layer_tokens,
    near_tie_tokens,
    permute,
    router_logits,
    scaled_projection,
    shared_expert,
    to_f64,
    topk_softmax,
)

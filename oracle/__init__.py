"""Plain CPU oracle of the MoE layer forward pass (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does.
"""
from .moe_oracle import (  # noqa: F401
    combine, combine_dedup, coselection, correlated_placement, partition, swap_gain,
    within_rank_coselection, dense_forward, dispatch, dispatch_dedup, dispatch_layout, expand,
    expert_ffn, layer_forward, layout_stats, shared_expert, rank_of_expert, route, route_sigmoid_bias, silu, slot_of_expert,
    swiglu_mlp, token_outputs, widen_bf16,
)

"""CPU oracle of the FusedMoE layer forward (test infrastructure only; see moe_oracle)."""
from .moe_oracle import (  # noqa: F401
    router_logits, score, group_score, route_token, select_experts, decision_margins,
    moe_align_block_size, round_bf16, silu, swiglu_mlp, expert_mlp, experts_combine, fused_moe,
    fused_moe_rows,
)
from .fp8_oracle import (  # noqa: F401
    e4m3_value, e4m3_round, e4m3_code, quant_group, dequant_group, quant_dequant,
    dequant_block, expert_mlp_fp8, experts_combine_fp8, fused_moe_fp8,
)
from .fp4_oracle import (  # noqa: F401
    e2m1_value, e2m1_round, e2m1_code, pack_fp4, unpack_fp4, weight_dequant, expert_act_fp4,
    expert_down_fp4, expert_mlp_fp4,
    experts_combine_fp4, fused_moe_fp4,
)

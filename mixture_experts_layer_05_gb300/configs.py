"""The five synthetic FusedMoE workloads (shapes, routing flags, value distributions).

Every field name follows the FusedMoE constructor on the vLLM ``fused_moe/layer``
page (``FusedMoE.__init__`` arguments: num_experts, top_k, hidden_size,
intermediate_size, renormalize, use_grouped_topk, num_expert_group, topk_group,
scoring_func, routed_scaling_factor) and, for the shared expert, the sglang
``models/deepseek_v2.py`` page (``DeepseekV2MoE.__init__``: the shared expert is one
``DeepseekV2MLP`` whose intermediate size is ``moe_intermediate_size *
n_shared_experts``).

This module holds shapes and distributions only: no routing or expert arithmetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field, asdict


@dataclass(frozen=True)
class MoEWorkload:
    name: str
    num_experts: int
    top_k: int
    hidden_size: int
    intermediate_size: int
    renormalize: bool
    use_grouped_topk: bool = False
    num_expert_group: int = 0
    topk_group: int = 0
    scoring_func: str = "softmax"          # "softmax" | "sigmoid"
    routed_scaling_factor: float = 1.0
    has_bias: bool = False                 # e_score_correction_bias present
    bias_std: float = 0.0
    shared_intermediate_size: int = 0      # 0 = no shared expert
    x_std: float = 1.0                     # hidden states ~ N(0, x_std)
    w_std: float = 0.02                    # expert weights ~ N(0, w_std), bf16
    logit_std: float = 1.0                 # router logits ~ N(0, logit_std), fp32
    zipf_s: float = 0.0                    # >0: Zipf(s) popularity offsets on logits
    zipf_beta: float = 0.0                 # scale of the Zipf log-offsets
    token_counts: tuple = field(default=())

    def as_dict(self) -> dict:
        return asdict(self)

    @property
    def expert_bytes(self) -> int:
        """bf16 bytes of one routed expert (w13 + w2)."""
        return 3 * self.hidden_size * self.intermediate_size * 2


TINY = MoEWorkload(
    name="tiny", num_experts=8, top_k=2, hidden_size=128, intermediate_size=256,
    renormalize=True, x_std=0.02, token_counts=(16,),
)

MIXTRAL = MoEWorkload(
    name="mixtral", num_experts=8, top_k=2, hidden_size=4096, intermediate_size=14336,
    renormalize=True, token_counts=(1, 16, 128, 1024, 4096),
)

# DeepSeek-V2: 160 routed experts, 2 shared experts of moe_intermediate 1536 each
# fold into one dense SwiGLU of intermediate 2 * 1536 = 3072.
DSV2 = MoEWorkload(
    name="dsv2", num_experts=160, top_k=6, hidden_size=5120, intermediate_size=1536,
    renormalize=False, use_grouped_topk=True, num_expert_group=8, topk_group=3,
    scoring_func="softmax", routed_scaling_factor=16.0, shared_intermediate_size=3072,
    token_counts=(1, 64, 512, 4096),
)

DSV3 = MoEWorkload(
    name="dsv3", num_experts=256, top_k=8, hidden_size=7168, intermediate_size=2048,
    renormalize=True, use_grouped_topk=True, num_expert_group=8, topk_group=4,
    scoring_func="sigmoid", routed_scaling_factor=2.5, has_bias=True, bias_std=0.1,
    shared_intermediate_size=2048, token_counts=(1, 32, 256, 2048, 8192),
)

# DeepSeek-V3 shapes with Zipf(1.2) expert popularity: logits get
# beta * log(rank^-s) added, rank drawn by a seeded permutation of the experts.
# beta = 0.5 makes the hottest expert receive about 16x the mean load while ~200
# of the 256 experts stay active (checked by a CPU test with the oracle's routing).
SKEW = MoEWorkload(
    name="skew", num_experts=256, top_k=8, hidden_size=7168, intermediate_size=2048,
    renormalize=True, use_grouped_topk=True, num_expert_group=8, topk_group=4,
    scoring_func="sigmoid", routed_scaling_factor=2.5, has_bias=True, bias_std=0.1,
    shared_intermediate_size=2048, zipf_s=1.2, zipf_beta=0.5,
    token_counts=tuple(2 ** i for i in range(15)),
)

WORKLOADS = {w.name: w for w in (TINY, MIXTRAL, DSV2, DSV3, SKEW)}


def get(name: str) -> MoEWorkload:
    return WORKLOADS[name]


def shrink(w: MoEWorkload, **overrides) -> MoEWorkload:
    """Same routing flags, smaller shapes (for tests that must finish on the oracle)."""
    d = w.as_dict()
    d.update(overrides)
    return MoEWorkload(**d)

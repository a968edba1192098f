"""Seeded random layer configurations against the oracle (GPU): routing flavour, expert and
group counts, top-k, shared expert, batch size (decode and prefill paths), bf16, FP8 or
NVFP4 weights. Routing must match bit for bit; the output stays within the layer's bound.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_05_gb300 import binding, configs, inputs
from tests.moe_cases import check_close, oracle_cfg, tokens

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _random_workload(rng: np.random.Generator, fp8: bool) -> configs.MoEWorkload:
    grouped = bool(rng.integers(2))
    if grouped:
        G = int(rng.choice([2, 4, 8]))
        E = G * int(rng.choice([2, 4, 8]))
        g = int(rng.integers(1, G + 1))
        k = int(rng.integers(1, min(8, g * (E // G)) + 1))
        sigmoid = bool(rng.integers(2))
        has_bias = sigmoid or bool(rng.integers(2))
    else:
        G = g = 0
        E = int(rng.choice([4, 8, 16, 32, 64]))
        k = int(rng.integers(1, min(8, E) + 1))
        sigmoid = False
        has_bias = bool(rng.integers(2))
    H = int(rng.choice([256, 512] if fp8 else [128, 256, 384]))
    I = int(rng.choice([128, 256, 384]))
    Is = int(rng.choice([0, 128, 256]))
    return configs.MoEWorkload(
        name=f"fuzz{E}_{k}_{H}_{I}", num_experts=E, top_k=k, hidden_size=H, intermediate_size=I,
        renormalize=bool(rng.integers(2)), use_grouped_topk=grouped, num_expert_group=G,
        topk_group=g, scoring_func="sigmoid" if sigmoid else "softmax",
        routed_scaling_factor=float(rng.choice([1.0, 2.5])), has_bias=has_bias,
        bias_std=0.1 if has_bias else 0.0, shared_intermediate_size=Is)


CASES = [(seed, fp8) for seed in range(40) for fp8 in (False, True)]


@pytest.mark.parametrize("seed,fp8", CASES, ids=[f"{s}-{'fp8' if f else 'bf16'}" for s, f in CASES])
def test_fuzz_layer(cuda_lib, seed, fp8):
    rng = np.random.default_rng(1000 + seed + (500 if fp8 else 0))
    w = _random_workload(rng, fp8)
    T = int(rng.choice([1, 2, 5, 16, 33, 150, 700]))
    if fp8:
        wts = inputs.make_fp8_weights(w, seed)
        names = ("w13_q", "w2_q", "shared_w13_q", "shared_w2_q")
    else:
        wts = inputs.make_weights(w, seed)
        names = ("w13", "w2", "shared_w13", "shared_w2")
    x, logits = tokens(w, T, wts["bias"], seed)
    d = {n: (None if v is None else v.to(DEV)) for n, v in wts.items()}
    kw = {}
    if fp8:
        kw = dict(w13_scale=d["w13_s"], w2_scale=d["w2_s"], shared_w13_scale=d["shared_w13_s"],
                  shared_w2_scale=d["shared_w2_s"])
    cfg = binding.config_from_workload(w, weight_quant="fp8" if fp8 else None)
    layer = binding.FusedMoE(cfg, d[names[0]], d[names[1]], d["bias"], d[names[2]], d[names[3]],
                             max_tokens=T, **kw)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    if fp8:
        y_ref, parts = oracle.fused_moe_fp8(x, logits, wts["bias"], wts["w13_q"], wts["w13_s"],
                                            wts["w2_q"], wts["w2_s"], wts["shared_w13_q"],
                                            wts["shared_w13_s"], wts["shared_w2_q"],
                                            wts["shared_w2_s"], return_parts=True,
                                            **oracle_cfg(w))
    else:
        y_ref, parts = oracle.fused_moe(x, logits, wts["bias"], wts["w13"], wts["w2"],
                                        wts["shared_w13"], wts["shared_w2"], return_parts=True,
                                        **oracle_cfg(w))
    lay = binding.moe_forward_workspace_layout(cfg, T)
    ids = layer.workspace[lay.topk_ids:lay.topk_ids + T * w.top_k * 4].view(torch.int32)
    assert np.array_equal(ids.cpu().numpy().reshape(T, w.top_k), parts["topk_ids"]), w
    check_close(y, y_ref, f"{w} T={T}")


FP4_CASES = list(range(24))


@pytest.mark.parametrize("seed", FP4_CASES, ids=[f"{s}-nvfp4" for s in FP4_CASES])
def test_fuzz_layer_nvfp4(cuda_lib, seed):
    """The NVFP4 layer on seeded random configurations: routing bit-exact, the act's
    quantization decisions equal to the oracle's away from rounding midpoints, y within the
    bound of the oracle's second GEMM and combine on the GPU's act (test_gpu_fp4)."""
    from tests.test_gpu_fp4 import _check_layer, _fp4_layer
    rng = np.random.default_rng(3000 + seed)
    w = _random_workload(rng, True)
    T = int(rng.choice([1, 2, 5, 16, 33, 150, 700]))
    wts = inputs.make_fp4_weights(w, seed)
    x, logits = tokens(w, T, wts["bias"], seed)
    layer = _fp4_layer(w, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    _check_layer(w, wts, layer, x, logits, y, T)

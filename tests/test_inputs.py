"""The seeded input generator: determinism, shapes, logit spread, margins, Zipf skew."""
import numpy as np
import torch

import oracle
from mixture_experts_layer_05_gb300 import configs, inputs
from tests.moe_cases import oracle_cfg, tokens


def test_deterministic_and_shaped():
    w = configs.TINY
    a = inputs.make_weights(w, 0)
    b = inputs.make_weights(w, 0)
    assert a["w13"].shape == (8, 512, 128) and a["w13"].dtype == torch.bfloat16
    assert a["w2"].shape == (8, 128, 256)
    assert torch.equal(a["w13"], b["w13"]) and torch.equal(a["w2"], b["w2"])
    x1, l1 = inputs.make_tokens(w, 16, 0)
    x2, l2 = inputs.make_tokens(w, 16, 0)
    assert torch.equal(x1, x2) and torch.equal(l1, l2)
    assert x1.dtype == torch.bfloat16 and l1.dtype == torch.float32
    assert abs(float(a["w13"].float().std()) - 0.02) < 2e-3
    assert abs(float(x1.float().std()) - 0.02) < 6e-3


def test_logit_rows_spread():
    lg = inputs.normal((64, 256), 1.0, 5)
    sp = inputs.spread_rows(lg)
    s, _ = torch.sort(sp.double(), dim=-1)
    assert float((s[:, 1:] - s[:, :-1]).min()) >= inputs.LOGIT_GAP * (1 - 1e-3)
    assert torch.equal(torch.argsort(sp, dim=-1, stable=True), torch.argsort(lg, dim=-1, stable=True))


def test_margin_redraw():
    w = configs.shrink(configs.DSV3, hidden_size=64, intermediate_size=64,
                       shared_intermediate_size=0)
    bias = inputs.make_weights(w, 0)["bias"]
    x, lg = tokens(w, 64, bias)
    m = oracle.decision_margins(lg, bias, **oracle_cfg(w))
    assert m.min() >= inputs.LOGIT_GAP


def test_zipf_skew_load():
    w = configs.shrink(configs.SKEW, hidden_size=64, intermediate_size=64,
                       shared_intermediate_size=0)
    bias = inputs.make_weights(w, 0)["bias"]
    _, lg = inputs.make_tokens(w, 512, 0)
    _, ids = oracle.select_experts(lg, bias, **oracle_cfg(w))
    cnt = np.bincount(ids.reshape(-1), minlength=w.num_experts)
    assert cnt.max() >= 10 * cnt.mean()


def test_fp4_weights_deterministic_shaped_and_scaled():
    w = configs.shrink(configs.DSV3, hidden_size=256, intermediate_size=128,
                       shared_intermediate_size=128)
    a = inputs.make_fp4_weights(w, 0)
    b = inputs.make_fp4_weights(w, 0)
    E, H, I = w.num_experts, w.hidden_size, w.intermediate_size
    assert a["w13"].shape == (E, 2 * I, H // 2) and a["w13"].dtype == torch.uint8
    assert a["w13_sf"].shape == (E, 2 * I, H // 16) and a["w13_sf"].dtype == torch.float8_e4m3fn
    assert a["w2"].shape == (E, H, I // 2) and a["w2_sf"].shape == (E, H, I // 16)
    assert a["shared_w13"].shape == (2 * I, H // 2) and a["shared_s2"].shape == (2,)
    for k in ("w13", "w13_sf", "w2", "w2_sf", "w13_s2", "shared_w2"):
        assert torch.equal(a[k].view(torch.uint8) if a[k].dtype == torch.float8_e4m3fn else a[k],
                           b[k].view(torch.uint8) if b[k].dtype == torch.float8_e4m3fn else b[k])
    sf = a["w13_sf"].view(torch.uint8)
    assert int(sf.min()) >= 0x30 and int(sf.max()) < 0x40       # e4m3 0.5 .. 1.875
    # the bias is the bf16 workload's rounded to bf16
    assert torch.equal(a["bias"], inputs.make_weights(w, 0)["bias"].to(torch.bfloat16).float())
    # the weights the codes stand for have about the bf16 workloads' rms
    W = oracle.weight_dequant(a["w13"][0], a["w13_sf"][0], float(a["w13_s2"][0]))
    assert 0.5 * w.w_std < float(np.sqrt(np.mean(W ** 2))) < 1.5 * w.w_std
    assert a["input_scale"] > 0 and a["act_scale"] > 0 and a["shared_act_scale"] > 0

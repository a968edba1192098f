"""Parity of the FP8 (w8a8, 128 x 128 block) CUDA path with the CPU oracle, on the GPU.

The quantized layer of the sglang ``models/deepseek_v2.py`` page: the input quantized once
per token and group of 128 columns (bit-exact against the oracle: the scale and the
quotient are both single fp32 divisions, the e4m3 conversion round-to-nearest-even), e4m3
weights with fp32 block scales, the act re-quantized before w2. Routing must match bit
for bit; the output within |y - y_ref| <= 2e-2 |y_ref| + 1e-2 rms(y_ref) (the oracle's act
is fp64, the kernel's fp32, so an act code may differ by one e4m3 step at a rounding
boundary; the bound absorbs it).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_05_gb300 import binding, configs, inputs
from tests.moe_cases import (check_close, check_routing_valid, gate_logit_error_bound,
                              oracle_cfg, tokens)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _values(q: torch.Tensor) -> np.ndarray:
    return oracle.e4m3_value(q.view(torch.uint8).cpu().numpy())


# ------------------------------------------------------------------ the input quant
@pytest.mark.parametrize("R,H", [(1, 256), (37, 384), (300, 7168)])
def test_quant_per_token_group_bitexact(cuda_lib, R, H):
    g = torch.Generator().manual_seed(R * 7 + H)
    x = torch.randn(R, H, generator=g) * torch.exp2(torch.randint(-20, 21, (R, 1), generator=g))
    x[0, :128] = 0.0                                            # an all-zero group
    if R > 2:
        x[1, 5] = 3.0e4                                         # one outlier in a group
        x[2] = torch.linspace(-1.0, 1.0, H) * 1e-30             # tiny magnitudes
    x = x.to(torch.bfloat16)
    q, s = binding.moe_quant_fp8_per_token_group(x.to(DEV))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle.quant_group(x)
    np.testing.assert_array_equal(s.cpu().numpy().T, s_ref)
    np.testing.assert_array_equal(_values(q), q_ref)


# ------------------------------------------------------------------ the layer, small shapes
def _fp8_layer(w, wts, T):
    cfg = binding.config_from_workload(w, weight_quant="fp8")
    d = {k: (None if v is None else v.to(DEV)) for k, v in wts.items()}
    layer = binding.FusedMoE(cfg, d["w13_q"], d["w2_q"], d["bias"], d["shared_w13_q"],
                             d["shared_w2_q"], max_tokens=max(T, 1), w13_scale=d["w13_s"],
                             w2_scale=d["w2_s"], shared_w13_scale=d["shared_w13_s"],
                             shared_w2_scale=d["shared_w2_s"])
    return layer, d


class _Host:
    """Per-expert slices copied to the host on demand (the oracle indexes w[e])."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].cpu()


def _oracle(w, wts, x, logits, bias, **kw):
    h = lambda n: None if wts[n] is None else wts[n].cpu()
    return oracle.fused_moe_fp8(x, logits, bias, _Host(wts["w13_q"]), _Host(wts["w13_s"]),
                                _Host(wts["w2_q"]), _Host(wts["w2_s"]), h("shared_w13_q"),
                                h("shared_w13_s"), h("shared_w2_q"), h("shared_w2_s"),
                                **oracle_cfg(w), **kw)


def _shrink(w, **kw):
    return configs.shrink(w, **kw)


SMALL = {
    "mixtral": _shrink(configs.MIXTRAL, hidden_size=512, intermediate_size=384),
    "dsv2": _shrink(configs.DSV2, hidden_size=512, intermediate_size=128,
                    shared_intermediate_size=256),
    "dsv3": _shrink(configs.DSV3, hidden_size=512, intermediate_size=256,
                    shared_intermediate_size=256),
}


def _routing_from_ws(layer, T, k):
    lay = binding.moe_forward_workspace_layout(layer.cfg, T)
    ws = layer.workspace
    ids = ws[lay.topk_ids:lay.topk_ids + T * k * 4].view(torch.int32).cpu().numpy()
    return ids.reshape(T, k), lay


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("T", [1, 16, 203, 600])
def test_fp8_forward_small(cuda_lib, name, T):
    w = SMALL[name]
    wts = inputs.make_fp8_weights(w, 0)
    x, logits = tokens(w, T, wts["bias"])
    layer, _ = _fp8_layer(w, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    y_ref, parts = _oracle(w, wts, x, logits, wts["bias"], return_parts=True)
    ids, lay = _routing_from_ws(layer, T, w.top_k)
    assert np.array_equal(ids, parts["topk_ids"])
    check_close(y, y_ref, f"fp8 {name} T={T}")
    # the routed act in the workspace: every real row's 128-column groups are e4m3 codes
    # whose largest magnitude is 448 (the group quant's defining property)
    ws = layer.workspace
    npp = int(ws[lay.num_tokens_post_padded:lay.num_tokens_post_padded + 4].view(torch.int32))
    srt = ws[lay.sorted_token_ids:lay.sorted_token_ids + npp * 4].view(torch.int32).cpu()
    rows = torch.nonzero(srt < T * w.top_k).flatten()
    I = w.intermediate_size
    act = ws[lay.act:lay.act + npp * I].view(npp, I)[rows.to(DEV)]
    a = np.abs(_values(act)).reshape(len(rows), I // 128, 128)
    assert (a.max(axis=2) == 448.0).all()


def test_fp8_deterministic(cuda_lib):
    w = SMALL["dsv3"]
    wts = inputs.make_fp8_weights(w, 0)
    x, logits = tokens(w, 300, wts["bias"])
    layer, _ = _fp8_layer(w, wts, 300)
    y1 = layer(x.to(DEV), logits.to(DEV)).clone()
    y2 = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)


# ------------------------------------------------------------------ decode sizes (split-K)
SPLIT = _shrink(configs.DSV3, num_experts=16, num_expert_group=4, topk_group=2, top_k=4,
                hidden_size=2048, intermediate_size=1024, shared_intermediate_size=1024)


@pytest.mark.parametrize("T", [1, 3, 17, 64])
def test_fp8_split_k(cuda_lib, T):
    """Few tiles and 16 K blocks: moe_forward cuts K into several splits."""
    wts = inputs.make_fp8_weights(SPLIT, 0)
    x, logits = tokens(SPLIT, T, wts["bias"])
    layer, _ = _fp8_layer(SPLIT, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    check_close(y, _oracle(SPLIT, wts, x, logits, wts["bias"]), f"fp8 split-K T={T}")
    assert torch.equal(y, layer(x.to(DEV), logits.to(DEV)))


# ------------------------------------------------------------------ full shapes, sampled
FULL = [("mixtral", 1, 1), ("dsv3", 1, 1), ("dsv3", 16, 2), ("dsv3", 2048, 3), ("dsv2", 64, 2)]


@pytest.mark.parametrize("name,T,n_sample", FULL)
def test_fp8_full_shapes_sampled(cuda_lib, name, T, n_sample):
    w = configs.WORKLOADS[name]
    torch.cuda.empty_cache()
    wts = inputs.make_fp8_weights(w, 0, device=DEV)
    bias_cpu = None if wts["bias"] is None else wts["bias"].cpu()
    x, logits = tokens(w, T, bias_cpu)
    layer, _ = _fp8_layer(w, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    _, ids_ref = oracle.select_experts(logits, bias_cpu, **oracle_cfg(w))
    ids, _ = _routing_from_ws(layer, T, w.top_k)
    assert np.array_equal(ids, ids_ref)
    rng = np.random.default_rng(T)
    rows = sorted({0, T - 1, *rng.choice(T, size=max(n_sample - 2, 0), replace=False).tolist()})
    rows = rows[:n_sample]
    y_ref = _oracle(w, wts, x[rows], logits[rows], bias_cpu)
    check_close(y[rows], y_ref, f"fp8 {name} T={T} rows {rows}")
    del layer, wts
    torch.cuda.empty_cache()


def test_fp8_cuda_graph_replay(cuda_lib):
    w = SMALL["dsv3"]
    wts = inputs.make_fp8_weights(w, 0)
    T = 37
    x, logits = tokens(w, T, wts["bias"])
    layer, _ = _fp8_layer(w, wts, T)
    xd, ld = x.to(DEV), logits.to(DEV)
    y_eager = layer(xd, ld).clone()
    out = torch.empty_like(y_eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        layer(xd, ld, out=out, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        layer(xd, ld, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, y_eager)


# ------------------------------------------------------------------ edge cases and options
def test_fp8_empty_batch_and_single_expert(cuda_lib):
    w = SMALL["mixtral"]
    layer, _ = _fp8_layer(w, inputs.make_fp8_weights(w, 0), 4)
    out = torch.full((0, w.hidden_size), 1.0, dtype=torch.bfloat16, device=DEV)
    layer(torch.empty(0, w.hidden_size, dtype=torch.bfloat16, device=DEV),
          torch.empty(0, w.num_experts, device=DEV), out=out)          # T = 0: a no-op
    # E = 1, k = 1: one dense fp8 SwiGLU MLP over more than one row block
    w1 = _shrink(configs.MIXTRAL, num_experts=1, top_k=1, hidden_size=512, intermediate_size=256)
    wts = inputs.make_fp8_weights(w1, 0)
    x, logits = tokens(w1, 200, None)
    layer1, _ = _fp8_layer(w1, wts, 200)
    y = layer1(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer1.device_status() == binding.OK
    check_close(y, _oracle(w1, wts, x, logits, None), "fp8 E=1 k=1")


def test_fp8_skewed_routing(cuda_lib):
    """Zipf-skewed DeepSeek-V3 routing (small shapes): hot experts span several row blocks."""
    w = _shrink(configs.SKEW, hidden_size=512, intermediate_size=256, shared_intermediate_size=256)
    wts = inputs.make_fp8_weights(w, 0)
    x, logits = tokens(w, 300, wts["bias"])
    layer, _ = _fp8_layer(w, wts, 300)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    check_close(y, _oracle(w, wts, x, logits, wts["bias"]), "fp8 skew T=300")


@pytest.mark.parametrize("T", [1, 77])
def test_fp8_from_gate_weight(cuda_lib, T):
    """The router GEMM in front of the fp8 layer: logits = x @ W_gate^T in fp32 first. Rows
    whose decision margin exceeds 1e-4 (far above the fp32 logit error) must route exactly
    like the oracle and match its output; closer rows must hold a valid routing for logits
    within the GEMM's fp32 error bound and match the oracle's fp8 experts and combine run
    on the GPU's own ids and weights."""
    w = SMALL["dsv3"]
    wts = inputs.make_fp8_weights(w, 0)
    gate = inputs.normal((w.num_experts, w.hidden_size), w.hidden_size ** -0.5,
                         inputs.tensor_seed(w.name, "gate", 0), torch.bfloat16)
    x = inputs.normal((T, w.hidden_size), 1.0, 5, torch.bfloat16)
    layer, _ = _fp8_layer(w, wts, T)
    y = layer(x.to(DEV), gate_weight=gate.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    logits = oracle.router_logits(x, gate)
    safe = oracle.decision_margins(logits, wts["bias"], **oracle_cfg(w)) >= 1e-4
    ids, lay = _routing_from_ws(layer, T, w.top_k)
    tw = layer.workspace[lay.topk_weights:lay.topk_weights + T * w.top_k * 4] \
        .view(torch.float32).cpu().numpy().reshape(T, w.top_k)
    check_routing_valid(w, ids, tw, logits, wts["bias"], gate_logit_error_bound(x, gate),
                        f"fp8 gate T={T}")
    rows = np.flatnonzero(safe).tolist()
    if rows:
        y_ref, parts = _oracle(w, wts, x[rows], logits[rows], wts["bias"], return_parts=True)
        assert np.array_equal(ids[rows], parts["topk_ids"])
        check_close(y[rows], y_ref, f"fp8 gate T={T}")
    close = np.flatnonzero(~safe).tolist()
    if close:
        y_own = oracle.experts_combine_fp8(x[close], tw[close], ids[close], wts["w13_q"],
                                           wts["w13_s"], wts["w2_q"], wts["w2_s"],
                                           wts["shared_w13_q"], wts["shared_w13_s"],
                                           wts["shared_w2_q"], wts["shared_w2_s"])
        check_close(y[close], y_own, f"fp8 gate T={T}, close rows on the GPU's routing")
    if T > 1:
        assert safe.mean() > 0.9


def test_fp8_stage_events_in_a_graph(cuda_lib):
    w = SMALL["dsv3"]
    wts = inputs.make_fp8_weights(w, 0)
    x, logits = tokens(w, 16, wts["bias"])
    layer, _ = _fp8_layer(w, wts, 16)
    xd, ld = x.to(DEV), logits.to(DEV)
    y_eager = layer(xd, ld).clone()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(binding.NUM_STAGE_EVENTS)]
    out = torch.empty_like(y_eager)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        layer(xd, ld, out=out, events=evs)
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, y_eager)
    times = [evs[i].elapsed_time(evs[i + 1]) for i in range(len(evs) - 1)]
    assert all(t >= 0 for t in times) and sum(times) > 0

"""Pins of the oracle's expert-MLP variants (CPU only).

The variants are the FusedMoE constructor's ``with_bias`` / ``is_gated`` /
``gemm1_alpha`` / ``gemm1_clamp_limit`` / ``apply_router_weight_on_input`` (sglang
``fused_moe_triton/layer.py`` page) and ``DeepseekV2MLP``'s ``swiglu_limit`` (sglang
``models/deepseek_v2.py`` page). Each pin checks a hand-worked value, a closed form or
a reduction to a torch routine; planted mistakes must trip at least one pin.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
from oracle import moe_oracle as om


def _cfg(**kw):
    base = dict(num_experts=4, top_k=2, renormalize=True, use_grouped_topk=False,
                num_expert_group=0, topk_group=0, scoring_func="softmax",
                routed_scaling_factor=1.0)
    base.update(kw)
    return base


def pin_clamp_hand_example():
    """x = 1, gate weight 10, up weight -9, limit 7: act = 7 sigmoid(7) (-7)."""
    o = oracle.expert_mlp(np.array([[1.0]]), np.array([[10.0], [-9.0]]), np.array([[1.0]]),
                          swiglu_limit=7.0)
    want = 7.0 / (1.0 + math.exp(-7.0)) * -7.0
    assert abs(o[0, 0] - want) < 1e-12
    # alpha 2 without a limit: act = g sigmoid(2 g) u, g = 0.5, u = 3
    o = oracle.expert_mlp(np.array([[1.0]]), np.array([[0.5], [3.0]]), np.array([[2.0]]),
                          gemm1_alpha=2.0)
    assert abs(o[0, 0] - 2.0 * 0.5 / (1.0 + math.exp(-1.0)) * 3.0) < 1e-12


def pin_clamp_reduces_to_plain():
    rng = np.random.default_rng(20)
    h = rng.normal(size=(5, 6))
    w13, w2 = rng.normal(size=(8, 6)), rng.normal(size=(6, 4))
    plain = oracle.swiglu_mlp(h, w13, w2)
    big = oracle.expert_mlp(h, w13, w2, swiglu_limit=1e9, gemm1_alpha=1.0)
    np.testing.assert_allclose(big, plain, rtol=1e-14)
    # the clamp binds: the largest gate value is cut to the limit, up is cut on both sides
    lim = 0.5
    W13, H_ = torch.tensor(w13), torch.tensor(h)
    g = torch.clamp(H_ @ W13[:4].T, max=lim)
    u = torch.clamp(H_ @ W13[4:].T, min=-lim, max=lim)
    ref = (torch.nn.functional.silu(g) * u) @ torch.tensor(w2).T
    np.testing.assert_allclose(oracle.expert_mlp(h, w13, w2, swiglu_limit=lim), ref.numpy(),
                               rtol=1e-12, atol=1e-14)


def pin_bias_dense():
    """E = 1, top_k = 1: the layer is torch's linear-with-bias SwiGLU MLP."""
    rng = np.random.default_rng(21)
    x = rng.normal(size=(6, 8))
    w13, w2 = rng.normal(size=(1, 10, 8)), rng.normal(size=(1, 8, 5))
    b13, b2 = rng.normal(size=(1, 10)), rng.normal(size=(1, 8))
    y = oracle.fused_moe(x, rng.normal(size=(6, 1)), None, w13, w2, w13_bias=b13, w2_bias=b2,
                         act_dtype=None, **_cfg(num_experts=1, top_k=1))
    X = torch.tensor(x)
    F = torch.nn.functional
    g = F.linear(X, torch.tensor(w13[0, :5]), torch.tensor(b13[0, :5]))
    u = F.linear(X, torch.tensor(w13[0, 5:]), torch.tensor(b13[0, 5:]))
    ref = F.linear(F.silu(g) * u, torch.tensor(w2[0]), torch.tensor(b2[0]))
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-13)


def pin_bias_zero_weights():
    """Zero weights: every expert outputs silu(bg) * bu pushed through w2 plus b2."""
    rng = np.random.default_rng(22)
    E, n = 4, 3
    b13 = rng.normal(size=(E, 2 * n))
    b2 = rng.normal(size=(E, n))
    w13 = np.zeros((E, 2 * n, n))
    w2 = np.stack([np.eye(n)] * E)
    x = rng.normal(size=(5, n))
    logits = rng.normal(size=(5, E))
    y = oracle.fused_moe(x, logits, None, w13, w2, w13_bias=b13, w2_bias=b2, act_dtype=None, **_cfg())
    W, ids = oracle.select_experts(logits, None, **_cfg())
    for t in range(5):
        want = sum(W[t, j] * (om.silu(b13[e, :n]) * b13[e, n:] + b2[e])
                   for j, e in enumerate(ids[t]))
        np.testing.assert_allclose(y[t], want, rtol=1e-12)


def pin_non_gated_dense():
    rng = np.random.default_rng(23)
    x = rng.normal(size=(4, 6))
    w1, w2 = rng.normal(size=(1, 5, 6)), rng.normal(size=(1, 6, 5))
    y = oracle.fused_moe(x, rng.normal(size=(4, 1)), None, w1, w2, gated=False,
                         act_dtype=None, **_cfg(num_experts=1, top_k=1))
    ref = torch.nn.functional.silu(torch.tensor(x) @ torch.tensor(w1[0]).T) @ \
        torch.tensor(w2[0]).T
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12)


def pin_router_weight_on_input():
    """Identity-like experts: y = sum_j silu(a w_j x) (b w_j x) elementwise."""
    rng = np.random.default_rng(24)
    E, n = 4, 5
    a = rng.uniform(0.5, 2.0, E)
    b = rng.uniform(-2.0, 2.0, E)
    w13 = np.stack([np.vstack([a[e] * np.eye(n), b[e] * np.eye(n)]) for e in range(E)])
    w2 = np.stack([np.eye(n)] * E)
    x = rng.normal(size=(6, n))
    logits = rng.normal(size=(6, E))
    y = oracle.fused_moe(x, logits, None, w13, w2, apply_router_weight_on_input=True, act_dtype=None, **_cfg())
    W, ids = oracle.select_experts(logits, None, **_cfg())
    for t in range(6):
        want = sum(om.silu(a[e] * W[t, j] * x[t]) * (b[e] * W[t, j] * x[t])
                   for j, e in enumerate(ids[t]))
        np.testing.assert_allclose(y[t], want, rtol=1e-12)


def pin_shared_expert_clamped_unbiased():
    """The shared expert takes the SwiGLU limit (DeepseekV2MLP) but no expert bias."""
    rng = np.random.default_rng(25)
    x = rng.normal(size=(3, 4))
    sw13, sw2 = rng.normal(size=(6, 4)), rng.normal(size=(4, 3))
    w13, w2 = np.zeros((2, 4, 4)), np.zeros((2, 4, 2))
    y = oracle.fused_moe(x, rng.normal(size=(3, 2)), None, w13, w2, sw13, sw2,
                         w13_bias=np.zeros((2, 4)), w2_bias=np.zeros((2, 4)),
                         swiglu_limit=0.3, act_dtype=None, **_cfg(num_experts=2, top_k=1))
    np.testing.assert_allclose(y, oracle.expert_mlp(x, sw13, sw2, swiglu_limit=0.3),
                               rtol=1e-12, atol=1e-15)


def pin_router_weight_on_input_bf16():
    """The weighted input is a tensor of the layer dtype: identity-like experts give
    y = sum_j bf16(silu(a r) (b r)) with r = bf16(w_j x), both roundings to nearest even."""
    rng = np.random.default_rng(26)
    E, n = 4, 5
    a = rng.uniform(0.5, 2.0, E)
    b = rng.uniform(-2.0, 2.0, E)
    w13 = np.stack([np.vstack([a[e] * np.eye(n), b[e] * np.eye(n)]) for e in range(E)])
    w2 = np.stack([np.eye(n)] * E)
    x = rng.normal(size=(6, n)) * 2.0
    logits = rng.normal(size=(6, E))
    y = oracle.fused_moe(x, logits, None, w13, w2, apply_router_weight_on_input=True, **_cfg())
    W, ids = oracle.select_experts(logits, None, **_cfg())
    bf = lambda v: torch.tensor(v, dtype=torch.float32).to(torch.bfloat16).double().numpy()
    for t in range(6):
        want = 0.0
        for j, e in enumerate(ids[t]):
            r = bf((W[t, j] * x[t]).astype(np.float32))
            want = want + bf((om.silu(a[e] * r) * (b[e] * r)).astype(np.float32))
        # float32 detours: the exact fp64 values round through fp32 first; compare loosely
        np.testing.assert_allclose(y[t], want, rtol=2e-7, atol=1e-7)
    y_exact = oracle.fused_moe(x, logits, None, w13, w2, apply_router_weight_on_input=True,
                               act_dtype=None, **_cfg())
    assert np.abs(y - y_exact).max() > 1e-4


PINS = [pin_clamp_hand_example, pin_clamp_reduces_to_plain, pin_bias_dense,
        pin_bias_zero_weights, pin_non_gated_dense, pin_router_weight_on_input,
        pin_router_weight_on_input_bf16,
        pin_shared_expert_clamped_unbiased]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_variant_pin(pin):
    pin()


_orig_expert = om.expert_mlp


def _clamp_gate_both_sides(h, w13_e, w2_e, *, swiglu_limit=None, **kw):
    if swiglu_limit is None:
        return _orig_expert(h, w13_e, w2_e, **kw)
    W13 = np.asarray(w13_e, dtype=np.float64)
    I = W13.shape[0] // 2
    z = np.atleast_2d(h) @ W13.T
    g = np.clip(z[:, :I], -swiglu_limit, swiglu_limit)
    u = np.minimum(z[:, I:], swiglu_limit)
    return (om.silu(g) * u) @ np.asarray(w2_e, dtype=np.float64).T


def _drop_b13(h, w13_e, w2_e, *, b13_e=None, **kw):
    return _orig_expert(h, w13_e, w2_e, **kw)


def _alpha_ignored(h, w13_e, w2_e, *, gemm1_alpha=1.0, **kw):
    return _orig_expert(h, w13_e, w2_e, **kw)


@pytest.mark.parametrize("fn", [_clamp_gate_both_sides, _drop_b13, _alpha_ignored])
def test_planted_variant_mistake_is_caught(monkeypatch, fn):
    monkeypatch.setattr(om, "expert_mlp", fn)
    monkeypatch.setattr(oracle, "expert_mlp", fn)
    caught = 0
    for pin in PINS:
        try:
            pin()
        except AssertionError:
            caught += 1
    assert caught, fn.__name__


def test_planted_weight_on_both_sides_is_caught(monkeypatch):
    orig = om.fused_moe

    def both(*a, apply_router_weight_on_input=False, **kw):
        y = orig(*a, apply_router_weight_on_input=apply_router_weight_on_input, **kw)
        if apply_router_weight_on_input:        # also weight the output: a plausible slip
            W, _ = oracle.select_experts(a[1], a[2], **{k: v for k, v in kw.items()
                                                        if k in _cfg()})
            y = y * W.sum(axis=1, keepdims=True) * 0.5
        return y

    monkeypatch.setattr(oracle, "fused_moe", both)
    with pytest.raises(AssertionError):
        pin_router_weight_on_input()


def test_router_logits_is_a_matmul():
    """The router GEMM reduces to torch's matmul of the bf16 operands widened to fp64."""
    g = torch.Generator().manual_seed(30)
    x = torch.randn(9, 64, generator=g).to(torch.bfloat16)
    wg = torch.randn(12, 64, generator=g).to(torch.bfloat16)
    ref = (x.double() @ wg.double().T).numpy()
    np.testing.assert_allclose(oracle.router_logits(x, wg), ref, rtol=1e-15, atol=0)
    # a transposed operand would not even have the right shape
    assert oracle.router_logits(x, wg).shape == (9, 12)
    # hand-worked: x = (1, 2), gate rows (3, 4) and (5, 6) -> logits 11, 17
    np.testing.assert_array_equal(oracle.router_logits(np.array([[1.0, 2.0]]),
                                                       np.array([[3.0, 4.0], [5.0, 6.0]])),
                                  [[11.0, 17.0]])


def test_planted_unrounded_weighted_input_is_caught(monkeypatch):
    """A layer that rounds the act but leaves the weighted input rows exact fails the
    bf16 weight-on-input pin."""
    def combine(x, topk_weights, topk_ids, w13, w2, shared_w13=None, shared_w2=None, *,
                return_parts=False, apply_router_weight_on_input=False, top_k=None,
                act_dtype="bf16", **kw):
        X = om._f64(x)
        W = np.atleast_2d(np.asarray(topk_weights, dtype=np.float64))
        ids = np.atleast_2d(np.asarray(topk_ids))
        y = np.zeros_like(X)
        for t in range(X.shape[0]):
            for j in range(ids.shape[1]):
                h = X[t:t + 1] * (W[t, j] if apply_router_weight_on_input else 1.0)
                o = om.expert_mlp(h, w13[ids[t, j]], w2[ids[t, j]], act_dtype=act_dtype)[0]
                y[t] += o if apply_router_weight_on_input else W[t, j] * o
        return y

    monkeypatch.setattr(om, "experts_combine", combine)
    with pytest.raises(AssertionError):
        pin_router_weight_on_input_bf16()

"""Pins of the NVFP4 oracle (CPU only).

The format and the fp4_quantize steps (blocks of 16 e2m1 values with an e4m3 scale and an
fp32 per-tensor scale, as FlashInferFP4MoE quantizes its hidden states on the sglang
fused_moe_triton/layer.py page) are checked against hand-worked values, every code's value
from its bit fields, the format's error bound, exact special cases and a layer of
identity-like experts; planted mistakes must each be caught by some pin.
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest
import torch

import oracle
from oracle import fp4_oracle as f4
from oracle import moe_oracle as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fp4_hand_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def pin_code_values():
    """Every 4-bit code decodes from its fields: sign bit 3, exponent bits 1..2 (bias 1),
    mantissa bit 0; exponent 0 is subnormal (mantissa * 0.5)."""
    for c in range(16):
        s, e, m = c >> 3, (c >> 1) & 3, c & 1
        mag = m * 0.5 if e == 0 else 2.0 ** (e - 1) * (1 + m / 2)
        want = -mag if s else mag
        assert f4.e2m1_value(c) == want, (c, f4.e2m1_value(c), want)


def pin_hand_rounding():
    g = _golden()
    for r in g["rounding"]:
        assert f4.e2m1_round(r["x"]) == r["q"], r
    p = g["packing"]
    assert f4.pack_fp4(np.array(p["codes"])).tolist() == p["bytes"]
    assert f4.unpack_fp4(np.array(p["bytes"], dtype=np.uint8)).tolist() == p["codes"]


def pin_hand_blocks():
    for b in _golden()["blocks"]:
        q, sf = f4.quantize(np.array([b["x"]]), b["g"])
        assert sf.tolist() == [[b["sf"]]], (b["name"], sf)
        assert q[0].tolist() == b["q"], (b["name"], q[0])
        if b["name"] == "scale_rounds_up":
            np.testing.assert_allclose(f4.dequantize(q, sf, b["g"])[0, 0], 7.68, rtol=1e-12)


def pin_rounding_properties():
    """e2m1_round lands on the grid, is odd-symmetric, monotone, leaves grid values alone, and
    errs by at most half the local grid step (up to 6; beyond, it saturates)."""
    rng = np.random.default_rng(31)
    v = np.concatenate([rng.uniform(-7, 7, 20000), np.linspace(-6, 6, 2401)])
    q = f4.e2m1_round(v)
    assert np.isin(np.abs(q), f4.E2M1_MAGNITUDES).all()
    np.testing.assert_array_equal(f4.e2m1_round(-v), -q)
    order = np.argsort(v)
    assert (np.diff(q[order]) >= 0).all()
    grid = np.concatenate([-f4.E2M1_MAGNITUDES, f4.E2M1_MAGNITUDES])
    np.testing.assert_array_equal(f4.e2m1_round(grid), grid)
    a = np.abs(v)
    step = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    inside = a <= 6
    assert (np.abs(q - v)[inside] <= step[inside] / 2 + 1e-12).all()
    assert (np.abs(q[~inside]) == 6).all()


def pin_quantize_error_bound():
    """Dequantized blocks are within half an e2m1 step (times sf / g) of x, or, where the
    block scale rounded down, saturated at 6 sf / g; the block's largest value uses the top
    of the range (|q| >= 4)."""
    rng = np.random.default_rng(32)
    x = rng.normal(size=(40, 64)) * np.exp2(rng.integers(-6, 6, size=(40, 1)))
    for g in (1.0, 37.5, 300.0):
        q, sf = f4.quantize(x, g)
        dq = f4.dequantize(q, sf, g)
        S = np.repeat(sf, 16, axis=1) / np.float32(g)
        xr = np.abs(x.astype(np.float32).astype(np.float64)) / np.where(S > 0, S, 1)
        step = np.where(xr < 2, 0.5, np.where(xr < 4, 1.0, 2.0))
        ok = (np.abs(dq - x) <= step / 2 * S * (1 + 1e-6) + 1e-300) | (np.abs(q) == 6)
        assert ok.all()
        blocks = np.abs(q).reshape(40, 4, 16).max(axis=2)
        assert (blocks >= 4).all()


def pin_weight_dequant():
    """w = q * sf * s2 with the codes unpacked low nibble first and the e4m3 scales decoded."""
    codes = np.array([[1, 2, 3, 15] + [0] * 12])              # 0.5, 1, 1.5, -6
    packed = f4.pack_fp4(codes)
    sf = torch.tensor([[2.0]]).to(torch.float8_e4m3fn)
    w = f4.weight_dequant(packed, sf, 0.25)
    np.testing.assert_array_equal(w[0, :4], [0.25, 0.5, 0.75, -3.0])
    assert (w[0, 4:] == 0).all()


def _identity_layer():
    """Two experts whose w13 gate block is the identity, up block twice the identity and w2
    the identity (e2m1 codes 2 = 1.0 and 4 = 2.0 on the diagonals, block scales 1), with
    per-expert scales s2."""
    n = 16
    eye = np.eye(n)
    codes = np.where(eye > 0, 2, 0)                       # e2m1 code 2 = 1.0
    twice = np.where(eye > 0, 4, 0)                       # e2m1 code 4 = 2.0
    w13 = np.stack([f4.pack_fp4(np.vstack([codes, twice])) for _ in range(2)])
    w2 = np.stack([f4.pack_fp4(codes) for _ in range(2)])
    one = torch.ones(2, 2 * n, 1).to(torch.float8_e4m3fn)
    one2 = torch.ones(2, n, 1).to(torch.float8_e4m3fn)
    return {"w13": w13, "w13_sf": one, "w2": w2, "w2_sf": one2,
            "w13_s2": np.array([1.0, 0.5]), "w2_s2": np.array([1.0, 2.0]),
            "input_scale": 2.0, "act_scale": 3.0}


def pin_identity_layer():
    """With these weights the layer is, per slot, quantize(silu(s xq) * (2 s xq)) * s2' with xq
    the quantized input: written out with the oracle's own quantize as the only step."""
    w = _identity_layer()
    rng = np.random.default_rng(33)
    x = rng.normal(size=(3, 16))
    ids = np.array([[0, 1], [1, 0], [0, 1]])
    tw = np.array([[0.7, 0.3], [0.6, 0.4], [0.5, 0.5]])
    y = f4.experts_combine_fp4(x, tw, ids, w)
    xq = f4.quant_dequant(x, 2.0)
    for t in range(3):
        want = 0.0
        for j in range(2):
            e = ids[t, j]
            z = xq[t] * w["w13_s2"][e]                   # gate = s2 xq, up = 2 s2 xq
            act = om.silu(z) * (2 * z)
            want = want + tw[t, j] * f4.quant_dequant(act[None], 3.0)[0] * w["w2_s2"][e]
        np.testing.assert_allclose(y[t], want, rtol=1e-12, atol=1e-15)


def pin_layer_near_exact_layer():
    """The fp4 layer equals the exact bf16-oracle layer on the dequantized input and weights
    up to the act quantization alone (|dy| within the act's quantization error pushed through
    w2), and the difference is not zero (the act is quantized)."""
    w = _identity_layer()
    rng = np.random.default_rng(34)
    x = rng.normal(size=(4, 16))
    logits = rng.normal(size=(4, 2))
    cfg = dict(num_experts=2, top_k=1, renormalize=True, use_grouped_topk=False,
               num_expert_group=0, topk_group=0, scoring_func="softmax",
               routed_scaling_factor=1.0)
    y = f4.fused_moe_fp4(x, logits, None, w, **cfg)
    W13 = np.stack([f4.weight_dequant(w["w13"][e], w["w13_sf"][e], w["w13_s2"][e]) for e in range(2)])
    W2 = np.stack([f4.weight_dequant(w["w2"][e], w["w2_sf"][e], w["w2_s2"][e]) for e in range(2)])
    xq = f4.quant_dequant(x, 2.0)
    y_ref = om.fused_moe(xq, logits, None, W13, W2, act_dtype=None, **cfg)
    diff = np.abs(y - y_ref)
    assert diff.max() > 0
    # per element: at most |w2| (2) times the act's half step at its scale (<= 6 sf / g / 6 * 2 / 2)
    act_amax = np.abs(y_ref).max()
    assert diff.max() <= act_amax * 2.0 / 6.0 + 1e-12


ALL_PINS = [pin_code_values, pin_hand_rounding, pin_hand_blocks, pin_rounding_properties,
            pin_quantize_error_bound, pin_weight_dequant, pin_identity_layer,
            pin_layer_near_exact_layer]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_fp4_pin(pin):
    pin()


def _round_half_up(v):
    v = np.asarray(v, dtype=np.float64)
    G = f4.E2M1_MAGNITUDES
    a = np.minimum(np.abs(v), 6.0)
    hi = np.minimum(np.searchsorted(G, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    pick = np.where(a - G[lo] < G[hi] - a, lo, hi)
    return np.copysign(G[pick], v)


def _unpack_high_first(p):
    p = np.asarray(p, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p >> 4
    out[..., 1::2] = p & 15
    return out


_orig_quantize = f4.quantize


def _scale_not_rounded(x, g, block=16):
    X = np.atleast_2d(om._f64(x)).astype(np.float32)
    R, C = X.shape
    B = X.reshape(R, C // block, block)
    amax = np.max(np.abs(B), axis=2).astype(np.float64)
    sf = g * amax / 6.0                                   # exact, not an e4m3 value
    r = np.where(sf > 0, g / np.where(sf > 0, sf, 1), 0)
    return f4.e2m1_round(B * r[:, :, None]).reshape(R, C), sf


def _inverted_global(x, g, block=16):
    return _orig_quantize(x, 1.0 / g, block)


def _weight_no_s2(packed, scales, scale2):
    return _orig_wd(packed, scales, 1.0)


_orig_wd = f4.weight_dequant


def _act_not_quantized(xq, w13_packed, w13_sf, w13_s2, w2_packed, w2_sf, w2_s2, act_scale):
    W13 = f4.weight_dequant(w13_packed, w13_sf, w13_s2)
    W2 = f4.weight_dequant(w2_packed, w2_sf, w2_s2)
    z = np.atleast_2d(xq) @ W13.T
    I = W13.shape[0] // 2
    return (om.silu(z[:, :I]) * z[:, I:]) @ W2.T


def _gate_up_swapped(xq, w13_packed, w13_sf, w13_s2, w2_packed, w2_sf, w2_s2, act_scale):
    W13 = f4.weight_dequant(w13_packed, w13_sf, w13_s2)
    W2 = f4.weight_dequant(w2_packed, w2_sf, w2_s2)
    z = np.atleast_2d(xq) @ W13.T
    I = W13.shape[0] // 2
    return f4.quant_dequant(om.silu(z[:, I:]) * z[:, :I], act_scale) @ W2.T


@pytest.mark.parametrize("name,fn", [("e2m1_round", _round_half_up),
                                     ("unpack_fp4", _unpack_high_first),
                                     ("quantize", _scale_not_rounded),
                                     ("quantize", _inverted_global),
                                     ("weight_dequant", _weight_no_s2),
                                     ("expert_mlp_fp4", _act_not_quantized),
                                     ("expert_mlp_fp4", _gate_up_swapped)],
                         ids=["half_up", "high_nibble_first", "scale_unrounded",
                              "inverted_global_scale", "no_weight_scale_2", "act_unquantized",
                              "gate_up_swapped"])
def test_planted_fp4_mistake_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(f4, name, fn)
    caught = []
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError):
            caught.append(pin.__name__)
    assert caught, f"no pin caught the planted mistake in {name}"

"""Pins of the FP8 (w8a8, block-128) oracle (CPU only).

The fp8 layer is the sglang ``models/deepseek_v2.py`` page's quantized DeepSeek MoE:
per-token-group-128 activation quant (``DeepseekV2MoE._maybe_quant_moe_input_once``,
``DeepseekV2MLP.forward``'s post-SiLU quant), [128, 128] block weights with fp32 scales
(``DeepseekV2MoE._compute_moe_quant_once_enabled``), dtype ``torch.float8_e4m3fn``.

Each pin checks the format's own definition against torch's float8 conversion (a library
routine), a hand-worked value, an error bound of the format, or a closed form of the
layer; planted mistakes must each trip a pin.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import fp8_oracle as fo
from oracle import moe_oracle as om


def _torch_e4m3(v) -> np.ndarray:
    """torch's float32 -> float8_e4m3fn -> float64 round trip."""
    t = torch.as_tensor(np.asarray(v, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).to(torch.float64).numpy()


def _finite_values() -> np.ndarray:
    v = oracle.e4m3_value(np.arange(256))
    return np.unique(v[np.isfinite(v)])


# ---------------------------------------------------------------- the format
def pin_e4m3_value_matches_torch():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.e4m3_value(np.arange(256))
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
    assert np.isnan(got).sum() == 2                       # 0x7F and 0xFF only
    assert np.nanmax(got) == 448.0 and np.nanmin(np.abs(got[got != 0])) == 2.0 ** -9


def pin_e4m3_round_matches_torch():
    vals = _finite_values()
    pos = vals[vals > 0]
    mids = (pos[:-1] + pos[1:]) / 2                       # exact ties, fp32-representable
    rng = np.random.default_rng(40)
    rand = np.sign(rng.normal(size=200000)) * np.exp2(rng.uniform(-12, np.log2(448), 200000))
    for v in (vals, mids, -mids, rand.astype(np.float32)):
        np.testing.assert_array_equal(oracle.e4m3_round(v), _torch_e4m3(v))


def pin_e4m3_hand_values():
    """Hand-worked: 448 = 1.75 * 2^8 is code 0x7E; 1 = 0x38; 2^-9 = 0x01 (smallest
    subnormal); 1.0625 lies halfway between 1 and 1.125 and goes to the even mantissa
    (1); 1.1875 lies halfway between 1.125 and 1.25 and goes to 1.25."""
    assert oracle.e4m3_code([448.0, 1.0, 2.0 ** -9, -2.0]).tolist() == [0x7E, 0x38, 0x01, 0xC0]
    np.testing.assert_array_equal(oracle.e4m3_round([1.0625, 1.1875, 500.0, -1e9, 2.0 ** -11]),
                                  [1.0, 1.25, 448.0, -448.0, 0.0])


# ---------------------------------------------------------------- group quant
def pin_quant_group_hand_example():
    """A group whose largest magnitude is 56: scale 56 / 448 = 0.125 exactly, and every
    element divides to an exact e4m3 value except 0.4125 / 0.125 = 3.3 -> 3.25."""
    x = np.zeros((1, 256))
    x[0, :5] = [56.0, -28.0, 1.0, 0.4125, -0.0625]
    x[0, 128] = 3.0                                       # second group: scale 3/448
    q, s = oracle.quant_group(x)
    assert s[0, 0] == 0.125
    assert s[0, 1] == float(np.float32(3.0) / np.float32(448.0))
    np.testing.assert_array_equal(q[0, :5], [448.0, -224.0, 8.0, 3.25, -0.5])
    assert q[0, 128] == 448.0 and not q[0, 129:].any()


def pin_quant_group_properties():
    rng = np.random.default_rng(41)
    R = 128                                               # as many rows as a group is wide
    x = torch.tensor(rng.normal(size=(R, 384)) * np.exp2(rng.integers(-8, 8, (R, 1))),
                     dtype=torch.bfloat16)
    x[3, 128:256] = 0.0                                   # an all-zero group
    q, s = oracle.quant_group(x)
    X = x.double().numpy()
    G = X.reshape(R, 3, 128)
    amax = np.abs(G).max(axis=2)
    nz = amax > 0
    want_s = np.where(nz, (amax.astype(np.float32) / np.float32(448)).astype(np.float64),
                      float(np.float32(1e-10) / np.float32(448)))
    np.testing.assert_array_equal(s, want_s)
    Q = np.abs(q.reshape(R, 3, 128))
    np.testing.assert_array_equal(Q.max(axis=2)[nz], 448.0)   # the group max hits 448
    assert not Q[~nz].any()
    # dequantization error within half an e4m3 spacing of the quotient
    quot = np.abs(X) / np.repeat(s, 128, axis=1)
    half = np.where(quot >= 2.0 ** -6, quot * 2.0 ** -4, 2.0 ** -10) * (1 + 1e-6)
    err = np.abs(oracle.dequant_group(q, s) - X) / np.repeat(s, 128, axis=1)
    assert np.all(err <= half)


# ---------------------------------------------------------------- block weights
def pin_dequant_block_indexing():
    """Code 0x38 (= 1) everywhere on a [256, 384] matrix and scale[i, j] = 10 i + j + 1:
    w[n, k] = 10 (n // 128) + k // 128 + 1."""
    codes = np.full((256, 384), 0x38, dtype=np.uint8)
    scale = np.array([[1.0, 2.0, 3.0], [11.0, 12.0, 13.0]])
    w = oracle.dequant_block(codes, scale)
    assert w[0, 0] == 1.0 and w[127, 383] == 3.0 and w[128, 0] == 11.0 and w[255, 200] == 12.0
    codes[5, 300] = 0xC0                                  # -2
    assert oracle.dequant_block(codes, scale)[5, 300] == -6.0


# ---------------------------------------------------------------- the layer
def _cfg(**kw):
    base = dict(num_experts=4, top_k=2, renormalize=True, use_grouped_topk=False,
                num_expert_group=0, topk_group=0, scoring_func="softmax",
                routed_scaling_factor=1.0)
    base.update(kw)
    return base


def _eye_codes(n):
    return np.where(np.eye(n, dtype=bool), 0x38, 0x00).astype(np.uint8)


def pin_layer_output_on_act_grid():
    """E = 1, k = 1, w13 = [Id; Id], w2 = Id (unit scales): y = dequant(quant(silu(xd) xd)),
    so y / s_act lies on the e4m3 grid with its largest magnitude exactly 448, and equals
    torch's float8 rounding of the same quotient."""
    rng = np.random.default_rng(42)
    n = 128
    x = torch.tensor(rng.normal(size=(3, n)), dtype=torch.bfloat16)
    w13 = np.concatenate([_eye_codes(n), _eye_codes(n)])[None]
    w2 = _eye_codes(n)[None]
    one = np.ones((1, 1, 1))
    y = oracle.fused_moe_fp8(x, rng.normal(size=(3, 1)), None, w13, np.ones((1, 2, 1)), w2,
                             one, **_cfg(num_experts=1, top_k=1))
    xd = oracle.quant_dequant(x)
    act = (xd / (1 + np.exp(-xd)) * xd).astype(np.float32)
    s = (np.abs(act).max(axis=1) / np.float32(448)).astype(np.float32).astype(np.float64)
    quot = (act / s[:, None].astype(np.float32)).astype(np.float32)
    np.testing.assert_array_equal(y, _torch_e4m3(quot) * s[:, None])
    assert np.all(np.abs(y / s[:, None]).max(axis=1) == 448.0)
    assert np.isin(np.abs(y / s[:, None]), _finite_values()).all()


def _dequant_stack(q, s):
    return np.stack([oracle.dequant_block(q[e], s[e]) for e in range(q.shape[0])])


def _small_fp8_case(seed=43, E=4, k=2, H=256, I=256, Is=128, T=6):
    rng = np.random.default_rng(seed)
    g = torch.Generator().manual_seed(seed)
    codes = lambda *sh: (torch.randn(*sh, generator=g) * 112).clamp(-448, 448).to(
        torch.float8_e4m3fn).view(torch.uint8).numpy()
    sc = lambda *sh: rng.uniform(0.8, 1.2, sh) * 0.02 * 4 / 448
    d = dict(w13_q=codes(E, 2 * I, H), w13_s=sc(E, 2 * I // 128, H // 128),
             w2_q=codes(E, H, I), w2_s=sc(E, H // 128, I // 128),
             sw13_q=codes(2 * Is, H), sw13_s=sc(2 * Is // 128, H // 128),
             sw2_q=codes(H, Is), sw2_s=sc(H // 128, Is // 128))
    x = torch.tensor(rng.normal(size=(T, H)), dtype=torch.bfloat16)
    logits = rng.normal(size=(T, E))
    return x, logits, d


def pin_layer_near_bf16_layer_on_dequantized_operands():
    """The fp8 layer equals the bf16-oracle layer run on the dequantized input and
    weights up to the act quant alone: |dy| <= sum_j w_j |W2| (half e4m3 spacing of act),
    and the difference is not zero (the act quant is applied)."""
    x, logits, d = _small_fp8_case()
    cfg = _cfg()
    y = oracle.fused_moe_fp8(x, logits, None, d["w13_q"], d["w13_s"], d["w2_q"], d["w2_s"],
                             d["sw13_q"], d["sw13_s"], d["sw2_q"], d["sw2_s"], **cfg)
    xd = oracle.quant_dequant(x)
    W13, W2 = _dequant_stack(d["w13_q"], d["w13_s"]), _dequant_stack(d["w2_q"], d["w2_s"])
    S13 = oracle.dequant_block(d["sw13_q"], d["sw13_s"])
    S2 = oracle.dequant_block(d["sw2_q"], d["sw2_s"])
    y_ref = om.fused_moe(xd, logits, None, W13, W2, S13, S2, act_dtype=None, **cfg)
    W, ids = om.select_experts(logits, None, **cfg)

    def act_err(h, w13):
        z = h @ w13.T
        I = w13.shape[0] // 2
        act = om.silu(z[:, :I]) * z[:, I:]
        s = np.repeat(np.abs(act).reshape(len(h), -1, 128).max(axis=2) / 448, 128, axis=1)
        return np.abs(act) * 2.0 ** -4 + 2.0 ** -10 * s + 1e-12

    bound = np.zeros_like(y)
    for t in range(len(x)):
        for j in range(cfg["top_k"]):
            e = ids[t, j]
            bound[t] += W[t, j] * (np.abs(W2[e]) @ act_err(xd[t:t + 1], W13[e])[0])
        bound[t] += np.abs(S2) @ act_err(xd[t:t + 1], S13)[0]
    assert np.all(np.abs(y - y_ref) <= bound)
    assert np.abs(y - y_ref).max() > 1e-6 * np.abs(y_ref).max()


def pin_layer_expert_relabeling():
    """Permuting the expert labels (weights, scales and logit columns together) leaves y."""
    x, logits, d = _small_fp8_case(seed=44)
    perm = np.array([2, 0, 3, 1])
    args = lambda dd, lg: (x, lg, None, dd["w13_q"], dd["w13_s"], dd["w2_q"], dd["w2_s"])
    y0 = oracle.fused_moe_fp8(*args(d, logits), **_cfg())
    dp = {k: (v[perm] if k in ("w13_q", "w13_s", "w2_q", "w2_s") else v) for k, v in d.items()}
    y1 = oracle.fused_moe_fp8(*args(dp, logits[:, perm]), **_cfg())
    np.testing.assert_allclose(y1, y0, rtol=1e-13, atol=1e-15)


def pin_layer_w2_scale_linearity():
    """Doubling every w2 block scale doubles the routed output exactly (no shared)."""
    x, logits, d = _small_fp8_case(seed=45)
    a = (x, logits, None, d["w13_q"], d["w13_s"], d["w2_q"])
    y1 = oracle.fused_moe_fp8(*a, d["w2_s"], **_cfg())
    y2 = oracle.fused_moe_fp8(*a, 2 * d["w2_s"], **_cfg())
    np.testing.assert_array_equal(y2, 2 * y1)


PINS = [pin_e4m3_value_matches_torch, pin_e4m3_round_matches_torch, pin_e4m3_hand_values,
        pin_quant_group_hand_example, pin_quant_group_properties, pin_dequant_block_indexing,
        pin_layer_output_on_act_grid, pin_layer_near_bf16_layer_on_dequantized_operands,
        pin_layer_expert_relabeling, pin_layer_w2_scale_linearity]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_fp8_pin(pin):
    pin()


# ---------------------------------------------------------------- planted mistakes
_orig_quant, _orig_round, _orig_dequant_block = fo.quant_group, fo.e4m3_round, fo.dequant_block


def _quant_inverted_scale(x, group=128):
    q, s = _orig_quant(x, group)
    return q, 1.0 / s


def _quant_by_column(x, group=128):
    X = np.atleast_2d(om._f64(x))
    if X.shape[0] % group:                  # the wrong axis only applies where it fits
        return _orig_quant(x, group)
    q, s = _orig_quant(X.T, group)
    return q.T, s.T.repeat(group, axis=0)[: X.shape[0]]


def _round_half_up(v):
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), 448.0)
    _, ex = np.frexp(a)
    quantum = np.exp2(np.maximum(ex - 1, -6) - 3.0)
    return np.copysign(np.minimum(np.floor(a / quantum + 0.5) * quantum, 448.0), v)


def _dequant_block_transposed(q_codes, scale, block=128):
    S = np.asarray(scale, dtype=np.float64)
    if S.shape[0] == S.shape[1]:
        return _orig_dequant_block(q_codes, S.T, block)
    return _orig_dequant_block(q_codes, S[::-1], block)


def _expert_no_act_quant(xd, w13_q, w13_s, w2_q, w2_s):
    W13, W2 = fo.dequant_block(w13_q, w13_s), fo.dequant_block(w2_q, w2_s)
    z = np.atleast_2d(xd) @ W13.T
    I = W13.shape[0] // 2
    return (om.silu(z[:, :I]) * z[:, I:]) @ W2.T


@pytest.mark.parametrize("name,fn", [("quant_group", _quant_inverted_scale),
                                     ("quant_group", _quant_by_column),
                                     ("e4m3_round", _round_half_up),
                                     ("dequant_block", _dequant_block_transposed),
                                     ("expert_mlp_fp8", _expert_no_act_quant)])
def test_planted_fp8_mistake_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(fo, name, fn)
    monkeypatch.setattr(oracle, name, fn)
    caught = 0
    for pin in PINS:
        try:
            pin()
        except (AssertionError, ValueError):
            caught += 1
    assert caught, f"{name} <- {fn.__name__}"

"""CPU oracle of the NVFP4 FusedMoE layer (w4a4): plain, slow, fp64, written from the pages.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module: only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of ``bench.py`` may use it.
It shares no code with the CUDA path.

The layer is the one ``FlashInferFP4MoE`` runs on the sglang ``fused_moe_triton/layer.py``
page: the hidden states are quantized each forward with ``fp4_quantize(hidden_states,
w13_input_scale_quant, 16, use_ue8m0=False, ...)`` into packed fp4 values ([T, H / 2]
bytes) and one fp8-e4m3 scale per 16 values ([T, H / 16]); the expert weights are fp4 with
e4m3 block scales (``gemm1_weights`` / ``gemm1_weights_scale``, ``gemm2_*``) and a
per-tensor fp32 scale (the same page's weight loader takes fp4's per-tensor scale from the
``weight_scale_2`` tensors); ``trtllm_fp4_block_scale_moe`` multiplies each GEMM's output by
a per-expert scalar (``output1_scale_gate_scalar`` / ``output2_scale_scalar``) and
quantizes the activation before the second GEMM with its own scale
(``output1_scale_scalar``).

The pages print the call sites, not the arithmetic. Readings used here (NVFP4 as the format
is published: fp4 e2m1 values, blocks of 16 with an e4m3 scale, a second fp32 scale per
tensor):

- e2m1: sign, 2 exponent bits (bias 1), 1 mantissa bit: magnitudes 0, 0.5, 1, 1.5, 2, 3, 4,
  6 (codes 0..7, bit 3 the sign); rounding to nearest, ties to the even code (mantissa bit
  0), saturating at 6.
- Packing: element 2i in the low nibble of byte i, element 2i + 1 in the high nibble.
- ``fp4_quantize(x, g)`` per row and block of 16 consecutive values, every step one fp32
  operation: amax = max |x|; sf = e4m3(g * (amax / 6)) (round to nearest even, saturating
  at 448); r = g / sf (0 when sf is 0); q = e2m1(x * r). Dequantized, the block holds
  q * sf / g: the block scale maps its largest value to about 6, the per-tensor scale g
  keeps the block scales inside e4m3's range.
- Weights: w = q * sf * s2 with e2m1 codes q, e4m3 block scales sf per 16 values along K
  and a per-expert fp32 scale s2 (``weight_scale_2``).
- The layer: z = xq @ w13^T with xq = dequantized quantize(x, g1) (quantized once, the same
  for every expert of the token); act = silu(gate) * up; aq = dequantized
  quantize(fp32(act), g2); o = aq @ w2^T; y = sum_j weight_j o_j over slots ascending, plus
  the shared expert computed the same way with its own scales, unscaled.
- fp64 everywhere except the quantization steps, which take the fp32 operations the
  format's definition names; the quantized codes and block scales are therefore exact
  decisions the GPU path must reproduce bit for bit on the same fp32 inputs.
"""
from __future__ import annotations

import numpy as np

from . import moe_oracle as _mo
from . import fp8_oracle as _f8

FP4_BLOCK = 16
E2M1_MAX = 6.0
E2M1_MAGNITUDES = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


# ---------------------------------------------------------------- the e2m1 format
def e2m1_value(codes) -> np.ndarray:
    """Value of each 4-bit e2m1 code (bit 3 the sign, bits 0..2 the magnitude index)."""
    c = np.asarray(codes, dtype=np.int64) & 15
    mag = E2M1_MAGNITUDES[c & 7]
    return np.where(c & 8, -mag, mag)


def e2m1_round(v) -> np.ndarray:
    """Nearest e2m1 value of each value (fp64 in, exact values out): magnitudes past 6
    saturate to 6; a value halfway between two grid points goes to the one with mantissa
    bit 0, i.e. the even code (0, 1, 2 or 4)."""
    v = np.asarray(v, dtype=np.float64)
    G = E2M1_MAGNITUDES
    a = np.minimum(np.abs(v), E2M1_MAX)
    hi = np.minimum(np.searchsorted(G, a, side="left"), 7)   # first grid point >= a
    lo = np.maximum(hi - 1, 0)
    dlo, dhi = a - G[lo], G[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(G[hi] == a, hi, pick)
    return np.copysign(G[pick], v)


def e2m1_code(values) -> np.ndarray:
    """The 4-bit code of each exact e2m1 value."""
    v = np.asarray(values, dtype=np.float64)
    idx = np.searchsorted(E2M1_MAGNITUDES, np.abs(v))
    if not np.array_equal(E2M1_MAGNITUDES[np.minimum(idx, 7)], np.abs(v)):
        raise ValueError("not e2m1 values")
    return (idx | np.where(np.signbit(v) & (v != 0), 8, 0)).astype(np.uint8)


def pack_fp4(codes) -> np.ndarray:
    """Codes [..., 2n] -> bytes [..., n]: element 2i in the low nibble of byte i."""
    c = np.asarray(codes, dtype=np.uint8) & 15
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


def unpack_fp4(packed) -> np.ndarray:
    """Bytes [..., n] -> codes [..., 2n] (low nibble first)."""
    p = np.asarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (2 * p.shape[-1],), dtype=np.uint8)
    out[..., 0::2] = p & 15
    out[..., 1::2] = p >> 4
    return out


# ---------------------------------------------------------------- fp4_quantize
def quantize(x, global_scale: float, block: int = FP4_BLOCK):
    """(q values [R, C] fp64, block scales [R, C / block] e4m3 values fp64) of fp4_quantize
    with per-tensor scale g: per block, sf = e4m3(g * (amax / 6)), r = g / sf, q = e2m1(x * r),
    each step one fp32 operation."""
    X = np.atleast_2d(_mo._f64(x)).astype(np.float32)
    R, C = X.shape
    if C % block:
        raise ValueError("columns must be a multiple of the block size")
    g = np.float32(global_scale)
    B = X.reshape(R, C // block, block)
    amax = np.max(np.abs(B), axis=2)
    sfv = (g * (amax / np.float32(E2M1_MAX)).astype(np.float32)).astype(np.float32)
    sf = _f8.e4m3_round(np.minimum(sfv.astype(np.float64), _f8.FP8_MAX))
    sf32 = sf.astype(np.float32)
    with np.errstate(divide="ignore"):
        r = np.where(sf32 > 0, (g / np.where(sf32 > 0, sf32, np.float32(1))).astype(np.float32),
                     np.float32(0))
    prod = (B * r[:, :, None]).astype(np.float32)
    q = e2m1_round(prod.astype(np.float64)).reshape(R, C)
    return q, sf


def dequantize(q, sf, global_scale: float, block: int = FP4_BLOCK) -> np.ndarray:
    """q * sf / g, the block scale broadcast over its 16 values (fp64, exact products)."""
    Q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    S = np.atleast_2d(np.asarray(sf, dtype=np.float64))
    return Q * np.repeat(S, block, axis=1) / np.float64(np.float32(global_scale))


def quant_dequant(x, global_scale: float) -> np.ndarray:
    q, sf = quantize(x, global_scale)
    return dequantize(q, sf, global_scale)


# ---------------------------------------------------------------- weights
def weight_dequant(packed, scales, scale2) -> np.ndarray:
    """One [N, K] fp4 weight: packed codes [N, K / 2] bytes, e4m3 block scales [N, K / 16]
    (float8_e4m3fn tensor or uint8 codes), fp32 per-tensor scale: w = q * sf * s2."""
    if hasattr(packed, "detach"):
        packed = packed.detach().cpu().numpy()
    if hasattr(scales, "detach"):
        import torch
        t = scales.detach().cpu()
        scales = (t.view(torch.uint8) if t.dtype != torch.uint8 else t).numpy()
    q = e2m1_value(unpack_fp4(packed))
    sf = _f8.e4m3_value(np.arange(256))[np.asarray(scales, dtype=np.uint8)]
    return q * np.repeat(sf, FP4_BLOCK, axis=1) * np.float64(np.float32(scale2))


# ---------------------------------------------------------------- the layer
def expert_act_fp4(xq, w13_packed, w13_sf, w13_s2) -> np.ndarray:
    """The first half of an NVFP4 expert on dequantized input rows xq [n, H]:
    z = xq @ W13^T, act = silu(gate) * up (fp64, before its quantization)."""
    W13 = weight_dequant(w13_packed, w13_sf, w13_s2)
    z = np.atleast_2d(xq) @ W13.T
    I = W13.shape[0] // 2
    return _mo.silu(z[:, :I]) * z[:, I:]


def expert_down_fp4(aq, w2_packed, w2_sf, w2_s2) -> np.ndarray:
    """The second GEMM of an NVFP4 expert on dequantized act rows aq [n, I]: o = aq @ W2^T."""
    return np.atleast_2d(aq) @ weight_dequant(w2_packed, w2_sf, w2_s2).T


def expert_mlp_fp4(xq, w13_packed, w13_sf, w13_s2, w2_packed, w2_sf, w2_s2, act_scale) -> np.ndarray:
    """One NVFP4 expert on already-dequantized input rows xq [n, H]: z = xq @ W13^T,
    act = silu(gate) * up, aq = dequantized fp4_quantize(fp32(act), act_scale), o = aq @ W2^T."""
    act = expert_act_fp4(xq, w13_packed, w13_sf, w13_s2)
    return expert_down_fp4(quant_dequant(act, act_scale), w2_packed, w2_sf, w2_s2)


def experts_combine_fp4(x, topk_weights, topk_ids, w, *, return_parts=False):
    """y [T, H] fp64 of the NVFP4 experts and the combine for a routing given as input.

    ``w`` holds the layer's tensors: w13 / w13_sf / w13_s2 (per expert), w2 / w2_sf / w2_s2,
    input_scale (g1), act_scale (g2), and, for a shared expert, shared_w13, shared_w13_sf,
    shared_w13_s2, shared_w2, shared_w2_sf, shared_w2_s2, shared_input_scale,
    shared_act_scale.
    """
    X = _mo._f64(x)
    T, H = X.shape
    W = np.atleast_2d(np.asarray(topk_weights, dtype=np.float64))
    ids = np.atleast_2d(np.asarray(topk_ids, dtype=np.int64))
    k = ids.shape[1]
    xq = quant_dequant(X, w["input_scale"]) if T else np.zeros((0, H))
    o = np.zeros((T, k, H), dtype=np.float64)
    for e in sorted(set(ids.reshape(-1).tolist())):
        rows = [(t, j) for t in range(T) for j in range(k) if ids[t, j] == e]
        out = expert_mlp_fp4(xq[[t for t, _ in rows]], w["w13"][e], w["w13_sf"][e],
                             float(w["w13_s2"][e]), w["w2"][e], w["w2_sf"][e],
                             float(w["w2_s2"][e]), w["act_scale"])
        for (t, j), r in zip(rows, out):
            o[t, j] = r
    y = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            y[t] += W[t, j] * o[t, j]
    shared = None
    if w.get("shared_w13") is not None and T:
        xs = quant_dequant(X, w["shared_input_scale"])
        shared = expert_mlp_fp4(xs, w["shared_w13"], w["shared_w13_sf"],
                                float(w["shared_w13_s2"]), w["shared_w2"], w["shared_w2_sf"],
                                float(w["shared_w2_s2"]), w["shared_act_scale"])
        y = y + shared
    if return_parts:
        return y, {"topk_weights": W, "topk_ids": ids, "expert_out": o, "shared": shared,
                   "x_dequant": xq}
    return y


def fused_moe_fp4(x, logits, bias, w, *, return_parts=False, **cfg):
    """y [T, H] fp64 of the NVFP4 layer: routing as the bf16 layer, then
    ``experts_combine_fp4``."""
    W, ids = _mo.select_experts(logits, bias, **cfg)
    return experts_combine_fp4(x, W, ids, w, return_parts=return_parts)

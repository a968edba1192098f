"""CPU oracle of the FP8 (w8a8, block-128) FusedMoE layer forward.

TEST INFRASTRUCTURE ONLY, like ``moe_oracle``: nothing on the product path imports it;
it shares no code with the CUDA path.

What the pages fix (sglang ``models/deepseek_v2.py`` page):

* ``DeepseekV2MoE._moe_quant_once_enabled`` / ``_maybe_quant_moe_input_once``: the MoE
  input is quantized once per layer to fp8 per token and per group of 128 consecutive
  hidden columns, and that one quantized tensor feeds both the shared expert's fp8 GEMM
  and the routed experts.
* ``DeepseekV2MoE._compute_moe_quant_once_enabled``: routed and shared expert weights are
  fp8 with a [128, 128] weight block size and fp32 scales (the non-UE8M0 path); the
  routed experts take a dynamic per-token-group-128 fp8 activation quant.
* ``DeepseekV2MLP.forward`` (the fast path for fp8 ``down_proj`` weights with
  ``weight_scale_inv``): the SiLU-and-mul output is quantized per token group of 128
  before the fp8 down GEMM (``silu_and_mul_contig_post_quant`` with
  ``quant_group_size=128``), and that GEMM writes bf16.
* The fp8 type is ``torch.float8_e4m3fn`` (named in the same passages).

What the pages leave open, and the reading taken here:

* The e4m3fn value set (``e4m3_value``): 1 sign bit, 4 exponent bits with bias 7, 3
  mantissa bits, subnormals below 2^-6, no infinities, the largest finite value 448 and
  the codes 0x7F / 0xFF reserved for NaN (the OCP 8-bit floating point format that the
  dtype's name refers to). Rounding to it (``e4m3_round``) is round-to-nearest-even,
  saturating at +-448.
* The group quant (``quant_group``): for each row and group, ``amax = max |x|``,
  ``s = max(amax, 1e-10) / 448`` and ``q = e4m3(clip(x / s, -448, 448))``, all in fp32
  (the group's largest magnitude lands on the largest finite code; the floor 1e-10
  keeps an all-zero group defined). The scale is the dequantization factor: x ~ q * s.
* The block weights (``dequant_block``): ``w[n, k] = q[n, k] * s[n // 128, k // 128]``:
  ``weight_scale_inv`` is the factor that multiplies the code back.
* A w8a8 GEMM is the product of the two dequantized operands (each K block's partial
  product times its two scales is the same sum regrouped); the oracle forms it in fp64.

Everything else (routing, align, SwiGLU, combine, the unscaled shared expert) is the
bf16 layer's, taken from ``moe_oracle``.
"""
from __future__ import annotations

import numpy as np

from . import moe_oracle as _mo

FP8_MAX = 448.0
GROUP = 128
SCALE_FLOOR = 1e-10


# ---------------------------------------------------------------- the e4m3fn format
def e4m3_value(code) -> np.ndarray:
    """Value of each e4m3fn byte (fp64; NaN for 0x7F and 0xFF)."""
    c = np.asarray(code, dtype=np.int64) & 0xFF
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    v = sign * np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, v)


def e4m3_round(v) -> np.ndarray:
    """Nearest e4m3fn value (ties to even mantissa), saturating at +-448 (fp64 result)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.minimum(np.abs(v), FP8_MAX)
    _, ex = np.frexp(a)                         # a = f * 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, -6)                  # unbiased exponent, subnormals share 2^-6
    quantum = np.exp2(e - 3.0)                  # spacing of the 3-bit mantissa
    r = np.round(a / quantum) * quantum         # a / quantum is exact; np.round is RNE
    r = np.minimum(r, FP8_MAX)
    return np.copysign(r, v)


def e4m3_code(v) -> np.ndarray:
    """Byte of each value already on the e4m3fn grid (|v| <= 448), -0 as 0x80."""
    v = np.asarray(v, dtype=np.float64)
    table = e4m3_value(np.arange(256))
    out = np.zeros(v.shape, dtype=np.uint8)
    flat, res = v.reshape(-1), out.reshape(-1)
    for i, x in enumerate(flat):
        hits = np.nonzero(table == x)[0]
        if x == 0.0:
            res[i] = 0x80 if np.signbit(x) else 0x00
        elif hits.size:
            res[i] = hits[0]
        else:
            raise ValueError(f"{x!r} is not an e4m3fn value")
    return out


# ---------------------------------------------------------------- per-token-group quant
def quant_group(x, group: int = GROUP):
    """Per row, per group of ``group`` consecutive columns: fp32 scale and e4m3 values.

    Returns ``(q, s)``: ``q [R, C]`` fp64 holding e4m3 values (the codes' values), ``s
    [R, C // group]`` fp64 holding fp32 scales. The scale and the quotient are formed in
    fp32, one rounding each, as a per-token-group quant kernel computes them.
    """
    X = np.atleast_2d(_mo._f64(x)).astype(np.float32)
    R, C = X.shape
    if C % group:
        raise ValueError("columns must be a multiple of the group size")
    G = X.reshape(R, C // group, group)
    amax = np.max(np.abs(G), axis=2) if C else np.zeros((R, 0), np.float32)
    s = (np.maximum(amax, np.float32(SCALE_FLOOR)) / np.float32(FP8_MAX)).astype(np.float32)
    quot = (G / s[:, :, None]).astype(np.float32)
    quot = np.clip(quot, -FP8_MAX, FP8_MAX)
    q = e4m3_round(quot.astype(np.float64)).reshape(R, C)
    return q, s.astype(np.float64)


def dequant_group(q, s, group: int = GROUP) -> np.ndarray:
    """x ~ q * s, the scale of a row's group broadcast over its columns (fp64, exact)."""
    Q = np.atleast_2d(np.asarray(q, dtype=np.float64))
    S = np.atleast_2d(np.asarray(s, dtype=np.float64))
    return Q * np.repeat(S, group, axis=1)


def quant_dequant(x, group: int = GROUP) -> np.ndarray:
    q, s = quant_group(x, group)
    return dequant_group(q, s, group)


# ---------------------------------------------------------------- block-128 weights
def dequant_block(q_codes, scale, block: int = GROUP) -> np.ndarray:
    """w[n, k] = value(q[n, k]) * scale[n // block, k // block] for one [N, K] matrix.

    ``q_codes`` are e4m3fn bytes (uint8 array or a torch float8 / uint8 tensor).
    """
    if hasattr(q_codes, "detach"):
        import torch
        t = q_codes.detach().cpu()
        if t.dtype != torch.uint8:
            t = t.view(torch.uint8)
        q_codes = t.numpy()
    V = e4m3_value(np.arange(256))[np.asarray(q_codes, dtype=np.uint8)]  # value of each code
    S = _mo._f64(scale)
    N, K = V.shape
    if S.shape != ((N + block - 1) // block, (K + block - 1) // block):
        raise ValueError(f"scale shape {S.shape} does not tile [{N}, {K}] by {block}")
    return V * np.repeat(np.repeat(S, block, axis=0)[:N], block, axis=1)[:, :K]


# ---------------------------------------------------------------- one expert, the layer
def expert_mlp_fp8(xd, w13_q, w13_s, w2_q, w2_s) -> np.ndarray:
    """One fp8 expert on already-dequantized input rows ``xd [n, H]``.

    z = xd @ W13^T with W13 the dequantized [2I, H] block weights; act = silu(gate) * up;
    act is quantized per token group of 128 (fp32 decisions) and dequantized; the output
    is that act times the dequantized W2^T.
    """
    W13 = dequant_block(w13_q, w13_s)
    W2 = dequant_block(w2_q, w2_s)
    z = np.atleast_2d(xd) @ W13.T
    I = W13.shape[0] // 2
    act = _mo.silu(z[:, :I]) * z[:, I:]
    return quant_dequant(act) @ W2.T


def experts_combine_fp8(x, topk_weights, topk_ids, w13_q, w13_s, w2_q, w2_s,
                        shared_w13_q=None, shared_w13_s=None, shared_w2_q=None,
                        shared_w2_s=None, *, return_parts=False, top_k=None):
    """y [T, H] fp64 of the fp8 experts and the combine for a routing given as input (the
    precomputed top-k of ``FusedMoE.forward(hidden_states, topk_output)``): x is quantized
    once per token and group of 128 and feeds the routed and the shared experts."""
    X = _mo._f64(x)
    T, H = X.shape
    W = np.atleast_2d(np.asarray(topk_weights, dtype=np.float64))
    ids = np.atleast_2d(np.asarray(topk_ids, dtype=np.int64))
    k = ids.shape[1] if top_k is None else top_k
    xd = quant_dequant(X) if T else np.zeros((0, H))
    o = np.zeros((T, k, H), dtype=np.float64)
    for e in sorted(set(ids.reshape(-1).tolist())):
        rows = [(t, j) for t in range(T) for j in range(k) if ids[t, j] == e]
        out = expert_mlp_fp8(xd[[t for t, _ in rows]], w13_q[e], w13_s[e], w2_q[e], w2_s[e])
        for (t, j), r in zip(rows, out):
            o[t, j] = r
    y = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            y[t] += W[t, j] * o[t, j]
    shared = None
    if shared_w13_q is not None:
        shared = (expert_mlp_fp8(xd, shared_w13_q, shared_w13_s, shared_w2_q, shared_w2_s)
                  if T else np.zeros((0, H)))
        y = y + shared
    if return_parts:
        return y, {"topk_weights": W, "topk_ids": ids, "expert_out": o, "shared": shared,
                   "x_dequant": xd}
    return y


def fused_moe_fp8(x, logits, bias, w13_q, w13_s, w2_q, w2_s, shared_w13_q=None,
                  shared_w13_s=None, shared_w2_q=None, shared_w2_s=None, *,
                  return_parts=False, **cfg):
    """y [T, H] fp64 of the fp8 layer: routing as the bf16 layer, then
    ``experts_combine_fp8``."""
    W, ids = _mo.select_experts(logits, bias, **cfg)
    return experts_combine_fp8(x, W, ids, w13_q, w13_s, w2_q, w2_s, shared_w13_q,
                               shared_w13_s, shared_w2_q, shared_w2_s,
                               return_parts=return_parts, top_k=cfg["top_k"])

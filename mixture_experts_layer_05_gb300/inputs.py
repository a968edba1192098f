"""Seeded synthetic inputs for the FusedMoE layer forward.

This module serves both the CUDA path and the oracle. It draws random numbers and
shapes them (seeds, normal draws, an order-preserving spread of each logit row, Zipf
popularity offsets, redraws of rows a caller rejects); it holds none of the layer's
arithmetic (no scoring, no top-k, no expert math). Rows whose routing decision is too
close to call are rejected by a caller-supplied ``margin_fn`` (the tests pass the
oracle's), so this module never needs to know how routing works.

Layouts follow the FusedMoE weight layout on the vLLM ``fused_moe/layer`` page
(``FusedMoE._load_w13`` / ``_load_w2``): ``w13 [E, 2I, H]`` with the gate (w1) rows
first and the up (w3) rows second, ``w2 [E, H, I]``; router logits ``[T, E]`` fp32 and
``e_score_correction_bias [E]`` fp32 as in ``MoEGate`` on the sglang
``models/deepseek_v2.py`` page.
"""
from __future__ import annotations

import zlib

import torch

from .configs import MoEWorkload

LOGIT_GAP = 1e-3


def tensor_seed(workload: str, tensor: str, seed: int = 0) -> int:
    """Stable per-tensor seed: crc32 of "workload/tensor" xor the run seed."""
    return (zlib.crc32(f"{workload}/{tensor}".encode()) ^ int(seed)) & 0x7FFFFFFF


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, dtype=torch.float32, device="cpu",
           clamp: float | None = None) -> torch.Tensor:
    """N(0, std) draws in fp32 (clamped to +-clamp if given), rounded once to ``dtype``;
    drawn in slices of the first dim."""
    device = torch.device(device)
    out = torch.empty(shape, dtype=dtype, device=device)
    g = _gen(seed, device)
    if len(shape) == 0 or shape[0] == 0:
        return out
    per = 1
    for s in shape[1:]:
        per *= s
    rows = max(1, (1 << 26) // max(per, 1))          # <= 256 MB of fp32 per slice
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        tmp = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device,
                          dtype=torch.float32)
        if std != 1.0:
            tmp.mul_(std)
        if clamp is not None:
            tmp.clamp_(-clamp, clamp)
        out[r0:r1].copy_(tmp)
    return out


def make_weights(w: MoEWorkload, seed: int = 0, device="cpu") -> dict:
    """Expert weights (bf16), correction bias (fp32) and shared-expert weights."""
    E, H, I = w.num_experts, w.hidden_size, w.intermediate_size
    out = {
        "w13": normal((E, 2 * I, H), w.w_std, tensor_seed(w.name, "w13", seed),
                      torch.bfloat16, device),
        "w2": normal((E, H, I), w.w_std, tensor_seed(w.name, "w2", seed),
                     torch.bfloat16, device),
        "bias": None, "shared_w13": None, "shared_w2": None,
    }
    if w.has_bias:
        out["bias"] = normal((E,), w.bias_std, tensor_seed(w.name, "bias", seed),
                             torch.float32, device)
    Is = w.shared_intermediate_size
    if Is:
        out["shared_w13"] = normal((2 * Is, H), w.w_std,
                                   tensor_seed(w.name, "shared_w13", seed),
                                   torch.bfloat16, device)
        out["shared_w2"] = normal((H, Is), w.w_std, tensor_seed(w.name, "shared_w2", seed),
                                  torch.bfloat16, device)
    return out


def make_expert_extras(w: MoEWorkload, seed: int = 0, gated: bool = True, bias_std: float = 0.1,
                       device="cpu") -> dict:
    """Per-expert biases (bf16 ~N(0, bias_std)) and, when not gated, a w1-only weight
    stack ``w1 [E, I, H]`` (bf16 ~N(0, w_std)) for the layer's optional variants."""
    E, H, I = w.num_experts, w.hidden_size, w.intermediate_size
    out = {
        "w13_bias": normal((E, (2 if gated else 1) * I), bias_std,
                           tensor_seed(w.name, "w13_bias", seed), torch.bfloat16, device),
        "w2_bias": normal((E, H), bias_std, tensor_seed(w.name, "w2_bias", seed),
                          torch.bfloat16, device),
    }
    if not gated:
        out["w1"] = normal((E, I, H), w.w_std, tensor_seed(w.name, "w1", seed), torch.bfloat16,
                           device)
    return out


def spread_rows(logits: torch.Tensor, gap: float = LOGIT_GAP) -> torch.Tensor:
    """Move values apart, order preserved, so that within each row any two differ by >= gap.

    Sort each row, then raise each value to at least its predecessor + gap (a running
    maximum of v_i - i*gap, plus i*gap), and put the values back in place.
    """
    if logits.numel() == 0:
        return logits
    v, order = torch.sort(logits.double(), dim=-1, stable=True)
    ramp = torch.arange(v.shape[-1], dtype=torch.float64) * gap
    v = torch.cummax(v - ramp, dim=-1).values + ramp
    out = torch.empty_like(v)
    out.scatter_(-1, order, v)
    return out.to(logits.dtype)


def zipf_offsets(w: MoEWorkload, seed: int = 0) -> torch.Tensor:
    """Per-expert logit offsets beta * log(rank^-s) over a seeded rank permutation."""
    E = w.num_experts
    if w.zipf_s <= 0:
        return torch.zeros(E, dtype=torch.float32)
    g = _gen(tensor_seed(w.name, "zipf_rank", seed), "cpu")
    rank = torch.randperm(E, generator=g) + 1                    # rank of expert e
    off = -w.zipf_s * w.zipf_beta * torch.log(rank.double())
    return off.float()


def _draw_logits(w: MoEWorkload, n: int, tag: str, seed: int) -> torch.Tensor:
    lg = normal((n, w.num_experts), w.logit_std, tensor_seed(w.name, tag, seed))
    if w.zipf_s > 0:
        lg += zipf_offsets(w, seed)
    return spread_rows(lg)


def make_tokens(w: MoEWorkload, T: int, seed: int = 0, margin_fn=None,
                min_margin: float = LOGIT_GAP, max_redraws: int = 64):
    """Hidden states ``x [T, H]`` bf16 and router logits ``[T, E]`` fp32 (on the CPU).

    Logit rows are spread so that any two entries differ by >= ``LOGIT_GAP``. If
    ``margin_fn(logits) -> [T] margins`` is given, rows whose margin is below
    ``min_margin`` are redrawn (deterministically, from derived seeds).
    """
    x = normal((T, w.hidden_size), w.x_std, tensor_seed(w.name, f"x/T{T}", seed),
               torch.bfloat16)
    logits = _draw_logits(w, T, f"logits/T{T}", seed)
    if margin_fn is not None and T > 0:
        rows = torch.arange(T)
        for r in range(max_redraws):
            bad = rows[torch.as_tensor(margin_fn(logits[rows])) < min_margin]
            if bad.numel() == 0:
                break
            logits[bad] = _draw_logits(w, int(bad.numel()), f"logits/T{T}/redraw{r}", seed)
            rows = bad
        else:
            raise RuntimeError("could not draw router logits with the requested margin")
    return x, logits


FP8_BLOCK = 128


def fp8_codes(shape, seed: int, code_std: float = 112.0, device="cpu") -> torch.Tensor:
    """Random e4m3fn numbers (torch.float8_e4m3fn): N(0, code_std) draws, clamped to the
    format's finite range +-448 and converted to the nearest fp8 value."""
    return normal(shape, code_std, seed, torch.float8_e4m3fn, device, clamp=448.0)


def make_fp8_weights(w: MoEWorkload, seed: int = 0, device="cpu") -> dict:
    """FP8 block-128 expert weights as a checkpoint stores them: e4m3fn codes
    ``w13_q [E, 2I, H]``, ``w2_q [E, H, I]`` and one fp32 scale per 128 x 128 block
    (``w13_s [E, 2I/128, H/128]``, ``w2_s [E, H/128, I/128]``), plus the shared expert's.

    Codes ~ N(0, 112) and scales ~ U(0.8, 1.2) * w_std * 4 / 448, so the weights the
    codes stand for are about N(0, w_std) like the bf16 workloads'. The bias is the bf16
    workload's (fp32).
    """
    E, H, I = w.num_experts, w.hidden_size, w.intermediate_size
    B = FP8_BLOCK
    base = w.w_std * 4.0 / 448.0

    def scales(shape, tag):
        g = _gen(tensor_seed(w.name, tag, seed), "cpu")
        s = (0.8 + 0.4 * torch.rand(shape, generator=g, dtype=torch.float32)) * base
        return s.to(device)

    out = {
        "w13_q": fp8_codes((E, 2 * I, H), tensor_seed(w.name, "fp8/w13", seed), device=device),
        "w13_s": scales((E, 2 * I // B, H // B), "fp8/w13_s"),
        "w2_q": fp8_codes((E, H, I), tensor_seed(w.name, "fp8/w2", seed), device=device),
        "w2_s": scales((E, H // B, I // B), "fp8/w2_s"),
        "bias": None, "shared_w13_q": None, "shared_w13_s": None, "shared_w2_q": None,
        "shared_w2_s": None,
    }
    if w.has_bias:
        out["bias"] = normal((E,), w.bias_std, tensor_seed(w.name, "bias", seed),
                             torch.float32, device)
    Is = w.shared_intermediate_size
    if Is:
        out["shared_w13_q"] = fp8_codes((2 * Is, H), tensor_seed(w.name, "fp8/shared_w13", seed),
                                        device=device)
        out["shared_w13_s"] = scales((2 * Is // B, H // B), "fp8/shared_w13_s")
        out["shared_w2_q"] = fp8_codes((H, Is), tensor_seed(w.name, "fp8/shared_w2", seed),
                                       device=device)
        out["shared_w2_s"] = scales((H // B, Is // B), "fp8/shared_w2_s")
    return out


def fp4_packed(shape, seed: int, device="cpu") -> torch.Tensor:
    """Random packed e2m1 pairs: uniform bytes (every 4-bit code equally likely) of
    ``shape`` (the last dim is half the value count), drawn on ``device``."""
    g = _gen(seed, torch.device(device))
    return torch.randint(0, 256, shape, generator=g, dtype=torch.uint8, device=device)


def fp4_block_scales(shape, seed: int, device="cpu") -> torch.Tensor:
    """Random e4m3fn block scales (torch.float8_e4m3fn): byte codes uniform in [0x30, 0x40),
    the e4m3 values 0.5 .. 1.875, drawn on ``device``."""
    g = _gen(seed, torch.device(device))
    return torch.randint(0x30, 0x40, shape, generator=g, dtype=torch.uint8,
                         device=device).view(torch.float8_e4m3fn)


def make_fp4_weights(w: MoEWorkload, seed: int = 0, device="cpu") -> dict:
    """NVFP4 expert weights as a checkpoint stores them: packed e2m1 codes ``w13 [E, 2I, H/2]``,
    ``w2 [E, H, I/2]`` (uint8, low nibble first), e4m3 block scales per 16 values along K
    (``w13_sf [E, 2I, H/16]``, ``w2_sf [E, H, I/16]``) and per-expert fp32 scales
    ``w13_s2 [E]``, ``w2_s2 [E]``; the shared expert's the same way (``shared_s2 [2]``).

    Uniform codes have an rms of 2.93 and the block scales of about 1.1, so the per-expert
    scales, U(0.8, 1.2) * w_std / 3.2, make the weights the codes stand for about w_std in
    rms like the bf16 workloads'. The per-tensor scales of the input and the act are the
    usual calibration form 448 * 6 / (expected amax): input amax 4 x_std, act amax
    8 rms(z)^2 with rms(z) = sqrt(H) x_std w_std; the shared expert's are 0.75 and 1.25
    times those. The bias is the bf16 workload's, rounded to bf16 as the FP4 layer of the
    pages casts it.
    """
    E, H, I = w.num_experts, w.hidden_size, w.intermediate_size
    base = w.w_std / 3.2

    def s2(shape, tag):
        g = _gen(tensor_seed(w.name, tag, seed), "cpu")
        return ((0.8 + 0.4 * torch.rand(shape, generator=g, dtype=torch.float32)) * base).to(device)

    rms_z = (H ** 0.5) * w.x_std * w.w_std
    g_in = 448.0 * 6.0 / (4.0 * w.x_std)
    g_act = 448.0 * 6.0 / (8.0 * rms_z * rms_z)
    out = {
        "w13": fp4_packed((E, 2 * I, H // 2), tensor_seed(w.name, "fp4/w13", seed), device),
        "w13_sf": fp4_block_scales((E, 2 * I, H // 16), tensor_seed(w.name, "fp4/w13_sf", seed),
                                   device),
        "w13_s2": s2((E,), "fp4/w13_s2"),
        "w2": fp4_packed((E, H, I // 2), tensor_seed(w.name, "fp4/w2", seed), device),
        "w2_sf": fp4_block_scales((E, H, I // 16), tensor_seed(w.name, "fp4/w2_sf", seed),
                                  device),
        "w2_s2": s2((E,), "fp4/w2_s2"),
        "input_scale": float(torch.tensor(g_in, dtype=torch.float32)),
        "act_scale": float(torch.tensor(g_act, dtype=torch.float32)),
        "bias": None, "shared_w13": None, "shared_w13_sf": None, "shared_w2": None,
        "shared_w2_sf": None, "shared_s2": None, "shared_input_scale": 0.0,
        "shared_act_scale": 0.0,
    }
    if w.has_bias:
        out["bias"] = normal((E,), w.bias_std, tensor_seed(w.name, "bias", seed),
                             torch.bfloat16, device).float()
    Is = w.shared_intermediate_size
    if Is:
        out["shared_w13"] = fp4_packed((2 * Is, H // 2), tensor_seed(w.name, "fp4/sw13", seed),
                                       device)
        out["shared_w13_sf"] = fp4_block_scales((2 * Is, H // 16),
                                                tensor_seed(w.name, "fp4/sw13_sf", seed), device)
        out["shared_w2"] = fp4_packed((H, Is // 2), tensor_seed(w.name, "fp4/sw2", seed), device)
        out["shared_w2_sf"] = fp4_block_scales((H, Is // 16),
                                               tensor_seed(w.name, "fp4/sw2_sf", seed), device)
        out["shared_s2"] = s2((2,), "fp4/shared_s2")
        out["shared_input_scale"] = float(torch.tensor(0.75 * g_in, dtype=torch.float32))
        out["shared_act_scale"] = float(torch.tensor(1.25 * g_act, dtype=torch.float32))
    return out

"""Parity of the NVFP4 (w4a4, 16-value blocks) CUDA path with the CPU oracle, on the GPU.

The FlashInferFP4MoE layer of the sglang ``fused_moe_triton/layer.py`` page. The input
quantization (``fp4_quantize``) is bit-exact against the oracle: every step is one fp32
operation on the same bf16 inputs. The weight preparation is a byte permutation, checked
byte for byte. The act is quantized from the kernel's fp32 sums, the oracle's from fp64, so
a block scale or a code can land on the other side of a rounding midpoint: the test takes
the GPU's quantized act from the workspace and requires it to equal the oracle's
quantization except at decisions within ACT_REL of a midpoint, then requires the output to
equal the oracle's second GEMM and combine of that act within the layer's bound. Routing
must match bit for bit.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import fp4_oracle as f4
from mixture_experts_layer_05_gb300 import binding, configs, inputs
from tests.moe_cases import check_close, oracle_cfg, tokens

pytestmark = pytest.mark.gpu

DEV = "cuda"
# relative error allowed on the kernel's fp32 act (fp32 sums of exact products over K
# values, the split-K sum, the SiLU): decisions nearer a midpoint than this may go either way
ACT_REL = 1e-4


# ------------------------------------------------------------------ the input quant
@pytest.mark.parametrize("R,H,g", [(1, 64, 1.0), (37, 384, 448.0 * 6 / 4), (300, 7168, 672.0),
                                   (5, 128, 1e-30), (9, 256, 1e30)])
def test_quant_nvfp4_bitexact(cuda_lib, R, H, g):
    gen = torch.Generator().manual_seed(R * 7 + H)
    x = torch.randn(R, H, generator=gen) * torch.exp2(torch.randint(-20, 21, (R, 1), generator=gen))
    x[0, :16] = 0.0                                             # an all-zero block
    if R > 2:
        x[1, 5] = 3.0e4                                         # one outlier in a block
        x[2] = torch.linspace(-1.0, 1.0, H) * 1e-30             # tiny magnitudes
    x = x.to(torch.bfloat16)
    q, sf = binding.moe_quant_nvfp4(x.to(DEV), g)
    torch.cuda.synchronize()
    q_ref, sf_ref = f4.quantize(x.float().numpy(), g)
    np.testing.assert_array_equal(oracle.e4m3_value(sf.view(torch.uint8).cpu().numpy()), sf_ref)
    vals = f4.e2m1_value(f4.unpack_fp4(q.cpu().numpy()))
    np.testing.assert_array_equal(vals, q_ref)   # values: -0 and +0 are both zero


def test_quant_nvfp4_rejects_bad_arguments(cuda_lib):
    x = torch.zeros(2, 40, dtype=torch.bfloat16, device=DEV)
    q = torch.empty(2, 20, dtype=torch.uint8, device=DEV)
    sf = torch.empty(2, 3, dtype=torch.uint8, device=DEV)
    lib = binding.load()
    assert lib.moe_quant_nvfp4(2, 40, x.data_ptr(), 1.0, q.data_ptr(), sf.data_ptr(), None) == \
        binding.ERR_INVALID_ARG                                  # H not a multiple of 16
    x = torch.zeros(2, 32, dtype=torch.bfloat16, device=DEV)
    for g in (0.0, -1.0, float("inf"), float("nan")):
        assert lib.moe_quant_nvfp4(2, 32, x.data_ptr(), g, q.data_ptr(), sf.data_ptr(), None) \
            == binding.ERR_INVALID_ARG


# ------------------------------------------------------------------ the weight layout
def _prepared_ref(packed: np.ndarray, scales: np.ndarray) -> np.ndarray:
    rows, kh = packed.shape
    K = 2 * kh
    out = np.zeros((rows // 128, K // 64, 4608), dtype=np.uint8)
    for t in range(rows // 128):
        for kb in range(K // 64):
            for h in range(2):
                for r in range(128):
                    out[t, kb, h * 2048 + r * 16: h * 2048 + r * 16 + 16] = \
                        packed[t * 128 + r, kb * 32 + h * 16: kb * 32 + h * 16 + 16]
            for r in range(128):
                out[t, kb, 4096 + r * 4: 4096 + r * 4 + 4] = scales[t * 128 + r, kb * 4: kb * 4 + 4]
    return out.reshape(-1)


@pytest.mark.parametrize("rows,K", [(128, 64), (256, 192)])
def test_prepare_weight_layout(cuda_lib, rows, K):
    packed = inputs.fp4_packed((rows, K // 2), 11, DEV)
    scales = inputs.fp4_block_scales((rows, K // 16), 12, DEV)
    out = binding.moe_nvfp4_prepare_weight(packed, scales)
    torch.cuda.synchronize()
    assert out.numel() == rows * K * 9 // 16 == binding.moe_nvfp4_prepared_bytes(rows, K)
    ref = _prepared_ref(packed.cpu().numpy(), scales.view(torch.uint8).cpu().numpy())
    np.testing.assert_array_equal(out.cpu().numpy(), ref)


def test_prepare_weight_rejects_bad_shapes(cuda_lib):
    assert binding.moe_nvfp4_prepared_bytes(100, 64) == 0
    assert binding.moe_nvfp4_prepared_bytes(128, 48) == 0
    lib = binding.load()
    b = torch.zeros(4096, dtype=torch.uint8, device=DEV)
    assert lib.moe_nvfp4_prepare_weight(128, 40, b.data_ptr(), b.data_ptr(), b.data_ptr(),
                                        None) == binding.ERR_INVALID_ARG


# ------------------------------------------------------------------ the layer
def _prep(packed, sf):
    """[..., N, K/2] codes and [..., N, K/16] scales -> the prepared stack."""
    return binding.moe_nvfp4_prepare_weight(packed.reshape(-1, packed.shape[-1]).contiguous(),
                                            sf.reshape(-1, sf.shape[-1]).contiguous())


def _fp4_layer(w, wts, T):
    cfg = binding.config_from_workload(w, weight_quant="nvfp4")
    d = wts
    kw = dict(w13_weight_scale_2=d["w13_s2"].to(DEV), w2_weight_scale_2=d["w2_s2"].to(DEV),
              input_scale=d["input_scale"], act_scale=d["act_scale"])
    sw13 = sw2 = None
    if w.shared_intermediate_size:
        sw13 = _prep(d["shared_w13"].to(DEV), d["shared_w13_sf"].to(DEV))
        sw2 = _prep(d["shared_w2"].to(DEV), d["shared_w2_sf"].to(DEV))
        kw.update(shared_weight_scale_2=d["shared_s2"].to(DEV),
                  shared_input_scale=d["shared_input_scale"],
                  shared_act_scale=d["shared_act_scale"])
    bias = None if d["bias"] is None else d["bias"].to(DEV)
    layer = binding.FusedMoE(cfg, _prep(d["w13"].to(DEV), d["w13_sf"].to(DEV)),
                             _prep(d["w2"].to(DEV), d["w2_sf"].to(DEV)), bias, sw13, sw2,
                             max_tokens=max(T, 1), **kw)
    return layer


def _oracle_w(wts):
    return {"w13": wts["w13"], "w13_sf": wts["w13_sf"], "w13_s2": wts["w13_s2"].cpu().numpy(),
            "w2": wts["w2"], "w2_sf": wts["w2_sf"], "w2_s2": wts["w2_s2"].cpu().numpy(),
            "input_scale": wts["input_scale"], "act_scale": wts["act_scale"]}


def _act_decisions_ok(act_ref: np.ndarray, gpu_vals: np.ndarray, g: float, what: str) -> int:
    """GPU act rows (f16 values q * sf) against the oracle's quantization of act_ref (fp64):
    equal, except blocks holding a decision (the block scale's e4m3 rounding, or a value's
    e2m1 rounding) within ACT_REL of its midpoint, whose GPU values must then be a valid
    quantization of act_ref moved by at most ACT_REL. Returns the number of such blocks."""
    q, sf = f4.quantize(act_ref, g)
    ref = q * np.repeat(sf, 16, axis=1)
    bad = ref != gpu_vals
    if not bad.any():
        return 0
    R, C = act_ref.shape
    blocks = np.argwhere(bad.reshape(R, C // 16, 16).any(axis=2))
    for r, b in blocks:
        a = act_ref[r, 16 * b:16 * b + 16]
        amax = np.abs(a).max()
        lo, hi = a - ACT_REL * amax, a + ACT_REL * amax
        # the GPU's block must be the quantization of some act within the band: try the
        # scale decision both ways and each value's rounding both ways
        ok = False
        for amx in (amax * (1 - ACT_REL), amax, amax * (1 + ACT_REL)):
            # the block scale an act with this amax gets, then the codes of the band
            _, sfa = f4.quantize(np.array([[amx] + [0.0] * 15]), g)
            s = float(sfa[0, 0])
            gv = gpu_vals[r, 16 * b:16 * b + 16]
            if s == 0:
                ok = ok or not gv.any()
                continue
            rr = float(np.float32(g) / np.float32(s))
            ql, qh = f4.e2m1_round(lo * rr), f4.e2m1_round(hi * rr)
            qg = gv / s
            on_grid = np.isin(np.abs(qg), f4.E2M1_MAGNITUDES).all()
            ok = ok or (on_grid and bool(np.all((qg >= ql) & (qg <= qh))))
        assert ok, (f"{what}: act row {r} block {b} differs from the oracle away from any "
                    f"rounding midpoint: gpu {gpu_vals[r, 16 * b:16 * b + 16]} ref "
                    f"{ref[r, 16 * b:16 * b + 16]}")
    assert len(blocks) <= max(2, bad.size // 1000), f"{what}: {len(blocks)} blocks differ"
    return len(blocks)


def _check_layer(w, wts, layer, x, logits, y, T):
    """Routing bit-exact, act decisions, and y against the oracle's down GEMM + combine of
    the GPU's act."""
    k, I, Is = w.top_k, w.intermediate_size, w.shared_intermediate_size
    ow = _oracle_w(wts)
    W, ids = oracle.select_experts(logits, wts["bias"], **oracle_cfg(w))
    lay = binding.moe_forward_workspace_layout(layer.cfg, T)
    ws = layer.workspace
    gid = ws[lay.topk_ids:lay.topk_ids + T * k * 4].view(torch.int32).cpu().numpy().reshape(T, k)
    assert np.array_equal(gid, ids), "routing differs"
    npp = int(ws[lay.num_tokens_post_padded:lay.num_tokens_post_padded + 4].view(torch.int32))
    srt = ws[lay.sorted_token_ids:lay.sorted_token_ids + npp * 4].view(torch.int32).cpu().numpy()
    act = ws[lay.act:lay.act + npp * I * 2].view(torch.float16).view(npp, I).double().cpu().numpy()
    xq = f4.quant_dequant(x.float().numpy(), wts["input_scale"])
    g2 = wts["act_scale"]
    o = np.zeros((T, k, w.hidden_size))
    flips = 0
    for e in sorted(set(ids.reshape(-1).tolist())):
        slots = [(t, j) for t in range(T) for j in range(k) if ids[t, j] == e]
        rows = [int(np.nonzero(srt == t * k + j)[0][0]) for t, j in slots]
        a_ref = f4.expert_act_fp4(xq[[t for t, _ in slots]], wts["w13"][e], wts["w13_sf"][e],
                                  float(ow["w13_s2"][e]))
        flips += _act_decisions_ok(a_ref, act[rows], g2, f"expert {e}")
        out = f4.expert_down_fp4(act[rows] / np.float64(np.float32(g2)), wts["w2"][e],
                                 wts["w2_sf"][e], float(ow["w2_s2"][e]))
        for (t, j), v in zip(slots, out):
            o[t, j] = v
    y_ref = np.einsum("tj,tjh->th", W, o)
    if Is:
        act_s = ws[lay.act_shared:lay.act_shared + T * Is * 2].view(torch.float16).view(T, Is)
        act_s = act_s.double().cpu().numpy()
        xs = f4.quant_dequant(x.float().numpy(), wts["shared_input_scale"])
        s2 = wts["shared_s2"].cpu().numpy()
        a_ref = f4.expert_act_fp4(xs, wts["shared_w13"], wts["shared_w13_sf"], float(s2[0]))
        flips += _act_decisions_ok(a_ref, act_s, wts["shared_act_scale"], "shared")
        y_ref = y_ref + f4.expert_down_fp4(
            act_s / np.float64(np.float32(wts["shared_act_scale"])), wts["shared_w2"],
            wts["shared_w2_sf"], float(s2[1]))
    check_close(y, y_ref, f"nvfp4 {w.name} T={T}")
    return flips


def _shrink(w, **kw):
    return configs.shrink(w, **kw)


SMALL = {
    "mixtral": _shrink(configs.MIXTRAL, hidden_size=512, intermediate_size=384),
    "dsv2": _shrink(configs.DSV2, hidden_size=512, intermediate_size=128,
                    shared_intermediate_size=256),
    "dsv3": _shrink(configs.DSV3, hidden_size=512, intermediate_size=256,
                    shared_intermediate_size=256),
    "tiny": configs.TINY,
}


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("T", [1, 16, 203, 600])
def test_fp4_forward_small(cuda_lib, name, T):
    w = SMALL[name]
    wts = inputs.make_fp4_weights(w, 0)
    x, logits = tokens(w, T, wts["bias"])
    layer = _fp4_layer(w, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    _check_layer(w, wts, layer, x, logits, y, T)


def test_fp4_forward_matches_whole_oracle(cuda_lib):
    """Where no act decision sits near a midpoint, the layer equals the oracle's whole NVFP4
    layer (fused_moe_fp4) within the bound."""
    w = SMALL["dsv3"]
    wts = inputs.make_fp4_weights(w, 0)
    x, logits = tokens(w, 16, wts["bias"])
    layer = _fp4_layer(w, wts, 16)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    if _check_layer(w, wts, layer, x, logits, y, 16) == 0:
        ow = _oracle_w(wts)
        ow.update(shared_w13=wts["shared_w13"], shared_w13_sf=wts["shared_w13_sf"],
                  shared_w13_s2=float(wts["shared_s2"][0]), shared_w2=wts["shared_w2"],
                  shared_w2_sf=wts["shared_w2_sf"], shared_w2_s2=float(wts["shared_s2"][1]),
                  shared_input_scale=wts["shared_input_scale"],
                  shared_act_scale=wts["shared_act_scale"])
        y_ref = f4.fused_moe_fp4(x.float().numpy(), logits, wts["bias"], ow, **oracle_cfg(w))
        check_close(y, y_ref, "nvfp4 whole layer")


def test_fp4_graph_replay(cuda_lib):
    """The NVFP4 forward captured once in a CUDA graph and replayed on new tokens."""
    w = SMALL["dsv3"]
    T = 5
    wts = inputs.make_fp4_weights(w, 0)
    layer = _fp4_layer(w, wts, T)
    xd = torch.zeros(T, w.hidden_size, dtype=torch.bfloat16, device=DEV)
    ld = torch.zeros(T, w.num_experts, dtype=torch.float32, device=DEV)
    yd = torch.empty_like(xd)
    layer(xd, ld, out=yd)                                    # warm-up outside the capture
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        layer(xd, ld, out=yd)
    for seed in (1, 2):
        x, logits = tokens(w, T, wts["bias"], seed=seed)
        xd.copy_(x.to(DEV))
        ld.copy_(logits.to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        _check_layer(w, wts, layer, x, logits, yd.clone(), T)


def test_fp4_forward_rejects_bad_arguments(cuda_lib):
    w = SMALL["mixtral"]
    wts = inputs.make_fp4_weights(w, 0)
    layer = _fp4_layer(w, wts, 4)
    x = torch.zeros(4, w.hidden_size, dtype=torch.bfloat16, device=DEV)
    lg = torch.zeros(4, w.num_experts, dtype=torch.float32, device=DEV)
    bad = dict(layer.scales)
    bad["act_scale"] = 0.0
    with pytest.raises(binding.GbmoeError):
        binding.moe_forward_ex(layer.cfg, x, lg, None, layer.w13, layer.w2, None, None,
                               torch.empty_like(x), layer.workspace, **bad)
    bad = dict(layer.scales)
    bad["w2_weight_scale_2"] = None
    with pytest.raises((binding.GbmoeError, ValueError)):
        binding.moe_forward_ex(layer.cfg, x, lg, None, layer.w13, layer.w2, None, None,
                               torch.empty_like(x), layer.workspace, **bad)


# ------------------------------------------------------------------ full sizes
FULL = [("dsv3", 1), ("dsv3", 8), ("mixtral", 1), ("dsv2", 3)]


@pytest.mark.parametrize("name,T", FULL, ids=[f"{n}-{t}" for n, t in FULL])
def test_fp4_forward_full_size(cuda_lib, name, T):
    w = configs.WORKLOADS[name]
    wts = inputs.make_fp4_weights(w, 0, device=DEV)
    x, logits = tokens(w, T, None if wts["bias"] is None else wts["bias"].cpu())
    layer = _fp4_layer(w, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    wts = dict(wts)
    if wts["bias"] is not None:
        wts["bias"] = wts["bias"].cpu()
    _check_layer(w, wts, layer, x, logits, y, T)

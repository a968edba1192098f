"""The C ABI on the host: every declared symbol is exported, argument validation
returns the documented status before anything touches a GPU, workspace sizing.

No compute call runs here (these tests need no GPU)."""
import ctypes
import os
import re
import subprocess

import pytest

from mixture_experts_layer_05_gb300 import binding, configs
from mixture_experts_layer_05_gb300 import build as build_mod

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "gbmoe.h")


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return binding.load()


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\w[\w ]*?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_declarations_match_binding():
    assert sorted(binding.EXPORTS) == _declared()


def test_every_declared_symbol_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    for name in _declared():
        assert name in exported, name
        assert hasattr(lib, name)


def _cfg(**kw):
    d = dict(num_experts=8, top_k=2, hidden_size=128, intermediate_size=256)
    d.update(kw)
    return binding.make_config(**d)


def _topk(lib, cfg, T=4, logits=1, w=1, ids=1):
    P = ctypes.c_void_p
    return lib.moe_topk(ctypes.byref(cfg), T, P(logits), None, P(w), P(ids), None)


def test_topk_validation(lib):
    ok = _cfg()
    # T = 0 is a no-op, before any pointer is looked at
    assert lib.moe_topk(ctypes.byref(ok), 0, None, None, None, None, None) == binding.OK
    assert lib.moe_topk(None, 4, None, None, None, None, None) == binding.ERR_INVALID_ARG
    assert lib.moe_topk(ctypes.byref(ok), 4, None, None, None, None, None) == binding.ERR_INVALID_ARG
    assert _topk(lib, ok, T=-1) == binding.ERR_INVALID_ARG
    # sigmoid scoring needs grouped routing (FusedMoE constructor)
    assert _topk(lib, _cfg(scoring_func="sigmoid")) == binding.ERR_UNSUPPORTED
    # grouped routing needs both group arguments
    assert _topk(lib, _cfg(use_grouped_topk=True, num_expert_group=4)) == binding.ERR_INVALID_ARG
    assert _topk(lib, _cfg(use_grouped_topk=True, topk_group=2)) == binding.ERR_INVALID_ARG
    assert _topk(lib, _cfg(use_grouped_topk=True, num_expert_group=3, topk_group=1)) == \
        binding.ERR_INVALID_ARG                                   # E % G != 0
    assert _topk(lib, _cfg(use_grouped_topk=True, num_expert_group=4, topk_group=5)) == \
        binding.ERR_INVALID_ARG                                   # g > G
    assert _topk(lib, _cfg(top_k=3, use_grouped_topk=True, num_expert_group=8, topk_group=2)) == \
        binding.ERR_INVALID_ARG                                   # k > g * E/G
    assert _topk(lib, _cfg(top_k=9)) == binding.ERR_INVALID_ARG   # k > E
    assert _topk(lib, _cfg(top_k=0)) == binding.ERR_INVALID_ARG
    assert _topk(lib, _cfg(num_experts=2000, top_k=2)) == binding.ERR_INVALID_ARG
    assert _topk(lib, _cfg(routed_scaling_factor=float("nan"))) == binding.ERR_INVALID_ARG


def _fwd(lib, cfg, T=4, ws_bytes=1 << 40, ptr=256, shared=False, events=None, nev=0):
    P = ctypes.c_void_p
    sw = P(ptr) if shared else None
    return lib.moe_forward_events(ctypes.byref(cfg), T, P(ptr), P(ptr), None, P(ptr), P(ptr), sw,
                                  sw, P(ptr), P(ptr), ws_bytes, events, nev, None)


def test_forward_validation(lib):
    ok = _cfg()
    assert _fwd(lib, _cfg(activation=1)) == binding.ERR_UNSUPPORTED     # only silu
    assert _fwd(lib, _cfg(is_act_and_mul=2)) == binding.ERR_INVALID_ARG
    # the clamp, alpha and a shared expert need the gated form
    assert _fwd(lib, _cfg(is_act_and_mul=0, swiglu_limit=7.0)) == binding.ERR_UNSUPPORTED
    assert _fwd(lib, _cfg(is_act_and_mul=0, gemm1_alpha=1.7)) == binding.ERR_UNSUPPORTED
    assert _fwd(lib, _cfg(is_act_and_mul=0, shared_intermediate_size=128),
                shared=True) == binding.ERR_UNSUPPORTED
    assert _fwd(lib, _cfg(swiglu_limit=-1.0)) == binding.ERR_INVALID_ARG
    assert _fwd(lib, _cfg(gemm1_alpha=float("nan"))) == binding.ERR_INVALID_ARG
    assert _fwd(lib, _cfg(hidden_size=96)) == binding.ERR_UNSUPPORTED    # H % 128
    assert _fwd(lib, _cfg(intermediate_size=200)) == binding.ERR_UNSUPPORTED
    assert _fwd(lib, _cfg(hidden_size=0)) == binding.ERR_INVALID_ARG
    assert _fwd(lib, ok, T=-3) == binding.ERR_INVALID_ARG
    assert _fwd(lib, ok, ptr=258) == binding.ERR_INVALID_ARG             # bf16 not 16-B aligned
    assert _fwd(lib, ok, shared=True) == binding.ERR_INVALID_ARG         # shared weights, I_s = 0
    assert _fwd(lib, _cfg(shared_intermediate_size=128)) == binding.ERR_INVALID_ARG
    assert _fwd(lib, ok, nev=5) == binding.ERR_INVALID_ARG               # events NULL, count 5
    need = lib.moe_forward_workspace_size(ctypes.byref(ok), 4)
    assert need > 0
    assert _fwd(lib, ok, ws_bytes=need - 1) == binding.ERR_WORKSPACE
    assert _fwd(lib, ok, T=0) == binding.OK                               # empty batch: no-op


def test_align_validation(lib):
    P = ctypes.c_void_p
    f = lib.moe_align_block_size
    assert f(P(256), 0, 2, 8, 16, None, None, None, None, 0, None) == binding.OK
    assert f(None, 4, 2, 8, 16, P(256), P(256), P(256), P(256), 1 << 30, None) == \
        binding.ERR_INVALID_ARG
    assert f(P(256), 4, 2, 8, 0, P(256), P(256), P(256), P(256), 1 << 30, None) == \
        binding.ERR_INVALID_ARG                                   # block size 0
    assert f(P(256), 4, 9, 8, 16, P(256), P(256), P(256), P(256), 1 << 30, None) == \
        binding.ERR_INVALID_ARG                                   # k > E
    need = lib.moe_align_block_size_workspace_size(4, 2, 8)
    assert f(P(256), 4, 2, 8, 16, P(256), P(256), P(256), P(256), need - 1, None) == \
        binding.ERR_WORKSPACE
    assert f(P(256), 4, 2, 8, 16, P(256), P(256), P(256), P(257), need, None) == \
        binding.ERR_WORKSPACE                                     # misaligned workspace


def test_workspace_sizes_monotone(lib):
    for w in configs.WORKLOADS.values():
        cfg = binding.config_from_workload(w)
        sizes = [lib.moe_forward_workspace_size(ctypes.byref(cfg), T) for T in (0, 1, 16, 4096)]
        assert all(s > 0 for s in sizes) and sizes == sorted(sizes), (w.name, sizes)
        lay = binding.moe_forward_workspace_layout(cfg, 16)
        assert lay.total == sizes[2]
        offs = [lay.status, lay.topk_weights, lay.topk_ids, lay.sorted_token_ids, lay.expert_ids,
                lay.num_tokens_post_padded, lay.act]
        assert offs == sorted(offs) and all(o % 256 == 0 for o in offs)
    assert lib.moe_forward_block_size(ctypes.byref(binding.config_from_workload(configs.TINY)),
                                      16) in (16, 32, 64, 128)


def test_device_status_validation(lib):
    v = ctypes.c_int32(0)
    assert lib.moe_get_device_status(None, ctypes.byref(v), None) == binding.ERR_INVALID_ARG
    P = ctypes.c_void_p
    assert lib.moe_selftest_bounded_wait(None, 1000, None) == binding.ERR_INVALID_ARG
    assert lib.moe_selftest_bounded_wait(P(257), 1000, None) == binding.ERR_INVALID_ARG
    assert lib.moe_selftest_bounded_wait(P(256), -1, None) == binding.ERR_INVALID_ARG


def test_launch_count_host(lib):
    bad = binding.make_config(num_experts=8, top_k=2, hidden_size=100, intermediate_size=256)
    assert lib.moe_forward_num_launches(ctypes.byref(bad), 4) == -1
    for w in configs.WORKLOADS.values():
        cfg = binding.config_from_workload(w)
        counts = [lib.moe_forward_num_launches(ctypes.byref(cfg), T) for T in (1, 16, 64, 4096)]
        assert all(4 <= c <= 9 for c in counts), (w.name, counts)
        # from the gate weight: small batches route inside the same launch, others add one
        for T, c in zip((1, 16, 64, 4096), counts):
            small = T <= 16 and T * w.top_k <= 2048
            assert lib.moe_forward_num_launches_ex(ctypes.byref(cfg), T, 1) == c + (0 if small else 1)
            assert lib.moe_forward_num_launches_ex(ctypes.byref(cfg), T, 0) == c


def _fwd_ex(lib, cfg, T=4, ptr=256, **fields):
    P = ctypes.c_void_p
    a = binding.ForwardArgs()
    for n in ("hidden_states", "router_logits", "w13_weight", "w2_weight", "output", "workspace"):
        setattr(a, n, ptr)
    a.workspace_bytes = 1 << 40
    for n, v in fields.items():
        setattr(a, n, v)
    return lib.moe_forward_ex(ctypes.byref(cfg), T, ctypes.byref(a), None)


def test_fp8_validation(lib):
    fp8 = dict(weight_quant="fp8", hidden_size=256)
    scales = dict(w13_scale=256, w2_scale=256)
    # the fp8 layer is the plain gated SiLU one, H a multiple of 256
    assert _fwd_ex(lib, _cfg(weight_quant="fp8"), **scales) == binding.ERR_UNSUPPORTED  # H 128
    assert _fwd_ex(lib, _cfg(swiglu_limit=7.0, **fp8), **scales) == binding.ERR_UNSUPPORTED
    assert _fwd_ex(lib, _cfg(gemm1_alpha=1.5, **fp8), **scales) == binding.ERR_UNSUPPORTED
    assert _fwd_ex(lib, _cfg(is_act_and_mul=0, **fp8), **scales) == binding.ERR_UNSUPPORTED
    assert _fwd_ex(lib, _cfg(apply_router_weight_on_input=True, **fp8),
                   **scales) == binding.ERR_UNSUPPORTED
    assert _fwd_ex(lib, _cfg(**fp8), w13_bias=256, **scales) == binding.ERR_UNSUPPORTED
    assert _fwd_ex(lib, _cfg(weight_quant=7)) == binding.ERR_INVALID_ARG
    # scales: required with fp8 weights, rejected without
    assert _fwd_ex(lib, _cfg(**fp8), w13_scale=256) == binding.ERR_INVALID_ARG
    assert _fwd_ex(lib, _cfg(hidden_size=256), **scales) == binding.ERR_INVALID_ARG
    ok = _cfg(**fp8)
    need = lib.moe_forward_workspace_size(ctypes.byref(ok), 4)
    assert need > 0 and _fwd_ex(lib, ok, workspace_bytes=need - 1, **scales) == \
        binding.ERR_WORKSPACE
    assert _fwd_ex(lib, ok, T=0, **scales) == binding.OK
    lay = binding.moe_forward_workspace_layout(ok, 4)
    assert lay.act_scale > lay.act and lay.act_scale % 256 == 0
    assert binding.moe_forward_workspace_layout(_cfg(hidden_size=256), 4).act_scale == 0
    # the standalone quant
    q = lib.moe_quant_fp8_per_token_group
    P = ctypes.c_void_p
    assert q(4, 100, P(256), P(256), P(256), None) == binding.ERR_INVALID_ARG    # H % 128
    assert q(4, 128, P(258), P(256), P(256), None) == binding.ERR_INVALID_ARG    # x alignment
    assert q(-1, 128, P(256), P(256), P(256), None) == binding.ERR_INVALID_ARG
    assert q(0, 128, None, None, None, None) == binding.OK


def test_fp8_workspace_fits_regions(lib):
    """The fp8 rows + scales fit the bf16-sized regions for every workload and batch size,
    including the smallest shared expert (T = 1, I_s = 128)."""
    for w in configs.WORKLOADS.values():
        if w.hidden_size % 256:
            continue
        cfg = binding.config_from_workload(w, weight_quant="fp8")
        for T in (1, 2, 16, 300, 4096):
            lay = binding.moe_forward_workspace_layout(cfg, T)
            assert lay.total > lay.act_scale > lay.act
    tiny = _cfg(weight_quant="fp8", hidden_size=256, shared_intermediate_size=128)
    assert lib.moe_forward_workspace_size(ctypes.byref(tiny), 1) > 0


def test_workspace_size_nondecreasing_in_tokens(lib):
    """A workspace sized for max_tokens serves every smaller batch: the layout of T tokens
    (split-K partials, fused-reduce counters and all) never needs more than that of T + 1."""
    for w in configs.WORKLOADS.values():
        for quant in (None, "fp8"):
            if quant and w.hidden_size % 256:
                continue
            cfg = binding.config_from_workload(w, weight_quant=quant)
            sizes = [lib.moe_forward_workspace_size(ctypes.byref(cfg), T)
                     for T in list(range(0, 200)) + [256, 1000, 4096]]
            assert all(a <= b for a, b in zip(sizes, sizes[1:])), (w.name, quant)


def test_nvfp4_validation(lib):
    fp4 = dict(weight_quant="nvfp4")
    sc = dict(w13_weight_scale_2=256, w2_weight_scale_2=256, input_scale=448.0, act_scale=100.0)
    # the NVFP4 layer is the plain gated SiLU one
    assert _fwd_ex(lib, _cfg(swiglu_limit=7.0, **fp4), **sc) == binding.ERR_UNSUPPORTED
    assert _fwd_ex(lib, _cfg(gemm1_alpha=1.5, **fp4), **sc) == binding.ERR_UNSUPPORTED
    assert _fwd_ex(lib, _cfg(is_act_and_mul=0, **fp4), **sc) == binding.ERR_UNSUPPORTED
    assert _fwd_ex(lib, _cfg(apply_router_weight_on_input=True, **fp4),
                   **sc) == binding.ERR_UNSUPPORTED
    assert _fwd_ex(lib, _cfg(**fp4), w13_bias=256, **sc) == binding.ERR_UNSUPPORTED
    # per-expert scales and positive finite per-tensor scales are required, and only here
    for bad in (dict(w2_weight_scale_2=None), dict(input_scale=0.0), dict(act_scale=-1.0),
                dict(act_scale=float("inf")), dict(input_scale=float("nan"))):
        assert _fwd_ex(lib, _cfg(**fp4), **{**sc, **bad}) == binding.ERR_INVALID_ARG, bad
    assert _fwd_ex(lib, _cfg(), w13_weight_scale_2=256) == binding.ERR_INVALID_ARG
    assert _fwd_ex(lib, _cfg(**fp4), w13_scale=256, **sc) == binding.ERR_INVALID_ARG
    # a shared expert needs its own scales
    shared = _cfg(shared_intermediate_size=128, **fp4)
    assert _fwd_ex(lib, shared, shared_w13=256, shared_w2=256, **sc) == binding.ERR_INVALID_ARG
    ok = _cfg(**fp4)
    need = lib.moe_forward_workspace_size(ctypes.byref(ok), 4)
    assert need > 0 and _fwd_ex(lib, ok, workspace_bytes=need - 1, **sc) == binding.ERR_WORKSPACE
    assert _fwd_ex(lib, ok, T=0, **sc) == binding.OK
    # the first GEMM's fp32 partials are sized for every batch, prefill included
    assert lib.moe_forward_workspace_size(ctypes.byref(ok), 4096) > \
        lib.moe_forward_workspace_size(ctypes.byref(_cfg()), 4096)
    # the standalone quant and the weight preparation
    q = lib.moe_quant_nvfp4
    P = ctypes.c_void_p
    assert q(4, 40, P(256), 1.0, P(256), P(256), None) == binding.ERR_INVALID_ARG   # H % 16
    assert q(4, 64, P(258), 1.0, P(256), P(256), None) == binding.ERR_INVALID_ARG   # x align
    assert q(4, 64, P(256), 0.0, P(256), P(256), None) == binding.ERR_INVALID_ARG   # g
    assert q(0, 64, None, 1.0, None, None, None) == binding.OK
    assert binding.moe_nvfp4_prepared_bytes(256, 7168) == 256 * 7168 * 9 // 16
    assert binding.moe_nvfp4_prepared_bytes(128, 64) == 4608
    for rows, K in ((0, 64), (100, 64), (128, 96), (128, -64)):
        assert binding.moe_nvfp4_prepared_bytes(rows, K) == 0
    prep = lib.moe_nvfp4_prepare_weight
    assert prep(100, 64, P(256), P(256), P(256), None) == binding.ERR_INVALID_ARG
    assert prep(128, 64, P(264), P(256), P(256), None) == binding.ERR_INVALID_ARG
    assert prep(128, 64, None, P(256), P(256), None) == binding.ERR_INVALID_ARG

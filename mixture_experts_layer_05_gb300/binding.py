"""Python binding of libgbmoe.so: the C ABI of ``include/gbmoe.h`` with the same names.

Argument marshalling only: torch tensors become device pointers, the current torch
CUDA stream becomes the ``stream`` argument, and a negative status raises
``GbmoeError``. Every step of the layer runs in the library's kernels; there is no
fallback of any kind, and loading fails loudly when the library is not built.
"""
from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgbmoe.so")

STATUS = {0: "GBMOE_OK", -1: "GBMOE_ERR_INVALID_ARG", -2: "GBMOE_ERR_UNSUPPORTED",
          -3: "GBMOE_ERR_WORKSPACE", -4: "GBMOE_ERR_CUDA", -5: "GBMOE_ERR_DEVICE_CHECK",
          -6: "GBMOE_ERR_TIMEOUT"}
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_DEVICE_CHECK, ERR_TIMEOUT = \
    0, -1, -2, -3, -4, -5, -6
SCORE = {"softmax": 0, "sigmoid": 1}
QUANT = {None: 0, "none": 0, "fp8": 1, "fp8_block128": 1, "nvfp4": 2}
NUM_STAGE_EVENTS = 5

# every entry point declared in include/gbmoe.h
EXPORTS = ("moe_topk", "moe_align_block_size_workspace_size", "moe_align_block_size",
           "moe_align_block_size_no_workspace",
           "moe_forward_workspace_size", "moe_forward_block_size", "moe_forward",
           "moe_forward_events", "moe_forward_workspace_layout", "moe_get_device_status",
           "moe_forward_num_launches", "moe_forward_num_launches_ex",
           "moe_selftest_bounded_wait", "moe_forward_ex",
           "moe_router_logits", "moe_quant_fp8_per_token_group", "moe_quant_nvfp4",
           "moe_nvfp4_prepared_bytes", "moe_nvfp4_prepare_weight", "gbmoe_version")


class GbmoeError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} returned {STATUS.get(code, code)}")
        self.code = code


class Config(ctypes.Structure):
    """gbmoe_config_t."""
    _fields_ = [("num_experts", ctypes.c_int32), ("top_k", ctypes.c_int32),
                ("hidden_size", ctypes.c_int32), ("intermediate_size", ctypes.c_int32),
                ("renormalize", ctypes.c_int32), ("use_grouped_topk", ctypes.c_int32),
                ("num_expert_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
                ("scoring_func", ctypes.c_int32), ("routed_scaling_factor", ctypes.c_float),
                ("activation", ctypes.c_int32), ("is_act_and_mul", ctypes.c_int32),
                ("shared_intermediate_size", ctypes.c_int32), ("swiglu_limit", ctypes.c_float),
                ("gemm1_alpha", ctypes.c_float),
                ("apply_router_weight_on_input", ctypes.c_int32),
                ("weight_quant", ctypes.c_int32)]


class ForwardArgs(ctypes.Structure):
    """gbmoe_forward_args_t."""
    _fields_ = [("hidden_states", ctypes.c_void_p), ("router_logits", ctypes.c_void_p),
                ("e_score_correction_bias", ctypes.c_void_p), ("w13_weight", ctypes.c_void_p),
                ("w2_weight", ctypes.c_void_p), ("shared_w13", ctypes.c_void_p),
                ("shared_w2", ctypes.c_void_p), ("w13_bias", ctypes.c_void_p),
                ("w2_bias", ctypes.c_void_p), ("output", ctypes.c_void_p),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t),
                ("events", ctypes.c_void_p), ("num_events", ctypes.c_int32),
                ("gate_weight", ctypes.c_void_p), ("w13_scale", ctypes.c_void_p),
                ("w2_scale", ctypes.c_void_p), ("shared_w13_scale", ctypes.c_void_p),
                ("shared_w2_scale", ctypes.c_void_p),
                ("w13_weight_scale_2", ctypes.c_void_p), ("w2_weight_scale_2", ctypes.c_void_p),
                ("shared_weight_scale_2", ctypes.c_void_p), ("input_scale", ctypes.c_float),
                ("act_scale", ctypes.c_float), ("shared_input_scale", ctypes.c_float),
                ("shared_act_scale", ctypes.c_float)]


class WorkspaceLayout(ctypes.Structure):
    """gbmoe_workspace_layout_t."""
    _fields_ = [(n, ctypes.c_size_t) for n in (
        "status", "topk_weights", "topk_ids", "sorted_token_ids", "expert_ids",
        "num_tokens_post_padded", "act", "act_scale", "total", "act_shared")]


def make_config(num_experts, top_k, hidden_size, intermediate_size, renormalize=True,
                use_grouped_topk=False, num_expert_group=0, topk_group=0,
                scoring_func="softmax", routed_scaling_factor=1.0, activation=0,
                is_act_and_mul=1, shared_intermediate_size=0, swiglu_limit=None,
                gemm1_alpha=1.0, apply_router_weight_on_input=False,
                weight_quant=None) -> Config:
    """weight_quant: None / "none", "fp8" (e4m3 weights with 128 x 128 fp32 block scales) or
    "nvfp4" (prepared e2m1 weights with e4m3 block scales and per-expert fp32 scales)."""
    return Config(int(num_experts), int(top_k), int(hidden_size), int(intermediate_size),
                  int(bool(renormalize)), int(bool(use_grouped_topk)), int(num_expert_group or 0),
                  int(topk_group or 0), SCORE.get(scoring_func, scoring_func),
                  float(routed_scaling_factor), int(activation), int(is_act_and_mul),
                  int(shared_intermediate_size or 0), float(swiglu_limit or 0.0),
                  float(gemm1_alpha), int(bool(apply_router_weight_on_input)),
                  QUANT.get(weight_quant, weight_quant))


def config_from_workload(w, **variants) -> Config:
    return make_config(w.num_experts, w.top_k, w.hidden_size, w.intermediate_size,
                       w.renormalize, w.use_grouped_topk, w.num_expert_group, w.topk_group,
                       w.scoring_func, w.routed_scaling_factor,
                       shared_intermediate_size=w.shared_intermediate_size, **variants)


_lib = None


def load() -> ctypes.CDLL:
    """Load libgbmoe.so (built by ``build()``); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built: run mixture_experts_layer_05_gb300.build"
                           ".build() (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    P, I32, SZ = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t
    CP = ctypes.POINTER(Config)
    sig = {
        "moe_topk": (I32, [CP, I32, P, P, P, P, P]),
        "moe_align_block_size_workspace_size": (SZ, [I32, I32, I32]),
        "moe_align_block_size": (I32, [P, I32, I32, I32, I32, P, P, P, P, SZ, P]),
        "moe_align_block_size_no_workspace": (I32, [P, I32, I32, I32, I32, P, P, P, P]),
        "moe_forward_workspace_size": (SZ, [CP, I32]),
        "moe_forward_block_size": (I32, [CP, I32]),
        "moe_forward": (I32, [CP, I32, P, P, P, P, P, P, P, P, P, SZ, P]),
        "moe_forward_events": (I32, [CP, I32, P, P, P, P, P, P, P, P, P, SZ, P, I32, P]),
        "moe_forward_workspace_layout": (I32, [CP, I32, ctypes.POINTER(WorkspaceLayout)]),
        "moe_get_device_status": (I32, [P, ctypes.POINTER(I32), P]),
        "moe_forward_num_launches": (I32, [CP, I32]),
        "moe_forward_num_launches_ex": (I32, [CP, I32, I32]),
        "moe_forward_ex": (I32, [CP, I32, ctypes.POINTER(ForwardArgs), P]),
        "moe_router_logits": (I32, [I32, I32, I32, P, P, P, P]),
        "moe_quant_fp8_per_token_group": (I32, [I32, I32, P, P, P, P]),
        "moe_quant_nvfp4": (I32, [I32, I32, P, ctypes.c_float, P, P, P]),
        "moe_nvfp4_prepared_bytes": (SZ, [I32, I32]),
        "moe_nvfp4_prepare_weight": (I32, [I32, I32, P, P, P, P]),
        "moe_selftest_bounded_wait": (I32, [P, I32, P]),
        "gbmoe_version": (I32, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, code: int):
    if code != OK:
        raise GbmoeError(fn, code)


def _need(t, dtype, name):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {dtype} tensor")


def moe_topk(cfg: Config, router_logits, e_score_correction_bias, topk_weights, topk_ids,
             stream=None):
    _need(router_logits, torch.float32, "router_logits")
    _need(e_score_correction_bias, torch.float32, "e_score_correction_bias")
    _need(topk_weights, torch.float32, "topk_weights")
    _need(topk_ids, torch.int32, "topk_ids")
    _check("moe_topk", load().moe_topk(ctypes.byref(cfg), router_logits.shape[0],
                                       _p(router_logits), _p(e_score_correction_bias),
                                       _p(topk_weights), _p(topk_ids), _stream(stream)))


def moe_align_block_size_workspace_size(num_tokens, top_k, num_experts) -> int:
    return load().moe_align_block_size_workspace_size(num_tokens, top_k, num_experts)


def moe_align_block_size(topk_ids, num_experts, block_size, sorted_token_ids, expert_ids,
                         num_tokens_post_padded, workspace, stream=None):
    _need(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    _check("moe_align_block_size", load().moe_align_block_size(
        _p(topk_ids), T, k, num_experts, block_size, _p(sorted_token_ids), _p(expert_ids),
        _p(num_tokens_post_padded), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))


def moe_align_block_size_no_workspace(topk_ids, num_experts, block_size, sorted_token_ids,
                                      expert_ids, num_tokens_post_padded, stream=None):
    """moe_align_block_size with the library's built-in 1 MiB scratch (no workspace).

    For callers that may not allocate device memory (a host framework owns every
    allocation); calls that overlap on the GPU share that scratch and must not be issued.
    """
    _need(topk_ids, torch.int32, "topk_ids")
    T, k = topk_ids.shape
    _check("moe_align_block_size_no_workspace", load().moe_align_block_size_no_workspace(
        _p(topk_ids), T, k, num_experts, block_size, _p(sorted_token_ids), _p(expert_ids),
        _p(num_tokens_post_padded), _stream(stream)))


def moe_forward_workspace_size(cfg: Config, max_num_tokens: int) -> int:
    n = load().moe_forward_workspace_size(ctypes.byref(cfg), max_num_tokens)
    if n == 0:
        raise GbmoeError("moe_forward_workspace_size", ERR_INVALID_ARG)
    return n


def moe_forward_block_size(cfg: Config, num_tokens: int) -> int:
    return load().moe_forward_block_size(ctypes.byref(cfg), num_tokens)


def moe_forward_workspace_layout(cfg: Config, num_tokens: int) -> WorkspaceLayout:
    out = WorkspaceLayout()
    _check("moe_forward_workspace_layout",
           load().moe_forward_workspace_layout(ctypes.byref(cfg), num_tokens, ctypes.byref(out)))
    return out


def alloc_workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A uint8 workspace; its status word (first 256 bytes) starts at zero."""
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    ws[:256].zero_()
    return ws


def moe_forward(cfg: Config, hidden_states, router_logits, e_score_correction_bias, w13_weight,
                w2_weight, shared_w13, shared_w2, output, workspace, events=None, stream=None):
    _need(hidden_states, torch.bfloat16, "hidden_states")
    _need(router_logits, torch.float32, "router_logits")
    _need(e_score_correction_bias, torch.float32, "e_score_correction_bias")
    for t, n in ((w13_weight, "w13_weight"), (w2_weight, "w2_weight"), (shared_w13, "shared_w13"),
                 (shared_w2, "shared_w2"), (output, "output")):
        _need(t, torch.bfloat16, n)
    lib = load()
    args = [ctypes.byref(cfg), hidden_states.shape[0], _p(hidden_states), _p(router_logits),
            _p(e_score_correction_bias), _p(w13_weight), _p(w2_weight), _p(shared_w13),
            _p(shared_w2), _p(output), _p(workspace),
            workspace.numel() * workspace.element_size()]
    if events is None:
        _check("moe_forward", lib.moe_forward(*args, _stream(stream)))
    else:
        for ev in events:                  # torch creates the CUDA event on first record
            if ev is not None and not ev.cuda_event:
                ev.record()
        arr = (ctypes.c_void_p * len(events))(
            *[None if ev is None else ev.cuda_event for ev in events])
        _check("moe_forward_events",
               lib.moe_forward_events(*args, arr, len(events), _stream(stream)))


def moe_forward_num_launches(cfg: Config, num_tokens: int) -> int:
    return load().moe_forward_num_launches(ctypes.byref(cfg), num_tokens)


def moe_forward_num_launches_ex(cfg: Config, num_tokens: int, from_gate_weight: bool) -> int:
    return load().moe_forward_num_launches_ex(ctypes.byref(cfg), num_tokens,
                                              int(bool(from_gate_weight)))


def moe_selftest_bounded_wait(workspace, timeout_us: int, stream=None):
    _check("moe_selftest_bounded_wait",
           load().moe_selftest_bounded_wait(_p(workspace), timeout_us, _stream(stream)))


def moe_router_logits(hidden_states, gate_weight, router_logits, stream=None):
    """router_logits [T, E] fp32 = hidden_states [T, H] @ gate_weight [E, H]^T (tensor cores)."""
    _need(hidden_states, torch.bfloat16, "hidden_states")
    _need(gate_weight, torch.bfloat16, "gate_weight")
    _need(router_logits, torch.float32, "router_logits")
    T, H = hidden_states.shape
    _check("moe_router_logits", load().moe_router_logits(
        T, H, gate_weight.shape[0], _p(hidden_states), _p(gate_weight), _p(router_logits),
        _stream(stream)))


def _fp8_bytes(t, name):
    """e4m3 weights as passed to the library: float8_e4m3fn or uint8 storage."""
    if t is None:
        return None
    if not t.is_cuda or not t.is_contiguous() or t.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise ValueError(f"{name} must be a contiguous CUDA float8_e4m3fn (or uint8) tensor")
    return t


NVFP4_KEYS = ("w13_weight_scale_2", "w2_weight_scale_2", "shared_weight_scale_2",
              "input_scale", "act_scale", "shared_input_scale", "shared_act_scale")


def moe_forward_ex(cfg: Config, hidden_states, router_logits, e_score_correction_bias,
                   w13_weight, w2_weight, shared_w13, shared_w2, output, workspace,
                   w13_bias=None, w2_bias=None, events=None, stream=None, gate_weight=None,
                   w13_scale=None, w2_scale=None, shared_w13_scale=None, shared_w2_scale=None,
                   w13_weight_scale_2=None, w2_weight_scale_2=None, shared_weight_scale_2=None,
                   input_scale=0.0, act_scale=0.0, shared_input_scale=0.0,
                   shared_act_scale=0.0):
    """moe_forward with the optional per-expert biases, stage events, (router_logits None)
    the gate weight whose router GEMM runs first, or quantized experts: (cfg.weight_quant
    fp8) e4m3 weights with their fp32 128 x 128 block scales; (nvfp4) prepared fp4 weights
    (moe_nvfp4_prepare_weight) with fp32 per-expert scales and the per-tensor scales."""
    _need(hidden_states, torch.bfloat16, "hidden_states")
    _need(router_logits, torch.float32, "router_logits")
    _need(e_score_correction_bias, torch.float32, "e_score_correction_bias")
    weights = ((w13_weight, "w13_weight"), (w2_weight, "w2_weight"), (shared_w13, "shared_w13"),
               (shared_w2, "shared_w2"))
    if cfg.weight_quant == QUANT["fp8"]:
        for t, n in weights:
            _fp8_bytes(t, n)
        for t, n in ((w13_scale, "w13_scale"), (w2_scale, "w2_scale"),
                     (shared_w13_scale, "shared_w13_scale"), (shared_w2_scale, "shared_w2_scale")):
            _need(t, torch.float32, n)
        weights = ()
    elif cfg.weight_quant == QUANT["nvfp4"]:
        for t, n in weights:
            _need(t, torch.uint8, n)
        for t, n in ((w13_weight_scale_2, "w13_weight_scale_2"),
                     (w2_weight_scale_2, "w2_weight_scale_2"),
                     (shared_weight_scale_2, "shared_weight_scale_2")):
            _need(t, torch.float32, n)
        weights = ()
    for t, n in weights + ((w13_bias, "w13_bias"), (w2_bias, "w2_bias"),
                           (output, "output"), (gate_weight, "gate_weight")):
        _need(t, torch.bfloat16, n)
    arr = None
    if events is not None:
        for ev in events:
            if ev is not None and not ev.cuda_event:
                ev.record()
        arr = (ctypes.c_void_p * len(events))(
            *[None if ev is None else ev.cuda_event for ev in events])
    ptr = lambda t: None if t is None else t.data_ptr()
    a = ForwardArgs(ptr(hidden_states), ptr(router_logits), ptr(e_score_correction_bias),
                    ptr(w13_weight), ptr(w2_weight), ptr(shared_w13), ptr(shared_w2),
                    ptr(w13_bias), ptr(w2_bias), ptr(output), ptr(workspace),
                    workspace.numel() * workspace.element_size(),
                    ctypes.cast(arr, ctypes.c_void_p) if arr is not None else None,
                    0 if events is None else len(events), ptr(gate_weight), ptr(w13_scale),
                    ptr(w2_scale), ptr(shared_w13_scale), ptr(shared_w2_scale),
                    ptr(w13_weight_scale_2), ptr(w2_weight_scale_2),
                    ptr(shared_weight_scale_2), float(input_scale), float(act_scale),
                    float(shared_input_scale), float(shared_act_scale))
    _check("moe_forward_ex", load().moe_forward_ex(ctypes.byref(cfg), hidden_states.shape[0],
                                                   ctypes.byref(a), _stream(stream)))


def moe_quant_fp8_per_token_group(x, q=None, scale=None, stream=None):
    """Per-token-group-128 e4m3 quant of bf16 rows: q [R, H] float8_e4m3fn and the
    group-major fp32 scales scale [H / 128, R]; returns (q, scale)."""
    _need(x, torch.bfloat16, "x")
    R, H = x.shape
    if q is None:
        q = torch.empty(R, H, dtype=torch.float8_e4m3fn, device=x.device)
    if scale is None:
        scale = torch.empty(H // 128, R, dtype=torch.float32, device=x.device)
    _fp8_bytes(q, "q")
    _need(scale, torch.float32, "scale")
    _check("moe_quant_fp8_per_token_group", load().moe_quant_fp8_per_token_group(
        R, H, _p(x), _p(q), _p(scale), _stream(stream)))
    return q, scale


def moe_quant_nvfp4(x, global_scale: float, q=None, sf=None, stream=None):
    """fp4_quantize(x, g, 16) of bf16 rows: packed e2m1 codes q [R, H / 2] uint8 (low nibble
    first) and e4m3 block scales sf [R, H / 16] (float8_e4m3fn); returns (q, sf)."""
    _need(x, torch.bfloat16, "x")
    R, H = x.shape
    if q is None:
        q = torch.empty(R, H // 2, dtype=torch.uint8, device=x.device)
    if sf is None:
        sf = torch.empty(R, H // 16, dtype=torch.float8_e4m3fn, device=x.device)
    _need(q, torch.uint8, "q")
    _fp8_bytes(sf, "sf")
    _check("moe_quant_nvfp4", load().moe_quant_nvfp4(R, H, _p(x), float(global_scale), _p(q),
                                                     _p(sf), _stream(stream)))
    return q, sf


def moe_nvfp4_prepared_bytes(rows: int, K: int) -> int:
    return int(load().moe_nvfp4_prepared_bytes(rows, K))


def moe_nvfp4_prepare_weight(packed, block_scale, out=None, stream=None):
    """The GEMMs' layout of one fp4 weight stack: packed [rows, K / 2] uint8 codes and
    block_scale [rows, K / 16] e4m3 (float8_e4m3fn or uint8) -> out (uint8, returned)."""
    _need(packed, torch.uint8, "packed")
    _fp8_bytes(block_scale, "block_scale")
    rows, K = packed.shape[0], packed.shape[1] * 2
    nbytes = moe_nvfp4_prepared_bytes(rows, K)
    if nbytes == 0:
        raise GbmoeError("moe_nvfp4_prepared_bytes", ERR_INVALID_ARG)
    if out is None:
        out = torch.empty(nbytes, dtype=torch.uint8, device=packed.device)
    _need(out, torch.uint8, "out")
    _check("moe_nvfp4_prepare_weight", load().moe_nvfp4_prepare_weight(
        rows, K, _p(packed), _p(block_scale), _p(out), _stream(stream)))
    return out


def moe_get_device_status(workspace, stream=None) -> int:
    v = ctypes.c_int32(0)
    _check("moe_get_device_status",
           load().moe_get_device_status(_p(workspace), ctypes.byref(v), _stream(stream)))
    return v.value


class FusedMoE:
    """The layer with its weights resident on the GPU and a workspace sized for max_tokens."""

    def __init__(self, cfg: Config, w13_weight, w2_weight, e_score_correction_bias=None,
                 shared_w13=None, shared_w2=None, max_tokens: int = 1, w13_bias=None,
                 w2_bias=None, w13_scale=None, w2_scale=None, shared_w13_scale=None,
                 shared_w2_scale=None, **nvfp4):
        self.cfg = cfg
        self.w13, self.w2 = w13_weight, w2_weight
        self.bias, self.shared_w13, self.shared_w2 = e_score_correction_bias, shared_w13, shared_w2
        self.w13_bias, self.w2_bias = w13_bias, w2_bias
        self.scales = dict(w13_scale=w13_scale, w2_scale=w2_scale,
                           shared_w13_scale=shared_w13_scale, shared_w2_scale=shared_w2_scale)
        unknown = set(nvfp4) - set(NVFP4_KEYS)
        if unknown:
            raise TypeError(f"unexpected arguments {sorted(unknown)}")
        self.scales.update(nvfp4)  # nvfp4: per-expert and per-tensor scales
        self.max_tokens = 0
        self.workspace = None
        self.reserve(max_tokens)

    def reserve(self, max_tokens: int):
        if max_tokens > self.max_tokens:
            dev = self.w13.device
            self.workspace = alloc_workspace(moe_forward_workspace_size(self.cfg, max_tokens), dev)
            self.max_tokens = max_tokens

    def __call__(self, hidden_states, router_logits=None, out=None, events=None, stream=None,
                 gate_weight=None):
        """Forward from router logits, or (router_logits None) from the gate weight."""
        T = hidden_states.shape[0]
        self.reserve(T)
        if out is None:
            out = torch.empty_like(hidden_states)
        if gate_weight is not None or router_logits is None or self.cfg.weight_quant:
            moe_forward_ex(self.cfg, hidden_states, router_logits if gate_weight is None else None,
                           self.bias, self.w13, self.w2, self.shared_w13, self.shared_w2, out,
                           self.workspace, w13_bias=self.w13_bias, w2_bias=self.w2_bias,
                           events=events, stream=stream, gate_weight=gate_weight, **self.scales)
        elif self.w13_bias is None and self.w2_bias is None:
            moe_forward(self.cfg, hidden_states, router_logits, self.bias, self.w13, self.w2,
                        self.shared_w13, self.shared_w2, out, self.workspace, events=events,
                        stream=stream)
        else:
            moe_forward_ex(self.cfg, hidden_states, router_logits, self.bias, self.w13, self.w2,
                           self.shared_w13, self.shared_w2, out, self.workspace,
                           w13_bias=self.w13_bias, w2_bias=self.w2_bias, events=events,
                           stream=stream)
        return out

    def device_status(self) -> int:
        return moe_get_device_status(self.workspace)


class HostPipeline:
    """Runs a FusedMoE layer over batches held in pinned host memory.

    Three CUDA streams and double-buffered device tensors: batch i's host-to-device copy
    runs while batch i-1 computes, and batch i-1's device-to-host copy while batch i
    computes. Every batch still pays its own copies; they are only overlapped.
    """

    def __init__(self, layer: FusedMoE, max_tokens: int, gate_weight=None):
        dev = layer.w13.device
        self.gate = gate_weight                       # route from the gate weight: no logits
        H = layer.cfg.hidden_size
        E = layer.cfg.num_experts
        layer.reserve(max_tokens)
        self.layer = layer
        self.h2d, self.comp, self.d2h = (torch.cuda.Stream(dev) for _ in range(3))
        self.x = [torch.empty(max_tokens, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.l = [torch.empty(max_tokens, E, dtype=torch.float32, device=dev) for _ in range(2)]
        self.y = [torch.empty(max_tokens, H, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        self.in_ready = [torch.cuda.Event() for _ in range(2)]
        self.comp_done = [torch.cuda.Event() for _ in range(2)]
        self.d2h_done = [torch.cuda.Event() for _ in range(2)]

    def run(self, xs, logits, ys):
        """Forward of every (xs[i], logits[i]) host batch into the host tensor ys[i]."""
        for i in range(len(xs)):
            b = i & 1
            T = xs[i].shape[0]
            x, lg, y = self.x[b][:T], self.l[b][:T], self.y[b][:T]
            self.h2d.wait_event(self.comp_done[b])         # batch i-2 no longer reads x[b]
            with torch.cuda.stream(self.h2d):
                x.copy_(xs[i], non_blocking=True)
                if self.gate is None:
                    lg.copy_(logits[i], non_blocking=True)
                self.in_ready[b].record(self.h2d)
            self.comp.wait_event(self.in_ready[b])
            self.comp.wait_event(self.d2h_done[b])         # batch i-2 has left y[b]
            if self.gate is None:
                self.layer(x, lg, out=y, stream=self.comp)
            else:
                self.layer(x, out=y, stream=self.comp, gate_weight=self.gate)
            self.comp_done[b].record(self.comp)
            self.d2h.wait_event(self.comp_done[b])
            with torch.cuda.stream(self.d2h):
                ys[i].copy_(y, non_blocking=True)
                self.d2h_done[b].record(self.d2h)
        return ys

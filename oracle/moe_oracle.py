"""CPU oracle of the FusedMoE layer forward: plain, slow, fp64, written from the pages.

TEST INFRASTRUCTURE ONLY. Nothing on the product path imports this module: only the
tests, ``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of ``bench.py``
may use it. It shares no code with the CUDA path.

What it computes, step by step, and where each step is defined:

1. Scores (``score``): softmax or sigmoid of the fp32 router logits. vLLM
   ``fused_moe/layer`` page, ``FusedMoE.select_experts`` (the three routing branches)
   and the constructor check that a non-softmax scoring function needs grouped top-k;
   the logits are fp32 as ``MoEGate.forward`` returns them (sglang
   ``models/deepseek_v2.py`` page).
2. Selection keys: the score plus ``e_score_correction_bias`` when one is given
   (``fused_topk_bias`` / ``grouped_topk`` in ``select_experts``; the fp32 bias of
   ``MoEGate.__init__``).
3. Grouped top-k (``grouped_topk`` in ``select_experts``, kwargs num_expert_group /
   topk_group in ``DeepseekV2MoE.__init__``): experts fall into ``num_expert_group``
   contiguous groups; the ``topk_group`` groups with the largest group score survive.
   The pages do not define the group score. Reading used here: without a bias the
   largest score in the group; with a bias (the "noaux_tc" method) the sum of the two
   largest keys in the group.
4. Top-k over the surviving experts by key, ties to the lower expert index, emitted in
   descending key order.
5. Weights are the unbiased scores of the chosen experts, divided by their sum when
   ``renormalize`` (the ``renormalize`` flag of the FusedMoE constructor), then
   multiplied by ``routed_scaling_factor`` (``select_experts`` scales after the biased
   and grouped paths; the factor is 1 on the plain path in every workload here).
6. Align (``moe_align_block_size``): a stable counting sort of the flat indices
   ``f = t*top_k + j`` by expert, each expert's run padded to a multiple of the block
   size with the sentinel ``T*top_k``; one expert id per block; the padded total.
   The pages name the FusedMoE call but not this step; its outputs are defined by
   their names (sorted_token_ids, expert_ids, num_tokens_post_padded).
7. Expert MLP (``swiglu_mlp``): ``w13[e]`` rows [0, I) are the gate (w1) and rows
   [I, 2I) the up projection (w3) (``FusedMoE._load_w13``); ``act = silu(gate) * up``
   (``SiluAndMul`` in ``DeepseekV2MLP``); ``o = w2[e] @ act`` with ``w2 [E, H, I]``
   (``FusedMoE._load_w2``). ``act``, the tensor between the two GEMMs, is held in the
   layer's dtype, bf16: ``DeepseekV2MLP.forward`` hands ``act_fn(gate_up)`` (or the buffer
   ``gate_up.new_empty(...)`` that ``silu_and_mul_clamp`` fills) to ``down_proj``, and the
   activations entering ``FusedMoE`` are the model dtype (``moe_in_dtype`` on the vLLM
   page). The layer functions therefore round ``act`` to the nearest bf16 value, ties to
   even (``round_bf16``), and compute everything else exactly.
8. Combine: ``y[t] = sum_j w[t, j] * o[t, j]`` over j ascending, plus the shared expert
   (one dense SwiGLU, ``DeepseekV2MLP``) added without the routed scaling factor
   (``DeepseekV2MoE.forward_normal`` / ``maybe_fuse_routed_scale_and_shared_add``).

Everything is fp64 (bf16 inputs widened exactly) except the bf16 act of step 7. Parity
of every function is pinned by the CPU tests (brute force, closed forms, invariants, hand-worked examples).
"""
from __future__ import annotations

import numpy as np


def _f64(a) -> np.ndarray:
    """Exact widening of a torch tensor (any float dtype) or array to fp64 numpy."""
    if hasattr(a, "detach"):
        import torch
        return a.detach().to("cpu", torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


# ---------------------------------------------------------------- 1. scores
def score(logits_row: np.ndarray, scoring_func: str) -> np.ndarray:
    """Softmax or sigmoid of one row of router logits (fp64)."""
    l = np.asarray(logits_row, dtype=np.float64)
    if scoring_func == "softmax":
        z = np.exp(l - l.max())
        return z / z.sum()
    if scoring_func == "sigmoid":
        return 1.0 / (1.0 + np.exp(-l))
    raise ValueError(f"unknown scoring_func {scoring_func!r}")


# ---------------------------------------------------------------- 3. group score
def group_score(scores_g: np.ndarray, keys_g: np.ndarray, with_bias: bool) -> float:
    """Group score: max score (no bias) or sum of the two largest keys (with bias)."""
    if with_bias:
        top = np.sort(keys_g)[::-1]
        return float(top[0] + (top[1] if len(top) > 1 else 0.0))
    return float(np.max(scores_g))


def _rank_desc(values: np.ndarray, candidates) -> list:
    """Candidates ordered by value descending, ties to the lower index."""
    return sorted(candidates, key=lambda i: (-values[i], i))


# ---------------------------------------------------------------- 0. router GEMM
def router_logits(x, gate_weight) -> np.ndarray:
    """logits [T, E] = x [T, H] @ gate_weight [E, H]^T in fp64 (``MoEGate.forward`` on the
    sglang ``models/deepseek_v2.py`` page: bf16 operands, fp32 logits)."""
    return _f64(x) @ _f64(gate_weight).T


# ---------------------------------------------------------------- 2-5. routing of one token
def route_token(logits_row, bias, *, num_experts, top_k, renormalize,
                use_grouped_topk=False, num_expert_group=0, topk_group=0,
                scoring_func="softmax", routed_scaling_factor=1.0):
    """(weights [k] fp64, ids [k] int, info) for one token."""
    E = num_experts
    s = score(logits_row, scoring_func)
    q = s + _f64(bias) if bias is not None else s.copy()
    eligible = list(range(E))
    kept_groups = None
    gscores = None
    if use_grouped_topk:
        G = num_expert_group
        size = E // G
        gscores = np.array([group_score(s[g * size:(g + 1) * size], q[g * size:(g + 1) * size],
                                        bias is not None) for g in range(G)])
        kept_groups = _rank_desc(gscores, range(G))[:topk_group]
        eligible = [e for e in range(E) if e // size in kept_groups]
    ids = _rank_desc(q, eligible)[:top_k]
    w = np.array([s[e] for e in ids], dtype=np.float64)
    if renormalize:
        w = w / w.sum()
    w = w * routed_scaling_factor
    info = {"scores": s, "keys": q, "eligible": eligible, "kept_groups": kept_groups,
            "group_scores": gscores}
    return w, np.array(ids, dtype=np.int64), info


def select_experts(logits, bias, **cfg):
    """Route every token: (topk_weights [T,k] fp64, topk_ids [T,k] int64)."""
    L = _f64(logits)
    T, k = L.shape[0], cfg["top_k"]
    W = np.zeros((T, k), dtype=np.float64)
    ids = np.zeros((T, k), dtype=np.int64)
    for t in range(T):
        W[t], ids[t], _ = route_token(L[t], bias, **cfg)
    return W, ids


def decision_margins(logits, bias, **cfg) -> np.ndarray:
    """Per token, the smallest gap at any routing decision that shapes the outputs.

    Decisions: which groups survive (the gap between the last kept and the first
    dropped group score) and the order of the top_k + 1 best eligible keys. Gaps are
    measured in logit units for softmax keys without a bias (log ratio of scores) and
    in key units otherwise.
    """
    L = _f64(logits)
    T = L.shape[0]
    out = np.full(T, np.inf)
    k = cfg["top_k"]
    soft_log = cfg.get("scoring_func", "softmax") == "softmax" and bias is None
    for t in range(T):
        _, _, info = route_token(L[t], bias, **cfg)
        q = info["keys"]
        qs = np.log(q) if soft_log else q
        m = np.inf
        if info["kept_groups"] is not None:
            g = info["group_scores"]
            gs = np.log(g) if soft_log else g
            order = _rank_desc(gs, range(len(gs)))
            nk = len(info["kept_groups"])
            if nk < len(order):
                m = min(m, gs[order[nk - 1]] - gs[order[nk]])
        order = _rank_desc(qs, info["eligible"])[: k + 1]
        for a, b in zip(order[:-1], order[1:]):
            m = min(m, qs[a] - qs[b])
        out[t] = m
    return out


# ---------------------------------------------------------------- 6. align
def moe_align_block_size(topk_ids, num_experts: int, block_size: int):
    """(sorted_token_ids, expert_ids, num_tokens_post_padded) by a stable counting sort."""
    flat = np.asarray(topk_ids, dtype=np.int64).reshape(-1)
    n = flat.size
    sentinel = n
    counts = np.zeros(num_experts, dtype=np.int64)
    for e in flat:
        counts[e] += 1
    padded = [((c + block_size - 1) // block_size) * block_size for c in counts]
    total = int(sum(padded))
    sorted_ids = np.full(total, sentinel, dtype=np.int64)
    expert_ids = np.zeros(total // block_size, dtype=np.int64)
    start = 0
    starts = []
    for e in range(num_experts):
        starts.append(start)
        for b in range(padded[e] // block_size):
            expert_ids[start // block_size + b] = e
        start += padded[e]
    fill = list(starts)
    for f in range(n):                          # ascending f: stable within an expert
        e = flat[f]
        sorted_ids[fill[e]] = f
        fill[e] += 1
    return sorted_ids, expert_ids, total


# ---------------------------------------------------------------- 7. expert MLP
BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127        # largest finite bfloat16


def round_bf16(a) -> np.ndarray:
    """Nearest bfloat16 value of each fp64 value, ties to even: 8 significant bits over
    fp32's exponent range (spacing 2^(e-7) for 2^e <= |a| < 2^(e+1), e >= -126; 2^-133 below
    2^-126), values past the largest finite bf16 to +-inf. Written from the format."""
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)                               # a = m 2^e with 1/2 <= |m| < 1
    e = np.maximum(e, -125)                          # subnormal spacing stays 2^-133
    q = np.ldexp(np.rint(np.ldexp(a, 8 - e)), e - 8)  # rint: ties to even
    return np.where(np.abs(q) > BF16_MAX, np.copysign(np.inf, a), q)


def silu(z: np.ndarray) -> np.ndarray:
    return z / (1.0 + np.exp(-z))


def swiglu_mlp(h: np.ndarray, w13_e, w2_e) -> np.ndarray:
    """o = w2 @ (silu(w1 @ h) * (w3 @ h)) for rows h [n, H]; w13_e [2I, H], w2_e [H, I]."""
    return expert_mlp(h, w13_e, w2_e)


def expert_mlp(h, w13_e, w2_e, *, b13_e=None, b2_e=None, gated=True, swiglu_limit=None,
               gemm1_alpha=1.0, act_dtype=None) -> np.ndarray:
    """One expert's MLP with the layer's optional variants (sglang ``fused_moe_triton/layer``
    page, ``FusedMoE.__init__``: ``with_bias``, ``is_gated``, ``gemm1_alpha``,
    ``gemm1_clamp_limit``; ``DeepseekV2MLP.forward``: ``swiglu_limit``).

    z = h @ w13^T (+ b13). Gated: gate = z[:, :I], up = z[:, I:]; with a limit L,
    gate = min(gate, L) and up = clip(up, -L, L); act = gate * sigmoid(alpha * gate) * up.
    Not gated (w13_e is [I, H]): act = silu(z). o = act @ w2^T (+ b2).
    The pages name these parameters without their arithmetic; this is the reading the
    NPU clipped-SwiGLU call's arguments (alpha, limit, bias) point to.
    act_dtype "bf16" rounds act to bf16 (the layer's intermediate tensor); None keeps it exact.
    """
    W13 = _f64(w13_e)
    W2 = _f64(w2_e)
    h = np.atleast_2d(_f64(h))
    z = h @ W13.T
    if b13_e is not None:
        z = z + _f64(b13_e)
    if gated:
        I = W13.shape[0] // 2
        gate, up = z[:, :I], z[:, I:]
        if swiglu_limit is not None:
            gate = np.minimum(gate, swiglu_limit)
            up = np.clip(up, -swiglu_limit, swiglu_limit)
        act = gate / (1.0 + np.exp(-gemm1_alpha * gate)) * up
    else:
        act = silu(z)
    if act_dtype == "bf16":
        act = round_bf16(act)
    elif act_dtype is not None:
        raise ValueError(f"unknown act_dtype {act_dtype!r}")
    o = act @ W2.T
    if b2_e is not None:
        o = o + _f64(b2_e)
    return o


# ---------------------------------------------------------------- 8. the layer
def experts_combine(x, topk_weights, topk_ids, w13, w2, shared_w13=None, shared_w2=None, *,
                    return_parts=False, w13_bias=None, w2_bias=None, gated=True,
                    swiglu_limit=None, gemm1_alpha=1.0, apply_router_weight_on_input=False,
                    top_k=None, act_dtype="bf16"):
    """y [T, H] fp64 of the experts and the combine for a routing given as input.

    This is the layer behind a precomputed top-k (``FusedMoE.forward(hidden_states,
    topk_output)`` with a ``StandardTopKOutput(topk_weights, topk_ids, ...)`` on the sglang
    ``fused_moe_triton/layer.py`` page): each (token, slot) runs its expert's MLP, the
    outputs are summed with the routing weights over slots j ascending, then the shared
    expert is added unscaled. With ``apply_router_weight_on_input`` (FusedMoE constructor
    argument) the routing weight scales the expert's input instead of its output. The
    shared expert (``DeepseekV2MLP``: no bias, alpha 1) shares the SwiGLU limit. The
    tensors the layer holds between its steps are of its dtype (``act_dtype`` "bf16"): every
    expert's act, and with ``apply_router_weight_on_input`` the weighted input rows, are
    rounded to bf16 (None keeps them exact).
    """
    X = _f64(x)
    T, H = X.shape
    W = np.atleast_2d(np.asarray(topk_weights, dtype=np.float64))
    ids = np.atleast_2d(np.asarray(topk_ids, dtype=np.int64))
    k = ids.shape[1] if top_k is None else top_k
    o = np.zeros((T, k, H), dtype=np.float64)
    for e in sorted(set(ids.reshape(-1).tolist())):           # each expert's weights once
        rows = [(t, j) for t in range(T) for j in range(k) if ids[t, j] == e]
        h = X[[t for t, _ in rows]]
        if apply_router_weight_on_input:
            h = h * np.array([W[t, j] for t, j in rows])[:, None]
            if act_dtype == "bf16":
                h = round_bf16(h)            # the scaled input is a tensor of the layer dtype
        out = expert_mlp(h, w13[e], w2[e],
                         b13_e=None if w13_bias is None else w13_bias[e],
                         b2_e=None if w2_bias is None else w2_bias[e], gated=gated,
                         swiglu_limit=swiglu_limit, gemm1_alpha=gemm1_alpha,
                         act_dtype=act_dtype)
        for (t, j), r in zip(rows, out):
            o[t, j] = r
    y = np.zeros((T, H), dtype=np.float64)
    for t in range(T):
        for j in range(k):
            y[t] += o[t, j] if apply_router_weight_on_input else W[t, j] * o[t, j]
    shared = None
    if shared_w13 is not None:
        shared = (expert_mlp(X, shared_w13, shared_w2, swiglu_limit=swiglu_limit,
                             act_dtype=act_dtype) if T else np.zeros((0, H)))
        y = y + shared
    if return_parts:
        return y, {"topk_weights": W, "topk_ids": ids, "expert_out": o, "shared": shared}
    return y


def fused_moe(x, logits, bias, w13, w2, shared_w13=None, shared_w2=None, *,
              return_parts=False, w13_bias=None, w2_bias=None, gated=True, swiglu_limit=None,
              gemm1_alpha=1.0, apply_router_weight_on_input=False, act_dtype="bf16", **cfg):
    """y [T, H] fp64 = routed experts (weighted, combined) + shared expert: the routing of
    ``select_experts`` followed by ``experts_combine`` (act rounded to bf16 unless
    ``act_dtype`` is None)."""
    W, ids = select_experts(logits, bias, **cfg)
    return experts_combine(x, W, ids, w13, w2, shared_w13, shared_w2,
                           return_parts=return_parts, w13_bias=w13_bias, w2_bias=w2_bias,
                           gated=gated, swiglu_limit=swiglu_limit, gemm1_alpha=gemm1_alpha,
                           apply_router_weight_on_input=apply_router_weight_on_input,
                           top_k=cfg["top_k"], act_dtype=act_dtype)


def fused_moe_rows(x_rows, logits_rows, bias, w13, w2, shared_w13=None, shared_w2=None,
                   **cfg):
    """The layer for a few chosen tokens (each token's output depends on that token only)."""
    return fused_moe(x_rows, logits_rows, bias, w13, w2, shared_w13, shared_w2, **cfg)


"""Shared test helpers: workload -> oracle arguments, margin-checked inputs, tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from mixture_experts_layer_05_gb300 import configs, inputs

# |y - y_ref| <= REL * |y_ref| + ABS_RMS * rms(y_ref), per element.
REL = 2e-2
ABS_RMS = 1e-2


def oracle_cfg(w: configs.MoEWorkload) -> dict:
    return dict(num_experts=w.num_experts, top_k=w.top_k, renormalize=w.renormalize,
                use_grouped_topk=w.use_grouped_topk, num_expert_group=w.num_expert_group,
                topk_group=w.topk_group, scoring_func=w.scoring_func,
                routed_scaling_factor=w.routed_scaling_factor)


def margin_fn(w: configs.MoEWorkload, bias):
    cfg = oracle_cfg(w)
    return lambda logits: oracle.decision_margins(logits, bias, **cfg)


def tokens(w: configs.MoEWorkload, T: int, bias, seed: int = 0):
    """x, logits with every routing decision at least LOGIT_GAP from a tie."""
    return inputs.make_tokens(w, T, seed=seed, margin_fn=margin_fn(w, bias))


def check_close(y, y_ref, what="y"):
    """The layer's acceptance bound, element by element."""
    y = np.asarray(y.float().cpu() if hasattr(y, "float") else y, dtype=np.float64)
    y_ref = np.asarray(y_ref, dtype=np.float64)
    assert y.shape == y_ref.shape, (y.shape, y_ref.shape)
    if y_ref.size == 0:
        return
    rms = float(np.sqrt(np.mean(y_ref ** 2)))
    bound = REL * np.abs(y_ref) + ABS_RMS * rms
    err = np.abs(y - y_ref)
    bad = err > bound
    assert not np.isnan(y).any(), f"{what}: NaN in output"
    assert not bad.any(), (
        f"{what}: {int(bad.sum())}/{bad.size} elements out of bound; worst excess "
        f"{float((err - bound).max()):.3e}, rms(y_ref)={rms:.3e}, "
        f"first at {np.argwhere(bad)[0].tolist()}")


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().numpy()


def gate_logit_error_bound(x, gate) -> np.ndarray:
    """[T, E] bound on |fp32 logit - exact logit| of the router GEMM: H * 2^-24 * sum |x||w|
    (fp32 accumulation of H bf16 products, each exact in fp32)."""
    H = x.shape[1]
    return (x.double().abs() @ gate.double().abs().T).numpy() * (H * 2.0 ** -24)


def key_tolerance(w, logit_err: float) -> float:
    """How far a decision gap (in the units of ``oracle.decision_margins``) can move when every
    logit of the row moves by at most ``logit_err``: a log-score gap by 2 err (softmax), a
    biased softmax key by 2 err per key, a sigmoid key by err / 4 per key; 4 err covers all,
    plus 1e-6 for the fp32 rounding of the scores themselves."""
    return 4.0 * logit_err + 1e-6


def check_routing_valid(w, ids, tw, logits, bias, logit_err, what="routing"):
    """The GPU's routing of rows computed from logits known only within ``logit_err`` (per
    row) of the exact ``logits``: ids distinct, their groups among the topk_group best within
    tolerance, every group that must survive honoured, ids in non-increasing key order and
    no better unchosen expert in a surviving group (within tolerance), and the weights equal
    to the routing rule applied to the chosen ids (softmax or sigmoid scores, renormalized,
    times the scaling factor) within the scores' error."""
    cfg = oracle_cfg(w)
    E, k = w.num_experts, w.top_k
    soft_log = w.scoring_func == "softmax" and bias is None
    for t in range(ids.shape[0]):
        err = float(np.max(logit_err[t]))
        tau = key_tolerance(w, err)
        _, _, info = oracle.route_token(logits[t], bias, **cfg)
        s, q = info["scores"], info["keys"]
        key = np.log(q) if soft_log else q
        row = [int(e) for e in ids[t]]
        assert len(set(row)) == k and all(0 <= e < E for e in row), (what, t, row)
        for a, b in zip(row[:-1], row[1:]):
            assert key[a] >= key[b] - tau, (what, t, "order", a, b)
        kept_possible = set(range(E))
        if w.use_grouped_topk:
            G, g = w.num_expert_group, w.topk_group
            size = E // G
            gs = info["group_scores"]
            gk = np.log(gs) if soft_log else gs
            ranked = sorted(gk, reverse=True)
            chosen_groups = {e // size for e in row}
            assert len(chosen_groups) <= g, (what, t, "groups", chosen_groups)
            for x in chosen_groups:
                assert gk[x] >= ranked[g - 1] - 2 * tau, (what, t, "group", x)
            first_dropped = ranked[g] if g < G else -np.inf
            must = {x for x in range(G) if gk[x] > first_dropped + 2 * tau}
            surviving = chosen_groups | must
            kept_possible = {e for e in range(E) if e // size in surviving}
        worst = min(key[e] for e in row)
        for e in kept_possible - set(row):
            assert key[e] <= worst + tau, (what, t, "missed", e)
        want = s[row] / (s[row].sum() if w.renormalize else 1.0) * w.routed_scaling_factor
        rtol = 4.0 * err + (E + 2 * k + 16) * 2.0 ** -24
        np.testing.assert_allclose(tw[t], want, rtol=rtol, atol=0, err_msg=f"{what} row {t}")

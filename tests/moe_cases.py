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

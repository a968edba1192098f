"""Pins of the CPU oracle against things other than itself (CPU only).

Each pin checks the oracle against hand-worked values, exhaustive enumeration, closed
forms or invariants of the FusedMoE forward (routing as in ``FusedMoE.select_experts``
on the vLLM ``fused_moe/layer`` page; shared expert and scaling as in
``DeepseekV2MoE`` on the sglang ``models/deepseek_v2.py`` page). The last block plants
mistakes in the oracle and checks that some pin catches each one.
"""
from __future__ import annotations

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch
from scipy.special import expit, softmax

import oracle
from oracle import moe_oracle as om

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "routing_hand_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def _cfg(**kw):
    base = dict(num_experts=8, top_k=2, renormalize=True, use_grouped_topk=False,
                num_expert_group=0, topk_group=0, scoring_func="softmax",
                routed_scaling_factor=1.0)
    base.update(kw)
    return base


# ------------------------------------------------------------------ hand-worked examples
def pin_hand_routing():
    for case in _golden()["cases"]:
        logits = np.log(np.array(case["exp_logits"], dtype=np.float64))
        bias = None if case["bias"] is None else np.array(case["bias"])
        w, ids = oracle.select_experts(logits[None], bias, **_cfg(**case["cfg"]))
        assert ids[0].tolist() == case["ids"], (case["name"], ids[0].tolist())
        np.testing.assert_allclose(w[0], case["weights"], rtol=1e-12, err_msg=case["name"])


def pin_hand_align():
    a = _golden()["align"]
    s, e, n = oracle.moe_align_block_size(np.array(a["topk_ids"]), a["num_experts"],
                                          a["block_size"])
    assert s.tolist() == a["sorted_token_ids"]
    assert e.tolist() == a["expert_ids"]
    assert n == a["num_tokens_post_padded"]


def pin_hand_expert_mlp():
    m = _golden()["expert_mlp"]
    x = np.array([[math.log(m["x_exp0"]), m["x1"]]])
    out = oracle.swiglu_mlp(x, np.array(m["w13"]), np.array(m["w2"]))
    np.testing.assert_allclose(out[0] / math.log(3.0), m["out_over_ln3"], rtol=1e-12)


def test_hand_routing():
    pin_hand_routing()


def test_hand_align():
    pin_hand_align()


def test_hand_expert_mlp():
    pin_hand_expert_mlp()


# ------------------------------------------------------------------ brute force
def _brute_topk(keys, candidates, k):
    return set(max(itertools.combinations(candidates, k), key=lambda c: sum(keys[i] for i in c)))


def _brute_grouped(s, q, G, g, k, with_bias):
    E = len(s)
    size = E // G

    def gscore(grp):
        mem = range(grp * size, (grp + 1) * size)
        if with_bias:
            return max(q[a] + q[b] for a, b in itertools.combinations(mem, 2))
        return max(s[m] for m in mem)

    gs = [gscore(x) for x in range(G)]
    groups = set(max(itertools.combinations(range(G), g), key=lambda c: sum(gs[x] for x in c)))
    elig = [e for e in range(E) if e // size in groups]
    return _brute_topk(q, elig, k), groups


def pin_bruteforce_ungrouped(n_cases=60):
    rng = np.random.default_rng(1)
    for c in range(n_cases):
        E = int(rng.choice([4, 6, 8, 12]))
        k = int(rng.integers(1, min(E, 4) + 1))
        logits = rng.normal(size=E)
        bias = rng.normal(scale=0.1, size=E) if c % 2 else None
        w, ids, _ = oracle.route_token(logits, bias, **_cfg(num_experts=E, top_k=k))
        s = softmax(logits)
        q = s + bias if bias is not None else s
        assert set(ids.tolist()) == _brute_topk(q, range(E), k)
        assert all(q[a] > q[b] for a, b in zip(ids[:-1], ids[1:]))   # descending keys


def pin_bruteforce_grouped(n_cases=80):
    rng = np.random.default_rng(2)
    for c in range(n_cases):
        G = int(rng.choice([2, 3, 4]))
        size = int(rng.choice([2, 3, 4]))
        E = G * size
        g = int(rng.integers(1, G + 1))
        k = int(rng.integers(1, min(g * size, 4) + 1))
        sig = c % 2 == 1
        logits = rng.normal(size=E)
        bias = rng.normal(scale=0.1, size=E) if sig else None
        cfg = _cfg(num_experts=E, top_k=k, use_grouped_topk=True, num_expert_group=G,
                   topk_group=g, scoring_func="sigmoid" if sig else "softmax")
        w, ids, info = oracle.route_token(logits, bias, **cfg)
        s = expit(logits) if sig else softmax(logits)
        q = s + bias if bias is not None else s
        want_ids, want_groups = _brute_grouped(s, q, G, g, k, bias is not None)
        assert set(ids.tolist()) == want_ids, (c, ids, want_ids)
        assert set(info["kept_groups"]) == want_groups
        assert all(q[a] > q[b] for a, b in zip(ids[:-1], ids[1:]))


def test_bruteforce_ungrouped():
    pin_bruteforce_ungrouped()


def test_bruteforce_grouped():
    pin_bruteforce_grouped()


# ------------------------------------------------------------------ closed forms, special cases
def pin_renormalized_softmax_closed_form():
    rng = np.random.default_rng(3)
    for _ in range(30):
        logits = rng.normal(size=16)
        w, ids, _ = oracle.route_token(logits, None, **_cfg(num_experts=16, top_k=4))
        np.testing.assert_allclose(w, softmax(logits[ids]), rtol=1e-12)


def pin_sigmoid_weights_unbiased():
    rng = np.random.default_rng(4)
    for _ in range(30):
        logits = rng.normal(size=32)
        bias = rng.normal(scale=0.3, size=32)
        cfg = _cfg(num_experts=32, top_k=6, use_grouped_topk=True, num_expert_group=4,
                   topk_group=2, scoring_func="sigmoid", routed_scaling_factor=2.5)
        w, ids, _ = oracle.route_token(logits, bias, **cfg)
        want = expit(logits[ids])
        np.testing.assert_allclose(w, 2.5 * want / want.sum(), rtol=1e-12)


def pin_grouped_reduces_to_ungrouped():
    rng = np.random.default_rng(5)
    for _ in range(30):
        logits = rng.normal(size=12)
        bias = rng.normal(scale=0.1, size=12)
        for b in (None, bias):
            plain = oracle.route_token(logits, b, **_cfg(num_experts=12, top_k=3))
            for G, g in ((1, 1), (3, 3), (4, 4)):
                grp = oracle.route_token(logits, b, **_cfg(num_experts=12, top_k=3,
                                                           use_grouped_topk=True,
                                                           num_expert_group=G, topk_group=g))
                assert grp[1].tolist() == plain[1].tolist()
                np.testing.assert_allclose(grp[0], plain[0], rtol=1e-15)


def pin_routing_invariants():
    rng = np.random.default_rng(6)
    logits = rng.normal(size=(64, 32))
    bias = rng.normal(scale=0.1, size=32)
    for sig in (False, True):
        for renorm in (False, True):
            cfg = _cfg(num_experts=32, top_k=5, renormalize=renorm, use_grouped_topk=True,
                       num_expert_group=8, topk_group=3,
                       scoring_func="sigmoid" if sig else "softmax",
                       routed_scaling_factor=3.0)
            b = bias if sig else None
            W, ids = oracle.select_experts(logits, b, **cfg)
            for t in range(64):
                assert len(set(ids[t].tolist())) == 5
                assert len({e // 4 for e in ids[t]}) <= 3            # inside kept groups
                if renorm:
                    assert abs(W[t].sum() - 3.0) < 1e-12
                elif not sig:
                    assert W[t].sum() <= 3.0 + 1e-12


def test_closed_forms():
    pin_renormalized_softmax_closed_form()
    pin_sigmoid_weights_unbiased()


def test_grouped_special_cases():
    pin_grouped_reduces_to_ungrouped()


def test_routing_invariants():
    pin_routing_invariants()


# ------------------------------------------------------------------ align
def pin_align_bruteforce():
    rng = np.random.default_rng(7)
    for case in range(40):
        E = int(rng.integers(1, 20))
        k = int(rng.integers(1, min(E, 6) + 1))
        T = int(rng.integers(0, 50))
        bs = int(rng.choice([1, 2, 4, 16, 64]))
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), int)
        s, ex, n = oracle.moe_align_block_size(ids, E, bs)
        flat = ids.reshape(-1)
        # expected by a comparison sort on (expert, flat index)
        order = sorted(range(flat.size), key=lambda f: (flat[f], f))
        got = [f for f in s.tolist() if f != flat.size]
        assert got == order
        assert n == len(s) and n % bs == 0
        assert (s == flat.size).sum() == n - flat.size
        for p, f in enumerate(s.tolist()):
            if f != flat.size:
                assert flat[f] == ex[p // bs]
        assert all(a <= b for a, b in zip(ex[:-1], ex[1:]))
        counts = np.bincount(flat, minlength=E) if flat.size else np.zeros(E, int)
        for e in range(E):
            assert (ex == e).sum() * bs == -(-counts[e] // bs) * bs


def test_align_bruteforce():
    pin_align_bruteforce()


# ------------------------------------------------------------------ expert math
def _rand_layer(rng, E, H, I, Is=0):
    w13 = rng.normal(scale=0.3, size=(E, 2 * I, H))
    w2 = rng.normal(scale=0.3, size=(E, H, I))
    sw13 = rng.normal(scale=0.3, size=(2 * Is, H)) if Is else None
    sw2 = rng.normal(scale=0.3, size=(H, Is)) if Is else None
    return w13, w2, sw13, sw2


def pin_dense_swiglu_single_expert():
    """E=1, top_k=1, renormalize: the layer is one dense SwiGLU MLP (torch fp64)."""
    rng = np.random.default_rng(8)
    x = rng.normal(size=(7, 12))
    w13, w2, _, _ = _rand_layer(rng, 1, 12, 5)
    y = oracle.fused_moe(x, rng.normal(size=(7, 1)), None, w13, w2,
                         act_dtype=None, **_cfg(num_experts=1, top_k=1))
    X, W13, W2 = (torch.tensor(a) for a in (x, w13[0], w2[0]))
    ref = torch.nn.functional.silu(X @ W13[:5].T) * (X @ W13[5:].T) @ W2.T
    np.testing.assert_allclose(y, ref.numpy(), rtol=1e-12, atol=1e-14)


def pin_identity_like_experts():
    """w1 = a_e*Id, w3 = b_e*Id, w2 = Id: y = sum_j w_j silu(a x) (b x) elementwise."""
    rng = np.random.default_rng(9)
    E, n, T = 4, 6, 5
    a = rng.uniform(0.5, 2.0, E)
    b = rng.uniform(-2.0, 2.0, E)
    w13 = np.stack([np.vstack([a[e] * np.eye(n), b[e] * np.eye(n)]) for e in range(E)])
    w2 = np.stack([np.eye(n)] * E)
    x = rng.normal(size=(T, n))
    logits = rng.normal(size=(T, E))
    cfg = _cfg(num_experts=E, top_k=2)
    y = oracle.fused_moe(x, logits, None, w13, w2, act_dtype=None, **cfg)
    W, ids = oracle.select_experts(logits, None, **cfg)
    for t in range(T):
        for i in range(n):
            want = 0.0
            for j in range(2):
                e = ids[t, j]
                z = a[e] * x[t, i]
                want += W[t, j] * (z / (1.0 + math.exp(-z))) * (b[e] * x[t, i])
            assert abs(y[t, i] - want) <= 1e-12 * (1 + abs(want))


def pin_scaling_and_shared():
    """rsf scales the routed part only; zero w2 leaves exactly the shared expert."""
    rng = np.random.default_rng(10)
    E, H, I, Is, T = 6, 8, 4, 8, 9
    w13, w2, sw13, sw2 = _rand_layer(rng, E, H, I, Is)
    x = rng.normal(size=(T, H))
    logits = rng.normal(size=(T, E))
    c1 = _cfg(num_experts=E, top_k=2, routed_scaling_factor=1.0)
    c2 = _cfg(num_experts=E, top_k=2, routed_scaling_factor=2.5)
    y1 = oracle.fused_moe(x, logits, None, w13, w2, sw13, sw2, act_dtype=None, **c1)
    y2 = oracle.fused_moe(x, logits, None, w13, w2, sw13, sw2, act_dtype=None, **c2)
    shared = torch.nn.functional.silu(torch.tensor(x) @ torch.tensor(sw13[:Is]).T) \
        * (torch.tensor(x) @ torch.tensor(sw13[Is:]).T) @ torch.tensor(sw2).T
    shared = shared.numpy()
    np.testing.assert_allclose(y2 - shared, 2.5 * (y1 - shared), rtol=1e-10, atol=1e-12)
    y0 = oracle.fused_moe(x, logits, None, w13, np.zeros_like(w2), sw13, sw2, act_dtype=None, **c1)
    np.testing.assert_allclose(y0, shared, rtol=1e-12, atol=1e-14)


def pin_expert_relabeling():
    """Relabelling experts (weights, logits columns, bias together) leaves y unchanged."""
    rng = np.random.default_rng(11)
    E, H, I, T = 8, 8, 4, 6
    w13, w2, _, _ = _rand_layer(rng, E, H, I)
    x = rng.normal(size=(T, H))
    logits = rng.normal(size=(T, E))
    bias = rng.normal(scale=0.1, size=E)
    cfg = _cfg(num_experts=E, top_k=3, use_grouped_topk=True, num_expert_group=4,
               topk_group=2, scoring_func="sigmoid")
    # permute groups as blocks and experts inside each group
    gperm = rng.permutation(4)
    perm = np.concatenate([g * 2 + rng.permutation(2) for g in gperm])
    y = oracle.fused_moe(x, logits, bias, w13, w2, **cfg)
    yp = oracle.fused_moe(x, logits[:, perm], bias[perm], w13[perm], w2[perm], **cfg)
    np.testing.assert_allclose(yp, y, rtol=1e-12, atol=1e-14)


def test_dense_swiglu_single_expert():
    pin_dense_swiglu_single_expert()


def test_identity_like_experts():
    pin_identity_like_experts()


def test_scaling_and_shared():
    pin_scaling_and_shared()


def test_expert_relabeling():
    pin_expert_relabeling()


def test_empty_batch():
    W, ids = oracle.select_experts(np.zeros((0, 8)), None, **_cfg())
    assert W.shape == (0, 2) and ids.shape == (0, 2)
    s, e, n = oracle.moe_align_block_size(ids, 8, 16)
    assert n == 0 and s.size == 0 and e.size == 0
    y = oracle.fused_moe(np.zeros((0, 4)), np.zeros((0, 8)), None, np.zeros((8, 4, 4)),
                         np.zeros((8, 4, 2)), **_cfg())
    assert y.shape == (0, 4)


# ------------------------------------------------------------------ bf16 act
BF16 = os.path.join(os.path.dirname(__file__), "golden", "bf16_round_examples.json")


def _rne_bits(a):
    """bfloat16 rounding by bit surgery on the fp64 pattern (a second, independent way):
    keep the top 7 of the 52 stored fraction bits, rounding the dropped 45 to nearest, ties
    to even, by adding 2^44 - 1 plus the lowest kept bit; for normal fp32-range values."""
    a = np.asarray(a, dtype=np.float64)
    bits = a.view(np.uint64).copy()
    lsb = (bits >> np.uint64(45)) & np.uint64(1)
    bits = bits + np.uint64((1 << 44) - 1) + lsb
    bits &= ~np.uint64((1 << 45) - 1)
    return bits.view(np.float64)


def pin_round_bf16():
    """round_bf16 on hand-worked values (ties, subnormals), against bit surgery on random
    fp64 values, and against torch's float32 -> bfloat16 conversion on fp32 values."""
    with open(BF16) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        got = float(oracle.round_bf16(math.ldexp(*c["x"])))
        assert got == math.ldexp(*c["want"]), c
    rng = np.random.default_rng(13)
    v = rng.normal(size=4000) * np.exp2(rng.integers(-100, 100, size=4000))
    np.testing.assert_array_equal(oracle.round_bf16(v), _rne_bits(v))
    f32 = (rng.normal(size=4000) * 3.0).astype(np.float32)
    f32[:64] = (np.arange(64, dtype=np.float32) + 0.5) * np.float32(2.0 ** -7) + 1  # ties
    want = torch.from_numpy(f32).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(oracle.round_bf16(f32.astype(np.float64)), want)


def pin_layer_rounds_act_only():
    """Identity-like experts (w1 = a Id, w3 = b Id, w2 = Id) and a shared expert: the layer
    equals sum_j w_j bf16(silu(a x) (b x)) + bf16(silu(c x) (d x)), the act rounded and
    nothing else (gate, up and output exact)."""
    rng = np.random.default_rng(14)
    E, n, T = 4, 6, 7
    a = rng.uniform(0.5, 2.0, E)
    b = rng.uniform(-2.0, 2.0, E)
    w13 = np.stack([np.vstack([a[e] * np.eye(n), b[e] * np.eye(n)]) for e in range(E)])
    w2 = np.stack([np.eye(n)] * E)
    c, d = 1.3, -0.7
    sw13, sw2 = np.vstack([c * np.eye(n), d * np.eye(n)]), np.eye(n)
    x = rng.normal(size=(T, n)) * 3.0
    logits = rng.normal(size=(T, E))
    cfg = _cfg(num_experts=E, top_k=2)
    y = oracle.fused_moe(x, logits, None, w13, w2, sw13, sw2, **cfg)
    W, ids = oracle.select_experts(logits, None, **cfg)
    for t in range(T):
        want = _rne_bits(om.silu(c * x[t]) * (d * x[t]))
        for j in range(2):
            e = ids[t, j]
            want = want + W[t, j] * _rne_bits(om.silu(a[e] * x[t]) * (b[e] * x[t]))
        np.testing.assert_allclose(y[t], want, rtol=1e-13, atol=1e-15)
    # and the act really is rounded: the exact layer differs
    y_exact = oracle.fused_moe(x, logits, None, w13, w2, sw13, sw2, act_dtype=None, **cfg)
    assert np.abs(y - y_exact).max() > 1e-4


def test_round_bf16():
    pin_round_bf16()


def test_layer_rounds_act_only():
    pin_layer_rounds_act_only()


# ------------------------------------------------------------------ decision margins
MARGINS = os.path.join(os.path.dirname(__file__), "golden", "margin_hand_examples.json")


def pin_hand_margins():
    """decision_margins on hand-worked rows, one per kind of decision: a softmax top-k gap
    (logit units), a biased sigmoid key gap, a kept/dropped group gap under each group rule."""
    with open(MARGINS) as f:
        cases = json.load(f)["cases"]
    for case in cases:
        logits = np.log(np.array(case["exp_logits"], dtype=np.float64))[None]
        bias = None if case["bias"] is None else np.array(case["bias"])
        m = oracle.decision_margins(logits, bias, **_cfg(**case["cfg"]))
        assert abs(m[0] - case["margin"]) <= 1e-9, (case["name"], m[0], case["margin"])


def _decision_plain(logits, bias, cfg):
    """(kept groups, ordered ids) of one row by plain sorting, written apart from the oracle:
    scores by scipy, group scores (largest score, or the two largest biased keys), the
    topk_group best groups, then the top_k best eligible keys in descending order."""
    E, k = cfg["num_experts"], cfg["top_k"]
    s = expit(logits) if cfg["scoring_func"] == "sigmoid" else softmax(logits)
    q = s + bias if bias is not None else s
    elig = list(range(E))
    kept = None
    if cfg["use_grouped_topk"]:
        G, g = cfg["num_expert_group"], cfg["topk_group"]
        size = E // G
        gs = []
        for x in range(G):
            mem = q[x * size:(x + 1) * size] if bias is not None else s[x * size:(x + 1) * size]
            top = sorted(mem, reverse=True)
            gs.append(top[0] + top[1] if bias is not None else top[0])
        kept = frozenset(sorted(range(G), key=lambda x: (-gs[x], x))[:g])
        elig = [e for e in elig if e // size in kept]
    return kept, tuple(sorted(elig, key=lambda e: (-q[e], e))[:k])


def _perturbed(logits, bias, cfg, e, delta):
    """Move the selection key of expert e by delta: in logit units for softmax without a bias
    (shift the logit), in key units otherwise (shift the bias entry, or, for unbiased sigmoid
    scores, the logit that moves the score by delta). None if the score would leave (0, 1)."""
    lg = logits.copy()
    if bias is not None:
        b = bias.copy()
        b[e] += delta
        return lg, b
    if cfg["scoring_func"] == "softmax":
        lg[e] += delta
        return lg, None
    s = expit(lg[e]) + delta
    if not 0.0 < s < 1.0:
        return None
    lg[e] = math.log(s / (1.0 - s))
    return lg, None


def _brute_margin(logits, bias, cfg, span=4.0, steps=48):
    """Smallest move of one selection key that changes the decision, by bisection over each
    expert and direction (a key moved one way changes its rank monotonically)."""
    base = _decision_plain(logits, bias, cfg)
    best = math.inf
    for e in range(cfg["num_experts"]):
        for sign in (1.0, -1.0):
            def changed(d):
                p = _perturbed(logits, bias, cfg, e, sign * d)
                return p is not None and _decision_plain(p[0], p[1], cfg) != base
            hi = span
            if not changed(hi):
                # unbiased sigmoid: the score range caps the move; shrink to the largest valid
                while hi > 1e-6 and _perturbed(logits, bias, cfg, e, sign * hi) is None:
                    hi /= 2
                if not changed(hi):
                    continue
            lo = 0.0
            for _ in range(steps):
                mid = 0.5 * (lo + hi)
                if changed(mid):
                    hi = mid
                else:
                    lo = mid
            best = min(best, hi)
    return best


def pin_margins_bruteforce(n_cases=36):
    """decision_margins equals the smallest single-key move that changes which groups
    survive or which experts are chosen (in which order), on small random rows of every
    routing branch."""
    rng = np.random.default_rng(12)
    kinds = ["softmax", "softmax_bias", "softmax_grouped", "sigmoid_grouped_bias",
             "sigmoid_grouped"]
    for c in range(n_cases):
        kind = kinds[c % len(kinds)]
        G = int(rng.choice([2, 3, 4]))
        size = int(rng.choice([2, 3]))
        E = G * size
        grouped = "grouped" in kind
        g = int(rng.integers(1, G + 1)) if grouped else 0
        k = int(rng.integers(1, min((g * size) if grouped else E, 3) + 1))
        cfg = _cfg(num_experts=E, top_k=k, use_grouped_topk=grouped,
                   num_expert_group=G if grouped else 0, topk_group=g,
                   scoring_func="sigmoid" if kind.startswith("sigmoid") else "softmax")
        logits = rng.normal(size=E)
        bias = rng.normal(scale=0.1, size=E) if "bias" in kind else None
        m = oracle.decision_margins(logits[None], bias, **cfg)[0]
        want = _brute_margin(logits, bias, cfg)
        assert abs(m - want) <= 1e-9 * max(1.0, want), (c, kind, m, want)


def test_hand_margins():
    pin_hand_margins()


def test_margins_bruteforce():
    pin_margins_bruteforce()


# ------------------------------------------------------------------ planted mistakes
ALL_PINS = [pin_hand_routing, pin_hand_align, pin_hand_expert_mlp, pin_bruteforce_ungrouped,
            pin_bruteforce_grouped, pin_renormalized_softmax_closed_form,
            pin_sigmoid_weights_unbiased, pin_grouped_reduces_to_ungrouped,
            pin_routing_invariants, pin_align_bruteforce, pin_dense_swiglu_single_expert,
            pin_identity_like_experts, pin_scaling_and_shared, pin_expert_relabeling,
            pin_hand_margins, pin_margins_bruteforce, pin_round_bf16,
            pin_layer_rounds_act_only]


def _caught(monkeypatch, name, fn):
    monkeypatch.setattr(om, name, fn)
    caught = []
    for pin in ALL_PINS:
        try:
            pin()
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    return caught


def _swapped_gate_up(h, w13_e, w2_e):
    W13 = np.asarray(w13_e, dtype=np.float64)
    I = W13.shape[0] // 2
    return (om.silu(np.atleast_2d(h) @ W13[I:].T) * (np.atleast_2d(h) @ W13[:I].T)) \
        @ np.asarray(w2_e, dtype=np.float64).T


def _max_group_rule(scores_g, keys_g, with_bias):
    return float(np.max(keys_g))


def _biased_weights(logits_row, bias, **cfg):
    w, ids, info = _orig_route(logits_row, bias, **cfg)
    w = np.array([info["keys"][e] for e in ids])
    if cfg["renormalize"]:
        w = w / w.sum()
    return w * cfg.get("routed_scaling_factor", 1.0), ids, info


def _no_renorm(logits_row, bias, **cfg):
    return _orig_route(logits_row, bias, **dict(cfg, renormalize=False))


def _unstable_align(topk_ids, num_experts, block_size):
    s, e, n = _orig_align(topk_ids, num_experts, block_size)
    s = s.copy()
    for b in range(len(e)):                      # reverse each block: order no longer stable
        blk = s[b * block_size:(b + 1) * block_size]
        real = blk[blk != np.asarray(topk_ids).size]
        blk[:real.size] = real[::-1]
    return s, e, n


_orig_route = om.route_token
_orig_align = om.moe_align_block_size


@pytest.mark.parametrize("name,fn", [
    ("swiglu_mlp", _swapped_gate_up),
    ("group_score", _max_group_rule),
    ("route_token", _biased_weights),
    ("route_token", _no_renorm),
    ("moe_align_block_size", _unstable_align),
])
def test_planted_mistake_is_caught(monkeypatch, name, fn):
    # the package re-exports, so patch both the module and the package names
    monkeypatch.setattr(oracle, name, fn, raising=False)
    caught = _caught(monkeypatch, name, fn)
    assert caught, f"no pin caught a planted mistake in {name}"


def _margins_mutant(log_units=True, group_gap=True, extra=1):
    """A copy of decision_margins with one step changed: gaps in score units instead of
    logit units, the group gap left out, or the key order checked over top_k + extra."""
    def margins(logits, bias, **cfg):
        L = np.asarray(logits, dtype=np.float64)
        out = np.full(L.shape[0], np.inf)
        soft_log = log_units and cfg.get("scoring_func", "softmax") == "softmax" and bias is None
        for t in range(L.shape[0]):
            _, _, info = om.route_token(L[t], bias, **cfg)
            q = np.log(info["keys"]) if soft_log else info["keys"]
            m = np.inf
            if group_gap and info["kept_groups"] is not None:
                gsc = np.log(info["group_scores"]) if soft_log else info["group_scores"]
                order = om._rank_desc(gsc, range(len(gsc)))
                nk = len(info["kept_groups"])
                if nk < len(order):
                    m = min(m, gsc[order[nk - 1]] - gsc[order[nk]])
            order = om._rank_desc(q, info["eligible"])[: cfg["top_k"] + extra]
            for a, b in zip(order[:-1], order[1:]):
                m = min(m, q[a] - q[b])
            out[t] = m
        return out
    return margins


@pytest.mark.parametrize("mutant", [dict(log_units=False), dict(group_gap=False),
                                    dict(extra=2), dict(extra=0)],
                         ids=["score_units", "no_group_gap", "k_plus_2", "k_only"])
def test_planted_margin_mistake_is_caught(monkeypatch, mutant):
    fn = _margins_mutant(**mutant)
    monkeypatch.setattr(oracle, "decision_margins", fn, raising=False)
    caught = _caught(monkeypatch, "decision_margins", fn)
    assert caught, f"no pin caught the planted margin mistake {mutant}"


def test_margin_mutant_copy_is_faithful(monkeypatch):
    """The unmutated copy passes the margin pins (so each caught mutant is caught for its
    change, not for a difference in the copy)."""
    fn = _margins_mutant()
    monkeypatch.setattr(oracle, "decision_margins", fn, raising=False)
    monkeypatch.setattr(om, "decision_margins", fn)
    pin_hand_margins()
    pin_margins_bruteforce()



def _round_half_away(a):
    a = np.asarray(a, dtype=np.float64)
    _, e = np.frexp(a)
    e = np.maximum(e, -125)
    m = np.ldexp(a, 8 - e)
    return np.ldexp(np.sign(m) * np.floor(np.abs(m) + 0.5), e - 8)


def _expert_act_unrounded(h, w13_e, w2_e, **kw):
    kw.pop("act_dtype", None)
    return _orig_expert(h, w13_e, w2_e, **kw)


def _expert_rounds_gate_up(h, w13_e, w2_e, act_dtype=None, **kw):
    if act_dtype is None:
        return _orig_expert(h, w13_e, w2_e, **kw)
    W13 = om.round_bf16(np.atleast_2d(om._f64(h)) @ om._f64(w13_e).T)   # z rounded as well
    I = W13.shape[1] // 2
    act = om.round_bf16(om.silu(W13[:, :I]) * W13[:, I:])
    return act @ om._f64(w2_e).T


_orig_expert = om.expert_mlp


@pytest.mark.parametrize("name,fn", [("round_bf16", _round_half_away),
                                     ("expert_mlp", _expert_act_unrounded),
                                     ("expert_mlp", _expert_rounds_gate_up)],
                         ids=["half_away", "act_not_rounded", "gate_up_rounded"])
def test_planted_bf16_mistake_is_caught(monkeypatch, name, fn):
    monkeypatch.setattr(oracle, name, fn, raising=False)
    caught = _caught(monkeypatch, name, fn)
    assert caught, f"no pin caught the planted bf16 mistake in {name}"

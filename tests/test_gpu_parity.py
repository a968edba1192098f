"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on the GPU.

Routing (topk_ids) and align (sorted_token_ids, expert_ids, num_tokens_post_padded)
must match bit for bit; topk_weights within the fp32 rounding bound of a softmax over
E terms; the layer output within |y - y_ref| <= 2e-2 |y_ref| + 1e-2 rms(y_ref).
Inputs are seeded; every routing decision is at least 1e-3 from a tie.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_layer_05_gb300 import binding, configs, inputs
from tests.moe_cases import (check_close, check_routing_valid, gate_logit_error_bound,
                              oracle_cfg, tokens)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def weight_rtol(w) -> float:
    """fp32 softmax/sigmoid + renormalize vs fp64: (E + 2k + 16) units of 2^-24."""
    return (w.num_experts + 2 * w.top_k + 16) * 2.0 ** -24


def _small(w, **kw):
    return configs.shrink(w, **kw)


SMALL = {
    "tiny": configs.TINY,
    "mixtral": _small(configs.MIXTRAL, hidden_size=256, intermediate_size=384),
    "dsv2": _small(configs.DSV2, hidden_size=384, intermediate_size=128,
                   shared_intermediate_size=256),
    "dsv3": _small(configs.DSV3, hidden_size=256, intermediate_size=256,
                   shared_intermediate_size=256),
    "skew": _small(configs.SKEW, hidden_size=512, intermediate_size=128,
                   shared_intermediate_size=128),
}


def _routing(w, T, seed=0):
    wts = inputs.make_weights(_small(w, hidden_size=128, intermediate_size=128,
                                     shared_intermediate_size=0), seed)
    bias = wts["bias"]
    _, logits = tokens(w, T, bias, seed)
    return logits, bias


# ------------------------------------------------------------------ moe_topk
@pytest.mark.parametrize("name", list(configs.WORKLOADS))
@pytest.mark.parametrize("T", [1, 37, 1000])
def test_topk_bitexact(cuda_lib, name, T):
    w = configs.WORKLOADS[name]
    logits, bias = _routing(w, T)
    cfg = binding.config_from_workload(w)
    tw = torch.empty(T, w.top_k, dtype=torch.float32, device=DEV)
    ti = torch.empty(T, w.top_k, dtype=torch.int32, device=DEV)
    binding.moe_topk(cfg, logits.to(DEV), None if bias is None else bias.to(DEV), tw, ti)
    torch.cuda.synchronize()
    W, ids = oracle.select_experts(logits, bias, **oracle_cfg(w))
    assert np.array_equal(ti.cpu().numpy(), ids), "topk_ids differ"
    np.testing.assert_allclose(tw.cpu().numpy(), W, rtol=weight_rtol(w), atol=0)


@pytest.mark.parametrize("variant", ["softmax_bias_ungrouped", "sigmoid_grouped_nobias",
                                     "softmax_grouped_bias_renorm"])
def test_topk_other_branches(cuda_lib, variant):
    """The fused_topk_bias branch and the two other bias/scoring combinations."""
    base = dict(num_experts=64, top_k=4, renormalize=True)
    if variant == "softmax_bias_ungrouped":
        w = _small(configs.DSV3, scoring_func="softmax", use_grouped_topk=False, **base)
    elif variant == "sigmoid_grouped_nobias":
        w = _small(configs.DSV3, has_bias=False, num_expert_group=8, topk_group=2, **base)
    else:
        w = _small(configs.DSV2, has_bias=True, bias_std=0.01, num_expert_group=4, topk_group=2,
                   routed_scaling_factor=1.5, **base)
    logits, bias = _routing(w, 300)
    cfg = binding.config_from_workload(w)
    tw = torch.empty(300, 4, dtype=torch.float32, device=DEV)
    ti = torch.empty(300, 4, dtype=torch.int32, device=DEV)
    binding.moe_topk(cfg, logits.to(DEV), None if bias is None else bias.to(DEV), tw, ti)
    W, ids = oracle.select_experts(logits, bias, **oracle_cfg(w))
    assert np.array_equal(ti.cpu().numpy(), ids)
    np.testing.assert_allclose(tw.cpu().numpy(), W, rtol=weight_rtol(w), atol=0)


# ------------------------------------------------------------------ moe_align_block_size
def _align_gpu(ids_np, E, bs):
    T, k = ids_np.shape
    n = T * k
    max_sorted = n + E * (bs - 1)
    ids = torch.from_numpy(ids_np.astype(np.int32)).to(DEV)
    srt = torch.full((max_sorted,), -7, dtype=torch.int32, device=DEV)
    eid = torch.full((max_sorted // bs + 1,), -7, dtype=torch.int32, device=DEV)
    npp = torch.zeros(1, dtype=torch.int32, device=DEV)
    ws = binding.alloc_workspace(binding.moe_align_block_size_workspace_size(T, k, E))
    binding.moe_align_block_size(ids, E, bs, srt, eid, npp, ws)
    assert binding.moe_get_device_status(ws) == binding.OK
    return srt.cpu().numpy(), eid.cpu().numpy(), int(npp.item())


@pytest.mark.parametrize("T,k,E,bs,skew", [
    (1, 1, 1, 1, False), (1, 2, 8, 128, False), (5, 3, 7, 16, False), (16, 2, 8, 128, False),
    (1000, 8, 256, 64, False), (3000, 6, 160, 128, False), (4097, 2, 8, 32, True),
    (20000, 8, 256, 128, True), (700, 4, 1024, 16, False)])
def test_align_bitexact(cuda_lib, T, k, E, bs, skew):
    rng = np.random.default_rng(T * 31 + E)
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
        ids = np.stack([rng.choice(E, size=k, replace=False, p=p) for _ in range(T)])
    else:
        ids = np.stack([rng.permutation(E)[:k] for _ in range(T)])
    srt, eid, npp = _align_gpu(ids, E, bs)
    s_ref, e_ref, n_ref = oracle.moe_align_block_size(ids, E, bs)
    assert npp == n_ref
    assert np.array_equal(srt[:npp], s_ref)
    assert np.array_equal(eid[:npp // bs], e_ref)
    assert (eid[npp // bs:] == -1).all()


# ------------------------------------------------------------------ the layer, small shapes
def _layer(w, wts, T):
    cfg = binding.config_from_workload(w)
    d = {k: (None if v is None else v.to(DEV)) for k, v in wts.items()}
    return binding.FusedMoE(cfg, d["w13"], d["w2"], d["bias"], d["shared_w13"], d["shared_w2"],
                            max_tokens=max(T, 1)), d


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("T", [1, 2, 3, 4, 5, 16])
def test_forward_small_batch_align_bitexact(cuda_lib, name, T):
    """The one-CTA routing + align of small batches (a one-warp align for at most 32 rows,
    the per-warp slices above that) writes exactly the oracle's sorted_token_ids,
    expert_ids and num_tokens_post_padded into the forward's workspace."""
    w = SMALL[name]
    wts = inputs.make_weights(w, 0)
    x, logits = tokens(w, T, wts["bias"], 3)
    layer, _ = _layer(w, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    bs = binding.moe_forward_block_size(layer.cfg, T)
    y_ref, parts = oracle.fused_moe(x, logits, wts["bias"], wts["w13"], wts["w2"],
                                    wts["shared_w13"], wts["shared_w2"], return_parts=True,
                                    **oracle_cfg(w))
    s_ref, e_ref, n_ref = oracle.moe_align_block_size(parts["topk_ids"], w.num_experts, bs)
    lay = binding.moe_forward_workspace_layout(layer.cfg, T)
    ws = layer.workspace
    npp = int(ws[lay.num_tokens_post_padded:lay.num_tokens_post_padded + 4].view(torch.int32))
    assert npp == n_ref
    srt = ws[lay.sorted_token_ids:lay.sorted_token_ids + npp * 4].view(torch.int32).cpu().numpy()
    assert np.array_equal(srt, s_ref)
    max_blocks = (T * w.top_k + w.num_experts * (bs - 1)) // bs + 1
    eid = ws[lay.expert_ids:lay.expert_ids + max_blocks * 4].view(torch.int32).cpu().numpy()
    assert np.array_equal(eid[:npp // bs], e_ref)
    assert (eid[npp // bs:] == -1).all()
    check_close(y, y_ref, f"{name} T={T}")


def _routing_from_ws(layer, T, k):
    lay = binding.moe_forward_workspace_layout(layer.cfg, T)
    ws = layer.workspace
    ids = ws[lay.topk_ids:lay.topk_ids + T * k * 4].view(torch.int32).cpu().numpy()
    tw = ws[lay.topk_weights:lay.topk_weights + T * k * 4].view(torch.float32).cpu().numpy()
    return ids.reshape(T, k), tw.reshape(T, k)


@pytest.mark.parametrize("name", list(SMALL))
@pytest.mark.parametrize("T", [1, 16, 203])
def test_forward_small(cuda_lib, name, T):
    w = SMALL[name]
    wts = inputs.make_weights(w, 0)
    x, logits = tokens(w, T, wts["bias"])
    layer, d = _layer(w, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    y_ref, parts = oracle.fused_moe(x, logits, wts["bias"], wts["w13"], wts["w2"],
                                    wts["shared_w13"], wts["shared_w2"], return_parts=True,
                                    **oracle_cfg(w))
    ids, tw = _routing_from_ws(layer, T, w.top_k)
    assert np.array_equal(ids, parts["topk_ids"])
    np.testing.assert_allclose(tw, parts["topk_weights"], rtol=weight_rtol(w), atol=0)
    check_close(y, y_ref, f"{name} T={T}")


def test_forward_deterministic(cuda_lib):
    w = SMALL["dsv3"]
    wts = inputs.make_weights(w, 0)
    x, logits = tokens(w, 300, wts["bias"])
    layer, _ = _layer(w, wts, 300)
    y1 = layer(x.to(DEV), logits.to(DEV)).clone()
    y2 = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert torch.equal(y1, y2)
    assert layer.device_status() == binding.OK


def test_forward_empty_and_single_expert(cuda_lib):
    # empty batch: a no-op that leaves the output untouched
    w = SMALL["mixtral"]
    wts = inputs.make_weights(w, 0)
    layer, _ = _layer(w, wts, 4)
    out = torch.full((0, w.hidden_size), 1.0, dtype=torch.bfloat16, device=DEV)
    layer(torch.empty(0, w.hidden_size, dtype=torch.bfloat16, device=DEV),
          torch.empty(0, w.num_experts, device=DEV), out=out)
    # E = 1, k = 1: a dense SwiGLU MLP
    w1 = _small(configs.MIXTRAL, num_experts=1, top_k=1, hidden_size=256, intermediate_size=256)
    wts1 = inputs.make_weights(w1, 0)
    x, logits = tokens(w1, 130, None)
    layer1, _ = _layer(w1, wts1, 130)
    y = layer1(x.to(DEV), logits.to(DEV))
    y_ref = oracle.fused_moe(x, logits, None, wts1["w13"], wts1["w2"], **oracle_cfg(w1))
    check_close(y, y_ref, "E=1 k=1")
    assert layer1.device_status() == binding.OK


# ------------------------------------------------------------------ full sizes, sampled
class _Experts:
    """Expert slices copied to the host on demand (the oracle indexes w[e])."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, e):
        return self.t[e].cpu()


# every token count of the four layer workloads above decode sizes (decode sizes are checked
# token by token below)
FULL = [("mixtral", 128), ("mixtral", 1024), ("mixtral", 4096), ("dsv2", 64), ("dsv2", 512),
        ("dsv2", 4096), ("dsv3", 32), ("dsv3", 256), ("dsv3", 2048), ("dsv3", 8192),
        ("skew", 16384)]


def block_edge_tokens(sorted_ids, npp, bs, n, k):
    """Tokens owning the first and the last real row of every row block (so every active
    expert, every row-block position a GEMM tile starts or ends on, and the last row blocks
    that the w2 stream-K tail splits all appear)."""
    toks = set()
    for b in range(npp // bs):
        blk = sorted_ids[b * bs:(b + 1) * bs]
        real = blk[blk < n]
        if real.size:
            toks.add(int(real[0]) // k)
            toks.add(int(real[-1]) // k)
    return sorted(toks)


@pytest.mark.parametrize("name,T", FULL)
def test_forward_full_size_sampled(cuda_lib, name, T):
    """Full shapes: routing of every token bit-exact, the forward's own align
    (sorted_token_ids, expert_ids, num_tokens_post_padded in its workspace) equal to the
    oracle's at full size, and the output of the tokens at both ends of every row block
    against the oracle (all active experts; at least 256 tokens where the batch has them)."""
    w = configs.WORKLOADS[name]
    torch.cuda.empty_cache()
    wts = inputs.make_weights(w, 0, device=DEV)
    bias_cpu = None if wts["bias"] is None else wts["bias"].cpu()
    x, logits = tokens(w, T, bias_cpu)
    cfg = binding.config_from_workload(w)
    layer = binding.FusedMoE(cfg, wts["w13"], wts["w2"], wts["bias"], wts["shared_w13"],
                             wts["shared_w2"], max_tokens=T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    W, ids_ref = oracle.select_experts(logits, bias_cpu, **oracle_cfg(w))
    ids, tw = _routing_from_ws(layer, T, w.top_k)
    assert np.array_equal(ids, ids_ref)
    np.testing.assert_allclose(tw, W, rtol=weight_rtol(w), atol=0)
    # the forward's align at full size
    bs = binding.moe_forward_block_size(cfg, T)
    s_ref, e_ref, n_ref = oracle.moe_align_block_size(ids_ref, w.num_experts, bs)
    lay = binding.moe_forward_workspace_layout(cfg, T)
    ws = layer.workspace
    npp = int(ws[lay.num_tokens_post_padded:lay.num_tokens_post_padded + 4].view(torch.int32))
    assert npp == n_ref
    srt = ws[lay.sorted_token_ids:lay.sorted_token_ids + npp * 4].view(torch.int32).cpu().numpy()
    assert np.array_equal(srt, s_ref)
    eid = ws[lay.expert_ids:lay.expert_ids + (npp // bs) * 4].view(torch.int32).cpu().numpy()
    assert np.array_equal(eid, e_ref)
    rows = block_edge_tokens(srt, npp, bs, T * w.top_k, w.top_k)
    if len(rows) < min(T, 256):                     # top up with random tokens
        rest = np.setdiff1d(np.arange(T), rows)
        extra = np.random.default_rng(T).choice(rest, size=min(T, 256) - len(rows),
                                                replace=False)
        rows = sorted(set(rows) | set(extra.tolist()))
    assert set(np.unique(ids_ref[rows])) == set(np.unique(ids_ref))   # every active expert
    y_ref = oracle.fused_moe_rows(x[rows], logits[rows], bias_cpu, _Experts(wts["w13"]),
                                  _Experts(wts["w2"]),
                                  None if wts["shared_w13"] is None else wts["shared_w13"].cpu(),
                                  None if wts["shared_w2"] is None else wts["shared_w2"].cpu(),
                                  **oracle_cfg(w))
    check_close(y[rows], y_ref, f"{name} T={T} ({len(rows)} block-edge tokens)")
    del layer, wts
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ decode sizes (split-K)
SPLIT = _small(configs.MIXTRAL, num_experts=4, hidden_size=1024, intermediate_size=1024)
SPLIT_SHARED = _small(configs.DSV3, num_experts=16, num_expert_group=4, topk_group=2, top_k=4,
                      hidden_size=1024, intermediate_size=512, shared_intermediate_size=1024)


@pytest.mark.parametrize("w", [SPLIT, SPLIT_SHARED], ids=["routed", "routed+shared"])
@pytest.mark.parametrize("T", [1, 3, 17, 64])
def test_forward_split_k(cuda_lib, w, T):
    """Shapes whose few tiles make moe_forward cut K into several splits."""
    wts = inputs.make_weights(w, 0)
    x, logits = tokens(w, T, wts["bias"])
    layer, _ = _layer(w, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    y_ref = oracle.fused_moe(x, logits, wts["bias"], wts["w13"], wts["w2"], wts["shared_w13"],
                             wts["shared_w2"], **oracle_cfg(w))
    check_close(y, y_ref, f"split-K T={T}")
    y2 = layer(x.to(DEV), logits.to(DEV))
    assert torch.equal(y, y2)                       # fixed reduction order: deterministic


@pytest.mark.parametrize("name,T", [("mixtral", 1), ("mixtral", 16), ("dsv2", 1), ("dsv3", 1),
                                    ("dsv3", 8)])
def test_forward_decode_full_shapes(cuda_lib, name, T):
    """Full shapes at decode token counts, every token against the oracle."""
    w = configs.WORKLOADS[name]
    torch.cuda.empty_cache()
    wts = inputs.make_weights(w, 0, device=DEV)
    bias_cpu = None if wts["bias"] is None else wts["bias"].cpu()
    x, logits = tokens(w, T, bias_cpu)
    layer = binding.FusedMoE(binding.config_from_workload(w), wts["w13"], wts["w2"], wts["bias"],
                             wts["shared_w13"], wts["shared_w2"], max_tokens=T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    y_ref = oracle.fused_moe(x, logits, bias_cpu, _Experts(wts["w13"]), _Experts(wts["w2"]),
                             None if wts["shared_w13"] is None else wts["shared_w13"].cpu(),
                             None if wts["shared_w2"] is None else wts["shared_w2"].cpu(),
                             **oracle_cfg(w))
    check_close(y, y_ref, f"{name} T={T}")
    del layer, wts
    torch.cuda.empty_cache()


# ------------------------------------------------------------------ CTA-pair GEMMs (large T)
PAIR_ROUTED = _small(configs.MIXTRAL, num_experts=4, hidden_size=512, intermediate_size=384)
PAIR_SHARED = _small(configs.DSV3, num_experts=8, top_k=4, num_expert_group=4, topk_group=2,
                     hidden_size=256, intermediate_size=256, shared_intermediate_size=384)


@pytest.mark.parametrize("w,T", [(PAIR_ROUTED, 4096), (PAIR_ROUTED, 4501), (PAIR_SHARED, 4100),
                                 (PAIR_SHARED, 300)],
                         ids=["routed-4096", "routed-4501", "shared-4100", "shared-300"])
def test_forward_pair_mode(cuda_lib, w, T):
    """Experts averaging >= 128 rows: the token-N GEMMs on CTA pairs (cta_group::2), row
    blocks of 256 whose MMA width follows their real rows; the forward's align must match
    the oracle's at block size 256."""
    cfg = binding.config_from_workload(w)
    assert binding.moe_forward_block_size(cfg, T) == 256
    wts = inputs.make_weights(w, 0)
    x, logits = tokens(w, T, wts["bias"])
    layer, _ = _layer(w, wts, T)
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    y_ref, parts = oracle.fused_moe(x, logits, wts["bias"], wts["w13"], wts["w2"],
                                    wts["shared_w13"], wts["shared_w2"], return_parts=True,
                                    **oracle_cfg(w))
    lay = binding.moe_forward_workspace_layout(cfg, T)
    ws = layer.workspace
    npp = int(ws[lay.num_tokens_post_padded:lay.num_tokens_post_padded + 4].view(torch.int32))
    s_ref, e_ref, n_ref = oracle.moe_align_block_size(parts["topk_ids"], w.num_experts, 256)
    assert npp == n_ref
    srt = ws[lay.sorted_token_ids:lay.sorted_token_ids + npp * 4].view(torch.int32).cpu().numpy()
    assert np.array_equal(srt, s_ref)
    check_close(y, y_ref, f"pair T={T}")
    y2 = layer(x.to(DEV), logits.to(DEV))
    assert torch.equal(y, y2)


# ------------------------------------------------------------------ failure detection
def test_bounded_wait_times_out_and_context_survives(cuda_lib):
    """A wait that nothing completes gives up, reports GBMOE_ERR_TIMEOUT, and the
    context stays usable for the next forward."""
    ws = binding.alloc_workspace(256)
    binding.moe_selftest_bounded_wait(ws, 2000)          # 2 ms limit
    assert binding.moe_get_device_status(ws) == binding.ERR_TIMEOUT
    assert binding.moe_get_device_status(ws) == binding.OK   # the read resets the word
    w = SMALL["tiny"]
    wts = inputs.make_weights(w, 0)
    x, logits = tokens(w, 16, wts["bias"])
    layer, _ = _layer(w, wts, 16)
    y = layer(x.to(DEV), logits.to(DEV))
    y_ref = oracle.fused_moe(x, logits, None, wts["w13"], wts["w2"], **oracle_cfg(w))
    check_close(y, y_ref, "after timeout")
    assert layer.device_status() == binding.OK


def test_launch_count_matches_path(cuda_lib):
    """moe_forward_num_launches: fused small-batch path, gather, split-K reduce."""
    cfg = binding.config_from_workload(configs.MIXTRAL)
    n1 = binding.moe_forward_num_launches(cfg, 1)      # fused route+align+copy, w13, reduce, w2, combine
    n4096 = binding.moe_forward_num_launches(cfg, 4096)  # topk, 3 align, gather, w13, w2, combine
    assert n4096 == 8
    assert 4 <= n1 <= 6
    assert binding.moe_forward_num_launches(cfg, 0) == 0


def test_host_pipeline_matches_direct_calls(cuda_lib):
    """Overlapped host batches give exactly the outputs of one-at-a-time forwards."""
    w = SMALL["dsv3"]
    wts = inputs.make_weights(w, 0)
    layer, _ = _layer(w, wts, 300)
    batches = [tokens(w, T, wts["bias"], seed=s) for s, T in ((1, 300), (2, 17), (3, 255))]
    ys = [torch.empty(x.shape, dtype=x.dtype).pin_memory() for x, _ in batches]
    pipe = binding.HostPipeline(layer, 300)
    pipe.run([x.pin_memory() for x, _ in batches], [lg.pin_memory() for _, lg in batches], ys)
    torch.cuda.synchronize()
    for (x, lg), y in zip(batches, ys):
        assert torch.equal(y, layer(x.to(DEV), lg.to(DEV)).cpu())
    assert layer.device_status() == binding.OK


@pytest.mark.parametrize("name,T", [("dsv3", 1), ("dsv3", 300), ("mixtral", 16)])
def test_forward_cuda_graph_replay(cuda_lib, name, T):
    """moe_forward enqueues no host synchronisation or allocation: captured into a CUDA
    graph and replayed it gives the eager result bit for bit."""
    w = SMALL[name]
    wts = inputs.make_weights(w, 0)
    x, logits = tokens(w, T, wts["bias"])
    layer, _ = _layer(w, wts, T)
    xd, ld = x.to(DEV), logits.to(DEV)
    eager = layer(xd, ld).clone()
    out = torch.empty_like(xd)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        layer(xd, ld, out=out)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager)
    assert layer.device_status() == binding.OK


@pytest.mark.parametrize("name,T", [("dsv3", 1), ("dsv3", 4), ("mixtral", 1), ("split", 1),
                                    ("split_shared", 5), ("fused2", 1), ("dsv2", 16)])
def test_graph_replay_follows_new_routing(cuda_lib, name, T):
    """One captured decode forward replayed on batches that route to different experts:
    every replay must equal an eager forward and the oracle. The decode w2 GEMM reads the
    routing's expert blocks before it waits on the kernel in front of it (safe only because
    each GEMM lets its dependents start after its own wait); stale expert ids from the
    previous replay would show up here as a mismatch."""
    w = {"split": SPLIT, "split_shared": SPLIT_SHARED, "fused2": FUSED2}.get(name) or SMALL[name]
    wts = inputs.make_weights(w, 0)
    layer, _ = _layer(w, wts, T)
    batches = [tokens(w, T, wts["bias"], seed=s) for s in range(11, 15)]
    xd = batches[0][0].to(DEV)
    ld = batches[0][1].to(DEV)
    out = torch.empty_like(xd)
    layer(xd, ld, out=out)                          # eager call before the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cs):
        layer(xd, ld, out=out)
    seen = []
    for x, lg in batches:
        xd.copy_(x)
        ld.copy_(lg)
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        ids, _ = _routing_from_ws(layer, T, w.top_k)
        seen.append(ids.copy())
        eager = layer(x.to(DEV), lg.to(DEV))
        torch.cuda.synchronize()
        assert torch.equal(got, eager)
        y_ref, parts = oracle.fused_moe(x, lg, wts["bias"], wts["w13"], wts["w2"],
                                        wts["shared_w13"], wts["shared_w2"], return_parts=True,
                                        **oracle_cfg(w))
        assert np.array_equal(ids, parts["topk_ids"])
        check_close(got, y_ref, f"{name} T={T} replay")
    assert any(not np.array_equal(seen[0], s_) for s_ in seen[1:])   # the routing changed
    assert layer.device_status() == binding.OK


# ------------------------------------------------------------------ layer variants
VARIANTS = {
    "bias": dict(bias=True),
    "clamp_alpha": dict(swiglu_limit=0.25, gemm1_alpha=1.7),
    "bias_clamp": dict(bias=True, swiglu_limit=0.25),
    "non_gated": dict(gated=False),
    "non_gated_bias": dict(gated=False, bias=True),
    "weight_on_input": dict(apply_router_weight_on_input=True),
}
# two-way split-K of the first GEMM: its last split finishes the activation in the GEMM
FUSED2 = _small(configs.MIXTRAL, num_experts=8, hidden_size=512, intermediate_size=1024)
# experts averaging >= 128 rows: the token-N CTA-pair GEMMs (w1 too: I % 256 == 0)
TN = _small(configs.DSV3, num_experts=16, top_k=4, num_expert_group=4, topk_group=2,
            hidden_size=512, intermediate_size=256, shared_intermediate_size=256)
VARIANT_SHAPES = {
    "tn": TN,                     # token-N CTA-pair GEMMs, shared expert included
    "dsv3": SMALL["dsv3"],        # grouped sigmoid routing + shared expert
    "split": SPLIT,               # decode shapes: split-K and the split reduce kernel
    "fused2": FUSED2,             # decode shapes: split-K reduced inside the GEMM
}


def test_two_way_split_reduces_in_the_gemm(cuda_lib):
    """The two-split decode shape launches no separate reduce kernel: routing + align with
    the row copy, w13, w2, combine."""
    cfg = binding.config_from_workload(FUSED2)
    assert binding.moe_forward_num_launches(cfg, 1) == 4
    assert binding.moe_forward_num_launches(binding.config_from_workload(SPLIT), 1) == 5


# w2 with more tiles than SMs and a short last round: the stream-K tail splits those tiles
TAIL = _small(configs.MIXTRAL, hidden_size=2048, intermediate_size=512)


@pytest.mark.parametrize("use_bias", [False, True], ids=["plain", "bias"])
@pytest.mark.parametrize("T", [1024, 1100])
def test_forward_w2_stream_k_tail(cuda_lib, use_bias, T):
    """Prefill shapes whose w2 tiles leave a last round of at most half the SMs: those tiles
    run as K ranges summed by the last range (checked against the oracle and for run-to-run
    determinism)."""
    w = TAIL
    wts = inputs.make_weights(w, 0)
    x, logits = tokens(w, T, None)
    _, ids = oracle.select_experts(logits, None, **oracle_cfg(w))
    blocks = sum((c + 127) // 128 for c in np.bincount(ids.reshape(-1), minlength=w.num_experts))
    tiles = blocks * (w.hidden_size // 256)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert tiles >= sms and 0 < tiles % sms <= sms // 2      # the shape takes the tail path
    extra = inputs.make_expert_extras(w, 0) if use_bias else {}
    b13 = extra.get("w13_bias")
    b2 = extra.get("w2_bias")
    cfg = binding.config_from_workload(w)
    dv = lambda t: None if t is None else t.to(DEV)
    layer = binding.FusedMoE(cfg, wts["w13"].to(DEV), wts["w2"].to(DEV), max_tokens=T,
                             w13_bias=dv(b13), w2_bias=dv(b2))
    y = layer(x.to(DEV), logits.to(DEV)).clone()
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    rows = sorted({0, T - 1, *np.random.default_rng(T).choice(T, size=30, replace=False).tolist()})
    y_ref = oracle.fused_moe(x[rows], logits[rows], None, wts["w13"], wts["w2"],
                             w13_bias=b13, w2_bias=b2, **oracle_cfg(w))
    check_close(y[rows], y_ref, f"w2 tail T={T}")
    assert torch.equal(y, layer(x.to(DEV), logits.to(DEV)))


@pytest.mark.parametrize("vname", list(VARIANTS))
@pytest.mark.parametrize("sname,T", [("tn", 600), ("dsv3", 203), ("split", 1), ("split", 17),
                                     ("fused2", 1), ("fused2", 5)])
def test_forward_variants(cuda_lib, vname, sname, T):
    v = dict(VARIANTS[vname])
    w = VARIANT_SHAPES[sname]
    if sname == "tn":
        assert binding.moe_forward_block_size(binding.config_from_workload(w), T) == 256
    gated = v.pop("gated", True)
    use_bias = v.pop("bias", False)
    if not gated:
        w = configs.shrink(w, shared_intermediate_size=0)  # a shared expert needs gating
    wts = inputs.make_weights(w, 0)
    extra = inputs.make_expert_extras(w, 0, gated=gated)
    w13 = wts["w13"] if gated else extra["w1"]
    b13 = extra["w13_bias"] if use_bias else None
    b2 = extra["w2_bias"] if use_bias else None
    x, logits = tokens(w, T, wts["bias"])
    cfg = binding.config_from_workload(w, is_act_and_mul=int(gated), **v)
    dv = lambda t: None if t is None else t.to(DEV)
    layer = binding.FusedMoE(cfg, w13.to(DEV), wts["w2"].to(DEV), dv(wts["bias"]),
                             dv(wts["shared_w13"]), dv(wts["shared_w2"]), max_tokens=T,
                             w13_bias=dv(b13), w2_bias=dv(b2))
    y = layer(x.to(DEV), logits.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    y_ref = oracle.fused_moe(x, logits, wts["bias"], w13, wts["w2"], wts["shared_w13"],
                             wts["shared_w2"], w13_bias=b13, w2_bias=b2, gated=gated,
                             **v, **oracle_cfg(w))
    check_close(y, y_ref, f"{vname} {sname} T={T}")


def test_stage_events_eager_and_captured(cuda_lib):
    """moe_forward_events times stages eagerly and inside a CUDA graph replay."""
    w = SMALL["mixtral"]
    wts = inputs.make_weights(w, 0)
    x, logits = tokens(w, 64, None)
    layer, _ = _layer(w, wts, 64)
    xd, ld = x.to(DEV), logits.to(DEV)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(binding.NUM_STAGE_EVENTS)]
    layer(xd, ld, events=ev)
    torch.cuda.synchronize()
    assert all(ev[i].elapsed_time(ev[i + 1]) >= 0.0 for i in range(4))
    out = torch.empty_like(xd)
    gev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    for e in gev:
        e.record()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        layer(xd, ld, out=out, events=[None, gev[0], gev[1], None, None])
    g.replay()
    torch.cuda.synchronize()
    assert gev[0].elapsed_time(gev[1]) > 0.0
    assert layer.device_status() == binding.OK


# ------------------------------------------------------------------ router GEMM
def _gate(w, seed=0):
    """Gate weight ~N(0, 1/sqrt(H)) so that the logits of N(0, 1) hidden states are ~N(0, 1)."""
    return inputs.normal((w.num_experts, w.hidden_size), w.hidden_size ** -0.5,
                         inputs.tensor_seed(w.name, "gate", seed), torch.bfloat16)


@pytest.mark.parametrize("E,H,T", [(8, 4096, 1), (8, 4096, 300), (160, 5120, 64),
                                   (256, 7168, 129), (256, 7168, 1)])
def test_router_logits(cuda_lib, E, H, T):
    x = inputs.normal((T, H), 1.0, 1, torch.bfloat16)
    wg = inputs.normal((E, H), H ** -0.5, 2, torch.bfloat16)
    out = torch.full((T, E), float("nan"), device=DEV)
    binding.moe_router_logits(x.to(DEV), wg.to(DEV), out)
    torch.cuda.synchronize()
    ref = oracle.router_logits(x, wg)
    # fp32 accumulation over H products: |error| <= H * 2^-24 * sum |x| |w| (rounded up)
    bound = (x.double().abs() @ wg.double().abs().T).numpy() * (H * 2.0 ** -24) + 1e-30
    err = np.abs(out.cpu().numpy().astype(np.float64) - ref)
    assert (err <= bound).all(), float((err / bound).max())


@pytest.mark.parametrize("name,T", [("dsv3", 1), ("dsv3", 5), ("dsv3", 16), ("dsv3", 77),
                                    ("mixtral", 1), ("mixtral", 16), ("dsv2", 3), ("dsv2", 300),
                                    ("skew", 200), ("tiny", 16)])
def test_forward_from_gate_weight(cuda_lib, name, T):
    """moe_forward_ex with the gate weight: router GEMM (split-K at decode), routing,
    experts. Rows whose oracle decision margin exceeds 1e-4 (far above the fp32 logit
    error) must route exactly like the oracle and match its output. Closer rows must hold
    a valid routing for logits within the GEMM's fp32 error bound (groups, order, no better
    expert left out, weights), and their output must match the oracle's experts and combine
    run on the GPU's own ids and weights."""
    w = SMALL[name]
    wts = inputs.make_weights(w, 0)
    wg = _gate(w)
    x = inputs.normal((T, w.hidden_size), 1.0, 5, torch.bfloat16)
    layer, d = _layer(w, wts, T)
    y = layer(x.to(DEV), gate_weight=wg.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    logits = oracle.router_logits(x, wg)
    err = gate_logit_error_bound(x, wg)
    margins = oracle.decision_margins(logits, wts["bias"], **oracle_cfg(w))
    safe = margins >= 1e-4
    ids, tw = _routing_from_ws(layer, T, w.top_k)
    check_routing_valid(w, ids, tw, logits, wts["bias"], err, f"{name} T={T} gate")
    y_ref, parts = oracle.fused_moe(x, logits, wts["bias"], wts["w13"], wts["w2"],
                                    wts["shared_w13"], wts["shared_w2"], return_parts=True,
                                    **oracle_cfg(w))
    assert np.array_equal(ids[safe], parts["topk_ids"][safe])
    check_close(y.cpu()[torch.from_numpy(safe)], y_ref[safe], f"{name} T={T} gate")
    close = np.flatnonzero(~safe).tolist()
    if close:
        y_own = oracle.experts_combine(x[close], tw[close], ids[close], wts["w13"], wts["w2"],
                                       wts["shared_w13"], wts["shared_w2"])
        check_close(y[close], y_own, f"{name} T={T} gate, close rows on the GPU's routing")
    assert T == 1 or safe.mean() > 0.9


@pytest.mark.parametrize("T", [16, 64])
def test_forward_from_gate_weight_near_ties(cuda_lib, T):
    """Gate weights whose logits are built to land near routing ties: many rows fall under
    the 1e-4 margin, and every one of them must still hold a valid routing and the output
    of its own routing (T = 16: logits inside the routing launch; T = 64: the router
    GEMM)."""
    w = SMALL["dsv3"]
    wts = inputs.make_weights(w, 0)
    x = inputs.normal((T, w.hidden_size), 1.0, 6, torch.bfloat16)
    base = _gate(w)
    # twin experts 2e, 2e + 1: the same correction bias, and gate rows that differ in one
    # bf16 unit of one column, so their keys differ by about |x[:, 0] w| 2^-7 / 4 (every row
    # of this batch lands under the 1e-4 margin, most under 1e-5)
    wts["bias"][1::2] = wts["bias"][0::2]
    wg = base.clone()
    wg[1::2] = base[0::2]
    wg[1::2, 0] = (base[0::2, 0].float() * (1 + 2.0 ** -7)).to(torch.bfloat16)
    layer, _ = _layer(w, wts, T)
    y = layer(x.to(DEV), gate_weight=wg.to(DEV))
    torch.cuda.synchronize()
    assert layer.device_status() == binding.OK
    logits = oracle.router_logits(x, wg)
    margins = oracle.decision_margins(logits, wts["bias"], **oracle_cfg(w))
    assert (margins < 1e-4).sum() >= T // 2            # the construction produced close rows
    ids, tw = _routing_from_ws(layer, T, w.top_k)
    check_routing_valid(w, ids, tw, logits, wts["bias"], gate_logit_error_bound(x, wg),
                        "near ties")
    y_own = oracle.experts_combine(x, tw, ids, wts["w13"], wts["w2"], wts["shared_w13"],
                                   wts["shared_w2"])
    check_close(y, y_own, "near ties, on the GPU's routing")


@pytest.mark.parametrize("name", ["dsv3", "mixtral", "dsv2"])
def test_gate_weight_adds_no_launch_for_small_batches(cuda_lib, name):
    """With the gate weight, batches of at most 16 tokens compute the router logits inside
    their routing launch: the same number of kernels as from logits; larger ones add the
    router GEMM."""
    cfg = binding.config_from_workload(configs.WORKLOADS[name])
    for T in (1, 4, 16):
        assert binding.moe_forward_num_launches_ex(cfg, T, True) == \
            binding.moe_forward_num_launches(cfg, T)
    assert binding.moe_forward_num_launches_ex(cfg, 200, True) == \
        binding.moe_forward_num_launches(cfg, 200) + 1


@pytest.mark.parametrize("T", [1, 8])
def test_gate_weight_graph_replay(cuda_lib, T):
    """The fused router's arrival counter returns to zero after every forward: a captured
    forward from the gate weight replayed on new tokens equals eager calls."""
    w = SMALL["dsv3"]
    wts = inputs.make_weights(w, 0)
    wg = _gate(w).to(DEV)
    layer, _ = _layer(w, wts, T)
    xs = [inputs.normal((T, w.hidden_size), 1.0, 40 + s, torch.bfloat16) for s in range(3)]
    xd = xs[0].to(DEV)
    out = torch.empty_like(xd)
    layer(xd, gate_weight=wg, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    cs = torch.cuda.Stream()
    cs.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=cs):
        layer(xd, gate_weight=wg, out=out)
    for x in xs:
        xd.copy_(x)
        g.replay()
        torch.cuda.synchronize()
        got = out.clone()
        eager = layer(x.to(DEV), gate_weight=wg)
        torch.cuda.synchronize()
        assert torch.equal(got, eager)
    assert layer.device_status() == binding.OK

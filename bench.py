"""Benchmark of the FusedMoE layer forward on GB300 (one JSON line on stdout).

Default workload: the DeepSeek-V3-shaped MoE layer (H=7168, I=2048, E=256 routed experts,
top_k=8, sigmoid scores + e_score_correction_bias, grouped top-k 8/4, renormalize,
routed_scaling_factor 2.5, one shared expert of I=2048) at T=8192 tokens, the largest
workload that fits one GPU: bf16 weights ~N(0, 0.02) (22.5 GB, far larger than L2, so no
flush is needed between steps), activations ~N(0, 1), fp32 router logits ~N(0, 1), bias
~N(0, 0.1), seed = rank.

A step is one full forward through the C ABI (routing, align, gather, w13 GEMM +
SiLU*mul, w2 GEMM, combine) on inputs resident in HBM. W warm-up steps, then K
timed steps between a barrier + synchronize on both sides, CUDA events on the
launching stream, max over ranks; ``value`` = tokens of all ranks / that time.
``eager`` times the same steps launched without a graph; ``e2e`` is the same metric with
pinned host inputs copied in and the output copied out inside each timed step.
``--impl reference`` times the CPU oracle instead, on a bounded token sample per step.
``--sweep T1,T2,...`` prints one line per token count instead (the skewed-routing sweep).

Multi-GPU (torchrun): independent data-parallel replicas, each rank its own batch
and a full copy of the weights; no collective on the data path (weak scaling).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused-MoE layer tokens/s; TFLOP/s & HBM GB/s as % of GB300 roofline"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------- host-side logic
def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def rank_seed(rank: int) -> int:
    """Each replica draws its own batch (weights are the same on every rank)."""
    return int(rank)


def reduce_max(value: float, device=None) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(tokens_per_rank: int, world: int, ms_max: float) -> float:
    return tokens_per_rank * world / (ms_max / 1e3)


def layer_work(w, T: int, n_active: int, quant: str = "none") -> dict:
    """Algorithmic flops and bytes of one forward (no padding rows).

    bf16: weights, gathered rows and act 2 bytes per element. fp8 (w8a8, block 128):
    weights, gathered rows and act 1 byte per element plus one fp32 scale per 128 x 128
    weight block and per 128-element activation group. nvfp4 (w4a4, block 16): weights,
    gathered rows and act half a byte per element plus one e4m3 byte per 16 elements.
    """
    H, I, k, E, Is = w.hidden_size, w.intermediate_size, w.top_k, w.num_experts, \
        w.shared_intermediate_size
    wb = {"fp8": 1.0 + 4.0 / (128 * 128), "nvfp4": 0.5 + 1.0 / 16}.get(quant, 2.0)
    ab = {"fp8": 1.0 + 4.0 / 128, "nvfp4": 0.5 + 1.0 / 16}.get(quant, 2.0)
    flops_w13 = 4.0 * T * k * H * I + 4.0 * T * H * Is
    flops_w2 = 2.0 * T * k * H * I + 2.0 * T * H * Is
    w13_bytes = (n_active * 2 * I * H + 2 * Is * H) * wb
    w2_bytes = (n_active * H * I + H * Is) * wb
    act_bytes = (T * k * I + T * Is) * ab
    bytes_total = (w13_bytes + w2_bytes + T * H * 2 * 2 + T * E * 4 + T * k * 8
                   + 2 * act_bytes)
    return {"flops": flops_w13 + flops_w2, "flops_w13": flops_w13, "flops_w2": flops_w2,
            "bytes": float(bytes_total),
            "bytes_w13": float(w13_bytes + T * k * H * ab + act_bytes),
            "bytes_w2": float(w2_bytes + act_bytes + T * k * H * 4)}


KERNEL_SOURCES = {"gemm.cu": ("gemm.cu", "tc.cuh", "common.cuh", "kernels.h"),
                  "gemm_tn.cu": ("gemm_tn.cu", "tc.cuh", "common.cuh", "kernels.h"),
                  "gemm_fp8.cu": ("gemm_fp8.cu", "tc.cuh", "fp8.cuh", "common.cuh", "kernels.h"),
                  "gemm_fp4.cu": ("gemm_fp4.cu", "tc.cuh", "fp4.cuh", "common.cuh", "kernels.h")}

# tensor peak of each path's contraction dtype: the measured bf16 peak times the nominal
# dense ratio (e4m3 4.5 / 2.25, fp4 13.5 / 2.25 PFLOP/s)
QUANT_PEAK_RATIO = {"none": 1.0, "fp8": 2.0, "nvfp4": 6.0}
QUANT_DTYPE = {"none": "bf16", "fp8": "e4m3", "nvfp4": "e2m1"}
QUANT_TAG = {"none": "", "fp8": " w8a8 fp8 block-128", "nvfp4": " w4a4 nvfp4 block-16"}


def source_digest(source: str) -> str:
    """sha1 over the code of a GEMM translation unit and the headers it compiles in, with
    comments and blank lines dropped (a comment-only edit keeps the digest)."""
    import hashlib
    import re
    h = hashlib.sha1()
    for name in KERNEL_SOURCES.get(source, (source,)):
        with open(os.path.join(ROOT, "mixture_experts_layer_05_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(code.encode())
    return h.hexdigest()


def kernel_traffic(kernel: str, workload: str, tokens: int, source: str = "gemm.cu"):
    """DRAM bytes per launch of `kernel` from a committed ncu summary, if it was captured on
    this workload with the current kernel source (source_digest of csrc/<source> and its
    headers); else None.

    A summary states it on a line `traffic: <kernel> <workload> <tokens> <bytes> <digest>`.
    """
    import glob
    try:
        sha = source_digest(source)
    except OSError:
        return None
    for path in sorted(glob.glob(os.path.join(ROOT, "profiles", "*.md"))):
        with open(path) as f:
            for line in f:
                p = line.split()
                if len(p) == 6 and p[0] == "traffic:" and p[1] == kernel and p[2] == workload \
                        and p[3] == str(tokens) and p[5] == sha:
                    return float(p[4])
    return None


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict:
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    p = [x.strip() for x in line.split(",")]
                    if len(p) < 10:
                        continue
                    try:
                        ts = time.mktime(time.strptime(p[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                        ts += float("0." + p[0].split(".")[1]) if "." in p[0] else 0.0
                        rows.append((ts, float(p[2]), float(p[3]), p[6:10]))
                    except (ValueError, IndexError):
                        continue
        except OSError:
            pass
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        used = inside or rows[-20:]
        if not used:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in used for i, v in enumerate(r[3])
                          if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in used),
                "sm_max_mhz": max(r[2] for r in used), "reasons": reasons,
                "samples": len(used), "in_timed_region": bool(inside)}


# ---------------------------------------------------------------- arms
L2_BYTES = 129 * 2 ** 20          # GB300 L2


def routing_stats(layer, cfg, w, T) -> dict:
    """Routing facts of the last forward, read from its workspace: distinct experts, padded
    row count of the align, the rows the expert GEMMs' MMAs cover (the padded rows for
    128-row blocks; each 256-row block's real rows rounded up to 16 for the token-N GEMMs),
    and the per-expert load (rows routed to each expert) relative to the mean."""
    import torch
    from mixture_experts_layer_05_gb300 import binding
    lay = binding.moe_forward_workspace_layout(cfg, T)
    ids = layer.workspace[lay.topk_ids:lay.topk_ids + T * w.top_k * 4].view(torch.int32)
    cnt = torch.bincount(ids.long(), minlength=w.num_experts).cpu()
    npp = int(layer.workspace[lay.num_tokens_post_padded:lay.num_tokens_post_padded + 4]
              .view(torch.int32).item())
    bs = binding.moe_forward_block_size(cfg, T)
    if bs == 256:
        mma_rows = int(sum(c // 256 * 256 + (-(-(c % 256) // 16) * 16) for c in cnt.tolist()))
    else:
        mma_rows = npp
    mean = T * w.top_k / w.num_experts
    rel = cnt.double() / mean
    edges = [0.0, 0.5, 1.0, 2.0, 4.0, 8.0, 16.0]
    hist = {}
    for a, b in zip(edges, edges[1:] + [float("inf")]):
        n = int(((rel > a) & (rel <= b)).sum()) if a > 0 else int((rel <= b).sum())
        hist[f"({a:g},{b:g}]" if a > 0 else f"[0,{b:g}]"] = n
    return {"active_experts": int((cnt > 0).sum()), "rows_post_padded": npp,
            "block_rows": bs, "mma_rows": mma_rows,
            "mma_padding_frac": round(mma_rows / (T * w.top_k) - 1.0, 4),
            "max_load_over_mean": round(float(rel.max()), 3),
            "top8_loads": sorted(cnt.tolist(), reverse=True)[:8],
            "load_over_mean_hist": hist}


def roofline_of(work: dict, t_s: float, peaks: dict, peak_src: str, quant: str, kname: str,
                which: str = "w13") -> dict:
    """Roofline of one kernel (its algorithmic flops and bytes over its duration): bound by
    the larger of flops / tensor peak and bytes / HBM peak, both at the burst peak (a kernel
    inside a short step); the sustained tensor fraction is reported beside it. The tensor
    peak is that of the path's own contraction dtype (QUANT_PEAK_RATIO)."""
    ratio = QUANT_PEAK_RATIO[quant]
    burst = peaks["bf16_tflops"] * ratio
    sustained = peaks["bf16_tflops_sustained"] * ratio
    flops, byts = work[f"flops_{which}"], work[f"bytes_{which}"]
    t_tc, t_hbm = flops / (burst * 1e12), byts / (peaks["hbm_gbs"] * 1e9)
    tflops = flops / t_s / 1e12
    gbs = byts / t_s / 1e9
    src = f"{peak_src} bf16 burst (best of 10 cuBLAS GEMMs)" + (
        f" x {ratio:g}, the nominal {QUANT_DTYPE[quant]}/bf16 dense ratio" if ratio != 1.0 else "")
    if t_tc >= t_hbm:
        roof = {"kernel": kname, "bound": "tensor", "achieved": round(tflops, 1),
                "peak": round(burst, 1), "unit": "TFLOP/s", "frac": round(tflops / burst, 4),
                "peak_source": src}
    else:
        roof = {"kernel": kname, "bound": "hbm", "achieved": round(gbs, 1),
                "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4),
                "peak_source": f"{peak_src} HBM copy bandwidth"}
    roof.update({"tensor_frac_of_burst": round(tflops / burst, 4),
                 "tensor_frac_of_sustained": round(tflops / sustained, 4),
                 "hbm_frac": round(gbs / peaks["hbm_gbs"], 4),
                 "ridge_frac": round(max(t_tc, t_hbm) / t_s, 4),
                 "ms": round(t_s * 1e3, 4)})
    return roof


def make_layer(w, quant: str, dev, T: int):
    """Seeded weights of the workload and the resident layer: bf16, fp8 block-128 or nvfp4
    (prepared once, as a loader would)."""
    from mixture_experts_layer_05_gb300 import binding, inputs
    if quant == "fp8":
        wts = inputs.make_fp8_weights(w, 0, device=dev)
        cfg = binding.config_from_workload(w, weight_quant="fp8")
        layer = binding.FusedMoE(cfg, wts["w13_q"], wts["w2_q"], wts["bias"], wts["shared_w13_q"],
                                 wts["shared_w2_q"], max_tokens=T, w13_scale=wts["w13_s"],
                                 w2_scale=wts["w2_s"], shared_w13_scale=wts["shared_w13_s"],
                                 shared_w2_scale=wts["shared_w2_s"])
    elif quant == "nvfp4":
        wts = inputs.make_fp4_weights(w, 0, device=dev)
        cfg = binding.config_from_workload(w, weight_quant="nvfp4")

        def prep(q, sf):
            return binding.moe_nvfp4_prepare_weight(q.reshape(-1, q.shape[-1]),
                                                    sf.reshape(-1, sf.shape[-1]))
        kw = dict(w13_weight_scale_2=wts["w13_s2"], w2_weight_scale_2=wts["w2_s2"],
                  input_scale=wts["input_scale"], act_scale=wts["act_scale"])
        sw13 = sw2 = None
        if w.shared_intermediate_size:
            sw13 = prep(wts["shared_w13"], wts["shared_w13_sf"])
            sw2 = prep(wts["shared_w2"], wts["shared_w2_sf"])
            kw.update(shared_weight_scale_2=wts["shared_s2"],
                      shared_input_scale=wts["shared_input_scale"],
                      shared_act_scale=wts["shared_act_scale"])
        layer = binding.FusedMoE(cfg, prep(wts["w13"], wts["w13_sf"]), prep(wts["w2"], wts["w2_sf"]),
                                 wts["bias"], sw13, sw2, max_tokens=T, **kw)
    else:
        wts = inputs.make_weights(w, 0, device=dev)
        cfg = binding.config_from_workload(w)
        layer = binding.FusedMoE(cfg, wts["w13"], wts["w2"], wts["bias"], wts["shared_w13"],
                                 wts["shared_w2"], max_tokens=T)
    return wts, cfg, layer


def run_ours(args, w, T):
    import torch
    import torch.distributed as dist

    from mixture_experts_layer_05_gb300 import binding, inputs
    from mixture_experts_layer_05_gb300 import build as build_mod

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1 and not dist.is_initialized():
        dist.init_process_group("nccl", device_id=dev)
    build_mod.build()
    binding.load()

    quant = args.quant
    fp8 = quant == "fp8"
    x_cpu, logits_cpu = inputs.make_tokens(w, T, seed=rank_seed(rank))
    x, logits = x_cpu.to(dev), logits_cpu.to(dev)
    wts, cfg, layer = make_layer(w, quant, dev, T)
    out = torch.empty_like(x)
    stream = torch.cuda.current_stream()
    K, W = args.steps, args.warmup
    gate = None
    if args.router == "gate":
        # the router GEMM inside the forward: a synthetic gate ~N(0, 1/sqrt(H)), so the
        # logits of the N(0, 1) hidden states are about N(0, 1) as in the logits workloads
        gate = inputs.normal((w.num_experts, w.hidden_size), w.hidden_size ** -0.5,
                             inputs.tensor_seed(w.name, "gate", 0), torch.bfloat16, dev)

    def fwd(**kw):
        if gate is not None:
            return layer(x, gate_weight=gate, out=out, **kw)
        return layer(x, logits, out=out, **kw)

    for _ in range(W):
        fwd()
    torch.cuda.synchronize()

    # stage breakdown (informational, untimed): events at every stage boundary
    sevs = [[torch.cuda.Event(enable_timing=True) for _ in range(binding.NUM_STAGE_EVENTS)]
            for _ in range(W)]
    for i in range(W):
        fwd(events=sevs[i])
    torch.cuda.synchronize()
    stage = {n: statistics.mean(e[a].elapsed_time(e[b]) for e in sevs)
             for n, a, b in (("route_align_gather", 0, 1), ("w13_gemm", 1, 2),
                             ("w2_gemm", 2, 3), ("combine", 3, 4))}
    step_est_s = max(sum(stage.values()) * 1e-3, 1e-6)

    # timed region: K forwards captured once into a CUDA graph and replayed (no events in
    # it: a stage event would break the kernels' programmatic launch chain). The w13 GEMM's
    # duration for the roofline comes from a second graph of K forwards whose w13 launches
    # are bracketed by events, replayed untimed right after the timed region.
    wevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    for pair in wevs:
        for ev in pair:
            ev.record(stream)
    torch.cuda.synchronize()
    graph = graph_w13 = None
    try:
        graph = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.graph(graph, stream=cap):
            for i in range(K):
                fwd()
        graph_w13 = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_w13, stream=cap):
            for i in range(K):
                fwd(events=[None, wevs[i][0], wevs[i][1], None, None])
        torch.cuda.synchronize()
    except Exception as exc:                        # eager timing if capture is refused
        print(f"[bench] CUDA graph capture failed ({exc}); timing eager steps", file=sys.stderr)
        graph = graph_w13 = None
        torch.cuda.synchronize()

    def eager_steps():
        for i in range(K):
            fwd()

    def timed_steps():
        if graph is not None:
            graph.replay()
        else:
            eager_steps()

    def w13_steps():
        if graph_w13 is not None:
            graph_w13.replay()
        else:
            for i in range(K):
                fwd(events=[None, wevs[i][0], wevs[i][1], None, None])

    def warm(fn, seconds=0.5):
        """Back-to-back steps until the GPU settles in its loaded power state."""
        for _ in range(max(1, int(seconds / (step_est_s * K)))):
            fn()

    def timed(fn, s=None):
        """(ms per step, wall start, wall end) of one K-step call on `s`, device-timed."""
        s = s or stream
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        w0 = time.time()
        a.record(s)
        fn()
        b.record(s)
        torch.cuda.synchronize()
        return a.elapsed_time(b) / K, w0, time.time()

    if graph is not None:
        graph.replay()                               # one untimed replay of each graph
        graph_w13.replay()
    torch.cuda.synchronize()
    sampler = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if sampler else 0)
    warm(timed_steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    wall0 = time.time()
    t_start.record(stream)
    timed_steps()
    t_end.record(stream)
    torch.cuda.synchronize()
    wall1 = time.time()
    if world > 1:
        dist.barrier()
    ms = t_start.elapsed_time(t_end) / K
    ms_max = reduce_max(ms, dev)
    # the same K forwards launched eagerly, in the same loaded state (informational)
    warm(eager_steps, 0.2)
    eager_ms, ew0, ew1 = timed(eager_steps)
    w13_steps()                                     # untimed: the w13 events for the roofline
    torch.cuda.synchronize()
    status = layer.device_status()
    if status != binding.OK:
        raise RuntimeError(f"device status {binding.STATUS.get(status, status)} after the run")
    try:
        w13_ms = statistics.mean(a.elapsed_time(b) for a, b in wevs)
        w13_src = ("w13 GEMM bracketed by events in a graph of K forwards replayed right "
                   "after the timed region")
    except RuntimeError as exc:                     # events not readable: use the eager ones
        print(f"[bench] w13 events unreadable ({exc}); using the stage pass", file=sys.stderr)
        w13_ms = stage["w13_gemm"]
        w13_src = "w13 GEMM events of the eager stage pass"
        torch.cuda.synchronize()

    # end to end: pinned host inputs in, output out, inside each timed step; copies of
    # neighbouring steps overlap the forward (binding.HostPipeline)
    x_h = x_cpu.pin_memory()
    l_h = logits_cpu.pin_memory()
    y_h = [torch.empty(x_cpu.shape, dtype=x_cpu.dtype).pin_memory() for _ in range(2)]
    pipe = binding.HostPipeline(layer, T, gate_weight=gate)

    def e2e_run(n):
        pipe.run([x_h] * n, [l_h] * n, [y_h[i & 1] for i in range(n)])

    e2e_run(W)
    torch.cuda.synchronize()
    warm(lambda: e2e_run(K), 0.3)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    xw0 = time.time()
    e0.record(pipe.h2d)
    e2e_run(K)
    e1.record(pipe.d2h)
    torch.cuda.synchronize()
    xw1 = time.time()
    e2e_ms = reduce_max(e0.elapsed_time(e1) / K, dev)
    clocks = e_clocks = x_clocks = None
    if sampler:
        time.sleep(0.1)
        clocks = sampler.summary(wall0, wall1)
        e_clocks = sampler.summary(ew0, ew1)
        x_clocks = sampler.summary(xw0, xw1)
        sampler.stop()

    # cold L2 for working sets that fit in L2: each step after writing a buffer larger than
    # L2, the forward alone timed by events (informational)
    cold = None
    weight_bytes = sum(v.numel() * v.element_size() for v in wts.values() if hasattr(v, "numel"))
    if weight_bytes < 3 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(K)]
        for a, b in evs:
            flush.fill_(1.0)
            a.record(stream)
            fwd()
            b.record(stream)
        torch.cuda.synchronize()
        cold = {"ms_per_step": round(statistics.mean(a.elapsed_time(b) for a, b in evs), 4),
                "how": "eager forwards, a 258 MB buffer written before each, events around "
                       "the forward only"}

    rs = routing_stats(layer, cfg, w, T)
    work = layer_work(w, T, rs["active_experts"], quant)
    peaks, peak_src = load_peaks()
    # which w13 kernel the forward runs: the token-N CTA-pair GEMM when its blocks are 256
    tn = quant == "none" and binding.moe_forward_block_size(cfg, T) == 256
    kname = ("gemm_fp8_kernel<w13> (grouped e4m3 w13 GEMM + SiLU*mul + act quant)" if fp8
             else "gemm_fp4_kernel<w13> (grouped nvfp4 w13 GEMM, fp4 -> f16 into tensor memory, "
                  "weights on M)"
             if quant == "nvfp4"
             else "gemm_tn_kernel<w13> (grouped w13 GEMM + SiLU*mul, tokens on N, CTA pairs)"
             if tn else "gemm_kernel<w13> (grouped w13 GEMM + SiLU*mul)")
    value = aggregate_tokens_per_s(T, world, ms_max)
    ratio = QUANT_PEAK_RATIO[quant]

    res = None
    if rank == 0:
        # dominant kernel: the w13 grouped GEMM (two thirds of the flops and weight bytes)
        roof = roofline_of(work, w13_ms / 1e3, peaks, peak_src, quant, kname)
        roof["traffic"] = args.traffic if args.traffic is not None else (
            kernel_traffic("gemm_fp8_w13", w.name, T, "gemm_fp8.cu") if fp8
            else kernel_traffic("gemm_fp4_w13", w.name, T, "gemm_fp4.cu") if quant == "nvfp4"
            else kernel_traffic("gemm_tn_w13", w.name, T, "gemm_tn.cu") if tn
            else kernel_traffic("gemm_w13", w.name, T))
        step_s = ms_max / 1e3
        tc_burst = peaks["bf16_tflops"] * ratio
        res = {
            "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world,
            "steps": K, "warmup": W, "ms_per_step": round(ms_max, 4), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": QUANT_DTYPE[quant],
            "data": "synthetic",
            "config": {"workload": f"{w.name}: FusedMoE layer H={w.hidden_size} "
                                   f"I={w.intermediate_size} E={w.num_experts} k={w.top_k}"
                                   + (f" shared I={w.shared_intermediate_size}"
                                      if w.shared_intermediate_size else "")
                                   + QUANT_TAG[quant]
                                   + (", router GEMM from the gate weight" if gate is not None
                                      else ""),
                       "tokens_per_gpu": T, "global_batch": T * world,
                       "parallelism": f"dp{world} replicas",
                       "l2": ("inputs larger than L2 (expert weights streamed every step)"
                              if weight_bytes >= 3 * L2_BYTES else
                              "weights fit in L2: value is warm-L2; cold_l2 flushes L2"),
                       "seed": "weights 0, tokens = rank"},
            "layer": {"tflops": round(work["flops"] / step_s / 1e12, 1),
                      "tensor_frac_of_burst": round(work["flops"] / step_s / 1e12 / tc_burst, 4),
                      "hbm_gbs": round(work["bytes"] / step_s / 1e9, 1),
                      "hbm_frac": round(work["bytes"] / step_s / 1e9 / peaks["hbm_gbs"], 4),
                      "ridge_frac": round(max(work["flops"] / (tc_burst * 1e12),
                                              work["bytes"] / (peaks["hbm_gbs"] * 1e9))
                                          / step_s, 4),
                      **rs,
                      "stages_ms": {k: round(v, 4) for k, v in stage.items()},
                      "stages_note": "eager forwards with events at every stage boundary, "
                                     "outside the timed region"},
            "roofline": roof,
            "timing": {"value": "one CUDA-graph replay of K captured forwards, after >= 0.5 s "
                                "of back-to-back replays" if graph is not None
                                else "K eager forwards",
                       "roofline": w13_src},
            "eager": {"ms_per_step": round(eager_ms, 4),
                      "value": round(aggregate_tokens_per_s(T, 1, eager_ms), 1),
                      "clocks": e_clocks,
                      "note": "the same K forwards launched one by one (no graph), right after "
                              "the timed region"},
            "e2e": {"value": round(aggregate_tokens_per_s(T, world, e2e_ms), 1),
                    "unit": "tokens/s",
                    "h2d_bytes_per_step": x.numel() * 2 + (0 if gate is not None else logits.numel() * 4),
                    "d2h_bytes_per_step": out.numel() * 2, "ms_per_step": round(e2e_ms, 4),
                    "clocks": x_clocks},
            "gpu_launches": K * binding.moe_forward_num_launches_ex(cfg, T, gate is not None),
            "clocks": clocks,
        }
        if cold is not None:
            res["cold_l2"] = cold
        if args.cpu_baseline and world == 1:
            res["cpu_baseline"] = cpu_baseline(w, wts, x_cpu, logits_cpu, args.cpu_sample,
                                               quant=quant)
    return res


def run_sweep(args, w, token_counts):
    """One JSON line per token count: graph-replayed forwards on the same weights, with the
    routing's per-expert load histogram (the skewed-routing sweep)."""
    import torch

    from mixture_experts_layer_05_gb300 import binding, inputs
    from mixture_experts_layer_05_gb300 import build as build_mod

    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    build_mod.build()
    binding.load()
    quant = args.quant
    Tmax = max(token_counts)
    wts, cfg, layer = make_layer(w, quant, dev, Tmax)
    peaks, peak_src = load_peaks()
    ratio = QUANT_PEAK_RATIO[quant]
    K = args.steps
    for T in token_counts:
        x_cpu, l_cpu = inputs.make_tokens(w, T, seed=0)
        x, lg = x_cpu.to(dev), l_cpu.to(dev)
        out = torch.empty_like(x)
        for _ in range(max(3, args.warmup)):
            layer(x, lg, out=out)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        cs = torch.cuda.Stream()
        cs.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=cs):
            for _ in range(K):
                layer(x, lg, out=out)
        g.replay()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        g.replay()
        b.record()
        torch.cuda.synchronize()
        ms = a.elapsed_time(b) / K
        if layer.device_status() != binding.OK:
            raise RuntimeError(f"device status error at T={T}")
        rs = routing_stats(layer, cfg, w, T)
        work = layer_work(w, T, rs["active_experts"], quant)
        t = ms / 1e3
        print(json.dumps({
            "sweep": w.name, "tokens": T, "dtype": QUANT_DTYPE[quant],
            "ms_per_step": round(ms, 4), "tokens_per_s": round(T / t, 1),
            "layer_tflops": round(work["flops"] / t / 1e12, 1),
            "tensor_frac_of_burst": round(work["flops"] / t / 1e12
                                          / (peaks["bf16_tflops"] * ratio), 4),
            "hbm_frac": round(work["bytes"] / t / 1e9 / peaks["hbm_gbs"], 4),
            "ridge_frac": round(max(work["flops"] / (peaks["bf16_tflops"] * ratio * 1e12),
                                    work["bytes"] / (peaks["hbm_gbs"] * 1e9)) / t, 4),
            **rs}), flush=True)
        del g


def _host_weights(w, wts):
    return {k: (v.to("cpu") if hasattr(v, "to") else v) for k, v in wts.items()}


def oracle_cfg(w):
    return dict(num_experts=w.num_experts, top_k=w.top_k, renormalize=w.renormalize,
                use_grouped_topk=w.use_grouped_topk, num_expert_group=w.num_expert_group,
                topk_group=w.topk_group, scoring_func=w.scoring_func,
                routed_scaling_factor=w.routed_scaling_factor)


def _fp4_oracle_weights(hw) -> dict:
    """make_fp4_weights' tensors under the names the NVFP4 oracle takes."""
    o = {k: hw[k] for k in ("w13", "w13_sf", "w2", "w2_sf", "input_scale", "act_scale")}
    o["w13_s2"], o["w2_s2"] = hw["w13_s2"].numpy(), hw["w2_s2"].numpy()
    if hw.get("shared_w13") is not None:
        o.update(shared_w13=hw["shared_w13"], shared_w13_sf=hw["shared_w13_sf"],
                 shared_w2=hw["shared_w2"], shared_w2_sf=hw["shared_w2_sf"],
                 shared_w13_s2=float(hw["shared_s2"][0]), shared_w2_s2=float(hw["shared_s2"][1]),
                 shared_input_scale=hw["shared_input_scale"],
                 shared_act_scale=hw["shared_act_scale"])
    return o


def _oracle_layer(w, hw, x, logits, quant: str):
    import oracle
    if quant == "nvfp4":
        oracle.fused_moe_fp4(x, logits, hw["bias"], _fp4_oracle_weights(hw), **oracle_cfg(w))
    elif quant == "fp8":
        oracle.fused_moe_fp8(x, logits, hw["bias"], hw["w13_q"], hw["w13_s"], hw["w2_q"],
                             hw["w2_s"], hw["shared_w13_q"], hw["shared_w13_s"],
                             hw["shared_w2_q"], hw["shared_w2_s"], **oracle_cfg(w))
    else:
        oracle.fused_moe_rows(x, logits, hw["bias"], hw["w13"], hw["w2"], hw["shared_w13"],
                              hw["shared_w2"], **oracle_cfg(w))


def _oracle_rows(w, hw, x_cpu, logits_cpu, r0, n, quant="none"):
    t0 = time.perf_counter()
    _oracle_layer(w, hw, x_cpu[r0:r0 + n], logits_cpu[r0:r0 + n], quant)
    return time.perf_counter() - t0


def cpu_baseline(w, wts, x_cpu, logits_cpu, n_tokens: int, target_s: float = 12.0,
                 quant: str = "none") -> dict:
    """The CPU oracle, as it stands, on a leading sample of the batch sized to ~target_s."""
    hw = _host_weights(w, wts)
    T = x_cpu.shape[0]
    n = min(n_tokens, T)
    dt = _oracle_rows(w, hw, x_cpu, logits_cpu, 0, n, quant)
    for _ in range(4):                              # grow the sample to ~target_s of work
        if dt >= target_s / 2 or n >= T:
            break
        n = int(min(T, max(2 * n, n * target_s / max(dt, 1e-3))))
        dt = _oracle_rows(w, hw, x_cpu, logits_cpu, 0, n, quant)
    return {"value": round(n / dt, 4), "unit": "tokens/s",
            "cores": len(os.sched_getaffinity(0)), "kind": "oracle",
            "sample": f"first {n} of the step's {T} tokens, full weights, fp64 numpy "
                      f"(BLAS default threading), {dt:.1f} s"}


def run_reference(args, w, T):
    """The CPU oracle as the reference arm: each step routes and computes a bounded sample."""
    import torch

    from mixture_experts_layer_05_gb300 import inputs
    import oracle

    rank, world, _ = dist_env()
    if rank != 0:
        return None
    n = args.ref_sample if args.ref_sample > 0 else 1
    quant = args.quant
    # drawn where the GPU arm draws them (the same values), then held on the host; on a
    # machine without a GPU, drawn on the CPU. Only the oracle's work is timed.
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    make = {"fp8": inputs.make_fp8_weights, "nvfp4": inputs.make_fp4_weights}.get(
        quant, inputs.make_weights)
    hw = {key: (v.to("cpu") if hasattr(v, "to") else v)
          for key, v in make(w, 0, device=gen).items()}
    if gen == "cuda":
        torch.cuda.empty_cache()
    x_cpu, logits_cpu = inputs.make_tokens(w, T, seed=0)

    def step(i):
        r0 = (i * n) % max(T - n + 1, 1)
        _oracle_layer(w, hw, x_cpu[r0:r0 + n], logits_cpu[r0:r0 + n], quant)

    # size each step's sample so one step is ~1.5 s of oracle work (the whole run then
    # stays within a few minutes for the usual K, W)
    t0 = time.perf_counter()
    step(0)
    dt0 = time.perf_counter() - t0
    for _ in range(4):                              # a fixed cost per call makes one guess short
        if args.ref_sample > 0 or dt0 >= 0.75 or n >= T:
            break
        n = max(n + 1, min(T, int(n * 1.5 / max(dt0, 1e-3))))
        t0 = time.perf_counter()
        step(0)
        dt0 = time.perf_counter() - t0
    for i in range(args.warmup):
        step(i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        step(args.warmup + i)
    dt = (time.perf_counter() - t0) / args.steps
    value = n / dt
    cores = len(os.sched_getaffinity(0))
    sample = f"{n} token(s) of the {T}-token batch per step, full weights, fp64 numpy"
    return {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "tokens/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(dt * 1e3, 2), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": f"{w.name}: FusedMoE layer H={w.hidden_size} "
                                   f"I={w.intermediate_size} E={w.num_experts} k={w.top_k}"
                                   + QUANT_TAG[quant],
                       "tokens_per_gpu": T, "sample_tokens_per_step": n},
            "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="dsv3")
    ap.add_argument("--tokens", type=int, default=8192)
    ap.add_argument("--sweep", default=None,
                    help="comma-separated token counts: one JSON line per count (no contract "
                         "line); e.g. the skewed-routing sweep 1,2,4,...,16384")
    ap.add_argument("--quant", choices=["none", "fp8", "nvfp4"], default="none",
                    help="expert weights: bf16 (none), e4m3 with 128 x 128 fp32 block scales, "
                         "or nvfp4 (e2m1, e4m3 scales per 16 values, per-expert fp32 scales)")
    ap.add_argument("--cpu-sample", type=int, default=4,
                    help="initial oracle sample (tokens); grown to ~12 s of CPU work")
    ap.add_argument("--ref-sample", type=int, default=0,
                    help="tokens per reference step (0: sized to ~1.5 s per step)")
    ap.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    ap.add_argument("--router", choices=["logits", "gate"], default="logits",
                    help="router logits as input (the FusedMoE layer's signature), or the "
                         "gate weight with the router GEMM inside the forward")
    ap.add_argument("--num-experts", type=int, default=0,
                    help="reduced-expert stand-in of the workload (profiling captures only)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="dram bytes per launch of the dominant kernel from an ncu capture")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    from mixture_experts_layer_05_gb300 import configs
    w = configs.get(args.workload)
    if args.num_experts:
        # a reduced-expert stand-in of the same shapes (for counter captures that must stay
        # small): the same hidden, intermediate, top_k and group count, fewer experts
        w = configs.shrink(w, num_experts=args.num_experts, name=f"{w.name}-E{args.num_experts}")
    if args.sweep:
        run_sweep(args, w, [int(t) for t in args.sweep.split(",")])
        return
    res = run_reference(args, w, args.tokens) if args.impl == "reference" \
        else run_ours(args, w, args.tokens)
    if res is not None:
        print(json.dumps(res), flush=True)
    try:
        import torch.distributed as dist
        if dist.is_initialized():
            dist.destroy_process_group()
    except Exception:
        pass


if __name__ == "__main__":
    main()

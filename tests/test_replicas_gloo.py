"""The multi-GPU path is data-parallel replicas: host logic checked with 2 gloo ranks on CPU.

Each rank draws its own batch (seed = rank) against the same weights, times its own
steps, and the job reports the max step time over ranks and tokens of all ranks.
"""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench
from mixture_experts_layer_05_gb300 import configs, inputs


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    r, w, lr = bench.dist_env()
    ms = 1.0 + rank                                   # rank 1 is the slow one
    ms_max = bench.reduce_max(ms)
    x, logits = inputs.make_tokens(configs.TINY, 8, seed=bench.rank_seed(r))
    wts = inputs.make_weights(configs.TINY, 0)
    digest = float(logits.sum()), float(wts["w13"].float().sum())
    q.put((r, w, lr, ms_max, bench.aggregate_tokens_per_s(8, w, ms_max), digest))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, w0, l0, m0, v0, d0), (r1, w1, l1, m1, v1, d1) = out
    assert (r0, r1, w0, w1, l0, l1) == (0, 1, 2, 2, 0, 1)
    assert m0 == m1 == 2.0                            # max over ranks
    assert v0 == v1 == 8 * 2 / 2e-3                   # all ranks' tokens / max time
    assert d0[0] != d1[0]                             # each replica its own batch
    assert d0[1] == d1[1]                             # same weights everywhere


def test_single_process_identity():
    assert bench.reduce_max(3.5) == 3.5
    assert bench.aggregate_tokens_per_s(4096, 1, 2.0) == 4096 / 2e-3

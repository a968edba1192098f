"""moe_align_block_size_no_workspace against moe_align_block_size, through the C ABI.

The no-workspace variant serves callers that may not allocate device memory (a host
framework owns every allocation, so they have no workspace to pass); it keeps its
scratch in a fixed 1 MiB array inside the library. Its outputs must equal those of
the workspace entry point exactly (integer outputs), on two calls in a row, since
every call reuses the same array. This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_layer_05_gb300 import binding

pytestmark = pytest.mark.gpu


def _ids(T, k, E, seed, skew):
    rng = np.random.default_rng(seed)
    if skew:
        p = 1.0 / np.arange(1, E + 1) ** 1.2
        p /= p.sum()
        rows = [rng.choice(E, size=k, replace=False, p=p) for _ in range(T)]
    else:
        rows = [rng.permutation(E)[:k] for _ in range(T)]
    return torch.from_numpy(np.stack(rows).astype(np.int32)).cuda()


def _outputs(T, k, E, bs):
    max_sorted = T * k + E * (bs - 1)
    return (torch.full((max_sorted,), -7, dtype=torch.int32, device="cuda"),
            torch.full((max_sorted // bs + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.zeros(1, dtype=torch.int32, device="cuda"))


def _compare(lib, T, k, E, bs, seed, skew, ids=None):
    if ids is None:
        ids = _ids(T, k, E, seed, skew)
    ref = _outputs(T, k, E, bs)
    ws = binding.alloc_workspace(binding.moe_align_block_size_workspace_size(T, k, E))
    binding.moe_align_block_size(ids, E, bs, *ref, ws)
    got = _outputs(T, k, E, bs)
    P = ctypes.c_void_p
    rc = lib.moe_align_block_size_no_workspace(
        P(ids.data_ptr()), T, k, E, bs, P(got[0].data_ptr()), P(got[1].data_ptr()),
        P(got[2].data_ptr()), P(torch.cuda.current_stream().cuda_stream))
    assert rc == binding.OK
    torch.cuda.synchronize()
    npp = int(ref[2].item())
    assert int(got[2].item()) == npp
    assert torch.equal(got[0][:npp], ref[0][:npp])
    assert torch.equal(got[1], ref[1])


def test_no_workspace_matches_workspace_entry_point(cuda_lib):
    lib = cuda_lib
    # two calls in a row with different shapes share (and reuse) the built-in scratch
    _compare(lib, 3000, 6, 160, 128, seed=1, skew=True)
    _compare(lib, 517, 8, 256, 64, seed=2, skew=False)
    # a request beyond the 1 MiB scratch is rejected before anything is enqueued
    P = ctypes.c_void_p
    too_big = lib.moe_align_block_size_no_workspace(P(256), 1 << 20, 8, 1024, 128, P(256),
                                                    P(256), P(256), None)
    assert too_big == binding.ERR_WORKSPACE


def test_no_workspace_size_limit_is_exact(cuda_lib):
    """The scratch limit is inclusive: with E = 256, 1,048,576 flat indices (512 chunks of
    2048, exactly 1 MiB of counts and offsets) are accepted and match the workspace entry
    point; one token more needs a 513th chunk and is refused before anything is enqueued."""
    lib = cuda_lib
    T, k, E = 131072, 8, 256
    rng = np.random.default_rng(3)
    # k distinct experts per token: a random start plus k offsets 32 apart
    ids = (rng.integers(0, E, size=(T, 1)) + 32 * np.arange(k)[None, :]) % E
    _compare(lib, T, k, E, 128, 0, False, torch.from_numpy(ids.astype(np.int32)).cuda())
    P = ctypes.c_void_p
    refused = lib.moe_align_block_size_no_workspace(P(256), T + 1, k, E, 128, P(256), P(256),
                                                    P(256), None)
    assert refused == binding.ERR_WORKSPACE

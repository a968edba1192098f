"""GB300 (sm_103a) FusedMoE layer forward: CUDA kernels behind a small C ABI.

The library (``libgbmoe.so``, built by ``build.build()``) exports ``moe_topk``,
``moe_align_block_size`` and ``moe_forward``; ``binding`` calls them from Python.
"""
from . import configs, inputs  # noqa: F401

__all__ = ["configs", "inputs", "binding", "build"]

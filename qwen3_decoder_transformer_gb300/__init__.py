"""Qwen3-style dense decoder forward pass (prefill + KV-cached decode) on one GB300 (sm_103a).

The compute runs in the CUDA library built from ``csrc/`` and exposed through the C ABI in
``include/qwen3.h``; ``binding`` is its ctypes wrapper. PyTorch provides device memory and streams.
"""
from .configs import QWEN3_0P6B, QWEN3_8B, TINY, WORKLOADS  # noqa: F401

"""GB300-native joint RoPE attention for the FLUX.2 MMDiT denoiser.

The compute runs in the CUDA library built from ``csrc/`` (C-ABI declared in
``include/flux_attn.h``); ``binding`` marshals torch device tensors into it.
Importing this package does not load the library; the first call does, and
fails loudly when it is missing.
"""
from . import workloads  # noqa: F401

__all__ = ["workloads"]

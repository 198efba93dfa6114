"""GB300-native hot path of the FLUX.2 MMDiT denoiser's joint attention.

The compute runs in the CUDA library built from ``csrc/`` (C-ABI declared in
``include/flux_attn.h``); ``binding`` marshals torch device tensors into it:

- ``rope_tables`` / ``rope_tables_packed``: cos/sin tables from 4-axis ids;
- ``joint_rope_attention`` (and ``joint_rope_attention_tabled``): RoPE fused
  into the Q/K tile loads, softmax(QK^T / sqrt(128)) V over [txt ; img],
  optionally with the QK RMS normalisation before RoPE (``qk_norm=``);
- ``attention_extract`` / ``attention_cached``: the reference-image KV modes;
- ``qkv_mlp_proj``: the single-stream block's fused Q/K/V + SwiGLU-MLP input
  projection, writing Q, K, V in the attention's [B, S, H, 128] layout.

Importing this package does not load the library; the first call does, and
fails loudly when it is missing (there is no CPU path).
"""
from . import workloads  # noqa: F401

__all__ = ["workloads"]

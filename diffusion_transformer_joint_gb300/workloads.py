"""Seeded synthetic workloads for the joint RoPE attention.

This module draws inputs and nothing else: it holds none of the method's
arithmetic, so both the CUDA path's tests/bench and the oracle can take their
inputs from it.

Shapes follow the pages' workloads at 1024x1024: 512 text tokens (the text
encoders' maximum length) and 64x64 = 4096 image tokens (8x VAE downsampling,
then 2x2 patchify), head_dim 128, 24 / 32 / 48 heads for klein-4B / klein-9B /
dev-32B ("FLUX.2 [klein]" survey page, section "模型架构"; "FLUX.2 Klein 9B Base
宏观架构" trace page, cards 1 and 3). Multi-reference editing concatenates the
reference images' tokens with the noisy image tokens; here two 64x64
references are offset on the T axis by 10 and 20.

Position ids are (T, H, W, L): text token l gets (0, 0, 0, l), image token
(h, w) gets (0, h, w, 0) in row-major order (h outer), reference r gets
(t_r, h, w, 0). q, k and v are i.i.d. N(0, 1) drawn in fp32 with numpy's PCG64
generator from a per-tensor seed, then rounded to bf16 (round-to-nearest-even).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

HEAD_DIM = 128
AXES_DIMS = (32, 32, 32, 32)
ROPE_THETA = 2000.0


@dataclass(frozen=True)
class Workload:
    name: str
    index: int  # seeds are 1000*index + {1, 2, 3} for q, k, v
    B: int
    H: int
    S_txt: int
    grid: int  # image tokens form a grid x grid lattice
    ref_t: tuple = field(default_factory=tuple)  # T-axis offsets of reference images
    D: int = HEAD_DIM

    @property
    def S_img(self) -> int:
        return self.grid * self.grid * (1 + len(self.ref_t))

    @property
    def S(self) -> int:
        return self.S_txt + self.S_img

    @property
    def flops(self) -> int:
        """4*B*H*S^2*D: the two S x S x D contractions, 2 flops per multiply-add."""
        return 4 * self.B * self.H * self.S * self.S * self.D

    @property
    def io_bytes(self) -> int:
        """Algorithmic HBM bytes: q, k, v read once and out written once, bf16."""
        return 8 * self.B * self.S * self.H * self.D


WORKLOADS = {
    w.name: w
    for w in (
        Workload("tiny", 0, B=1, H=2, S_txt=16, grid=8),
        Workload("klein4b", 1, B=1, H=24, S_txt=512, grid=64),
        Workload("klein9b", 2, B=1, H=32, S_txt=512, grid=64),
        Workload("dev32b", 3, B=1, H=48, S_txt=512, grid=64),
        Workload("klein9b_edit2", 4, B=1, H=32, S_txt=512, grid=64, ref_t=(10, 20)),
    )
}


def txt_ids(S_txt: int) -> np.ndarray:
    ids = np.zeros((S_txt, 4), dtype=np.int32)
    ids[:, 3] = np.arange(S_txt, dtype=np.int32)
    return ids


def img_ids(grid: int, t: int = 0) -> np.ndarray:
    h, w = np.meshgrid(np.arange(grid, dtype=np.int32), np.arange(grid, dtype=np.int32),
                       indexing="ij")
    ids = np.zeros((grid * grid, 4), dtype=np.int32)
    ids[:, 0] = t
    ids[:, 1] = h.reshape(-1)
    ids[:, 2] = w.reshape(-1)
    return ids


def workload_ids(w: Workload):
    """(txt_ids [S_txt, 4], img_ids [S_img, 4]) int32; img_ids = noisy, then references."""
    parts = [img_ids(w.grid, 0)] + [img_ids(w.grid, t) for t in w.ref_t]
    return txt_ids(w.S_txt), np.ascontiguousarray(np.concatenate(parts, axis=0))


def normal_bf16(shape, seed: int, scale: float = 1.0):
    """i.i.d. N(0, scale^2) in fp32 from PCG64(seed), rounded to a bf16 torch CPU tensor."""
    import torch

    x = np.random.default_rng(seed).standard_normal(size=shape, dtype=np.float32)
    if scale != 1.0:
        x *= np.float32(scale)
    return torch.from_numpy(x).to(torch.bfloat16)


def workload_qkv(w: Workload, seed_offset: int = 0):
    """q, k, v as bf16 CPU tensors [B, S, H, D] from the workload's seeds."""
    shape = (w.B, w.S, w.H, w.D)
    base = 1000 * w.index + seed_offset
    return (normal_bf16(shape, base + 1), normal_bf16(shape, base + 2),
            normal_bf16(shape, base + 3))


MLP_RATIO = 3  # MLP width / hidden width of the FLUX.2 blocks


def proj_dims(w: Workload):
    """(M tokens, dim = hidden width = H * 128, mlp width) of the workload's
    single-stream input projection."""
    inner = w.H * w.D
    return w.B * w.S, inner, MLP_RATIO * inner


def proj_flops(w: Workload) -> int:
    """2 * M * dim * (3 * inner + 2 * mlp): one multiply-add per weight and token."""
    M, dim, mlp = proj_dims(w)
    return 2 * M * dim * (3 * dim + 2 * mlp)


def proj_inputs(w: Workload, seed_offset: int = 0):
    """x [M, dim] ~ N(0, 1) and W [3 dim + 2 mlp, dim] ~ N(0, 1/dim) as bf16 CPU
    tensors (synthetic activations and weights, seeds 1000*index + {11, 12})."""
    M, dim, mlp = proj_dims(w)
    base = 1000 * w.index + seed_offset
    return (normal_bf16((M, dim), base + 11),
            normal_bf16((3 * dim + 2 * mlp, dim), base + 12, scale=dim ** -0.5))


def random_ids(S: int, seed: int, low: int = -600, high: int = 600, n_axes: int = 4):
    """Arbitrary int32 ids (any value is a valid position) for edge-case tests."""
    rng = np.random.default_rng(seed)
    return rng.integers(low, high, size=(S, n_axes), dtype=np.int32)

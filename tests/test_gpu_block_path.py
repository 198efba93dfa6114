"""The hot path composed as the FLUX.2 blocks run it, against the oracle's
steps composed the same way.

Single-stream block ("Diffusers 中 Flux2Transformer2DModel 全面解析", section
内部架构双流块与单流块): one fused projection yields Q, K, V (and the SwiGLU
MLP input), Q and K are RMS-normalised and rotated, and the text and image
tokens attend jointly. Double-stream block (same section): the text and the
image stream have their own Q/K/V projections, and their outputs are
concatenated into one attention; here the two projections write straight into
the joint [txt ; img] layout (row offsets, no MLP half). q, k and v are stored
in bf16 between the projection and the attention on both sides: the
reference rounds the oracle's projection to bf16 before the oracle's
attention. Bar: max |gpu - reference| <= 1e-2, mean <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_joint_gb300 import binding, build
from diffusion_transformer_joint_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
EPS = 1e-6


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)


def _bar(got, ref):
    err = np.abs(got.float().cpu().numpy().astype(np.float64) - ref)
    assert np.isfinite(err).all()
    assert err.max() <= MAX_ABS, f"max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"mean abs err {err.mean():.3e}"


def test_single_stream_block_path():
    S_t, S_i, H, dim, mlp = 48, 208, 2, 256, 768
    S = S_t + S_i
    x = W.normal_bf16((S, dim), 1301)
    w = W.normal_bf16((3 * H * 128 + 2 * mlp, dim), 1302, scale=dim ** -0.5)
    ids = W.random_ids(S, 1303, 0, 200)
    rng = np.random.default_rng(1304)
    norm = [rng.uniform(0.5, 1.5, 128).astype(np.float32) for _ in range(4)]
    # GPU: projection -> joint attention with the QK norm
    q, k, v, act = binding.qkv_mlp_proj(x.cuda(), w.cuda(), H, mlp)
    out = binding.joint_rope_attention(q[None], k[None], v[None], torch.from_numpy(ids[:S_t]).cuda(),
                                       torch.from_numpy(ids[S_t:]).cuda(),
                                       qk_norm=tuple(torch.from_numpy(n).cuda() for n in norm) + (EPS,))
    torch.cuda.synchronize()
    # reference: the oracle's projection, stored in bf16, then the oracle's attention
    rq, rk, rv, ra = oracle.qkv_mlp_proj(x.float().numpy(), w.float().numpy(), H, 128, mlp)
    qs, ks, vs = (_bf16(t).float().numpy()[None] for t in (rq, rk, rv))
    ref = oracle.joint_rope_attention(qs, ks, vs, ids[:S_t], ids[S_t:], qk_norm=tuple(norm) + (EPS,))
    _bar(out, ref)


def test_double_stream_projections_write_the_joint_layout():
    S_t, S_i, H, dim = 40, 216, 2, 192
    S = S_t + S_i
    x_t = W.normal_bf16((S_t, dim), 1311)  # text stream hidden states
    x_i = W.normal_bf16((S_i, dim), 1312)  # image stream hidden states
    w_t = W.normal_bf16((3 * H * 128, dim), 1313, scale=dim ** -0.5)  # text Q/K/V projections
    w_i = W.normal_bf16((3 * H * 128, dim), 1314, scale=dim ** -0.5)  # image Q/K/V projections
    ids = W.random_ids(S, 1315, 0, 200)
    q, k, v = (torch.empty((1, S, H, 128), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    for xs, ws, lo, hi in ((x_t, w_t, 0, S_t), (x_i, w_i, S_t, S)):
        binding.qkv_mlp_proj(xs.cuda(), ws.cuda(), H, 0, q=q[0, lo:hi], k=k[0, lo:hi],
                             v=v[0, lo:hi])
    out = binding.joint_rope_attention(q, k, v, torch.from_numpy(ids[:S_t]).cuda(),
                                       torch.from_numpy(ids[S_t:]).cuda())
    torch.cuda.synchronize()
    parts = [oracle.qkv_mlp_proj(xs.float().numpy(), ws.float().numpy(), H, 128, 0)
             for xs, ws in ((x_t, w_t), (x_i, w_i))]
    rq, rk, rv = (np.concatenate([p[i] for p in parts])[None] for i in range(3))
    for got, ref in ((q, rq), (k, rk), (v, rv)):
        d = np.abs(got.float().cpu().numpy() - ref) - (2.0 ** -8 * np.abs(ref) + 1e-4)
        assert d.max() <= 0
    qs, ks, vs = (_bf16(t).float().numpy() for t in (rq, rk, rv))
    ref = oracle.joint_rope_attention(qs, ks, vs, ids[:S_t], ids[S_t:])
    _bar(out, ref)

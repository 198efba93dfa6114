"""GPU parity of the fused single-stream input projection against the oracle.

The single-stream block's to_qkv_mlp_proj ("Diffusers 中 Flux2Transformer2DModel
全面解析", sections 内部架构双流块与单流块, 激活函数与 FFN, 并行化支持): y = x W^T,
split into Q, K, V ([M, H, 128] each) and the SwiGLU activation
silu(gate) * linear of the MLP half. The kernel accumulates in fp32 and rounds
every output once to bf16, so the bar is |gpu - oracle| <= 2^-8 |oracle| + 1e-4
(twice the bf16 half-ulp, plus fp32 accumulation and exp error) for every
compared element.
"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_joint_gb300 import binding, build
from diffusion_transformer_joint_gb300 import workloads as W

pytestmark = pytest.mark.gpu

REL = 2.0 ** -8
ABS = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _check(got, ref, what):
    got = got.float().cpu().numpy().astype(np.float64).reshape(ref.shape)
    assert np.isfinite(got).all(), what
    err = np.abs(got - ref) - (REL * np.abs(ref) + ABS)
    assert err.max() <= 0, f"{what}: worst excess {err.max():.3e}"


def _inputs(M, dim, H, mlp, seed):
    x = W.normal_bf16((M, dim), seed)
    w = W.normal_bf16((3 * H * 128 + 2 * mlp, dim), seed + 1, scale=dim ** -0.5)
    return x, w


@pytest.mark.parametrize("M,dim,H,mlp", [
    (130, 128, 2, 768),   # two row blocks, ragged tail of 2 rows
    (1, 64, 1, 128),      # one token; 3 units: the last Q/K/V tile has one unit
    (300, 192, 3, 256),   # odd head count, three row blocks
    (257, 256, 2, 0),     # no MLP half
    (128, 64, 2, 384),    # exactly one row block
])
def test_proj_small_shapes_all_outputs(M, dim, H, mlp):
    x, w = _inputs(M, dim, H, mlp, 900 + M + dim)
    q, k, v, act = binding.qkv_mlp_proj(x.cuda(), w.cuda(), H, mlp)
    torch.cuda.synchronize()
    rq, rk, rv, ra = oracle.qkv_mlp_proj(x.float().numpy(), w.float().numpy(), H, 128, mlp)
    _check(q, rq, "q")
    _check(k, rk, "k")
    _check(v, rv, "v")
    if mlp:
        _check(act, ra, "act")


def test_proj_writes_nothing_past_the_outputs():
    M, dim, H, mlp = 77, 128, 2, 256
    x, w = _inputs(M, dim, H, mlp, 950)
    bufs = [torch.full((M + 64, H, 128), 7.0, dtype=torch.bfloat16, device="cuda")
            for _ in range(3)]
    abuf = torch.full((M + 64, mlp), 7.0, dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    binding.qkv_mlp_proj(x.cuda(), w.cuda(), H, mlp, q=bufs[0][:M], k=bufs[1][:M], v=bufs[2][:M],
                         act=abuf[:M], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for b in bufs:
        assert bool((b[M:] == 7.0).all())
    assert bool((abuf[M:] == 7.0).all())
    rq, _, _, ra = oracle.qkv_mlp_proj(x.float().numpy(), w.float().numpy(), H, 128, mlp)
    _check(bufs[0][:M], rq, "q")
    _check(abuf[:M], ra, "act")


def test_proj_is_deterministic():
    x, w = _inputs(300, 256, 2, 256, 960)
    a = binding.qkv_mlp_proj(x.cuda(), w.cuda(), 2, 256)
    b = binding.qkv_mlp_proj(x.cuda(), w.cuda(), 2, 256)
    torch.cuda.synchronize()
    for s, t in zip(a, b):
        assert torch.equal(s, t)


@pytest.mark.parametrize("name", ["klein4b", "klein9b", "dev32b"])
def test_proj_full_workload(name):
    """The workload's projection at full size: sampled token rows (every
    output feature) against the oracle, and every element against torch's
    bf16 matmul with the split and SwiGLU applied in fp32 (a whole-output
    check of the tile mapping; one bf16 rounding on each side)."""
    wl = W.WORKLOADS[name]
    M, dim, mlp = W.proj_dims(wl)
    H = wl.H
    x, w = W.proj_inputs(wl)
    xd, wd = x.cuda(), w.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, k, v, act = binding.qkv_mlp_proj(xd, wd, H, mlp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 127, 128, M - 1], rng.integers(0, M, 6)]))
    rq, rk, rv, ra = oracle.qkv_mlp_proj(x.float().numpy(), w.float().numpy(), H, 128, mlp,
                                         rows=rows)
    ri = torch.from_numpy(rows).cuda()
    _check(q[ri], rq, "q")
    _check(k[ri], rk, "k")
    _check(v[ri], rv, "v")
    _check(act[ri], ra, "act")
    inner = H * 128
    y = (xd.float() @ wd.float().T)
    for got, ref in ((q, y[:, :inner]), (k, y[:, inner:2 * inner]), (v, y[:, 2 * inner:3 * inner])):
        d = (got.reshape(M, inner).float() - ref).abs() - (2.0 ** -7 * ref.abs() + 1e-3)
        assert float(d.max()) <= 0
    g, u = y[:, 3 * inner:3 * inner + mlp], y[:, 3 * inner + mlp:]
    ra_all = torch.nn.functional.silu(g) * u
    d = (act.float() - ra_all).abs() - (2.0 ** -7 * ra_all.abs() + 1e-3)
    assert float(d.max()) <= 0

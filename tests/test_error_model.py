"""CPU checks of the test infrastructure behind the full-size and large-logit
GPU comparisons.

The rounding-error model (tests/error_model.py) is checked against a direct
simulation, in fp64, of the roundings it describes: (cos, sin) stored as
fp16, rotated q and k stored as bf16, the softmax weights stored as bf16 over
an unrounded denominator, the output stored as bf16. Its predicted sigma must
match the simulated error's spread, its bounds must hold, and a simulation
with one more mantissa bit dropped from the rotated rows must break them (the
bound is not so loose that any error passes).

The per-head runner (tests/oracle_parallel.py) must reproduce the oracle's
single call bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_joint_gb300 import workloads as W
from tests import error_model as EM
from tests.oracle_parallel import by_head


def _round_mantissa(x: torch.Tensor, bits: int) -> torch.Tensor:
    """Round fp64 values to `bits` stored mantissa bits (nearest, ties to even
    via the fp64 rounding of the scaled value)."""
    a = x.abs()
    e = torch.floor(torch.log2(torch.where(a > 0, a, torch.ones_like(a))))
    q = torch.pow(2.0, e - bits)
    return torch.where(a > 0, torch.round(x / q) * q, x)


def _simulate(q, k, v, ids, n_txt, rot_bits=7):
    c, s = oracle.rope_tables(ids)
    c16 = c.astype(np.float16).astype(np.float64)
    s16 = s.astype(np.float16).astype(np.float64)
    qr = _round_mantissa(torch.from_numpy(oracle.rope_apply(q.double().numpy(), c16, s16)), rot_bits)
    kr = _round_mantissa(torch.from_numpy(oracle.rope_apply(k.double().numpy(), c16, s16)), rot_bits)
    B, S, H, D = q.shape
    out = torch.empty((B, S, H, D), dtype=torch.float64)
    for h in range(H):
        z = qr[0, :, h] @ kr[0, :, h].T / np.sqrt(D)
        p = torch.exp(z - z.max(-1, keepdim=True).values)
        o = (p.to(torch.bfloat16).double() @ v[0, :, h].double()) / p.sum(-1, keepdim=True)
        out[0, :, h] = o.to(torch.bfloat16).double()
    return out.numpy()


def _case(scale):
    B, H, S = 1, 2, 300
    q = W.normal_bf16((B, S, H, 128), 3001, scale=scale)
    k = W.normal_bf16((B, S, H, 128), 3002)
    v = W.normal_bf16((B, S, H, 128), 3003)
    ids = W.random_ids(S, 3004, 0, 600)
    exact = oracle.joint_rope_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                        ids[:20], ids[20:])
    c, s = oracle.rope_tables(ids)
    qh = oracle.rope_apply(q.double().numpy(), c, s)
    kh = oracle.rope_apply(k.double().numpy(), c, s)
    sigma = EM.predicted_sigma(qh, kh, v.double().numpy(), exact,
                               EM.rotated_error_var(q.double().numpy(), c, s, qh),
                               EM.rotated_error_var(k.double().numpy(), c, s, kh))
    return q, k, v, ids, exact, sigma


@pytest.mark.parametrize("scale", [1.0, 8.0])
def test_model_matches_a_simulation_of_the_roundings(scale):
    q, k, v, ids, exact, sigma = _case(scale)
    sim = _simulate(q, k, v, ids, 20)
    err = np.abs(sim - exact)
    sig = sigma.numpy()
    live = sig > 0
    rms_ratio = float(np.sqrt(((err[live] / sig[live]) ** 2).mean()))
    assert 0.7 <= rms_ratio <= 1.3, rms_ratio
    EM.check(sim, exact, sigma, float(v.abs().max()))


def test_model_bound_rejects_a_coarser_rounding():
    q, k, v, ids, exact, sigma = _case(8.0)
    sim = _simulate(q, k, v, ids, 20, rot_bits=6)
    with pytest.raises(AssertionError):
        EM.check(sim, exact, sigma, float(v.abs().max()))


def test_kappa_is_the_relative_variance_of_a_bf16_rounding():
    x = torch.from_numpy(np.random.default_rng(5).standard_normal(2_000_000))
    e = x.to(torch.bfloat16).double() - x
    assert abs(float((e * e).mean() / (x * x).mean()) / EM.KAPPA - 1.0) < 0.03


def test_per_head_runner_reproduces_the_single_call():
    B, H, S_t, S_r, S_i = 1, 3, 20, 70, 90
    S = S_t + S_r + S_i
    q, k, v = (W.normal_bf16((B, S, H, 128), 3100 + i).float().numpy() for i in range(3))
    ids = W.random_ids(S, 3103, 0, 300)
    txt, ref, img = ids[:S_t], ids[S_t:S_t + S_r], ids[S_t + S_r:]
    whole = oracle.attention_extract(q, k, v, txt, ref, img)
    split = by_head(oracle.attention_extract, H, q, k, v, txt, ref, img)
    for a, b in zip(whole, split):
        assert np.array_equal(a, b)
    keep = np.r_[0:S_t, S_t + S_r:S]
    args = (q[:, keep], k[:, keep], v[:, keep], txt, img, whole[1], whole[2])
    assert np.array_equal(oracle.attention_cached(*args), by_head(oracle.attention_cached, H, *args))

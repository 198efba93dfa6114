"""First-order model of how far a bf16-operand attention kernel may land from
the exact (fp64) result, used as the a-priori bound of the tests that compare
large-logit cases with the plain oracle.

Definition being approximated ("Transformer架构解析FLUX.2-klein-base-9b-nvfp4",
section 2): o_i = sum_j w_ij v_j, w_ij = softmax_j(q^_i . k^_j / sqrt(D)), with
q^, k^ the RoPE-rotated (optionally RMS-normalised first) rows.

What the kernel rounds, and how it enters:
  1. Every rotated channel y of q^ and k^ is stored as bf16 (round to nearest
     even): error uniform within +-ulp(y)/2, ulp(y) = 2^(floor(log2|y|) - 7),
     variance ulp(y)^2 / 12.
  2. The (cos, sin) table is stored as fp16: each entry is off by up to half
     an fp16 ulp (2^(floor(log2|c|) - 10)), variance ulp16(c)^2 / 12. A pair
     (x0, x1) rotates to y0 = x0 c - x1 s, y1 = x0 s + x1 c, so the table adds
     x0^2 var(dc) + x1^2 var(ds) to var(y0) and x0^2 var(ds) + x1^2 var(dc)
     to var(y1).
  3. The softmax weights P are stored as bf16 for the P V product while the
     denominator sums the unrounded fp32 weights: a relative error with the
     variance KAPPA of one bf16 rounding.
  4. The output is rounded to bf16: variance ulp(o)^2 / 12.
  Everything else (fp32 accumulation, fp32 normalisation, the exp2
  instruction's relative error <= 2^-22 per weight) stays below 2^-21 max|v|,
  added as a fixed term.

Propagation (first order; roundings independent and zero-mean). Write e^q_i,
e^k_j for the channel errors of q^_i, k^_j and c_jd = v_jd - o_id. The logit
error is eps_ij = (e^q_i . k^_j + q^_i . e^k_j) / sqrt(D). A logit error moves
o_id by sum_j w_ij (eps_ij - sum_l w_il eps_il) c_jd; since sum_j w_ij c_jd = 0
this is
    sum_j w_ij c_jd (q^_i . e^k_j) / sqrt(D)      (independent over j)
  + e^q_i . (sum_j w_ij k^_j c_jd) / sqrt(D)       (shared over j),
with variances
    sum_j w_ij^2 c_jd^2 beta_ij,  beta_ij = sum_p q^_ip^2 var(e^k_jp) / D,
    sum_p var(e^q_ip) M_ipd^2 / D,  M_ipd = sum_j w_ij k^_jp c_jd.
The P rounding adds KAPPA sum_j w_ij^2 v_jd^2 and the output rounding
ulp(o_id)^2 / 12. sigma_id is the square root of the sum.

Bounds the tests assert, with N compared elements:
  - every element: |gpu - exact| <= Z(N) sigma_id + 2^-21 max|v|, with
    Z(N) = sqrt(2 ln(N / 1e-3)) (the level a maximum of N Gaussians exceeds
    with probability about 1e-3; uniform rounding terms have lighter tails);
  - the mean: mean |gpu - exact| <= RMS(sigma) (1 + 3 / sqrt(N)), since
    E|X| <= sqrt(E X^2) and the mean of N terms scatters by about RMS/sqrt(N).

KAPPA: a bf16 rounding's relative variance for values whose mantissas follow
the logarithmic (Benford) law, as Gaussian data do:
(2^-7)^2 / 12 * E[1/m^2] with E[1/m^2] = 3 / (8 ln 2) for m log-uniform on
[1, 2), i.e. 2^-14 / (32 ln 2) ~ 2.75e-6.
"""
from __future__ import annotations

import math

import numpy as np
import torch

KAPPA = 2.0 ** -14 / (32.0 * math.log(2.0))
FIXED = 2.0 ** -21


def _ulp_var(y: torch.Tensor, mant_bits: int) -> torch.Tensor:
    """Variance of round-to-nearest of y to a float with `mant_bits` stored
    mantissa bits: ulp(y)^2 / 12 (0 where y == 0)."""
    a = y.abs()
    e = torch.floor(torch.log2(torch.where(a > 0, a, torch.ones_like(a))))
    ulp = torch.pow(2.0, e - mant_bits)
    return torch.where(a > 0, ulp * ulp / 12.0, torch.zeros_like(a))


def rotated_error_var(x: np.ndarray, cos_t: np.ndarray, sin_t: np.ndarray,
                      yhat: np.ndarray) -> torch.Tensor:
    """Per-channel error variance of the kernel's bf16 rotated rows: x [B, S, H,
    D] the (normalised) rows before the rotation, yhat the exact rotated rows,
    cos_t / sin_t [S, D/2] the exact tables."""
    x = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    y = torch.from_numpy(np.ascontiguousarray(yhat, dtype=np.float64))
    c = torch.from_numpy(np.ascontiguousarray(cos_t, dtype=np.float64))[None, :, None, :]
    s = torch.from_numpy(np.ascontiguousarray(sin_t, dtype=np.float64))[None, :, None, :]
    vc, vs = _ulp_var(c, 10), _ulp_var(s, 10)
    x0, x1 = x[..., 0::2], x[..., 1::2]
    tab = torch.empty_like(x)
    tab[..., 0::2] = x0 * x0 * vc + x1 * x1 * vs
    tab[..., 1::2] = x0 * x0 * vs + x1 * x1 * vc
    return _ulp_var(y, 7) + tab


def predicted_sigma(qhat: np.ndarray, khat: np.ndarray, v: np.ndarray, o: np.ndarray,
                    var_q: torch.Tensor, var_k: torch.Tensor) -> torch.Tensor:
    """sigma [B, S, H, D] of the model above for exact rotated rows qhat, khat,
    values v, exact output o and channel error variances var_q, var_k (all
    [B, S, H, D]); one (batch, head) at a time."""
    qh = torch.from_numpy(np.ascontiguousarray(qhat, dtype=np.float64))
    kh = torch.from_numpy(np.ascontiguousarray(khat, dtype=np.float64))
    vv = torch.from_numpy(np.ascontiguousarray(v, dtype=np.float64))
    oo = torch.from_numpy(np.ascontiguousarray(o, dtype=np.float64))
    B, S, H, D = qh.shape
    sig2 = torch.empty_like(qh)
    for b in range(B):
        for h in range(H):
            q, k, val, out = qh[b, :, h], kh[b, :, h], vv[b, :, h], oo[b, :, h]
            w = torch.softmax(q @ k.T / math.sqrt(D), dim=-1)  # [S_q, S_k]
            w2 = w * w
            beta = (q * q) @ var_k[b, :, h].T / D
            a = w2 * beta
            t1 = a @ (val * val) - 2 * out * (a @ val) + out * out * a.sum(-1, keepdim=True)
            # M[i, p, d] = sum_j w_ij k_jp (v_jd - o_id)
            m = torch.einsum("ij,jp,jd->ipd", w, k, val) - (w @ k)[:, :, None] * out[:, None, :]
            t2 = torch.einsum("ip,ipd->id", var_q[b, :, h] / D, m * m)
            t3 = KAPPA * (w2 @ (val * val))
            t4 = _ulp_var(out, 7)
            sig2[b, :, h] = t1 + t2 + t3 + t4
    return sig2.sqrt()


def z_max(n: int) -> float:
    return math.sqrt(2.0 * math.log(n / 1e-3))


def check(got: np.ndarray, exact: np.ndarray, sigma: torch.Tensor, v_absmax: float):
    """Asserts both bounds; returns (max |err| / sigma-bound, mean / mean-bound)."""
    err = np.abs(np.asarray(got, dtype=np.float64) - exact)
    sig = sigma.numpy()
    n = err.size
    per_elem = z_max(n) * sig + FIXED * v_absmax
    worst = float((err / per_elem).max())
    mean_bound = float(np.sqrt((sig * sig).mean())) * (1.0 + 3.0 / math.sqrt(n))
    mean_ratio = float(err.mean()) / mean_bound
    assert np.isfinite(got).all()
    assert worst <= 1.0, (f"an element is {worst:.2f}x its bound: max err {err.max():.3e}, "
                          f"z {z_max(n):.2f}")
    assert mean_ratio <= 1.0, f"mean err {err.mean():.3e} > bound {mean_bound:.3e}"
    return worst, mean_ratio

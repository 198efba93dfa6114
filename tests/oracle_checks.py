"""Pins for the oracle: checks against what the pages and mathematics fix.

Each ``check_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees with an independent fact. None of them re-types the oracle's
formula: they use closed forms evaluated at high precision (mpmath), complex
exponentials instead of cos/sin tables, invariants of rotations and of the
softmax, torch's float64 scaled-dot-product attention (a library routine)
and brute-force loops on tiny inputs. tests/test_oracle_mutants.py plants
plausible mistakes in a copy of the oracle's C source and requires every one
of them to fail at least one check here.
"""
from __future__ import annotations

import cmath
import math

import numpy as np

FLUX_AXES = (32, 32, 32, 32)
FLUX_THETA = 2000.0


def _rng(seed):
    return np.random.default_rng(seed)


def _rand_ids(rng, S, n_axes=4, lo=-40, hi=600):
    return rng.integers(lo, hi, size=(S, n_axes)).astype(np.int32)


def rotate_complex(x, ids, axes_dims, theta):
    """Independent restatement of N-D RoPE with complex exponentials.

    x: [S, D] float64, ids: [S, n_axes]. Pair (2p, 2p+1) belongs to axis a and
    frequency index j; it is multiplied by exp(i * id_a * theta^(-2j/d_a)).
    """
    S, D = x.shape
    y = np.empty_like(x)
    for s in range(S):
        p = 0
        for a, d_a in enumerate(axes_dims):
            for j in range(d_a // 2):
                w = cmath.exp(1j * float(ids[s, a]) * theta ** (-(2.0 * j) / d_a))
                z = complex(x[s, 2 * p], x[s, 2 * p + 1]) * w
                y[s, 2 * p], y[s, 2 * p + 1] = z.real, z.imag
                p += 1
    return y


# ---------------------------------------------------------------- RoPE tables


def check_zero_ids_identity(orc):
    ids = np.zeros((5, 4), np.int32)
    c, s = orc.rope_tables(ids, FLUX_AXES, FLUX_THETA)
    assert c.shape == (5, 64) and np.all(c == 1.0) and np.all(s == 0.0)
    x = _rng(1).standard_normal((2, 5, 3, 128))
    y = orc.rope_apply(x, c, s)
    assert np.array_equal(x, y), "zero ids must leave q/k unchanged"


def check_frequencies_high_precision(orc):
    """cos/sin of id_a * theta^(-2j/d_a), per axis width, against mpmath."""
    import mpmath

    mpmath.mp.dps = 40
    for axes, theta, seed in ((FLUX_AXES, FLUX_THETA, 3), ((16, 48, 64), 10000.0, 4),
                              ((2, 6), 7.5, 5)):
        rng = _rng(seed)
        ids = _rand_ids(rng, 6, n_axes=len(axes))
        c, s = orc.rope_tables(ids, axes, theta)
        for t in range(ids.shape[0]):
            p = 0
            for a, d_a in enumerate(axes):
                for j in range(d_a // 2):
                    ang = mpmath.mpf(int(ids[t, a])) * mpmath.power(
                        mpmath.mpf(theta), -mpmath.mpf(2 * j) / d_a)
                    assert abs(c[t, p] - float(mpmath.cos(ang))) < 1e-12, (axes, t, a, j)
                    assert abs(s[t, p] - float(mpmath.sin(ang))) < 1e-12, (axes, t, a, j)
                    p += 1


def check_frequency_ratio(orc):
    """Along one axis the frequencies fall geometrically by theta^(-2/d_a)."""
    ids = np.array([[1, 1, 1, 1]], np.int32)
    c, s = orc.rope_tables(ids, FLUX_AXES, FLUX_THETA)
    ang = np.arctan2(s[0], c[0])  # all angles are in (0, 1], no wrap
    for a in range(4):
        seg = ang[16 * a:16 * a + 16]
        assert abs(seg[0] - 1.0) < 1e-15
        ratio = seg[1:] / seg[:-1]
        assert np.allclose(ratio, FLUX_THETA ** (-2.0 / 32), rtol=1e-12, atol=0)


# ------------------------------------------------------------- RoPE rotation


def check_rotation_keeps_norm(orc):
    rng = _rng(6)
    ids = _rand_ids(rng, 33)
    c, s = orc.rope_tables(ids, FLUX_AXES, FLUX_THETA)
    x = rng.standard_normal((2, 33, 3, 128))
    y = orc.rope_apply(x, c, s)
    assert np.allclose(np.linalg.norm(y, axis=-1), np.linalg.norm(x, axis=-1), rtol=1e-13)
    # each pair keeps its own length too
    px = np.hypot(x[..., 0::2], x[..., 1::2])
    py = np.hypot(y[..., 0::2], y[..., 1::2])
    assert np.allclose(px, py, rtol=1e-12, atol=1e-14)


def check_relative_position(orc):
    """RoPE(q, p) . RoPE(k, p') depends only on p' - p, axis by axis."""
    rng = _rng(7)
    n = 40
    p1, p2 = _rand_ids(rng, n), _rand_ids(rng, n)
    q = rng.standard_normal((1, n, 1, 128))
    k = rng.standard_normal((1, n, 1, 128))
    c1, s1 = orc.rope_tables(p1, FLUX_AXES, FLUX_THETA)
    c2, s2 = orc.rope_tables(p2, FLUX_AXES, FLUX_THETA)
    cd, sd = orc.rope_tables(p2 - p1, FLUX_AXES, FLUX_THETA)
    lhs = np.sum(orc.rope_apply(q, c1, s1) * orc.rope_apply(k, c2, s2), axis=-1)
    rhs = np.sum(q * orc.rope_apply(k, cd, sd), axis=-1)
    assert np.allclose(lhs, rhs, rtol=1e-10, atol=1e-10)


def check_rotation_complex_bruteforce(orc):
    rng = _rng(8)
    for axes, theta in ((FLUX_AXES, FLUX_THETA), ((16, 48, 64), 10000.0)):
        ids = _rand_ids(rng, 7, n_axes=len(axes))
        x = rng.standard_normal((1, 7, 1, sum(axes)))
        c, s = orc.rope_tables(ids, axes, theta)
        y = orc.rope_apply(x, c, s)[0, :, 0, :]
        ref = rotate_complex(x[0, :, 0, :], ids, axes, theta)
        assert np.allclose(y, ref, rtol=0, atol=1e-12)


def check_rotation_direction(orc):
    """Pair 0 of each axis turns by +id radians: (1, 0) -> (cos id, sin id)."""
    ids = np.array([[1, 2, 3, 4]], np.int32)
    c, s = orc.rope_tables(ids, FLUX_AXES, FLUX_THETA)
    x = np.zeros((1, 1, 1, 128))
    x[..., 0::2] = 1.0
    y = orc.rope_apply(x, c, s)[0, 0, 0]
    for a, idv in enumerate((1, 2, 3, 4)):
        ch = 2 * 16 * a
        assert abs(y[ch] - math.cos(idv)) < 1e-14 and abs(y[ch + 1] - math.sin(idv)) < 1e-14


# ----------------------------------------------------------------- attention


def _sdpa_f64(qh, kh, v):
    import torch

    q_t = torch.from_numpy(qh).permute(0, 2, 1, 3)  # [B, H, S, D]
    k_t = torch.from_numpy(kh).permute(0, 2, 1, 3)
    v_t = torch.from_numpy(v).permute(0, 2, 1, 3)
    o = torch.nn.functional.scaled_dot_product_attention(q_t, k_t, v_t)
    return o.permute(0, 2, 1, 3).contiguous().numpy()


def _rotate_all(x, ids, axes, theta):
    B, S, H, D = x.shape
    y = np.empty_like(x)
    for b in range(B):
        for h in range(H):
            y[b, :, h, :] = rotate_complex(x[b, :, h, :], ids, axes, theta)
    return y


def check_attention_vs_torch_sdpa(orc):
    rng = _rng(9)
    B, S_t, S_i, H, D = 2, 5, 32, 3, 128
    S = S_t + S_i
    txt, img = _rand_ids(rng, S_t), _rand_ids(rng, S_i)
    ids = np.concatenate([txt, img])
    for qscale in (1.0, 8.0):  # 8x makes the softmax peaked
        q = qscale * rng.standard_normal((B, S, H, D))
        k = rng.standard_normal((B, S, H, D))
        v = rng.standard_normal((B, S, H, D))
        out = orc.joint_rope_attention(q, k, v, txt, img, FLUX_AXES, FLUX_THETA, threads=3)
        ref = _sdpa_f64(_rotate_all(q, ids, FLUX_AXES, FLUX_THETA),
                        _rotate_all(k, ids, FLUX_AXES, FLUX_THETA), v)
        assert np.allclose(out, ref, rtol=0, atol=1e-11), np.abs(out - ref).max()


def check_attention_naive_loops(orc):
    """Triple loop with the textbook softmax exp(z)/sum exp(z), no max shift."""
    rng = _rng(10)
    axes, theta = (2, 2, 4), 50.0
    B, S, H, D = 1, 9, 2, 8
    ids = _rand_ids(rng, S, n_axes=3, lo=0, hi=20)
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    out = orc.joint_rope_attention(q, k, v, ids[:4], ids[4:], axes, theta, threads=1)
    ref = np.zeros_like(out)
    for b in range(B):
        for h in range(H):
            qh = rotate_complex(q[b, :, h, :], ids, axes, theta)
            kh = rotate_complex(k[b, :, h, :], ids, axes, theta)
            for i in range(S):
                w = [math.exp(sum(qh[i, c] * kh[j, c] for c in range(D)) / math.sqrt(D))
                     for j in range(S)]
                tot = sum(w)
                for c in range(D):
                    ref[b, i, h, c] = sum(w[j] * v[b, j, h, c] for j in range(S)) / tot
    assert np.allclose(out, ref, rtol=0, atol=1e-12), np.abs(out - ref).max()


def check_identical_keys_give_mean(orc):
    rng = _rng(11)
    B, S, H, D = 1, 23, 2, 128
    ids = np.tile(np.array([[3, 1, 4, 1]], np.int32), (S, 1))  # same position: same k^
    q = rng.standard_normal((B, S, H, D)) * 4
    k = np.broadcast_to(rng.standard_normal((B, 1, H, D)), (B, S, H, D)).copy()
    v = rng.standard_normal((B, S, H, D))
    out = orc.joint_rope_attention(q, k, v, ids[:3], ids[3:], FLUX_AXES, FLUX_THETA)
    assert np.allclose(out, np.broadcast_to(v.mean(axis=1, keepdims=True), out.shape),
                       rtol=0, atol=1e-13)


def check_constant_v_and_single_token(orc):
    rng = _rng(12)
    B, S, H, D = 2, 19, 2, 128
    txt, img = _rand_ids(rng, 4), _rand_ids(rng, 15)
    q, k = rng.standard_normal((B, S, H, D)), rng.standard_normal((B, S, H, D))
    out = orc.joint_rope_attention(q, k, np.ones((B, S, H, D)), txt, img)
    assert np.allclose(out, 1.0, rtol=0, atol=1e-13)
    q1, k1, v1 = (rng.standard_normal((B, 1, H, D)) for _ in range(3))
    out1 = orc.joint_rope_attention(q1, k1, v1, None, _rand_ids(rng, 1))
    assert np.allclose(out1, v1, rtol=0, atol=1e-15)


def check_translation_invariance(orc):
    rng = _rng(13)
    B, S, H, D = 1, 30, 2, 128
    txt, img = _rand_ids(rng, 6), _rand_ids(rng, 24)
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    shift = np.array([[7, -3, 11, 250]], np.int32)
    a = orc.joint_rope_attention(q, k, v, txt, img)
    b = orc.joint_rope_attention(q, k, v, txt + shift, img + shift)
    assert np.allclose(a, b, rtol=0, atol=1e-10)


def check_permutation_equivariance(orc):
    rng = _rng(14)
    B, S, H, D = 1, 26, 2, 128
    ids = _rand_ids(rng, S)
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    perm = rng.permutation(S)
    a = orc.joint_rope_attention(q, k, v, ids[:6], ids[6:])
    pi = ids[perm]
    b = orc.joint_rope_attention(q[:, perm], k[:, perm], v[:, perm], pi[:6], pi[6:])
    assert np.allclose(a[:, perm], b, rtol=0, atol=1e-12)


def check_rows_and_threads(orc):
    rng = _rng(15)
    B, S, H, D = 2, 40, 3, 128
    ids = _rand_ids(rng, S)
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    full1 = orc.joint_rope_attention(q, k, v, ids[:8], ids[8:], threads=1)
    full4 = orc.joint_rope_attention(q, k, v, ids[:8], ids[8:], threads=4)
    assert np.array_equal(full1, full4)
    rows = np.array([39, 0, 17, 17, 5])
    sub = orc.joint_rope_attention(q, k, v, ids[:8], ids[8:], rows=rows, threads=2)
    assert np.array_equal(sub, full1[:, rows])


# ------------------------------------------------------ QK RMS normalisation


def _torch_rms_norm(x, w, eps):
    import torch

    return torch.nn.functional.rms_norm(torch.from_numpy(x), (x.shape[-1],),
                                        weight=torch.from_numpy(w), eps=eps).numpy()


def check_rms_norm_mean_square(orc):
    """With unit weights the output's mean square is ms / (ms + eps) exactly
    (ms the input's mean square): 1 for large vectors, ms / eps for tiny ones."""
    rng = _rng(16)
    D = 128
    for scale in (1.0, 30.0, 1e-4):
        x = scale * rng.standard_normal((2, 7, 3, D))
        y = orc.rms_norm(x, np.ones(D), 1e-6)
        ms = (x * x).mean(axis=-1)
        assert np.allclose((y * y).mean(axis=-1), ms / (ms + 1e-6), rtol=1e-13, atol=0)


def check_rms_norm_vs_torch(orc):
    """torch's float64 rms_norm (a library routine) on random weights."""
    rng = _rng(17)
    D = 128
    w = rng.uniform(0.2, 2.0, D)
    for scale, eps in ((1.0, 1e-6), (1e-3, 1e-6), (5.0, 0.5)):
        x = scale * rng.standard_normal((1, 11, 2, D))
        y = orc.rms_norm(x, w, eps)
        assert np.allclose(y, _torch_rms_norm(x, w, eps), rtol=1e-13, atol=1e-15)


def check_qk_norm_attention_vs_sdpa(orc):
    """Attention with the QK norm: q and k normalised by torch's rms_norm with
    the text weights on the text tokens and the image weights on the others,
    rotated with complex exponentials, then torch's float64 SDPA."""
    rng = _rng(18)
    B, S_t, S_i, H, D = 1, 6, 27, 2, 128
    S = S_t + S_i
    txt, img = _rand_ids(rng, S_t), _rand_ids(rng, S_i)
    ids = np.concatenate([txt, img])
    q = 3.0 * rng.standard_normal((B, S, H, D))
    k = 0.5 * rng.standard_normal((B, S, H, D))
    v = rng.standard_normal((B, S, H, D))
    qw_t, kw_t, qw_i, kw_i = (rng.uniform(0.3, 2.5, D) for _ in range(4))
    eps = 1e-6
    qn = np.concatenate([_torch_rms_norm(q[:, :S_t], qw_t, eps),
                         _torch_rms_norm(q[:, S_t:], qw_i, eps)], axis=1)
    kn = np.concatenate([_torch_rms_norm(k[:, :S_t], kw_t, eps),
                         _torch_rms_norm(k[:, S_t:], kw_i, eps)], axis=1)
    ref = _sdpa_f64(_rotate_all(qn, ids, FLUX_AXES, FLUX_THETA),
                    _rotate_all(kn, ids, FLUX_AXES, FLUX_THETA), v)
    out = orc.joint_rope_attention(q, k, v, txt, img, FLUX_AXES, FLUX_THETA, threads=2,
                                   qk_norm=(qw_t, kw_t, qw_i, kw_i, eps))
    assert np.allclose(out, ref, rtol=0, atol=1e-11), np.abs(out - ref).max()
    # the norm removes any positive per-token scale of q and k (eps aside)
    scl = rng.uniform(0.5, 4.0, (B, S, 1, 1))
    out2 = orc.joint_rope_attention(q * scl, k / scl, v, txt, img, FLUX_AXES, FLUX_THETA,
                                    qk_norm=(qw_t, kw_t, qw_i, kw_i, 0.0))
    out3 = orc.joint_rope_attention(q, k, v, txt, img, FLUX_AXES, FLUX_THETA,
                                    qk_norm=(qw_t, kw_t, qw_i, kw_i, 0.0))
    assert np.allclose(out2, out3, rtol=0, atol=1e-12)


# ---------------------------------------------------- reference KV modes


def _sdpa_masked_f64(qh, kh, v, mask):
    """torch float64 SDPA with a boolean mask [S_q, S_k] (True = attend)."""
    import torch

    q_t = torch.from_numpy(qh).permute(0, 2, 1, 3)
    k_t = torch.from_numpy(kh).permute(0, 2, 1, 3)
    v_t = torch.from_numpy(v).permute(0, 2, 1, 3)
    o = torch.nn.functional.scaled_dot_product_attention(q_t, k_t, v_t,
                                                         attn_mask=torch.from_numpy(mask))
    return o.permute(0, 2, 1, 3).contiguous().numpy()


def check_extract_mode_vs_masked_sdpa(orc):
    """[txt ; ref ; img]: reference queries see reference keys only, the rest
    see every key (a boolean mask for torch's SDPA); the cache holds the
    reference keys rotated (complex exponentials) and their values."""
    rng = _rng(19)
    B, n_t, n_r, n_i, H, D = 2, 5, 11, 14, 2, 128
    S = n_t + n_r + n_i
    txt, ref, img = _rand_ids(rng, n_t), _rand_ids(rng, n_r), _rand_ids(rng, n_i)
    ids = np.concatenate([txt, ref, img])
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    out, ck, cv = orc.attention_extract(q, k, v, txt, ref, img)
    mask = np.ones((S, S), dtype=bool)
    mask[n_t:n_t + n_r, :] = False
    mask[n_t:n_t + n_r, n_t:n_t + n_r] = True
    kh = _rotate_all(k, ids, FLUX_AXES, FLUX_THETA)
    ref_out = _sdpa_masked_f64(_rotate_all(q, ids, FLUX_AXES, FLUX_THETA), kh, v, mask)
    assert np.allclose(out, ref_out, rtol=0, atol=1e-11), np.abs(out - ref_out).max()
    assert np.allclose(ck, kh[:, n_t:n_t + n_r], rtol=0, atol=1e-12)
    assert np.array_equal(cv, v[:, n_t:n_t + n_r])


def check_cached_mode_vs_concatenated_sdpa(orc):
    """[txt ; img] queries over keys [txt ; cache ; img] built explicitly."""
    rng = _rng(20)
    B, n_t, n_i, n_r, H, D = 1, 6, 21, 9, 3, 128
    S = n_t + n_i
    txt, img = _rand_ids(rng, n_t), _rand_ids(rng, n_i)
    ids = np.concatenate([txt, img])
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    ck, cv = rng.standard_normal((B, n_r, H, D)), rng.standard_normal((B, n_r, H, D))
    out = orc.attention_cached(q, k, v, txt, img, ck, cv)
    kh = _rotate_all(k, ids, FLUX_AXES, FLUX_THETA)
    keys = np.concatenate([kh[:, :n_t], ck, kh[:, n_t:]], axis=1)
    vals = np.concatenate([v[:, :n_t], cv, v[:, n_t:]], axis=1)
    ref_out = _sdpa_f64(_rotate_all(q, ids, FLUX_AXES, FLUX_THETA), keys, vals)
    assert np.allclose(out, ref_out, rtol=0, atol=1e-11), np.abs(out - ref_out).max()


def check_extract_then_cached_reproduces_rows(orc):
    """The cache's purpose: with the same text and image inputs, cached mode
    gives the text and image rows that extract mode gave."""
    rng = _rng(21)
    B, n_t, n_r, n_i, H, D = 1, 4, 10, 17, 2, 128
    txt, ref, img = _rand_ids(rng, n_t), _rand_ids(rng, n_r), _rand_ids(rng, n_i)
    S = n_t + n_r + n_i
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    out, ck, cv = orc.attention_extract(q, k, v, txt, ref, img)
    keep = np.r_[0:n_t, n_t + n_r:S]
    out2 = orc.attention_cached(q[:, keep], k[:, keep], v[:, keep], txt, img, ck, cv)
    assert np.allclose(out2, out[:, keep], rtol=0, atol=1e-12)
    # row subsets give the same rows
    rows = np.array([S - 1, 0, n_t + 3, n_t])
    sub, ck2, _ = orc.attention_extract(q, k, v, txt, ref, img, rows=rows)
    assert np.array_equal(sub, out[:, rows]) and np.array_equal(ck2, ck)
    sub2 = orc.attention_cached(q[:, keep], k[:, keep], v[:, keep], txt, img, ck, cv,
                                rows=np.array([2, 0]))
    assert np.array_equal(sub2, out2[:, [2, 0]])


def check_kv_modes_with_qk_norm(orc):
    """Extract and cached with the QK norm equal the plain modes on q and k
    normalised beforehand by torch's float64 rms_norm (text tokens with the
    text weights, reference and image tokens with the image weights)."""
    rng = _rng(43)
    B, H, D = 1, 2, 16
    S_t, S_r, S_i = 5, 9, 7
    S = S_t + S_r + S_i
    ids = _rand_ids(rng, S)
    txt, ref, img = ids[:S_t], ids[S_t:S_t + S_r], ids[S_t + S_r:]
    q, k, v = (rng.standard_normal((B, S, H, D)) for _ in range(3))
    ws = [rng.uniform(0.3, 1.7, D) for _ in range(4)]  # q txt, k txt, q img, k img
    eps = 1e-6

    def normed(x, w_txt, w_img, n_txt):
        y = np.empty_like(x)
        y[:, :n_txt] = _torch_rms_norm(x[:, :n_txt], w_txt, eps)
        y[:, n_txt:] = _torch_rms_norm(x[:, n_txt:], w_img, eps)
        return y

    axes = (4, 4, 4, 4)
    qn, kn = normed(q, ws[0], ws[2], S_t), normed(k, ws[1], ws[3], S_t)
    ref_out, ref_ck, ref_cv = orc.attention_extract(qn, kn, v, txt, ref, img, axes, 50.0)
    out, ck, cv = orc.attention_extract(q, k, v, txt, ref, img, axes, 50.0,
                                        qk_norm=tuple(ws) + (eps,))
    assert np.allclose(out, ref_out, rtol=1e-12, atol=1e-13)
    assert np.allclose(ck, ref_ck, rtol=1e-12, atol=1e-13) and np.array_equal(cv, ref_cv)
    keep = np.r_[0:S_t, S_t + S_r:S]
    q2, k2, v2 = q[:, keep], k[:, keep], v[:, keep]
    q2n, k2n = normed(q2, ws[0], ws[2], S_t), normed(k2, ws[1], ws[3], S_t)
    ref2 = orc.attention_cached(q2n, k2n, v2, txt, img, ck, cv, axes, 50.0)
    got2 = orc.attention_cached(q2, k2, v2, txt, img, ck, cv, axes, 50.0,
                                qk_norm=tuple(ws) + (eps,))
    assert np.allclose(got2, ref2, rtol=1e-12, atol=1e-13)


def _torch_silu(x):
    import torch

    return torch.nn.functional.silu(torch.from_numpy(np.asarray(x, dtype=np.float64))).numpy()


def check_proj_selection_weights(orc):
    """Weights whose rows are unit vectors select input channels: every output
    must be exactly the selected channel, placed where the split puts it
    (Q, K, V heads in [H, D] order, then the gate and linear halves), and the
    activation is torch's float64 silu of the gate times the linear half."""
    rng = _rng(40)
    M, dim, H, D, mlp = 5, 23, 3, 4, 7
    inner = H * D
    n_out = 3 * inner + 2 * mlp
    pick = rng.integers(0, dim, size=n_out)
    w = np.zeros((n_out, dim))
    w[np.arange(n_out), pick] = 1.0
    x = rng.standard_normal((M, dim))
    q, k, v, act = orc.qkv_mlp_proj(x, w, H, D, mlp)
    for t, base in ((q, 0), (k, inner), (v, 2 * inner)):
        for h in range(H):
            for d in range(D):
                assert np.array_equal(t[:, h, d], x[:, pick[base + h * D + d]])
    g = x[:, pick[3 * inner:3 * inner + mlp]]
    u = x[:, pick[3 * inner + mlp:]]
    assert np.allclose(act, _torch_silu(g) * u, rtol=1e-14, atol=1e-15)


def check_proj_vs_torch_matmul(orc):
    """Random weights: torch's float64 matmul and silu (library routines) on
    slices taken by their column ranges."""
    import torch

    rng = _rng(41)
    M, dim, H, D, mlp = 9, 64, 2, 8, 24
    inner = H * D
    x = rng.standard_normal((M, dim))
    w = rng.standard_normal((3 * inner + 2 * mlp, dim)) / math.sqrt(dim)
    y = (torch.from_numpy(x) @ torch.from_numpy(w).T).numpy()
    q, k, v, act = orc.qkv_mlp_proj(x, w, H, D, mlp)
    assert np.allclose(q.reshape(M, inner), y[:, :inner], rtol=1e-12, atol=1e-13)
    assert np.allclose(k.reshape(M, inner), y[:, inner:2 * inner], rtol=1e-12, atol=1e-13)
    assert np.allclose(v.reshape(M, inner), y[:, 2 * inner:3 * inner], rtol=1e-12, atol=1e-13)
    g, u = y[:, 3 * inner:3 * inner + mlp], y[:, 3 * inner + mlp:]
    assert np.allclose(act, _torch_silu(g) * u, rtol=1e-12, atol=1e-13)
    rows = np.array([M - 1, 0, 4])
    sq, sk, sv, sa = orc.qkv_mlp_proj(x, w, H, D, mlp, rows=rows)
    assert np.array_equal(sq, q[rows]) and np.array_equal(sa, act[rows])
    assert np.array_equal(sk, k[rows]) and np.array_equal(sv, v[rows])


def check_proj_silu_closed_forms(orc):
    """SiLU's closed forms through the projection: silu(0) = 0,
    silu(g) - silu(-g) = g, silu(g) -> g for large g and -> 0 for very
    negative g (a linear half of ones makes act = silu(gate))."""
    rng = _rng(42)
    H, D, mlp, dim = 1, 2, 6, 3
    inner = H * D
    w = np.zeros((3 * inner + 2 * mlp, dim))
    w[3 * inner:3 * inner + mlp, 0] = [0.0, 1.0, -1.0, 2.5, -2.5, 1.0]
    w[3 * inner + mlp:, 1] = 1.0  # the linear half reads channel 1
    for g0 in (0.7, -1.3, 3.1):
        x = np.array([[g0, 1.0, rng.standard_normal()]])
        _, _, _, a = orc.qkv_mlp_proj(x, w, H, D, mlp)
        a = a[0]
        assert a[0] == 0.0
        assert abs((a[1] - a[2]) - g0) < 1e-15
        assert abs((a[3] - a[4]) - 2.5 * g0) < 1e-14
        assert abs(a[5] - g0 / (1.0 + math.exp(-g0))) < 1e-15
    x = np.array([[60.0, 1.0, 0.0]])
    _, _, _, a = orc.qkv_mlp_proj(x, w, H, D, mlp)
    assert abs(a[0, 1] - 60.0) < 1e-12 and abs(a[0, 2]) < 1e-20


ALL_CHECKS = [
    check_zero_ids_identity,
    check_frequencies_high_precision,
    check_frequency_ratio,
    check_rotation_keeps_norm,
    check_relative_position,
    check_rotation_complex_bruteforce,
    check_rotation_direction,
    check_attention_vs_torch_sdpa,
    check_attention_naive_loops,
    check_identical_keys_give_mean,
    check_constant_v_and_single_token,
    check_translation_invariance,
    check_permutation_equivariance,
    check_rows_and_threads,
    check_rms_norm_mean_square,
    check_rms_norm_vs_torch,
    check_qk_norm_attention_vs_sdpa,
    check_extract_mode_vs_masked_sdpa,
    check_cached_mode_vs_concatenated_sdpa,
    check_extract_then_cached_reproduces_rows,
    check_kv_modes_with_qk_norm,
    check_proj_selection_weights,
    check_proj_vs_torch_matmul,
    check_proj_silu_closed_forms,
]

"""GPU parity of the reference-image KV modes against the oracle.

Extract mode ("Diffusers 中 Flux2Transformer2DModel 全面解析", section
参考图 KV 缓存机制): tokens [txt ; ref ; img], reference queries attend to
the reference keys only, text and image queries to every key, and the
reference tokens' rotated K and their V go to the cache. Cached mode: queries
[txt ; img] attend to the keys [txt ; cache ; img]. Bar: max |gpu - oracle|
<= 1e-2, mean <= 1e-3; the cache's K within the fp16 table and bf16 storage
rounding of the rotated values, its V bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_joint_gb300 import binding, build
from diffusion_transformer_joint_gb300 import workloads as W
from tests.oracle_parallel import by_head as _by_head

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _dev(x):
    if x is None:
        return None
    return x.cuda() if isinstance(x, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x)).cuda()


def _bar(got, ref):
    err = np.abs(got.astype(np.float64) - ref)
    assert np.isfinite(got).all()
    assert err.max() <= MAX_ABS, f"max abs err {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"mean abs err {err.mean():.3e}"


def _inputs(B, S, H, seed):
    return (W.normal_bf16((B, S, H, 128), seed), W.normal_bf16((B, S, H, 128), seed + 1),
            W.normal_bf16((B, S, H, 128), seed + 2))


def _check_cache_k(got, ref, k_raw):
    """The cached K is the kernel's rotated key: fp16 (cos, sin) table entries
    (relative error 2^-11 each, so up to (|x_2i| + |x_2i+1|) * 2^-11 on a
    pair's outputs, cancellation included) and one bf16 rounding (2^-9
    relative). Both bounds are doubled for slack."""
    pair = np.abs(k_raw.reshape(*k_raw.shape[:-1], -1, 2)).sum(-1)
    mag = np.repeat(pair, 2, axis=-1)
    assert np.all(np.abs(got - ref) <= 2.0 ** -8 * np.abs(ref) + 2.0 ** -10 * mag + 1e-6)


def _seg(ids, lo, n):
    return ids[lo:lo + n] if n else None


@pytest.mark.parametrize("B,H,S_t,S_r,S_i", [
    (1, 2, 16, 64, 64),     # tiny-like, segments tile-unaligned
    (1, 2, 0, 130, 70),     # no text; reference block crosses a tile
    (2, 3, 7, 121, 0),      # no image
    (1, 2, 100, 0, 300),    # no reference (plain attention, empty cache)
    (1, 1, 33, 200, 290),   # every boundary off the 128 and 256 grids
])
def test_extract_small_shapes(B, H, S_t, S_r, S_i):
    S = S_t + S_r + S_i
    q, k, v = _inputs(B, S, H, 600 + S)
    ids = W.random_ids(S, 604 + S, 0, 300)
    txt, ref, img = _seg(ids, 0, S_t), _seg(ids, S_t, S_r), _seg(ids, S_t + S_r, S_i)
    out, ck, cv = binding.attention_extract(_dev(q), _dev(k), _dev(v), _dev(txt), _dev(ref),
                                            _dev(img))
    torch.cuda.synchronize()
    r_out, r_ck, r_cv = oracle.attention_extract(q.float().numpy(), k.float().numpy(),
                                                 v.float().numpy(), txt, ref, img)
    _bar(out.float().cpu().numpy(), r_out)
    if S_r:
        _check_cache_k(ck.float().cpu().numpy(), r_ck, k[:, S_t:S_t + S_r].float().numpy())
        assert torch.equal(cv.cpu(), v[:, S_t:S_t + S_r])


@pytest.mark.parametrize("B,H,S_t,S_i,S_r", [
    (1, 2, 16, 64, 64),
    (2, 2, 0, 150, 33),
    (1, 3, 40, 0, 300),
    (1, 2, 77, 180, 0),
])
def test_cached_small_shapes(B, H, S_t, S_i, S_r):
    S = S_t + S_i
    q, k, v = _inputs(B, S, H, 700 + S + S_r)
    ck = W.normal_bf16((B, S_r, H, 128), 703 + S)
    cv = W.normal_bf16((B, S_r, H, 128), 704 + S)
    ids = W.random_ids(S, 705 + S, 0, 300)
    txt, img = _seg(ids, 0, S_t), _seg(ids, S_t, S_i)
    out = binding.attention_cached(_dev(q), _dev(k), _dev(v), _dev(txt), _dev(img), _dev(ck),
                                   _dev(cv))
    torch.cuda.synchronize()
    ref = oracle.attention_cached(q.float().numpy(), k.float().numpy(), v.float().numpy(), txt,
                                  img, ck.float().numpy(), cv.float().numpy())
    _bar(out.float().cpu().numpy(), ref)


def test_extract_then_cached_on_the_gpu():
    """The GPU's own cache, fed back: cached-mode rows match the oracle, and
    they match extract mode's text and image rows."""
    B, H, S_t, S_r, S_i = 1, 2, 40, 300, 213
    S = S_t + S_r + S_i
    q, k, v = _inputs(B, S, H, 801)
    ids = W.random_ids(S, 804, 0, 300)
    txt, ref, img = ids[:S_t], ids[S_t:S_t + S_r], ids[S_t + S_r:]
    out, ck, cv = binding.attention_extract(_dev(q), _dev(k), _dev(v), _dev(txt), _dev(ref),
                                            _dev(img))
    keep = np.r_[0:S_t, S_t + S_r:S]
    qk, kk, vk = q[:, keep].contiguous(), k[:, keep].contiguous(), v[:, keep].contiguous()
    out2 = binding.attention_cached(_dev(qk), _dev(kk), _dev(vk), _dev(txt), _dev(img), ck, cv)
    torch.cuda.synchronize()
    ref = oracle.attention_cached(qk.float().numpy(), kk.float().numpy(), vk.float().numpy(), txt,
                                  img, ck.float().cpu().numpy(), cv.float().cpu().numpy())
    _bar(out2.float().cpu().numpy(), ref)
    _bar(out2.float().cpu().numpy(), out[:, keep].float().cpu().numpy().astype(np.float64))


def test_two_reference_edit_workload_all_outputs():
    """The klein-9B two-reference edit shape as the KV pipeline runs it: one
    extract call over [txt 512 ; ref 8192 ; img 4096], then a cached call
    over [txt ; img] with that cache. Every output of both calls against the
    oracle; the whole cache against the oracle's."""
    w = W.WORKLOADS["klein9b_edit2"]
    S_t, S_i, S_r = w.S_txt, 4096, w.S_img - 4096
    q0, k0, v0 = W.workload_qkv(w)  # [txt ; img ; refs]: reorder to [txt ; refs ; img]
    order = np.r_[0:S_t, S_t + S_i:w.S, S_t:S_t + S_i]
    q, k, v = (x[:, order].contiguous() for x in (q0, k0, v0))
    t_ids, i_ids = W.workload_ids(w)
    ids = np.concatenate([t_ids, i_ids])[order]
    txt, ref, img = ids[:S_t], ids[S_t:S_t + S_r], ids[S_t + S_r:]
    out, ck, cv = binding.attention_extract(_dev(q), _dev(k), _dev(v), _dev(txt), _dev(ref),
                                            _dev(img))
    torch.cuda.synchronize()
    qn, kn, vn = q.float().numpy(), k.float().numpy(), v.float().numpy()
    r_out, r_ck, _ = _by_head(oracle.attention_extract, w.H, qn, kn, vn, txt, ref, img)
    _bar(out.float().cpu().numpy(), r_out)
    _check_cache_k(ck.float().cpu().numpy(), r_ck, kn[:, S_t:S_t + S_r])
    assert torch.equal(cv.cpu(), v[:, S_t:S_t + S_r])
    keep = np.r_[0:S_t, S_t + S_r:w.S]
    qk, kk, vk = q[:, keep].contiguous(), k[:, keep].contiguous(), v[:, keep].contiguous()
    out2 = binding.attention_cached(_dev(qk), _dev(kk), _dev(vk), _dev(txt), _dev(img), ck, cv)
    torch.cuda.synchronize()
    r2 = _by_head(oracle.attention_cached, w.H, qk.float().numpy(), kk.float().numpy(),
                  vk.float().numpy(), txt, img, ck.float().cpu().numpy(), cv.float().cpu().numpy())
    _bar(out2.float().cpu().numpy(), r2)


def _norm_weights(seed, eps=1e-6):
    rng = np.random.default_rng(seed)
    return [rng.uniform(0.5, 1.5, 128).astype(np.float32) for _ in range(4)], eps


def _normed(x, w_txt, w_img, n_txt, eps):
    """x / sqrt(mean x^2 + eps) * w per head vector, in float64 (for error bounds)."""
    x = x.astype(np.float64)
    r = 1.0 / np.sqrt((x * x).mean(axis=-1, keepdims=True) + eps)
    w = np.concatenate([np.broadcast_to(w_txt, (n_txt, 128)),
                        np.broadcast_to(w_img, (x.shape[1] - n_txt, 128))])[None, :, None, :]
    return x * r * w


@pytest.mark.parametrize("B,H,S_t,S_r,S_i", [(1, 2, 16, 64, 64), (1, 1, 33, 200, 290)])
def test_kv_modes_with_qk_norm(B, H, S_t, S_r, S_i):
    """Extract then cached with the QK RMS normalisation before RoPE: outputs
    against the oracle, the cache's K against the normalised, rotated keys,
    and cached mode fed with the GPU's own cache."""
    S = S_t + S_r + S_i
    q, k, v = _inputs(B, S, H, 1200 + S)
    ids = W.random_ids(S, 1204 + S, 0, 300)
    txt, ref, img = ids[:S_t], ids[S_t:S_t + S_r], ids[S_t + S_r:]
    ws, eps = _norm_weights(1205 + S)
    norm_dev = tuple(_dev(w) for w in ws) + (eps,)
    norm_np = tuple(ws) + (eps,)
    out, ck, cv = binding.attention_extract(_dev(q), _dev(k), _dev(v), _dev(txt), _dev(ref),
                                            _dev(img), qk_norm=norm_dev)
    torch.cuda.synchronize()
    r_out, r_ck, _ = oracle.attention_extract(q.float().numpy(), k.float().numpy(),
                                              v.float().numpy(), txt, ref, img, qk_norm=norm_np)
    _bar(out.float().cpu().numpy(), r_out)
    kn = _normed(k.float().numpy(), ws[1], ws[3], S_t, eps)[:, S_t:S_t + S_r]
    _check_cache_k(ck.float().cpu().numpy(), r_ck, kn)
    assert torch.equal(cv.cpu(), v[:, S_t:S_t + S_r])
    keep = np.r_[0:S_t, S_t + S_r:S]
    qk, kk, vk = q[:, keep].contiguous(), k[:, keep].contiguous(), v[:, keep].contiguous()
    out2 = binding.attention_cached(_dev(qk), _dev(kk), _dev(vk), _dev(txt), _dev(img), ck, cv,
                                    qk_norm=norm_dev)
    torch.cuda.synchronize()
    ref2 = oracle.attention_cached(qk.float().numpy(), kk.float().numpy(), vk.float().numpy(), txt,
                                   img, ck.float().cpu().numpy(), cv.float().cpu().numpy(),
                                   qk_norm=norm_np)
    _bar(out2.float().cpu().numpy(), ref2)
    _bar(out2.float().cpu().numpy(), out[:, keep].float().cpu().numpy().astype(np.float64))

"""The checked build of the library (compiled with -DFLUX_DEBUG) on the GPU.

In that build the attention kernel checks, before each shared-memory, TMEM,
TMA and global access site (the work queue, the K / V rings, the Q tiles, the
epilogue staging, the table copies, the exchange buffer and its publication
flags, the output rows), that the region, stage, lane quadrant, column range,
coordinates and rows it is about to use lie inside what the site may touch. A
failed check skips the access and puts FLUX_DEBUG_STATUS_BASE - site into the
status word; nothing traps. This is the memory-safety evidence for the
kernel's cross-CTA exchange protocol that a sanitizer would otherwise give.

Every case below (tiny, ragged, more work items than thread blocks, the QK
norm, a head range, a query-row slice, both KV modes, the caller-built table,
with and without the exchange buffer) must end with status 0 and give output
bit-identical to the release build's.
"""
import ctypes

import numpy as np
import pytest
import torch

from diffusion_transformer_joint_gb300 import binding, build
from diffusion_transformer_joint_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def libs():
    release = binding.load(build.build())
    checked = ctypes.CDLL(build.build_checked())
    for name in binding.EXPORTS + ("flux_status_string",):
        fn_r, fn_c = getattr(release, name), getattr(checked, name)
        fn_c.argtypes, fn_c.restype = fn_r.argtypes, fn_r.restype
    return release, checked


def _inputs(B, S, H, seed):
    q, k, v = (W.normal_bf16((B, S, H, 128), seed + i).cuda() for i in range(3))
    ids = torch.from_numpy(W.random_ids(S, seed + 3, 0, 300)).cuda()
    return q, k, v, ids


def _both(libs, monkeypatch, run):
    """run() with the checked library swapped in, then with the release one;
    run returns (outputs, status words)."""
    release, checked = libs
    monkeypatch.setattr(binding, "_lib", checked)
    outs_c, stats = run()
    torch.cuda.synchronize()
    monkeypatch.setattr(binding, "_lib", release)
    outs_r, _ = run()
    torch.cuda.synchronize()
    for st in stats:
        assert st == 0, f"checked build status {st}: {release.flux_status_string(st)}"
    for a, b in zip(outs_c, outs_r):
        assert torch.equal(a, b)


@pytest.mark.parametrize("B,H,S_txt,S_img", [
    (1, 2, 16, 64), (2, 3, 7, 121), (1, 3, 100, 413), (1, 160, 40, 216), (1, 9, 512, 3840)])
@pytest.mark.parametrize("share_k", [True, False])
def test_one_call_passes_every_check(libs, monkeypatch, B, H, S_txt, S_img, share_k):
    S = S_txt + S_img
    q, k, v, ids = _inputs(B, S, H, 6000 + S)

    def run():
        n = binding.workspace_shared_bytes(B, S, H) if share_k else binding.workspace_bytes(S)
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
        out = binding.joint_rope_attention(q, k, v, ids[:S_txt], ids[S_txt:], workspace=ws)
        return [out], [binding.query_status(ws)]

    _both(libs, monkeypatch, run)


def test_qk_norm_head_range_and_row_slice_pass_every_check(libs, monkeypatch):
    B, H, S, S_txt = 2, 7, 1000, 100
    q, k, v, ids = _inputs(B, S, H, 6100)
    rng = np.random.default_rng(6104)
    norm = tuple(torch.from_numpy(rng.uniform(0.5, 1.5, 128).astype(np.float32)).cuda()
                 for _ in range(4)) + (1e-6,)
    txt, img = ids[:S_txt], ids[S_txt:]

    def run():
        outs, stats = [], []
        ws = torch.zeros(binding.workspace_shared_bytes(B, S, H), dtype=torch.uint8, device="cuda")
        outs.append(binding.joint_rope_attention(q, k, v, txt, img, workspace=ws, qk_norm=norm))
        stats.append(binding.query_status(ws))
        ws = torch.zeros(binding.workspace_shared_bytes(B, S, 5), dtype=torch.uint8, device="cuda")
        out = torch.zeros_like(q)
        binding.joint_rope_attention_heads(q, k, v, txt, img, 1, 5, out=out, workspace=ws)
        outs.append(out)
        stats.append(binding.query_status(ws))
        ws = torch.zeros(binding.rows_workspace_bytes(B, 300, S, H), dtype=torch.uint8,
                         device="cuda")
        outs.append(binding.joint_rope_attention_rows(q[:, 100:400].contiguous(), 100, k, v, txt,
                                                      img, workspace=ws))
        stats.append(binding.query_status(ws))
        table = binding.rope_tables_packed(ids)
        status = torch.zeros(1, dtype=torch.int32, device="cuda")
        krot = torch.zeros(binding.krot_bytes(B, S, H), dtype=torch.uint8, device="cuda")
        outs.append(binding.joint_rope_attention_tabled(q, k, v, table, status, krot=krot))
        torch.cuda.synchronize()
        stats.append(int(status.item()))
        return outs, stats

    _both(libs, monkeypatch, run)


@pytest.mark.parametrize("B,H,S_t,S_r,S_i", [(1, 1, 33, 200, 290), (2, 2, 0, 130, 70)])
def test_kv_modes_pass_every_check(libs, monkeypatch, B, H, S_t, S_r, S_i):
    S = S_t + S_r + S_i
    q, k, v, ids = _inputs(B, S, H, 6200 + S)
    txt = ids[:S_t] if S_t else None
    ref, img = ids[S_t:S_t + S_r], ids[S_t + S_r:]
    keep = np.r_[0:S_t, S_t + S_r:S]

    def run():
        ws = torch.zeros(binding.extract_workspace_bytes(B, S_t, S_r, S_i, H), dtype=torch.uint8,
                         device="cuda")
        out, ck, cv = binding.attention_extract(q, k, v, txt, ref, img, workspace=ws)
        st1 = binding.query_status(ws)
        qk, kk, vk = (x[:, keep].contiguous() for x in (q, k, v))
        ws2 = torch.zeros(binding.cached_workspace_bytes(B, S_t, S_i, S_r, H), dtype=torch.uint8,
                          device="cuda")
        out2 = binding.attention_cached(qk, kk, vk, txt, img, ck, cv, workspace=ws2)
        return [out, ck, cv, out2], [st1, binding.query_status(ws2)]

    _both(libs, monkeypatch, run)

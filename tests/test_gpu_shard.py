"""GPU checks of the entry points that tensor- and sequence-parallel callers use
("Diffusers 中 Flux2Transformer2DModel 全面解析", section 并行化支持), run on one
GPU: each rank's call is made in turn on the same device.

Head parallel: flux_joint_rope_attention_heads over a rank's heads gives, bit
for bit, the full call's output for those heads and leaves every other head
of ``out`` untouched; the ranks' calls together rebuild the full output.

Sequence parallel: flux_joint_rope_attention_rows over a rank's query rows
(every key and value given) matches the oracle's rows within the bar
(max 1e-2, mean 1e-3); the ranks' calls together match the full call within
twice the bar (both are rounded; the key order of a row can differ).
"""
import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_joint_gb300 import binding, build, shard
from diffusion_transformer_joint_gb300 import workloads as W

pytestmark = pytest.mark.gpu

MAX_ABS = 1e-2
MEAN_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.load()


def _inputs(B, S, H, seed):
    q, k, v = (W.normal_bf16((B, S, H, 128), seed + i).cuda() for i in range(3))
    ids = torch.from_numpy(W.random_ids(S, seed + 3, 0, 300)).cuda()
    return q, k, v, ids


@pytest.mark.parametrize("B,H,S,S_txt", [(1, 2, 80, 16), (2, 7, 1000, 100), (1, 9, 4352, 512)])
def test_heads_entry_reproduces_the_full_call(B, H, S, S_txt):
    q, k, v, ids = _inputs(B, S, H, 5000 + S)
    txt, img = ids[:S_txt], ids[S_txt:]
    full = binding.joint_rope_attention(q, k, v, txt, img)
    for h0, n in ((0, 1), (H - 1, 1), (1, H - 1), (0, H)):
        for share_k in (True, False):
            out = torch.full_like(q, 7.0)
            binding.joint_rope_attention_heads(q, k, v, txt, img, h0, n, out=out,
                                               share_k=share_k)
            torch.cuda.synchronize()
            assert torch.equal(out[:, :, h0:h0 + n], full[:, :, h0:h0 + n]), (h0, n, share_k)
            rest = torch.cat([out[:, :, :h0], out[:, :, h0 + n:]], dim=2)
            assert bool((rest == 7.0).all()), "heads outside the range were written"


@pytest.mark.parametrize("world", [2, 3, 8])
def test_head_parallel_ranks_rebuild_the_klein9b_output(world):
    w = W.WORKLOADS["klein9b"]
    q, k, v = (t.cuda() for t in W.workload_qkv(w))
    txt, img = (torch.from_numpy(x).cuda() for x in W.workload_ids(w))
    full = binding.joint_rope_attention(q, k, v, txt, img)
    out = torch.full_like(q, 7.0)
    for r in range(world):
        h0, n = shard.head_range(r, world, w.H)
        binding.joint_rope_attention_heads(q, k, v, txt, img, h0, n, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, full)


def test_heads_entry_rejects_bad_ranges():
    q, k, v, ids = _inputs(1, 80, 4, 5100)
    for h0, n in ((-1, 2), (0, 0), (3, 2), (4, 1)):
        with pytest.raises(binding.FluxError):
            binding.joint_rope_attention_heads(q, k, v, ids[:16], ids[16:], h0, n)


def _oracle_rows(q, k, v, txt, img, rows):
    return oracle.joint_rope_attention(q.float().cpu().numpy(), k.float().cpu().numpy(),
                                       v.float().cpu().numpy(), txt.cpu().numpy(),
                                       img.cpu().numpy(), rows=rows)


@pytest.mark.parametrize("q0,n", [(0, 1), (999, 1), (100, 300), (128, 256), (5, 990), (0, 1000)])
def test_rows_entry_matches_the_oracle(q0, n):
    B, H, S, S_txt = 2, 3, 1000, 100
    q, k, v, ids = _inputs(B, S, H, 5200)
    txt, img = ids[:S_txt], ids[S_txt:]
    for share_k in (True, False):
        out = binding.joint_rope_attention_rows(q[:, q0:q0 + n].contiguous(), q0, k, v, txt, img,
                                                share_k=share_k)
        torch.cuda.synchronize()
        ref = _oracle_rows(q, k, v, txt, img, np.arange(q0, q0 + n))
        err = np.abs(out.float().cpu().numpy() - ref)
        assert err.max() <= MAX_ABS and err.mean() <= MEAN_ABS, (share_k, err.max(), err.mean())


def test_rows_entry_rejects_bad_slices():
    q, k, v, ids = _inputs(1, 80, 2, 5300)
    for q0, n in ((-1, 10), (75, 10), (80, 1)):
        with pytest.raises((binding.FluxError, ValueError)):
            binding.joint_rope_attention_rows(q[:, :max(n, 1)].contiguous(), q0, k, v, ids[:16],
                                              ids[16:])


@pytest.mark.parametrize("world", [2, 4])
def test_sequence_parallel_ranks_match_the_klein9b_output(world):
    """Each rank's query rows over the whole sequence's keys (the K / V its
    all-gather would deliver): put together, every output within twice the bar
    of the full call, and a sample of rows against the oracle."""
    w = W.WORKLOADS["klein9b"]
    q, k, v = (t.cuda() for t in W.workload_qkv(w))
    txt, img = (torch.from_numpy(x).cuda() for x in W.workload_ids(w))
    full = binding.joint_rope_attention(q, k, v, txt, img)
    parts = []
    for r in range(world):
        q0, n = shard.seq_range(r, world, w.S)
        parts.append(binding.joint_rope_attention_rows(q[:, q0:q0 + n].contiguous(), q0, k, v,
                                                       txt, img))
    got = torch.cat(parts, dim=1)
    torch.cuda.synchronize()
    err = (got.float() - full.float()).abs()
    assert float(err.max()) <= 2 * MAX_ABS and float(err.mean()) <= 2 * MEAN_ABS
    rows = np.unique(np.r_[0, w.S_txt - 1, w.S_txt, w.S // world - 1, w.S // world, w.S - 1])
    ref = _oracle_rows(q, k, v, txt, img, rows)
    e = np.abs(got[:, rows].float().cpu().numpy() - ref)
    assert e.max() <= MAX_ABS and e.mean() <= MEAN_ABS

"""The multi-rank host logic on CPU: two gloo ranks (world size 2) on 127.0.0.1.

Replicas: each rank runs the whole path on its own seeded inputs; the only
cross-rank step is the max-reduction of the timings.

Head parallel and sequence parallel (diffusion_transformer_joint_gb300.shard):
the head split covers every head exactly once; the sequence split's K / V
all-gather rebuilds the full tensors; and with the oracle standing in for each
rank's kernel call (there is no GPU here), the ranks' outputs put together
equal the oracle's output over the whole problem, bit for bit (every
(batch, head, query row) is computed independently).
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import sys

    sys.path.insert(0, ROOT)
    import bench
    from diffusion_transformer_joint_gb300 import workloads as W

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank measured a different time; every rank must see the slowest
        local_ms = 10.0 + 5.0 * rank
        t_max = bench.max_over_ranks(local_ms, dist, torch.device("cpu"))
        # replicas draw different inputs
        w = W.WORKLOADS["tiny"]
        q, _, _ = W.workload_qkv(w, seed_offset=bench.rank_seed_offset(rank))
        gathered = [torch.zeros_like(q.float()) for _ in range(world)]
        dist.all_gather(gathered, q.float())
        distinct = not torch.equal(gathered[0], gathered[1])
        results[rank] = (t_max, distinct)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time_and_distinct_inputs():
    world = 2
    manager = mp.Manager()
    results = manager.dict()
    mp.spawn(_worker, args=(world, _free_port(), results), nprocs=world, join=True)
    assert results[0][0] == results[1][0] == 15.0
    assert results[0][1] and results[1][1]


def test_head_and_sequence_splits_cover_everything_once():
    import sys

    sys.path.insert(0, ROOT)
    from diffusion_transformer_joint_gb300 import shard

    for n in (1, 2, 3, 24, 32, 48, 4608, 4609):
        for world in (1, 2, 3, 4, 8):
            seen = []
            for r in range(world):
                a, m = shard.even_range(r, world, n)
                seen.extend(range(a, a + m))
                assert m in (n // world, n // world + 1)
            assert seen == list(range(n))
    with pytest.raises(ValueError):
        shard.head_range(2, 2, 32)


def _split_worker(rank, world, port, mode, shape, results):
    import sys

    sys.path.insert(0, ROOT)
    import numpy as np

    import oracle
    from diffusion_transformer_joint_gb300 import shard
    from diffusion_transformer_joint_gb300 import workloads as W

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        B, H, S_txt, S = shape
        q, k, v = (W.normal_bf16((B, S, H, 128), 4000 + i).float() for i in range(3))
        ids = W.random_ids(S, 4003, 0, 200)
        txt, img = ids[:S_txt], ids[S_txt:]
        if mode == "heads":
            h0, n = shard.head_range(rank, world, H)
            sl = slice(h0, h0 + n)
            mine = oracle.joint_rope_attention(q[:, :, sl].numpy(), k[:, :, sl].numpy(),
                                               v[:, :, sl].numpy(), txt, img)
            # gather every rank's heads, padded to the largest share
            n_max = -(-H // world)
            buf = torch.zeros((B, S, n_max, 128), dtype=torch.float64)
            buf[:, :, :n] = torch.from_numpy(mine)
            parts = [torch.empty_like(buf) for _ in range(world)]
            dist.all_gather(parts, buf)
            full = torch.cat([p[:, :, :shard.head_range(r, world, H)[1]]
                              for r, p in enumerate(parts)], dim=2)
            gathered_ok = True
        else:
            q0, n = shard.seq_range(rank, world, S)
            kf = shard.gather_sequence(k[:, q0:q0 + n].contiguous(), S, dist)
            vf = shard.gather_sequence(v[:, q0:q0 + n].contiguous(), S, dist)
            gathered_ok = torch.equal(kf, k) and torch.equal(vf, v)
            # this rank's query rows only: the oracle reads q at the rows it is asked for
            q_mine = torch.zeros_like(q)
            q_mine[:, q0:q0 + n] = q[:, q0:q0 + n]
            mine = oracle.joint_rope_attention(q_mine.numpy(), kf.numpy(), vf.numpy(), txt, img,
                                               rows=np.arange(q0, q0 + n))
            full = shard.gather_sequence(torch.from_numpy(mine), S, dist)
        if rank == 0:
            ref = oracle.joint_rope_attention(q.numpy(), k.numpy(), v.numpy(), txt, img)
            results[0] = (gathered_ok, bool(np.array_equal(full.numpy(), ref)))
        else:
            results[rank] = (gathered_ok, True)
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("mode", ["heads", "seq"])
@pytest.mark.parametrize("shape", [(1, 2, 16, 80), (2, 3, 10, 81)])
def test_two_gloo_ranks_split_the_attention_like_the_whole(mode, shape):
    world = 2
    manager = mp.Manager()
    results = manager.dict()
    mp.spawn(_split_worker, args=(world, _free_port(), mode, shape, results), nprocs=world,
             join=True)
    assert results[0] == (True, True) and results[1][0]


def test_whole_job_value_is_weak_scaling_aggregate():
    import sys

    sys.path.insert(0, ROOT)
    import bench

    # 2 ranks x 10 steps x 1 TFLOP in 20 ms (slowest rank) -> 1000 TFLOP/s
    assert bench.whole_job_tflops(1e12, 2, 10, 20.0) == pytest.approx(1000.0)
    assert bench.max_over_ranks(3.5) == 3.5


def test_reference_arm_prints_a_line_on_cpu(capsys):
    import json
    import subprocess
    import sys

    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "tiny", "--steps", "2", "--warmup", "3"],
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["d2h_bytes_per_step"] == 0

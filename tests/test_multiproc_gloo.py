"""The bench's multi-rank host logic on CPU: two gloo ranks (world size 2).

On GPUs each rank is a replica of the whole path on its own seeded inputs
(heads and batches are independent units, so no data moves between
ranks); the only cross-rank step is the max-reduction of the timings. These
tests run that logic with the gloo backend on 127.0.0.1.
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

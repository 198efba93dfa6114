"""Host-side arithmetic of bench.py (no GPU): FLOP counts of the KV modes and
the projection, the edit workload's token split, percentiles, whole-job
throughput, and the profiled-traffic lookup."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402
from diffusion_transformer_joint_gb300 import workloads as W  # noqa: E402


def test_edit_workload_split_and_kv_flops():
    w = W.WORKLOADS["klein9b_edit2"]
    S_t, S_r, S_i = bench.kv_split(w)
    assert (S_t, S_r, S_i) == (512, 8192, 4096) and S_t + S_r + S_i == w.S
    per = 4 * w.B * w.H * w.D
    # extract: text and image queries see all keys, reference queries only the references
    assert bench.kv_flops(w, "extract") == per * (4608 * 12800 + 8192 * 8192)
    # cached: text and image queries over [txt ; cache ; img]
    assert bench.kv_flops(w, "cached") == per * 4608 * 12800
    # together less than full attention over all 12800 tokens, more than half of it
    assert 0.5 * w.flops < bench.kv_flops(w, "extract") < w.flops


def test_projection_flops_and_dims():
    w = W.WORKLOADS["klein9b"]
    M, dim, mlp = W.proj_dims(w)
    assert (M, dim, mlp) == (4608, 4096, 12288)
    assert W.proj_flops(w) == 2 * 4608 * 4096 * 36864


def test_percentiles_and_whole_job_throughput():
    xs = [float(i) for i in range(101)]
    assert bench._percentiles(xs, (10, 50, 90)) == [10.0, 50.0, 90.0]
    assert bench._percentiles([3.0], (10, 90)) == [3.0, 3.0]
    # 2 ranks x 1e12 FLOP x 4 steps in 8 ms -> 1000 TFLOP/s
    assert bench.whole_job_tflops(1e12, 2, 4, 8.0) == pytest.approx(1000.0)
    assert bench.rank_seed_offset(1, 2) != bench.rank_seed_offset(2, 1)


def test_profiled_traffic_is_none_or_positive():
    t = bench._profiled_traffic()
    assert t is None or t > 0
    p = bench._profiled_traffic(bench.PROJ_PROFILE_SUMMARY, bench.PROJ_SOURCE,
                                "dram_bytes_per_launch_klein9b")
    assert p is None or p > 0
    # a summary taken on another source reads as unknown
    assert bench._profiled_traffic(bench.PROJ_PROFILE_SUMMARY, bench.KERNEL_SOURCE,
                                   "dram_bytes_per_launch_klein9b") is None


def test_committed_profiles_are_of_the_current_kernel_sources():
    # the bench's traffic figures come from the ncu summaries in profiles/; each
    # summary records the hash of the source it was taken on, so a kernel edit
    # without a new capture shows up here instead of as a silent null
    w = W.WORKLOADS["klein9b"]
    attn = bench._profiled_traffic()
    assert attn is not None
    # DRAM traffic cannot be below the algorithmic bytes; far above them would
    # mean re-reads (the exchange buffer accounts for the measured extra)
    assert w.io_bytes <= attn <= 1.5 * w.io_bytes
    proj = bench._profiled_traffic(bench.PROJ_PROFILE_SUMMARY, bench.PROJ_SOURCE,
                                   "dram_bytes_per_launch_klein9b")
    M, dim, mlp = W.proj_dims(w)
    n_out = 3 * w.H * 128 + 2 * mlp
    proj_io = 2 * (M * dim + n_out * dim + M * (3 * w.H * 128 + mlp))
    assert proj is not None
    assert proj_io <= proj <= 1.5 * proj_io

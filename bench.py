"""Bench: joint RoPE attention TFLOP/s on the klein-9B 1024^2 shape.

One step is one pass of the whole hot path over one batch: the RoPE table
kernel for the joint ids, then the attention kernel (RoPE fused into the
Q/K tile loads, QK^T and PV on tcgen05, online softmax). FLOPs per step are
4 * B * H * S^2 * 128.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload klein9b] [--qk-norm] [--kv-mode extract|cached] [--proj]

Prints one JSON line (rank 0). With N > 1 (torchrun, one rank per GPU) every
rank runs the same-shaped workload on its own seeded inputs with no data
exchange (heads and batches are independent): weak scaling, and `value` is
all ranks' FLOPs over the slowest rank's time.

`--kv-mode extract|cached` times one reference-image KV-mode call per step on
the two-reference edit shape instead (tables, attention and, for extract, the
cache copies inside the call). `--proj` times the fused single-stream
QKV + SwiGLU-MLP input projection of the workload (one GEMM kernel per step).

`--impl reference` times the fp64 CPU oracle on the host cores instead, on a
bounded sample of query rows of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "joint RoPE-attention bf16 TFLOP/s at klein-9B 1024² shape; % dense-BF16 peak"
UNIT = "TFLOP/s"
L2_BYTES = 129 * 1024 * 1024
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "attention_klein9b_ncu.txt")
KERNEL_SOURCE = os.path.join(ROOT, "diffusion_transformer_joint_gb300", "csrc",
                             "attention_sm103a.cu")
PROJ_PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "qkv_mlp_proj_ncu.txt")
PROJ_SOURCE = os.path.join(ROOT, "diffusion_transformer_joint_gb300", "csrc", "proj_sm103a.cu")


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return p, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def _kernel_hash(source=KERNEL_SOURCE):
    """Hash of a kernel source's code: // comments, trailing blanks and blank
    lines are left out, so that a comment edit does not orphan a profile."""
    import re

    with open(source, encoding="utf-8") as f:
        lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in f]
    code = "\n".join(ln for ln in lines if ln)
    return hashlib.sha256(code.encode("utf-8")).hexdigest()[:16]


def _profiled_traffic(summary=PROFILE_SUMMARY, source=KERNEL_SOURCE,
                      key="dram_bytes_per_launch_klein9b"):
    """dram bytes per launch from a committed ncu summary, when it was taken
    on the current kernel source; else None."""
    try:
        vals = {}
        for line in open(summary):
            if ":" in line and not line.startswith("#"):
                k, v = line.split(":", 1)
                vals[k.strip()] = v.strip()
        if vals.get("kernel_source_sha256_16") != _kernel_hash(source):
            return None
        return float(vals[key])
    except (OSError, KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during a region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.idx = device_index
        self.proc = None
        self.path = os.path.join("/tmp", f"flux_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50", "-i", str(self.idx)], stdout=self.f, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, power = [], [], set(), []
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for n, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        busy = [s for s in sm if s > 0.5 * max(sm)] or sm
        return {"sm_mhz": statistics.median(busy), "sm_max_mhz": max(smax),
                "power_w_max": max(power) if power else None, "samples": len(sm),
                "reasons": sorted(reasons)}


def gpu_head_start(torch, stream=None):
    """Keep the device busy (about 1 ms of spinning) while the host enqueues the
    timed steps, so that the timed region measures the steps and not the host's
    latency in submitting the first one."""
    if stream is None:
        torch.cuda._sleep(2_000_000)
    else:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(2_000_000)


# ------------------------------------------------- multi-rank host logic


def rank_seed_offset(rank: int, set_index: int = 0) -> int:
    """Seed offset of a rank's input set: every rank runs its own replica."""
    return 100000 * rank + 17 * set_index


def max_over_ranks(x: float, dist=None, device=None) -> float:
    """The slowest rank's value (the whole job ends when it does)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(x)
    import torch

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(flops_per_rank_step: float, world: int, steps: int, t_max_ms: float) -> float:
    """All ranks' FLOPs over the slowest rank's time (weak scaling)."""
    return world * flops_per_rank_step * steps / (t_max_ms * 1e-3) / 1e12


# ------------------------------------------------------------------ ours


def run_ours(args, rank, world, local_rank):
    import torch

    from diffusion_transformer_joint_gb300 import binding
    from diffusion_transformer_joint_gb300 import build as cuda_build
    from diffusion_transformer_joint_gb300 import workloads as W

    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(cuda_build.LIB_PATH):
        cuda_build.build()
    if dist is not None:
        dist.barrier()
    binding.load()

    w = W.WORKLOADS[args.workload]
    txt_np, img_np = W.workload_ids(w)
    import numpy as np

    ids = torch.from_numpy(np.concatenate([txt_np, img_np])).to(dev)
    txt_d, img_d = ids[:w.S_txt], ids[w.S_txt:]
    set_bytes = 3 * w.B * w.S * w.H * w.D * 2
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes) + 1)
    sets = []
    for i in range(n_sets):
        q, k, v = W.workload_qkv(w, seed_offset=rank_seed_offset(rank, i))
        sets.append((q.to(dev), k.to(dev), v.to(dev), torch.empty_like(q, device=dev)))
    # the one-call workspace: status word, table, rotated-K exchange buffer
    ws = torch.zeros(binding.workspace_shared_bytes(w.B, w.S, w.H, w.D), dtype=torch.uint8,
                     device=dev)
    xbuf_bytes = binding.krot_bytes(w.B, w.S, w.H, w.D)
    qk_norm = None
    if args.qk_norm:  # synthetic learned weights in [0.5, 1.5), one vector per stream and tensor
        g = torch.Generator().manual_seed(7)
        qk_norm = tuple((0.5 + torch.rand(w.D, generator=g)).to(dev) for _ in range(4)) + (1e-6,)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        # one pass of the whole path: the table kernel, then the attention
        # kernel, whose start overlaps the table kernel (one C-ABI call)
        q, k, v, out = sets[i % n_sets]
        binding.joint_rope_attention(q, k, v, txt_d, img_d, out=out, workspace=ws,
                                     stream=stream, qk_norm=qk_norm)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()

    K = args.steps
    ev_start = torch.cuda.Event(enable_timing=True)
    ev_end = torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        gpu_head_start(torch, stream)
        with torch.cuda.stream(stream):
            ev_start.record(stream)
            for i in range(K):
                step(i)
            ev_end.record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    total_ms = ev_start.elapsed_time(ev_end)
    st = binding.query_status(ws, stream)
    if st != 0:
        raise RuntimeError(f"device status {st} after the timed steps")
    attn_ms = attention_launch_ms(w, sets, ids, binding, torch, dev, stream, K, qk_norm)

    t_max = max_over_ranks(total_ms, dist, dev)

    # end-to-end through the public one-call API with host buffers
    e2e = run_e2e(w, dev, K, args.warmup, binding, W, torch, np, txt_np, img_np, qk_norm)
    e2e["ms_per_step"] = max_over_ranks(e2e["ms_per_step"], dist, dev)

    if rank != 0:
        return None
    peaks, peak_src = _peaks()
    flops_step = w.flops
    value = whole_job_tflops(flops_step, world, K, t_max)
    attn_avg_ms = statistics.mean(attn_ms)
    achieved = flops_step / (attn_avg_ms * 1e-3) / 1e12
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    traffic = _profiled_traffic()
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": round(t_max / K, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v, FLUX.2 (T,H,W,L) ids)",
        "config": {
            "workload": f"{w.name}: B={w.B} H={w.H} S={w.S} ({w.S_txt} text + {w.S_img} image) "
                        f"head_dim={w.D} axes=(32,32,32,32) theta=2000 non-causal",
            "B": w.B, "H": w.H, "S": w.S, "S_txt": w.S_txt, "S_img": w.S_img, "head_dim": w.D,
            "parallelism": f"replicas x{world} (heads/batches independent, no collective)",
            "l2": f"inputs rotate over {n_sets} sets of {set_bytes / 2**20:.0f} MiB "
                  f"({n_sets * set_bytes / 2**20:.0f} MiB > 129 MiB L2)",
            "timed_region": "CUDA events around the K steps, enqueued behind a ~1 ms device "
                            "spin so that the host's submission latency is not timed",
            "step": "flux_joint_rope_attention: rope_tables kernel + attention kernel "
                    "(launched to overlap the table kernel's run), tables rebuilt every step",
            "k_rope": "rotated K tiles shared by the CTAs of a head through an exchange "
                      f"buffer ({xbuf_bytes / 2**20:.0f} MiB)",
            "qk_norm": ("fused QK RMS norm before RoPE (eps 1e-6, synthetic per-stream weights)"
                        if args.qk_norm else "none"),
        },
        "pct_peak": round(100.0 * value / world / peak, 2),
        "roofline": {
            "bound": "tensor",
            "kernel": "joint_rope_attention_kernel",
            "achieved": round(achieved, 2),
            "peak": peak,
            "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "frac_of_sustained": round(achieved / peak_sus, 4),
            "peak_source": f"{peak_src} bf16_tflops (burst)",
            "traffic": traffic,
            "algorithmic_flops_per_launch": flops_step,
            "algorithmic_bytes_per_launch": w.io_bytes,
            "avg_launch_ms": round(attn_avg_ms, 4),
            "launch_timing": f"{K} back-to-back launches of the attention kernel alone "
                             "(caller-built table), each between CUDA events on its stream, "
                             "right after the timed steps on the same inputs",
            "launch_ms_p10_p50_p90": [round(x, 4) for x in _percentiles(attn_ms, (10, 50, 90))],
        },
        "clocks": clocks.summary(),
        "e2e": {"value": round(whole_job_tflops(flops_step, world, 1, e2e["ms_per_step"]), 2),
                "unit": UNIT, "ms_per_step": round(e2e["ms_per_step"], 4),
                "h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"],
                "api": ("flux_joint_qknorm_rope_attention" if args.qk_norm else
                        "flux_joint_rope_attention") + " (one call: tables + attention)",
                "pipelining": PIPELINING},
        "gpu_launches": 2 * K,
    }
    if not args.no_cpu_baseline and world == 1:  # the oracle baseline is an N = 1 figure
        gpu_out = sets[0][3].float().cpu().numpy()  # the last output of the first input set
        norm_np = None
        if qk_norm is not None:
            norm_np = tuple(x.cpu().numpy() for x in qk_norm[:4]) + (qk_norm[4],)
        line["cpu_baseline"], line["parity"] = cpu_baseline(
            w, target_s=args.cpu_seconds, gpu_out=gpu_out, qk_norm=norm_np)
    return line


def attention_launch_ms(w, sets, ids, binding, torch, dev, stream, K, qk_norm):
    """Duration of each of K launches of the attention kernel alone (the
    tabled entry point on a table built once), between CUDA events recorded on
    its stream; the inputs rotate over the same sets as the timed steps."""
    table = binding.rope_tables_packed(ids, stream=stream)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    krot = torch.empty(binding.krot_bytes(w.B, w.S, w.H, w.D), dtype=torch.uint8, device=dev)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(K + 1)]
    with torch.cuda.stream(stream):
        for i in range(3):
            q, k, v, out = sets[i % len(sets)]
            binding.joint_rope_attention_tabled(q, k, v, table, status, out=out, stream=stream,
                                                krot=krot, qk_norm=qk_norm, s_txt=w.S_txt)
        for i in range(K):
            q, k, v, out = sets[i % len(sets)]
            evs[i].record(stream)
            binding.joint_rope_attention_tabled(q, k, v, table, status, out=out, stream=stream,
                                                krot=krot, qk_norm=qk_norm, s_txt=w.S_txt)
        evs[K].record(stream)
    stream.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status set during the attention launches")
    return [evs[i].elapsed_time(evs[i + 1]) for i in range(K)]


PIPELINING = ("two streams with their own buffers: a step's host-to-device copies overlap "
              "the previous step's kernels and copy back")


def two_lane_ms(torch, dev, K, warmup, lanes, one):
    """ms per step of one(i, lane) run for i < K, alternating between two lanes
    (dicts with their own "stream" and buffers): a step's copies overlap the
    other lane's kernels; within a lane the steps stay in order."""
    for i in range(max(2, warmup)):
        one(i, lanes[i % 2])
    torch.cuda.synchronize(dev)
    main = torch.cuda.current_stream(dev)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    gpu_head_start(torch, main)
    e0.record(main)
    for ln in lanes:
        ln["stream"].wait_event(e0)
    for i in range(K):
        one(i, lanes[i % 2])
    for ln in lanes:
        main.wait_stream(ln["stream"])
    e1.record(main)
    torch.cuda.synchronize(dev)
    return e0.elapsed_time(e1) / K


def run_e2e(w, dev, K, warmup, binding, W, torch, np, txt_np, img_np, qk_norm=None):
    """Same metric through the one-call API: every step copies its inputs from
    pinned host memory, runs the call and copies the output back. Steps
    alternate between two streams with their own device buffers and
    workspaces, so one step's host-to-device copies overlap the previous
    step's kernels and device-to-host copy (the copy engines and the SMs
    work at the same time); within a stream the steps stay in order."""
    q, k, v = W.workload_qkv(w, seed_offset=555)
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    htxt = torch.from_numpy(txt_np).pin_memory()
    himg = torch.from_numpy(img_np).pin_memory()
    lanes = []
    for _ in range(2):
        lane = {
            "in": [torch.empty_like(t, device=dev) for t in (hq, hk, hv, htxt, himg)],
            "ws": torch.zeros(binding.workspace_shared_bytes(w.B, w.S, w.H, w.D),
                              dtype=torch.uint8, device=dev),
            "hout": torch.empty_like(hq).pin_memory(),
            "stream": torch.cuda.Stream(device=dev),
        }
        lane["out"] = torch.empty_like(lane["in"][0])
        lanes.append(lane)

    def one(i, ln):
        st = ln["stream"]
        with torch.cuda.stream(st):
            for d, h in zip(ln["in"], (hq, hk, hv, htxt, himg)):
                d.copy_(h, non_blocking=True)
            dq, dk, dv, dtxt, dimg = ln["in"]
            binding.joint_rope_attention(dq, dk, dv, dtxt, dimg, out=ln["out"],
                                         workspace=ln["ws"], stream=st, qk_norm=qk_norm)
            ln["hout"].copy_(ln["out"], non_blocking=True)

    ms = two_lane_ms(torch, dev, K, warmup, lanes, one)
    for ln in lanes:
        if binding.query_status(ln["ws"], ln["stream"]) != 0:
            raise RuntimeError("device status set during the end-to-end steps")
    h2d = sum(t.numel() * t.element_size() for t in (hq, hk, hv, htxt, himg))
    d2h = lanes[0]["hout"].numel() * lanes[0]["hout"].element_size()
    return {"ms_per_step": ms, "h2d": h2d, "d2h": d2h}


# --------------------------------------------------------- reference-image KV modes


def kv_split(w):
    """An edit workload as the KV pipeline orders it, [txt ; refs ; img]:
    (S_txt, S_ref, S_img)."""
    S_i = w.grid * w.grid
    return w.S_txt, w.S_img - S_i, S_i


def kv_flops(w, mode):
    """Extract: text and image queries against all S keys, reference queries
    against the reference keys. Cached: text and image queries against
    [txt ; cache ; img]. 4 flops per (query, key, channel)."""
    S_t, S_r, S_i = kv_split(w)
    per = 4 * w.B * w.H * w.D
    if mode == "extract":
        return per * ((S_t + S_i) * w.S + S_r * S_r)
    return per * (S_t + S_i) * w.S


def _kv_host_inputs(w, mode, seed_offset, W, np):
    """bf16 CPU tensors and int32 ids of one KV-mode call (refs moved before img)."""
    S_t, S_r, S_i = kv_split(w)
    q, k, v = W.workload_qkv(w, seed_offset=seed_offset)  # [txt ; img ; refs]
    t_ids, i_ids = W.workload_ids(w)
    ids = np.concatenate([t_ids, i_ids])
    if mode == "extract":
        order = np.r_[0:S_t, S_t + S_i:w.S, S_t:S_t + S_i]
        q, k, v = (x[:, order].contiguous() for x in (q, k, v))
        ids = ids[order]
        return (q, k, v), (ids[:S_t], ids[S_t:S_t + S_r], ids[S_t + S_r:])
    keep = np.r_[0:S_t + S_i]
    q, k, v = (x[:, keep].contiguous() for x in (q, k, v))
    ck = W.normal_bf16((w.B, S_r, w.H, w.D), 1000 * w.index + seed_offset + 7)
    cv = W.normal_bf16((w.B, S_r, w.H, w.D), 1000 * w.index + seed_offset + 8)
    return (q, k, v, ck, cv), (ids[:S_t], ids[S_t:S_t + S_i])


def run_kv(args, rank, world, local_rank):
    """Time one KV-mode call per step (ids -> tables -> attention -> cache)."""
    import numpy as np
    import torch

    from diffusion_transformer_joint_gb300 import binding
    from diffusion_transformer_joint_gb300 import build as cuda_build
    from diffusion_transformer_joint_gb300 import workloads as W

    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(cuda_build.LIB_PATH):
        cuda_build.build()
    if dist is not None:
        dist.barrier()
    binding.load()
    w = W.WORKLOADS[args.workload]
    mode = args.kv_mode
    S_t, S_r, S_i = kv_split(w)
    if S_r == 0:
        raise SystemExit(f"--kv-mode needs a workload with reference images, not {w.name}")

    def to_dev(xs):
        return tuple(torch.from_numpy(np.ascontiguousarray(x)).to(dev)
                     if isinstance(x, np.ndarray) else x.to(dev) for x in xs)

    tensors0, ids_h = _kv_host_inputs(w, mode, rank_seed_offset(rank, 0), W, np)
    set_bytes = sum(t.numel() * 2 for t in tensors0)
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes) + 1)
    ids = to_dev(ids_h)
    sets = []
    for i in range(n_sets):
        ts = tensors0 if i == 0 else _kv_host_inputs(w, mode, rank_seed_offset(rank, i), W, np)[0]
        ts = to_dev(ts)
        outs = (torch.empty_like(ts[0]),)
        if mode == "extract":
            outs += tuple(torch.empty((w.B, S_r, w.H, w.D), dtype=torch.bfloat16, device=dev)
                          for _ in range(2))
        sets.append((ts, outs))
    n_ws = (binding.extract_workspace_bytes(w.B, S_t, S_r, S_i, w.H, w.D) if mode == "extract"
            else binding.cached_workspace_bytes(w.B, S_t, S_i, S_r, w.H, w.D))
    ws = torch.zeros(int(n_ws), dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(device=dev)
    qk_norm = None
    if args.qk_norm:  # synthetic learned weights in [0.5, 1.5), one vector per stream and tensor
        g = torch.Generator().manual_seed(7)
        qk_norm = tuple((0.5 + torch.rand(w.D, generator=g)).to(dev) for _ in range(4)) + (1e-6,)

    def call(ts, outs, st):
        if mode == "extract":
            binding.attention_extract(*ts, *ids, out=outs[0], cache_k=outs[1], cache_v=outs[2],
                                      workspace=ws, stream=st, qk_norm=qk_norm)
        else:
            q, k, v, ck, cv = ts
            binding.attention_cached(q, k, v, ids[0], ids[1], ck, cv, out=outs[0], workspace=ws,
                                     stream=st, qk_norm=qk_norm)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            call(*sets[i % n_sets], stream)
    stream.synchronize()
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(2_000_000)  # the host enqueues ahead (gpu_head_start)
            ev0.record(stream)
            for i in range(K):
                call(*sets[i % n_sets], stream)
            ev1.record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    if binding.query_status(ws, stream) != 0:
        raise RuntimeError("device status set during the timed steps")
    t_max = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)

    # end to end: pinned host inputs in, the call, the outputs (and cache) back
    h_in = tuple(t.pin_memory() for t in tensors0)
    h_ids = tuple(torch.from_numpy(np.ascontiguousarray(x)).pin_memory() for x in ids_h)
    lanes = []
    for li in range(2):
        lanes.append({
            "in": tuple(torch.empty_like(t, device=dev) for t in h_in),
            "ids": tuple(torch.empty_like(t, device=dev) for t in h_ids),
            "out": tuple(torch.empty_like(t) for t in sets[0][1]),
            "hout": tuple(torch.empty_like(t, device="cpu").pin_memory() for t in sets[0][1]),
            "ws": ws if li == 0 else torch.zeros_like(ws),
            "stream": stream if li == 0 else torch.cuda.Stream(device=dev),
        })

    def e2e_one(i, ln):
        st = ln["stream"]
        with torch.cuda.stream(st):
            for d, h in zip(ln["in"] + ln["ids"], h_in + h_ids):
                d.copy_(h, non_blocking=True)
            d_in, d_ids, d_out = ln["in"], ln["ids"], ln["out"]
            if mode == "extract":
                binding.attention_extract(*d_in, *d_ids, out=d_out[0], cache_k=d_out[1],
                                          cache_v=d_out[2], workspace=ln["ws"], stream=st,
                                          qk_norm=qk_norm)
            else:
                q, k, v, ck, cv = d_in
                binding.attention_cached(q, k, v, d_ids[0], d_ids[1], ck, cv, out=d_out[0],
                                         workspace=ln["ws"], stream=st, qk_norm=qk_norm)
            for h, d in zip(ln["hout"], d_out):
                h.copy_(d, non_blocking=True)

    e2e_step_ms = two_lane_ms(torch, dev, K, args.warmup, lanes, e2e_one)
    for ln in lanes:
        if binding.query_status(ln["ws"], ln["stream"]) != 0:
            raise RuntimeError("device status set during the end-to-end steps")
    h_out = lanes[0]["hout"]
    e2e_ms = max_over_ranks(e2e_step_ms, dist, dev)
    if rank != 0:
        return None

    peaks, peak_src = _peaks()
    flops = kv_flops(w, mode)
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    call_ms = t_max / K
    value = whole_job_tflops(flops, world, K, t_max)
    per_call = flops / (call_ms * 1e-3) / 1e12
    keys = "[txt ; refs ; img]" if mode == "extract" else "[txt ; cache ; img]"
    queries = "all S (refs against refs only)" if mode == "extract" else f"{S_t + S_i} (txt ; img)"
    return {
        "metric": f"{mode}-mode joint RoPE-attention bf16 TFLOP/s at the klein-9B two-reference "
                  "edit shape",
        "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(call_ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v and cache, FLUX.2 (T,H,W,L) ids)",
        "config": {
            "workload": f"{w.name} {mode}: B={w.B} H={w.H} text {S_t}, refs {S_r}, image {S_i}; "
                        f"queries {queries}, keys {keys}; head_dim={w.D} theta=2000",
            "B": w.B, "H": w.H, "S_txt": S_t, "S_ref": S_r, "S_img": S_i, "head_dim": w.D,
            "parallelism": f"replicas x{world} (no collective)",
            "l2": f"inputs rotate over {n_sets} sets of {set_bytes / 2**20:.0f} MiB "
                  f"({n_sets * set_bytes / 2**20:.0f} MiB > 129 MiB L2)",
            "step": ("two table kernels, the attention kernel over 3 segments, two cache copies"
                     if mode == "extract" else
                     "one table kernel, the attention kernel (cache read in place, not rotated)"),
            "qk_norm": ("fused QK RMS norm before RoPE (eps 1e-6, synthetic per-stream weights)"
                        if args.qk_norm else "none"),
        },
        "roofline": {
            "bound": "tensor", "kernel": "whole call (tables + attention + copies)",
            "achieved": round(per_call, 2), "peak": peak, "unit": "TFLOP/s",
            "frac": round(per_call / peak, 4),
            "peak_source": f"{peak_src} bf16_tflops (burst)", "traffic": None,
            "algorithmic_flops_per_launch": flops,
        },
        "clocks": clocks.summary(),
        "e2e": {"value": round(whole_job_tflops(flops, world, 1, e2e_ms), 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4),
                "h2d_bytes_per_step": sum(t.numel() * t.element_size() for t in h_in + h_ids),
                "d2h_bytes_per_step": sum(t.numel() * t.element_size() for t in h_out),
                "api": f"flux_joint_rope_attention_{mode}", "pipelining": PIPELINING},
        "gpu_launches": (3 if mode == "extract" else 2) * K,
    }


# --------------------------------------------------------- single-stream projection


def proj_cpu_baseline(w, target_s=10.0):
    """The oracle's projection on a bounded sample of token rows (every output
    feature of each row), timed on the host cores."""
    import numpy as np

    import oracle
    from diffusion_transformer_joint_gb300 import workloads as W

    M, dim, mlp = W.proj_dims(w)
    x, wt = W.proj_inputs(w)
    xn, wn = x.float().numpy().astype(np.float64), wt.float().numpy().astype(np.float64)
    t0 = time.perf_counter()
    oracle.qkv_mlp_proj(xn, wn, w.H, 128, mlp, rows=np.array([0]))
    per_row = max(time.perf_counter() - t0, 1e-6)
    n = int(max(2, min(M, target_s / per_row)))
    rows = np.linspace(0, M - 1, n).astype(np.int64)
    t0 = time.perf_counter()
    oracle.qkv_mlp_proj(xn, wn, w.H, 128, mlp, rows=rows)
    t = time.perf_counter() - t0
    flops = 2 * rows.size * dim * (3 * dim + 2 * mlp)
    return {"value": round(flops / t / 1e12, 6), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{rows.size} of {M} token rows x all {3 * dim + 2 * mlp} output features "
                      f"of {w.name}, fp64, one thread, {t:.1f} s"}


def run_proj(args, rank, world, local_rank):
    """Time the fused single-stream input projection (one kernel per step)."""
    import torch

    from diffusion_transformer_joint_gb300 import binding
    from diffusion_transformer_joint_gb300 import build as cuda_build
    from diffusion_transformer_joint_gb300 import workloads as W

    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(cuda_build.LIB_PATH):
        cuda_build.build()
    if dist is not None:
        dist.barrier()
    binding.load()
    w = W.WORKLOADS[args.workload]
    M, dim, mlp = W.proj_dims(w)
    H = w.H
    x_h, wt_h = W.proj_inputs(w, seed_offset=rank_seed_offset(rank, 0))
    wt = wt_h.to(dev)  # weights stay resident, as a model's do
    set_bytes = x_h.numel() * 2
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes) + 1)
    xs = [x_h.to(dev)] + [W.proj_inputs(w, seed_offset=rank_seed_offset(rank, i))[0].to(dev)
                          for i in range(1, n_sets)]
    q = torch.empty((M, H, 128), dtype=torch.bfloat16, device=dev)
    k, v = torch.empty_like(q), torch.empty_like(q)
    act = torch.empty((M, mlp), dtype=torch.bfloat16, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(i):
        binding.qkv_mlp_proj(xs[i % n_sets], wt, H, mlp, q=q, k=k, v=v, act=act, status=status,
                             stream=stream)

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(2_000_000)  # the host enqueues ahead (gpu_head_start)
            ev0.record(stream)
            for i in range(K):
                step(i)
            ev1.record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    if int(status.item()) != 0:
        raise RuntimeError("device status set during the timed steps")
    t_max = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)

    # end to end: the activations from pinned host memory, the four outputs back
    hx = x_h.pin_memory()
    lanes = []
    for li in range(2):
        outs = (q, k, v, act) if li == 0 else tuple(torch.empty_like(t) for t in (q, k, v, act))
        lanes.append({
            "x": torch.empty_like(hx, device=dev), "out": outs,
            "hout": tuple(torch.empty_like(t, device="cpu").pin_memory() for t in outs),
            "status": torch.zeros(1, dtype=torch.int32, device=dev),
            "stream": stream if li == 0 else torch.cuda.Stream(device=dev),
        })

    def e2e_one(i, ln):
        st = ln["stream"]
        with torch.cuda.stream(st):
            ln["x"].copy_(hx, non_blocking=True)
            oq, ok_, ov, oa = ln["out"]
            binding.qkv_mlp_proj(ln["x"], wt, H, mlp, q=oq, k=ok_, v=ov, act=oa,
                                 status=ln["status"], stream=st)
            for h, d in zip(ln["hout"], ln["out"]):
                h.copy_(d, non_blocking=True)

    e2e_step_ms = two_lane_ms(torch, dev, K, args.warmup, lanes, e2e_one)
    if any(int(ln["status"].item()) != 0 for ln in lanes):
        raise RuntimeError("device status set during the end-to-end steps")
    houts = lanes[0]["hout"]
    e2e_ms = max_over_ranks(e2e_step_ms, dist, dev)
    if rank != 0:
        return None
    peaks, peak_src = _peaks()
    flops = W.proj_flops(w)
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_sus = float(peaks.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"]))
    ms = t_max / K
    value = whole_job_tflops(flops, world, K, t_max)
    achieved = flops / (ms * 1e-3) / 1e12
    n_out = 3 * dim + 2 * mlp
    line = {
        "metric": f"fused single-stream QKV+MLP input projection bf16 TFLOP/s at the {w.name} shape",
        "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(ms, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 activations, N(0,1/dim) bf16 weights)",
        "config": {
            "workload": f"{w.name} to_qkv_mlp_proj: M={M} tokens, dim={dim}, H={H}, "
                        f"mlp={mlp}, W [{n_out}, {dim}]; epilogue split into Q/K/V "
                        "[B,S,H,128] + SwiGLU",
            "M": M, "dim": dim, "H": H, "mlp": mlp,
            "parallelism": f"replicas x{world} (no collective)",
            "l2": f"weights {wt.numel() * 2 / 2**20:.0f} MiB resident (> 129 MiB L2); "
                  f"activations rotate over {n_sets} sets of {set_bytes / 2**20:.0f} MiB",
            "step": "one fused projection kernel",
        },
        "roofline": {
            "bound": "tensor", "kernel": "qkv_mlp_proj_kernel", "achieved": round(achieved, 2),
            "peak": peak, "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
            "frac_of_sustained": round(achieved / peak_sus, 4),
            "peak_source": f"{peak_src} bf16_tflops (burst)",
            "traffic": _profiled_traffic(PROJ_PROFILE_SUMMARY, PROJ_SOURCE,
                                         f"dram_bytes_per_launch_{w.name}"),
            "algorithmic_flops_per_launch": flops,
            "algorithmic_bytes_per_launch": 2 * (M * dim + n_out * dim + M * (3 * dim + mlp)),
        },
        "clocks": clocks.summary(),
        "e2e": {"value": round(whole_job_tflops(flops, world, 1, e2e_ms), 2), "unit": UNIT,
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": hx.numel() * 2,
                "d2h_bytes_per_step": sum(h.numel() * 2 for h in houts),
                "api": "flux_qkv_mlp_proj (weights resident on the device)",
                "pipelining": PIPELINING},
        "gpu_launches": K,
    }
    if not args.no_cpu_baseline and world == 1:  # the oracle baseline is an N = 1 figure
        line["cpu_baseline"] = proj_cpu_baseline(w, target_s=args.cpu_seconds)
    return line


# --------------------------------------------------------- CPU baseline


def _oracle_sample(w, rows, threads, q, k, v, txt, img, qk_norm=None, result=None):
    import oracle

    t0 = time.perf_counter()
    out = oracle.joint_rope_attention(q, k, v, txt, img, rows=rows, threads=threads,
                                      qk_norm=qk_norm)
    if result is not None:
        result.append(out)
    return time.perf_counter() - t0


def _oracle_inputs(w):
    from diffusion_transformer_joint_gb300 import workloads as W

    q, k, v = W.workload_qkv(w)
    txt, img = W.workload_ids(w)
    return q.float().numpy(), k.float().numpy(), v.float().numpy(), txt, img


def _rows_for(w, seconds, threads, inputs):
    import numpy as np

    probe = np.arange(0, w.S, max(1, w.S // 32), dtype=np.int64)[:32]
    _oracle_sample(w, probe[:4], threads, *inputs)  # warm: threads, caches, page faults
    t = _oracle_sample(w, probe, threads, *inputs)
    per_row = t / probe.size
    n = int(max(16, min(w.S, seconds / max(per_row, 1e-9))))
    return np.linspace(0, w.S - 1, n).astype(np.int64)


def cpu_baseline(w, target_s=12.0, gpu_out=None, qk_norm=None):
    """The oracle as it stands, timed on the host cores on a bounded sample of
    query rows (all batch elements and heads of each row) of the workload.
    With ``gpu_out`` (the GPU's output for the same inputs, as a float array)
    the oracle's rows also check it: (baseline, parity) is returned."""
    import numpy as np

    import oracle

    threads = oracle.default_threads()
    inputs = _oracle_inputs(w)
    rows = _rows_for(w, target_s, threads, inputs)
    ref = []
    t = _oracle_sample(w, rows, threads, *inputs, qk_norm=qk_norm, result=ref)
    flops = 4 * w.B * w.H * rows.size * w.S * w.D
    base = {"value": round(flops / t / 1e12, 6), "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"{rows.size} of {w.S} query rows x all {w.B * w.H} (batch, head) pairs of "
                      f"{w.name} against all {w.S} keys, fp64, {t:.1f} s"}
    if gpu_out is None:
        return base
    err = np.abs(np.asarray(gpu_out, dtype=np.float64)[:, rows] - ref[0])
    parity = {"rows": int(rows.size), "elements": int(err.size),
              "max_abs": float(err.max()), "mean_abs": float(err.mean()),
              "bar": "max <= 1e-2, mean <= 1e-3",
              "pass": bool(err.max() <= 1e-2 and err.mean() <= 1e-3),
              "against": "fp64 oracle rows of the first input set, the timed steps' output"}
    return base, parity


def _percentiles(xs, ps):
    xs = sorted(xs)
    return [xs[min(len(xs) - 1, max(0, int(round(p / 100.0 * (len(xs) - 1)))))] for p in ps]


def cpu_report(seconds=3.0):
    """The oracle on every workload: a bounded sample of query rows timed with
    all host threads and with one (one head's rows for the one-thread run),
    as fp64 GFLOP/s. Printed as its own JSON line; no GPU is used."""
    import numpy as np

    import oracle
    from diffusion_transformer_joint_gb300 import workloads as W

    oracle.build()
    threads = oracle.default_threads()
    report = []
    for w in W.WORKLOADS.values():
        inputs = _oracle_inputs(w)
        rows = _rows_for(w, seconds, threads, inputs)
        t = _oracle_sample(w, rows, threads, *inputs)
        many = 4 * w.B * w.H * rows.size * w.S * w.D / t / 1e9
        q, k, v, txt, img = inputs  # one head, one thread
        one_head = [x[:, :, :1] for x in (q, k, v)]
        rows1 = np.linspace(0, w.S - 1, min(64, w.S)).astype(np.int64)
        t1 = _oracle_sample(w, rows1, 1, *one_head, txt, img)
        single = 4 * w.B * rows1.size * w.S * w.D / t1 / 1e9
        report.append({"workload": w.name, "S": w.S, "H": w.H,
                       "gflops_all_threads": round(many, 2), "threads": threads,
                       "rows_sampled": int(rows.size), "seconds": round(t, 2),
                       "gflops_one_thread": round(single, 3),
                       "one_thread_sample": f"{rows1.size} rows x 1 head"})
    return {"cpu_report": report, "kind": "oracle", "dtype": "f64"}


# ------------------------------------------- head- and sequence-parallel ranks


def run_sharded(args, rank, world, local_rank):
    """One klein-9B-shaped call split over the ranks (strong scaling: the whole
    job does one call's work per step).

    heads: rank r attends its contiguous range of heads of the same [B, S, H,
    128] inputs (flux_joint_rope_attention_heads); nothing moves between ranks.
    seq: rank r holds the q, k, v rows of its contiguous range of tokens; each
    step all-gathers K and V (NCCL), then attends its query rows over every
    key (flux_joint_rope_attention_rows). The gather is inside the step."""
    import numpy as np
    import torch

    from diffusion_transformer_joint_gb300 import binding, shard
    from diffusion_transformer_joint_gb300 import build as cuda_build
    from diffusion_transformer_joint_gb300 import workloads as W

    dist = None
    if world > 1:
        import torch.distributed as dist
    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    if rank == 0 or not os.path.exists(cuda_build.LIB_PATH):
        cuda_build.build()
    if dist is not None:
        dist.barrier()
    binding.load()
    w = W.WORKLOADS[args.workload]
    txt_np, img_np = W.workload_ids(w)
    ids = torch.from_numpy(np.concatenate([txt_np, img_np])).to(dev)
    txt_d, img_d = ids[:w.S_txt], ids[w.S_txt:]
    set_bytes = 3 * w.B * w.S * w.H * w.D * 2
    n_sets = max(2, -(-2 * L2_BYTES // set_bytes) + 1)
    stream = torch.cuda.Stream(device=dev)
    if args.shard == "heads":
        h0, n = shard.head_range(rank, world, w.H)
        flops_rank = w.flops * n // w.H
        sets = []
        for i in range(n_sets):  # every rank holds the same inputs (one call split by heads)
            q, k, v = W.workload_qkv(w, seed_offset=17 * i)
            sets.append((q.to(dev), k.to(dev), v.to(dev), torch.empty_like(q, device=dev)))
        ws = torch.zeros(binding.workspace_shared_bytes(w.B, w.S, n, w.D), dtype=torch.uint8,
                         device=dev)

        def step(i):
            q, k, v, out = sets[i % n_sets]
            binding.joint_rope_attention_heads(q, k, v, txt_d, img_d, h0, n, out=out,
                                               workspace=ws, stream=stream)
        part = f"heads {h0}..{h0 + n - 1} of {w.H} on rank {rank}"
    else:
        q0, n = shard.seq_range(rank, world, w.S)
        flops_rank = 4 * w.B * w.H * n * w.S * w.D
        sets = []
        for i in range(n_sets):
            q, k, v = W.workload_qkv(w, seed_offset=17 * i)
            sets.append(tuple(x[:, q0:q0 + n].contiguous().to(dev) for x in (q, k, v)))
        k_full = torch.empty((w.B, w.S, w.H, w.D), dtype=torch.bfloat16, device=dev)
        v_full = torch.empty_like(k_full)
        out = torch.empty((w.B, n, w.H, w.D), dtype=torch.bfloat16, device=dev)
        ws = torch.zeros(binding.rows_workspace_bytes(w.B, n, w.S, w.H, w.D), dtype=torch.uint8,
                         device=dev)

        def step(i):
            q, k, v = sets[i % n_sets]
            with torch.cuda.stream(stream):
                if dist is not None:
                    shard.gather_sequence(k, w.S, dist, out=k_full)
                    shard.gather_sequence(v, w.S, dist, out=v_full)
                else:
                    k_full.copy_(k)
                    v_full.copy_(v)
            binding.joint_rope_attention_rows(q, q0, k_full, v_full, txt_d, img_d, out=out,
                                              workspace=ws, stream=stream)
        part = f"query rows {q0}..{q0 + n - 1} of {w.S} on rank {rank}"

    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            step(i)
    stream.synchronize()
    K = args.steps
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local_rank) as clocks:
        with torch.cuda.stream(stream):
            torch.cuda._sleep(2_000_000)  # the host enqueues ahead (gpu_head_start)
            ev0.record(stream)
            for i in range(K):
                step(i)
            ev1.record(stream)
        torch.cuda.synchronize(dev)
    if dist is not None:
        dist.barrier()
    if binding.query_status(ws, stream) != 0:
        raise RuntimeError("device status set during the timed steps")
    t_max = max_over_ranks(ev0.elapsed_time(ev1), dist, dev)
    if rank != 0:
        return None
    peaks, peak_src = _peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    value = w.flops * K / (t_max * 1e-3) / 1e12  # one call's FLOPs per step, all ranks
    return {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(t_max / K, 4), "higher_is_better": True,
        "scaling": "strong", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v, FLUX.2 (T,H,W,L) ids)",
        "config": {
            "workload": f"{w.name}: B={w.B} H={w.H} S={w.S} ({w.S_txt} text + {w.S_img} image) "
                        f"head_dim={w.D} axes=(32,32,32,32) theta=2000 non-causal",
            "B": w.B, "H": w.H, "S": w.S,
            "parallelism": (f"head parallel x{world}: each rank attends its heads, no "
                            "collective" if args.shard == "heads" else
                            f"sequence parallel x{world}: K and V all-gathered every step, "
                            "each rank attends its query rows over every key"),
            "rank0": part,
            "l2": f"inputs rotate over {n_sets} sets",
            "flops_rank0_per_step": flops_rank,
        },
        "pct_peak": round(100.0 * value / world / peak, 2),
        "clocks": clocks.summary(),
        "e2e": None,
        "e2e_note": "end-to-end copies are measured on the replicas line (the default)",
        "gpu_launches": 2 * K,
    }


def run_reference(args, rank, world):
    """The oracle on the host cores: each step is a bounded sample of the same
    workload; the line carries the same metric and unit as ours."""
    if rank != 0:
        return None
    import oracle
    from diffusion_transformer_joint_gb300 import workloads as W

    oracle.build()
    w = W.WORKLOADS[args.workload]
    threads = oracle.default_threads()
    inputs = _oracle_inputs(w)
    budget_s = 150.0 / max(1, args.steps + args.warmup)
    rows = _rows_for(w, min(4.0, budget_s), threads, inputs)
    for _ in range(args.warmup):
        _oracle_sample(w, rows[:8], threads, *inputs)
    times = [_oracle_sample(w, rows, threads, *inputs) for _ in range(args.steps)]
    flops = 4 * w.B * w.H * rows.size * w.S * w.D
    tot = sum(times)
    value = flops * len(times) / tot / 1e12
    sample = (f"{rows.size} of {w.S} query rows x all {w.B * w.H} (batch, head) pairs of "
              f"{w.name} per step, fp64")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot / len(times), 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded N(0,1) bf16 q/k/v, FLUX.2 (T,H,W,L) ids)",
        "config": {"workload": f"{w.name}: B={w.B} H={w.H} S={w.S} ({w.S_txt} text + "
                               f"{w.S_img} image) head_dim={w.D} axes=(32,32,32,32) theta=2000 "
                               "non-causal", "B": w.B, "H": w.H, "S": w.S},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default="klein9b")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--kv-mode", choices=("extract", "cached"), default=None,
                    help="time a reference-image KV-mode call on an edit workload instead")
    ap.add_argument("--cpu-report", action="store_true",
                    help="time the fp64 oracle on every workload (all threads and one); no GPU")
    ap.add_argument("--proj", action="store_true",
                    help="time the fused single-stream QKV+MLP input projection instead")
    ap.add_argument("--qk-norm", action="store_true",
                    help="time the entry with the fused QK RMS normalisation before RoPE")
    ap.add_argument("--shard", choices=("replicas", "heads", "seq"), default="replicas",
                    help="replicas: every rank runs its own call (weak scaling, the default); "
                         "heads / seq: one call split over the ranks by heads or by tokens "
                         "(strong scaling)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    if args.gpus > 1 and "WORLD_SIZE" not in os.environ:
        # not started by a launcher: start one rank per GPU on this node
        import socket
        import subprocess

        with socket.socket() as sk:
            sk.bind(("127.0.0.1", 0))
            port = sk.getsockname()[1]
        cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1",
               f"--nproc-per-node={args.gpus}", "--master-addr", "127.0.0.1",
               f"--master-port={port}", os.path.abspath(__file__), *sys.argv[1:]]
        sys.exit(subprocess.run(cmd).returncode)
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world != args.gpus:
        ap.error(f"--gpus {args.gpus} but WORLD_SIZE is {world}")
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.cpu_report:
        line = cpu_report() if rank == 0 else None
    elif args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        if world > 1:
            import torch
            import torch.distributed as dist

            torch.cuda.set_device(local_rank)
            dist.init_process_group("nccl")
        if args.proj:
            line = run_proj(args, rank, world, local_rank)
        elif args.shard != "replicas":
            line = run_sharded(args, rank, world, local_rank)
        elif args.kv_mode is not None:
            if args.workload == "klein9b":
                args.workload = "klein9b_edit2"
            line = run_kv(args, rank, world, local_rank)
        else:
            line = run_ours(args, rank, world, local_rank)
        if world > 1:
            import torch.distributed as dist

            dist.destroy_process_group()
    if line is not None:
        print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()

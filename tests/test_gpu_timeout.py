"""Failure detection without a GPU fault: a bounded wait that runs out.

The test compiles a copy of the library in which the RoPE warps of every
CTA withhold their hand-off of key tile 0 (a barrier arrival that nothing
else provides; without the exchange buffer every K tile goes through them). The MMA thread's wait on it is bounded (about a
second of clock cycles); when it runs out the kernel raises its abort flag,
every other role leaves its loop, copies still in flight are waited for,
TMEM is released and FLUX_ERR_DEVICE_TIMEOUT lands in the status word. No
trap, no fault: afterwards the context is still usable and the regular
library computes the correct result on the same stream.
"""
import ctypes
import shutil
import subprocess
import time

import numpy as np
import pytest
import torch

import oracle
from diffusion_transformer_joint_gb300 import binding, build
from diffusion_transformer_joint_gb300 import workloads as W

pytestmark = pytest.mark.gpu

ANCHOR = "warp_arrive(bar(kBarKFull + s), lane);"
WITHHELD = "if (tj != 0) warp_arrive(bar(kBarKFull + s), lane);"


def _build_withholding_library(tmp_path):
    src = tmp_path / "csrc"
    shutil.copytree(build.CSRC, src)
    f = src / "attention_sm103a.cu"
    text = f.read_text()
    assert text.count(ANCHOR) == 1, "the K hand-off to patch was not found exactly once"
    f.write_text(text.replace(ANCHOR, WITHHELD))
    out = tmp_path / "libflux_attn_withheld.so"
    flags = [x for x in build.NVCC_FLAGS if x not in ("-Xptxas", "-v")]
    subprocess.run([build.nvcc(), *flags, "-I", build.INCLUDE, "-I", str(src),
                    *sorted(str(p) for p in src.glob("*.cu")), "-o", str(out)],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(str(out))
    V, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.flux_joint_rope_attention.argtypes = [V, V, V, V, I64, V, I64, I32, I32, I32, V, I32,
                                              ctypes.c_double, V, V, ctypes.c_size_t, V]
    lib.flux_joint_rope_attention.restype = I32
    lib.flux_query_status.argtypes = [V, V]
    lib.flux_query_status.restype = I32
    return lib


def test_bounded_wait_reports_timeout_and_context_survives(tmp_path):
    build.build()
    binding.load()
    lib = _build_withholding_library(tmp_path)
    w = W.WORKLOADS["tiny"]
    q, k, v = (t.cuda() for t in W.workload_qkv(w))
    txt_np, img_np = W.workload_ids(w)
    txt, img = (torch.from_numpy(x).cuda() for x in (txt_np, img_np))
    out = torch.zeros_like(q)
    ws = torch.zeros(binding.workspace_bytes(w.S), dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    axes = (ctypes.c_int32 * 4)(32, 32, 32, 32)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    t0 = time.time()
    rc = lib.flux_joint_rope_attention(P(q), P(k), P(v), P(txt), w.S_txt, P(img), w.S_img,
                                       w.B, w.H, w.D, axes, 4, 2000.0, P(out), P(ws),
                                       ws.numel(), ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    status = lib.flux_query_status(P(ws), ctypes.c_void_p(stream.cuda_stream))
    elapsed = time.time() - t0
    assert status == -7, f"expected FLUX_ERR_DEVICE_TIMEOUT, got {status}"
    assert elapsed < 60.0, f"bounded wait took {elapsed:.1f} s"
    # the context is usable: the regular library runs and is correct
    good = binding.joint_rope_attention(q, k, v, txt, img, workspace=ws)
    assert binding.query_status(ws) == 0
    ref = oracle.joint_rope_attention(q.float().cpu().numpy(), k.float().cpu().numpy(),
                                      v.float().cpu().numpy(), txt_np, img_np)
    assert np.abs(good.float().cpu().numpy() - ref).max() <= 1e-2


PROJ_ANCHOR = "if (lane == 0) mbar_arrive_cluster(acc_empty0 + 8u * static_cast<uint32_t>(buf));"
PROJ_WITHHELD = ("if (lane == 0 && lt != 0) "
                 "mbar_arrive_cluster(acc_empty0 + 8u * static_cast<uint32_t>(buf));")


def test_projection_bounded_wait_reports_timeout(tmp_path):
    """The fused projection's epilogue warps withhold the release of their
    first accumulator; a CTA pair with a third tile then waits for it in its
    MMA warp until the bounded wait runs out. 160 tiles over at most 76 CTA
    pairs give pair 0 a third tile."""
    build.build()
    binding.load()
    src = tmp_path / "csrc"
    shutil.copytree(build.CSRC, src)
    f = src / "proj_sm103a.cu"
    text = f.read_text()
    assert text.count(PROJ_ANCHOR) == 1, "the accumulator release was not found exactly once"
    f.write_text(text.replace(PROJ_ANCHOR, PROJ_WITHHELD))
    out = tmp_path / "libflux_proj_withheld.so"
    flags = [x for x in build.NVCC_FLAGS if x not in ("-Xptxas", "-v")]
    subprocess.run([build.nvcc(), *flags, "-I", build.INCLUDE, "-I", str(src),
                    *sorted(str(p) for p in src.glob("*.cu")), "-o", str(out)],
                   check=True, capture_output=True)
    lib = ctypes.CDLL(str(out))
    V, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.flux_qkv_mlp_proj.argtypes = [V, V, I64, I32, I32, I32, I64, V, V, V, V, V, V]
    lib.flux_qkv_mlp_proj.restype = I32
    M, dim, H, mlp = 1280, 64, 16, 1024  # 5 256-row blocks x (24 + 8) feature tiles
    x = W.normal_bf16((M, dim), 31).cuda()
    w = W.normal_bf16((3 * H * 128 + 2 * mlp, dim), 32, scale=dim ** -0.5).cuda()
    q, k, v = (torch.empty((M, H, 128), dtype=torch.bfloat16, device="cuda") for _ in range(3))
    act = torch.empty((M, mlp), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream()
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    t0 = time.time()
    rc = lib.flux_qkv_mlp_proj(P(x), P(w), M, dim, H, 128, mlp, P(q), P(k), P(v), P(act),
                               P(status), ctypes.c_void_p(stream.cuda_stream))
    assert rc == 0
    torch.cuda.synchronize()
    elapsed = time.time() - t0
    assert int(status.item()) == -7, f"expected FLUX_ERR_DEVICE_TIMEOUT, got {int(status.item())}"
    assert elapsed < 60.0, f"bounded wait took {elapsed:.1f} s"
    # the context is usable: the regular library runs and is correct
    status.zero_()
    gq, _, _, gact = binding.qkv_mlp_proj(x, w, H, mlp, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = np.array([0, 700, M - 1])
    rq, _, _, ra = oracle.qkv_mlp_proj(x.float().cpu().numpy(), w.float().cpu().numpy(), H, 128,
                                       mlp, rows=rows)
    gq_np = gq.float().cpu().numpy()[rows]
    assert np.all(np.abs(gq_np - rq) <= 2.0 ** -8 * np.abs(rq) + 1e-4)
    ga_np = gact.float().cpu().numpy()[rows]
    assert np.all(np.abs(ga_np - ra) <= 2.0 ** -8 * np.abs(ra) + 1e-4)

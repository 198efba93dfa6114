"""The library used from plain C: tests/c_abi/attention_from_c.c includes only
include/flux_attn.h and the CUDA runtime, allocates with cudaMalloc, calls the
one-call entry point and reads its status word. On the CPU the program must
compile warning-free as C11 and link against the built library; on the GPU its
output must equal the Python binding's bit for bit and the oracle's within the
bar (max 1e-2, mean 1e-3)."""
import os
import subprocess

import numpy as np
import pytest

from diffusion_transformer_joint_gb300 import binding, build
from diffusion_transformer_joint_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "c_abi", "attention_from_c.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _compile(tmp_path):
    lib = build.build()
    exe = tmp_path / "attention_from_c"
    libdir = os.path.dirname(lib)
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-Werror", "-I", build.INCLUDE,
           "-I", os.path.join(CUDA, "include"), SRC, "-o", str(exe), "-L", libdir, "-lflux_attn",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{libdir}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert _compile(tmp_path).exists()


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,S_txt,S_img", [(1, 2, 16, 64), (2, 3, 7, 300)])
def test_c_program_matches_binding_and_oracle(tmp_path, B, H, S_txt, S_img):
    import torch

    import oracle

    exe = _compile(tmp_path)
    S = S_txt + S_img
    q, k, v = (W.normal_bf16((B, S, H, 128), 7000 + S + i) for i in range(3))
    ids = W.random_ids(S, 7003 + S, 0, 300)
    for name, t in (("q", q), ("k", k), ("v", v)):
        t.contiguous().view(torch.int16).numpy().tofile(tmp_path / f"{name}.bin")
    ids[:S_txt].astype(np.int32).tofile(tmp_path / "txt_ids.bin")
    ids[S_txt:].astype(np.int32).tofile(tmp_path / "img_ids.bin")
    res = subprocess.run([str(exe), str(tmp_path), str(B), str(S_txt), str(S_img), str(H)],
                         capture_output=True, text=True, timeout=120)
    assert res.returncode == 0, res.stderr
    raw = np.fromfile(tmp_path / "out.bin", dtype=np.int16).reshape(B, S, H, 128)
    got = torch.from_numpy(raw).view(torch.bfloat16)
    ref_py = binding.joint_rope_attention(q.cuda(), k.cuda(), v.cuda(),
                                          torch.from_numpy(ids[:S_txt]).cuda(),
                                          torch.from_numpy(ids[S_txt:]).cuda())
    torch.cuda.synchronize()
    assert torch.equal(got, ref_py.cpu())
    ref = oracle.joint_rope_attention(q.float().numpy(), k.float().numpy(), v.float().numpy(),
                                      ids[:S_txt], ids[S_txt:])
    err = np.abs(got.float().numpy() - ref)
    assert err.max() <= 1e-2 and err.mean() <= 1e-3

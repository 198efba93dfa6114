"""Builds the CUDA library libflux_attn.so in-tree with nvcc for sm_103a.

Usage: ``python -m diffusion_transformer_joint_gb300.build [--force] [--checked]``.
``--checked`` builds libflux_attn_checked.so instead: the same library compiled
with -DFLUX_DEBUG, whose attention kernel checks its shared-memory, TMEM, TMA
and exchange-buffer accesses and reports a failed check in the status word
(the binding loads it when FLUX_ATTN_DEBUG=1).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_NAME = "libflux_attn.so"
LIB_PATH = os.path.join(BUILD_DIR, LIB_NAME)
CHECKED_LIB_PATH = os.path.join(BUILD_DIR, "libflux_attn_checked.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17", "--threads", "0",
    "-Xcompiler", "-fPIC,-O2", "-shared",
    "-Xptxas", "-v",
]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + sorted(
        glob.glob(os.path.join(CSRC, "*.h"))) + sorted(glob.glob(os.path.join(INCLUDE, "*.h")))


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, out: str = LIB_PATH, defines=(), verbose: bool = False) -> str:
    """Compile every csrc/*.cu into one shared library; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    if not force and os.path.exists(out):
        t = os.path.getmtime(out)
        if all(os.path.getmtime(p) <= t for p in _inputs()):
            return out
    tmp = out + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, "-I", INCLUDE, "-I", CSRC,
           *[f"-D{d}" for d in defines], *sources(), "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(os.path.dirname(out), "nvcc.log")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + res.stdout + res.stderr)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc failed (log: {log})")
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, out)
    return out


def build_checked(force: bool = False, out: str = CHECKED_LIB_PATH) -> str:
    """The checked library (-DFLUX_DEBUG) at ``out``; returns its path."""
    return build(force=force, out=out, defines=("FLUX_DEBUG",))


if __name__ == "__main__":
    if "--checked" in sys.argv:
        print(build_checked(force="--force" in sys.argv))
    else:
        print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""flux_joint_rope_attention_noalloc: the entry point for callers that cannot
allocate device memory (its scratch is a fixed device array inside the
library). Collected last on purpose: if it fails, a run that stops at the
first failure has already run every other test.

The GPU test calls the new entry point through the C-ABI twice in a row, on
different inputs, and compares each result with the regular entry point's
(which uses a caller-allocated workspace) at the suite's tolerance. It does
not depend on any earlier test, so it passes alone in a fresh process too.
"""
import ctypes

import pytest

from diffusion_transformer_joint_gb300 import binding, build
from diffusion_transformer_joint_gb300 import workloads as W

MAX_ABS = 1e-2
MEAN_ABS = 1e-3
MAX_TOKENS = 32768


def _noalloc(lib):
    fn = lib.flux_joint_rope_attention_noalloc
    V, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [V, V, V, V, I64, V, I64, I32, I32, I32, V, I32, ctypes.c_double, V, V]
    fn.restype = I32
    return fn


def _call(fn, q, k, v, txt, img, out, S_txt, S_img, stream=None):
    B, S, H, D = (q.shape if q is not None else (1, S_txt + S_img, 1, 128))
    axes = (ctypes.c_int32 * 4)(32, 32, 32, 32)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return fn(P(q), P(k), P(v), P(txt), S_txt, P(img), S_img, B, H, D, axes, 4, 2000.0, P(out),
              stream)


def test_noalloc_rejects_sequences_beyond_its_scratch():
    build.build()
    fn = _noalloc(binding.load())
    # rejected on the host before any pointer is used or any device is touched
    assert fn(ctypes.c_void_p(16), ctypes.c_void_p(32), ctypes.c_void_p(48), ctypes.c_void_p(64),
              16, ctypes.c_void_p(80), MAX_TOKENS, 1, 1, 128, (ctypes.c_int32 * 4)(32, 32, 32, 32),
              4, 2000.0, ctypes.c_void_p(96), None) == -2


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point_twice():
    import torch

    build.build()
    fn = _noalloc(binding.load())
    stream = torch.cuda.current_stream()
    for case, (name, seed_offset) in enumerate((("tiny", 0), ("klein4b", 7))):
        w = W.WORKLOADS[name]
        q, k, v = (t.cuda() for t in W.workload_qkv(w, seed_offset=seed_offset))
        txt, img = (torch.from_numpy(x).cuda() for x in W.workload_ids(w))
        expected = binding.joint_rope_attention(q, k, v, txt, img)
        got = torch.full_like(q, float("nan"))
        rc = _call(fn, q, k, v, txt, img, got, w.S_txt, w.S_img,
                   ctypes.c_void_p(stream.cuda_stream))
        assert rc == 0, binding.load().flux_status_string(rc)
        torch.cuda.synchronize()
        err = (got.float() - expected.float()).abs()
        assert torch.isfinite(got).all(), f"call {case}: non-finite output"
        assert err.max().item() <= MAX_ABS and err.mean().item() <= MEAN_ABS, \
            f"call {case}: max {err.max().item():.3e} mean {err.mean().item():.3e}"

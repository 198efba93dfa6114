"""flux_joint_rope_attention_noalloc: the entry point for callers that cannot
allocate device memory (a plugin whose host application owns all device
memory, or code that must not risk cudaMalloc's device synchronisation). Its
scratch is a fixed device array inside the library. Collected last on purpose:
if it fails, a run that stops at the first failure has already run every
other test.

The GPU test calls the entry point through the C-ABI several times in a row,
on different inputs, and compares each result with the regular entry point's
(which uses a caller-allocated workspace of the same, smallest size, so
neither uses the rotated-K exchange buffer): the two are bit-identical. After
each call the status word in the library's array reads FLUX_OK. One case
fills the array: a sequence of exactly the maximum number of tokens. The
test depends on no earlier test, so it passes alone in a fresh process too.
"""
import ctypes

import pytest

from diffusion_transformer_joint_gb300 import binding, build
from diffusion_transformer_joint_gb300 import workloads as W

MAX_TOKENS = 32768  # FLUX_NOALLOC_MAX_TOKENS
FLUX_ERR_SHAPE = -2


def _noalloc(lib):
    fn = lib.flux_joint_rope_attention_noalloc
    V, I64, I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    fn.argtypes = [V, V, V, V, I64, V, I64, I32, I32, I32, V, I32, ctypes.c_double, V, V]
    fn.restype = I32
    st = lib.flux_joint_rope_attention_noalloc_status
    st.argtypes = [V]
    st.restype = I32
    return fn, st


def _call(fn, q, k, v, txt, img, out, S_txt, S_img, stream=None):
    B, S, H, D = q.shape
    axes = (ctypes.c_int32 * 4)(32, 32, 32, 32)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    return fn(P(q), P(k), P(v), P(txt), S_txt, P(img), S_img, B, H, D, axes, 4, 2000.0, P(out),
              stream)


def _host_reject(fn, S_txt, S_img):
    # rejected on the host before any pointer is used or any device is touched
    p = lambda a: ctypes.c_void_p(a)
    return fn(p(16), p(32), p(48), p(64), S_txt, p(80), S_img, 1, 1, 128,
              (ctypes.c_int32 * 4)(32, 32, 32, 32), 4, 2000.0, p(96), None)


def test_noalloc_rejects_sequences_beyond_its_scratch():
    build.build()
    fn, _ = _noalloc(binding.load())
    assert _host_reject(fn, 16, MAX_TOKENS - 15) == FLUX_ERR_SHAPE
    assert _host_reject(fn, MAX_TOKENS + 1, 0) == FLUX_ERR_SHAPE
    # two sizes whose sum overflows int64 are rejected, not wrapped around
    assert _host_reject(fn, 2 ** 62, 2 ** 62) == FLUX_ERR_SHAPE
    assert _host_reject(fn, 2 ** 63 - 1, 1) == FLUX_ERR_SHAPE
    assert _host_reject(fn, -1, 16) == FLUX_ERR_SHAPE


def _cases():
    """(q, k, v, txt ids, img ids) on the GPU: the tiny and klein-4B workloads
    (different seeds) and a sequence of exactly the maximum length."""
    import torch

    for name, seed_offset in (("tiny", 0), ("klein4b", 7)):
        w = W.WORKLOADS[name]
        q, k, v = (t.cuda() for t in W.workload_qkv(w, seed_offset=seed_offset))
        txt, img = (torch.from_numpy(x).cuda() for x in W.workload_ids(w))
        yield name, q, k, v, txt, img
    S_txt, S = 512, MAX_TOKENS
    q, k, v = (W.normal_bf16((1, S, 1, 128), 2100 + i).cuda() for i in range(3))
    ids = torch.from_numpy(W.random_ids(S, 2103, 0, 200)).cuda()
    yield "max_tokens", q, k, v, ids[:S_txt], ids[S_txt:]


@pytest.mark.gpu
def test_noalloc_matches_regular_entry_point():
    import torch

    build.build()
    lib = binding.load()
    fn, status_fn = _noalloc(lib)
    stream = torch.cuda.current_stream()
    handle = ctypes.c_void_p(stream.cuda_stream)
    for name, q, k, v, txt, img in _cases():
        S_txt, S_img = txt.shape[0], img.shape[0]
        ws = torch.zeros(binding.workspace_bytes(S_txt + S_img), dtype=torch.uint8, device="cuda")
        expected = binding.joint_rope_attention(q, k, v, txt, img, workspace=ws)
        for call in range(2):
            got = torch.full_like(q, float("nan"))
            rc = _call(fn, q, k, v, txt, img, got, S_txt, S_img, handle)
            assert rc == 0, (name, call, lib.flux_status_string(rc))
            assert status_fn(handle) == 0, (name, call)
            torch.cuda.synchronize()
            assert torch.equal(got, expected), f"{name}, call {call}: differs from the regular entry"

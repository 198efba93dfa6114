"""The synthetic workloads against the hyper-parameters the pages print."""
import os

import numpy as np

from diffusion_transformer_joint_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "flux2_config.txt")


def _golden():
    vals = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].strip()
        if line:
            key, *rest = line.split()
            vals[key] = [int(x) for x in rest]
    return vals


def test_workloads_match_printed_config():
    g = _golden()
    assert W.HEAD_DIM == g["head_dim"][0]
    assert tuple(W.AXES_DIMS) == tuple(g["axes_dims"])
    assert W.ROPE_THETA == g["rope_theta"][0]
    for name, key in (("klein4b", "klein4b"), ("klein9b", "klein9b"), ("dev32b", "dev32b")):
        w = W.WORKLOADS[name]
        assert w.H == g["heads_" + key][0]
        assert w.H * w.D == g["hidden_" + key][0]
        assert w.S_txt == g["text_tokens"][0]
        assert w.grid * w.grid == g["image_tokens_1024"][0]
        assert w.S == 4608
    e = W.WORKLOADS["klein9b_edit2"]
    assert e.S == 512 + 3 * 4096 == 12800 and e.H == 32


def test_projection_dims_match_printed_config():
    g = _golden()
    for name in ("klein4b", "klein9b", "dev32b"):
        w = W.WORKLOADS[name]
        M, dim, mlp = W.proj_dims(w)
        assert dim == g["hidden_" + name][0] and M == w.S
        assert 10 * mlp == g["mlp_ratio_tenths"][0] * dim
        assert W.proj_flops(w) == 2 * M * dim * (3 * dim + g["mlp_halves"][0] * mlp)
    x, wt = W.proj_inputs(W.WORKLOADS["tiny"])
    assert tuple(x.shape) == (80, 256) and tuple(wt.shape) == (3 * 256 + 2 * 768, 256)


def test_ids_recipe():
    w = W.WORKLOADS["klein9b_edit2"]
    txt, img = W.workload_ids(w)
    assert txt.shape == (512, 4) and img.shape == (3 * 4096, 4)
    assert np.array_equal(txt[:, 3], np.arange(512)) and not txt[:, :3].any()
    assert np.array_equal(img[:4096, 0], np.zeros(4096))
    assert np.array_equal(img[4096:8192, 0], np.full(4096, 10))
    assert np.array_equal(img[8192:, 0], np.full(4096, 20))
    assert img[65, 1] == 1 and img[65, 2] == 1 and not img[:, 3].any()
    assert w.flops == 4 * 32 * 12800 * 12800 * 128


def test_inputs_are_seeded_bf16():
    import torch

    w = W.WORKLOADS["tiny"]
    q1, k1, v1 = W.workload_qkv(w)
    q2, _, _ = W.workload_qkv(w)
    assert q1.dtype == torch.bfloat16 and q1.shape == (1, 80, 2, 128)
    assert torch.equal(q1, q2) and not torch.equal(q1, k1)
    assert abs(float(q1.float().std()) - 1.0) < 0.1

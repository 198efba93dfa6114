"""The C-ABI library on the host: it loads, exports every declared symbol, and
rejects bad arguments with the documented status before touching a device."""
import ctypes
import os
import re

import pytest

from diffusion_transformer_joint_gb300 import binding, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def _declared_symbols():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names.update(re.findall(r"\b(flux_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_symbol_is_exported(lib):
    declared = _declared_symbols()
    assert set(binding.EXPORTS) <= set(declared)
    for name in declared:
        assert hasattr(lib, name), name


def _declared_signatures():
    """name -> (return type, [parameter types]) from the header, as C type strings."""
    sigs = {}
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for ret, name, params in re.findall(
                r"([A-Za-z_][A-Za-z0-9_ ]*?\**)\s*\b(flux_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
            types = []
            for prm in params.split(","):
                prm = prm.strip()
                types.append("ptr" if "*" in prm else prm.rsplit(None, 1)[0].replace("const ", ""))
            sigs[name] = ("ptr" if "*" in ret else ret.split()[-1], types)
    return sigs


_CTYPE_OF = {"ptr": (ctypes.c_void_p, ctypes.c_char_p), "int": (ctypes.c_int,),
             "int64_t": (ctypes.c_int64,), "size_t": (ctypes.c_size_t,),
             "double": (ctypes.c_double,), "float": (ctypes.c_float,)}


def test_binding_marshals_every_argument_as_declared(lib):
    # a wrong ctypes width (an int where the header has int64_t, a float for a
    # double) would pass garbage through the ABI without any error
    sigs = _declared_signatures()
    assert set(binding.EXPORTS) <= set(sigs)
    for name in binding.EXPORTS:
        ret, params = sigs[name]
        fn = getattr(lib, name)
        assert len(fn.argtypes) == len(params), name
        for i, (have, want) in enumerate(zip(fn.argtypes, params)):
            assert have in _CTYPE_OF[want], (name, i, have, want)
        assert fn.restype in _CTYPE_OF[ret], (name, fn.restype, ret)


def test_status_strings(lib):
    for code in binding.STATUS:
        assert lib.flux_status_string(code)
    assert lib.flux_status_string(12345) == b"unknown status"


def test_workspace_size(lib):
    assert lib.flux_joint_rope_attention_workspace(4608, 128) == 256 + 4608 * 64 * 4
    assert lib.flux_joint_rope_attention_workspace(80, 128) == 256 + 20480
    assert lib.flux_joint_rope_attention_workspace(1, 128) == 256 + 256
    assert lib.flux_joint_rope_attention_workspace(0, 128) == 0
    assert lib.flux_joint_rope_attention_workspace(10, 7) == 0


def test_krot_and_shared_workspace_sizes(lib):
    # flags: B*H*ceil(S/128)*4 words of 8 bytes, padded to 256; then rotated K
    # and rotated Q, each bf16 [B, S, H, 128]
    assert (lib.flux_joint_rope_attention_krot_bytes(1, 4608, 32, 128)
            == 36864 + 2 * 4608 * 32 * 256)
    assert lib.flux_joint_rope_attention_krot_bytes(1, 80, 2, 128) == 256 + 2 * 80 * 2 * 256
    # 2 * 3 * 2 tiles * 4 words * 8 B = 384 -> 512
    assert (lib.flux_joint_rope_attention_krot_bytes(2, 129, 3, 128)
            == 512 + 2 * 2 * 129 * 3 * 256)
    assert (lib.flux_joint_rope_attention_workspace_shared(1, 4608, 32, 128)
            == lib.flux_joint_rope_attention_workspace(4608, 128)
            + lib.flux_joint_rope_attention_krot_bytes(1, 4608, 32, 128))
    for B, S, H, D in ((0, 80, 2, 128), (1, 0, 2, 128), (1, 80, 0, 128), (1, 80, 2, 64)):
        assert lib.flux_joint_rope_attention_krot_bytes(B, S, H, D) == 0
        assert lib.flux_joint_rope_attention_workspace_shared(B, S, H, D) == 0


def _call(lib, **kw):
    args = dict(q=16, k=16 * 1024, v=32 * 1024, txt=None, S_txt=16, img=None, S_img=64, B=1, H=2,
                D=128, axes=(32, 32, 32, 32), theta=2000.0, out=48 * 1024 * 1024, ws=256 * 4096,
                ws_bytes=1 << 20)
    args.update(kw)
    axes = (ctypes.c_int32 * len(args["axes"]))(*args["axes"])
    P = lambda x: None if x is None else ctypes.c_void_p(x)
    txt = args["txt"] if "txt" in kw else 1024
    img = args["img"] if "img" in kw else 2048
    return lib.flux_joint_rope_attention(P(args["q"]), P(args["k"]), P(args["v"]), P(txt),
                                         args["S_txt"], P(img), args["S_img"], args["B"],
                                         args["H"], args["D"], axes, len(args["axes"]),
                                         args["theta"], P(args["out"]), P(args["ws"]),
                                         args["ws_bytes"], None)


# Every case fails a host-side check, so no pointer is dereferenced.
@pytest.mark.parametrize("kw,code", [
    (dict(q=None), -1),
    (dict(out=None), -1),
    (dict(txt=None), -1),
    (dict(S_txt=-1), -2),
    (dict(S_txt=0, S_img=0), -2),
    (dict(D=64), -2),
    (dict(B=0), -2),
    (dict(H=0), -2),
    (dict(axes=(32, 32, 32)), -3),
    (dict(axes=(33, 31, 32, 32)), -3),
    (dict(axes=(32, 32, 32, 32, 0)), -3),
    (dict(axes=(16,) * 9), -3),
    (dict(theta=0.0), -3),
    (dict(q=17), -4),
    (dict(out=16 + 1024), -9),
    (dict(ws=None), -5),
    (dict(ws=256 * 4096 + 16), -5),
    (dict(ws_bytes=100), -5),
    (dict(ws=256), -9),               # workspace overlaps q
    (dict(ws=48 * 1024 * 1024), -9),  # workspace overlaps out
])
def test_bad_arguments_rejected_on_host(lib, kw, code):
    assert _call(lib, **kw) == code


def test_rope_tables_bad_arguments(lib):
    axes = (ctypes.c_int32 * 4)(32, 32, 32, 32)
    P = ctypes.c_void_p
    assert lib.flux_rope_tables(None, 4, axes, 4, 2000.0, P(16), P(32), None) == -1
    assert lib.flux_rope_tables(P(16), 0, axes, 4, 2000.0, P(16), P(32), None) == -2
    bad = (ctypes.c_int32 * 2)(3, 4)
    assert lib.flux_rope_tables(P(16), 4, bad, 2, 2000.0, P(16), P(32), None) == -3
    assert lib.flux_rope_tables_packed(None, 4, axes, 4, 2000.0, P(16), None) == -1
    assert lib.flux_rope_tables_packed(P(16), 0, axes, 4, 2000.0, P(16), None) == -2
    assert lib.flux_rope_tables_packed(P(16), 4, bad, 2, 2000.0, P(16), None) == -3


def _tabled(lib, krot, krot_bytes, out=48 * 1024 * 1024):
    P = ctypes.c_void_p
    return lib.flux_joint_rope_attention_tabled(P(16), P(16 * 1024), P(32 * 1024), P(4096 * 256),
                                                1, 80, 2, 128, P(out), P(64), None if krot is None
                                                else P(krot), krot_bytes, None)


def test_tabled_exchange_buffer_checked_on_host(lib):
    need = lib.flux_joint_rope_attention_krot_bytes(1, 80, 2, 128)
    assert _tabled(lib, 256 * 8192 + 16, need) == -5      # not 256-byte aligned
    assert _tabled(lib, 256 * 8192, need - 1) == -5        # too small
    assert _tabled(lib, 256, need) == -9                   # overlaps q
    assert _tabled(lib, 48 * 1024 * 1024 + 256, need) == -9  # overlaps out


def test_qknorm_arguments_checked_on_host(lib):
    P = ctypes.c_void_p
    axes = (ctypes.c_int32 * 4)(32, 32, 32, 32)
    W = 8 * 4096  # fake 16-byte-aligned weight vectors

    def one_call(qt=W, kt=W + 512, qi=W + 1024, ki=W + 1536, eps=1e-6):
        return lib.flux_joint_qknorm_rope_attention(
            P(16), P(16 * 1024), P(32 * 1024), P(1024), 16, P(2048), 64, 1, 2, 128, axes, 4,
            2000.0, P(qt) if qt else None, P(kt) if kt else None, P(qi) if qi else None,
            P(ki) if ki else None, eps, P(48 * 1024 * 1024), P(256 * 4096), 1 << 20, None)

    assert one_call(qt=0) == -1
    assert one_call(ki=0) == -1
    assert one_call(kt=W + 8) == -4
    assert one_call(eps=-1.0) == -2
    assert one_call(eps=float("nan")) == -2

    def tab(s_txt):
        return lib.flux_joint_qknorm_rope_attention_tabled(
            P(16), P(16 * 1024), P(32 * 1024), P(4096 * 256), 1, 80, 2, 128, s_txt, P(W),
            P(W + 512), P(W + 1024), P(W + 1536), 1e-6, P(48 * 1024 * 1024), P(64), None, 0,
            None)

    assert tab(81) == -2
    assert tab(-1) == -2


def test_kv_mode_workspace_sizes_and_checks(lib):
    P = ctypes.c_void_p
    assert lib.flux_joint_rope_attention_extract_workspace(1, 512, 8192, 4096, 32, 128) > 0
    assert lib.flux_joint_rope_attention_extract_workspace(1, 0, 0, 0, 32, 128) == 0
    assert lib.flux_joint_rope_attention_extract_workspace(1, 5, 5, 5, 32, 64) == 0
    assert lib.flux_joint_rope_attention_cached_workspace(1, 512, 4096, 8192, 32, 128) > 0
    assert lib.flux_joint_rope_attention_cached_workspace(1, 0, 0, 8, 32, 128) == 0
    axes = (ctypes.c_int32 * 4)(32, 32, 32, 32)
    need = lib.flux_joint_rope_attention_extract_workspace(1, 16, 32, 32, 2, 128)

    def extract(ck=96 * 1024 * 1024, ws=256 * 65536, wsb=None, ref_ids=3072):
        return lib.flux_joint_rope_attention_extract(
            P(16), P(64 * 1024), P(128 * 1024), P(1024), 16, P(ref_ids) if ref_ids else None, 32,
            P(2048), 32, 1, 2, 128, axes, 4, 2000.0, P(48 * 1024 * 1024), P(ck) if ck else None,
            P(100 * 1024 * 1024), P(ws), need if wsb is None else wsb, None)

    assert extract(ck=0) == -1            # cache needed when S_ref > 0
    assert extract(ref_ids=0) == -1       # ids needed for a non-empty segment
    assert extract(wsb=need - 1) == -5    # workspace too small
    assert extract(ck=16) == -9           # cache overlaps q
    cneed = lib.flux_joint_rope_attention_cached_workspace(1, 16, 32, 8, 2, 128)
    assert lib.flux_joint_rope_attention_cached(
        P(16), P(64 * 1024), P(128 * 1024), P(1024), 16, P(2048), 32, None, P(200 * 1024), 8, 1,
        2, 128, axes, 4, 2000.0, P(48 * 1024 * 1024), P(256 * 65536), cneed, None) == -1
    assert lib.flux_joint_rope_attention_cached(
        P(16), P(64 * 1024), P(128 * 1024), P(1024), 16, P(2048), 32, P(300 * 1024),
        P(200 * 1024 + 8), 8, 1, 2, 128, axes, 4, 2000.0, P(48 * 1024 * 1024), P(256 * 65536),
        cneed, None) == -4


def test_qkv_mlp_proj_argument_checks(lib):
    P = ctypes.c_void_p
    MB = 1 << 20

    def call(x=16, w=64 * MB, M=100, dim=128, H=2, D=128, mlp=256, q=128 * MB, k=129 * MB,
             v=130 * MB, act=131 * MB, status=200 * MB):
        return lib.flux_qkv_mlp_proj(P(x) if x else None, P(w) if w else None, M, dim, H, D, mlp,
                                     P(q) if q else None, P(k) if k else None,
                                     P(v) if v else None, P(act) if act else None,
                                     P(status) if status else None, None)

    assert call(x=0) == -1
    assert call(status=0) == -1
    assert call(act=0) == -1               # the MLP half needs act
    assert call(D=64) == -2
    assert call(dim=96) == -2              # dim a multiple of 64
    assert call(mlp=200) == -2             # mlp a multiple of 128
    assert call(M=0) == -2
    assert call(q=128 * MB + 8) == -4
    assert call(k=128 * MB + 4096) == -9   # k overlaps q
    assert call(act=1024) == -9            # act overlaps x
    assert call(v=64 * MB + 64) == -9      # v overlaps w


def test_kv_modes_with_norm_argument_checks(lib):
    P = ctypes.c_void_p
    axes = (ctypes.c_int32 * 4)(32, 32, 32, 32)
    need = lib.flux_joint_rope_attention_extract_workspace(1, 16, 32, 32, 2, 128)
    w = [P(200 * 1024 * 1024 + 512 * i) for i in range(4)]

    def extract(weights=w, eps=1e-6):
        return lib.flux_joint_qknorm_rope_attention_extract(
            P(16), P(64 * 1024), P(128 * 1024), P(1024), 16, P(3072), 32, P(2048), 32, 1, 2, 128,
            axes, 4, 2000.0, *weights, eps, P(48 * 1024 * 1024), P(96 * 1024 * 1024),
            P(100 * 1024 * 1024), P(256 * 65536), need, None)

    assert extract(weights=[w[0], None, w[2], w[3]]) == -1       # every weight vector needed
    assert extract(weights=[P(200 * 1024 * 1024 + 4)] + w[1:]) == -4  # 16-byte aligned
    assert extract(eps=-1.0) == -2                                 # eps >= 0
    cneed = lib.flux_joint_rope_attention_cached_workspace(1, 16, 32, 8, 2, 128)
    assert lib.flux_joint_qknorm_rope_attention_cached(
        P(16), P(64 * 1024), P(128 * 1024), P(1024), 16, P(2048), 32, P(300 * 1024),
        P(200 * 1024), 8, 1, 2, 128, axes, 4, 2000.0, None, w[1], w[2], w[3], 1e-6,
        P(48 * 1024 * 1024), P(256 * 65536), cneed, None) == -1


def test_norm_weight_shapes_checked_in_the_binding():
    # the kernels read 128 fp32 weights through each pointer: a shorter vector
    # is refused before anything reaches the library
    import torch

    good = torch.ones(128)
    with pytest.raises(ValueError, match="shape"):
        binding._norm_args((torch.ones(64), good, good, good, 1e-6), "cpu")
    with pytest.raises(ValueError, match="shape"):
        binding._norm_args((good, good, good, torch.ones(2, 128), 1e-6), "cpu")
    with pytest.raises(ValueError, match="qk_norm must be"):
        binding._norm_args((good, good, good, 1e-6), "cpu")
    # right shapes pass that check and stop at the device check (no CPU path)
    with pytest.raises(ValueError, match="CUDA"):
        binding._norm_args((good, good, good, good, 1e-6), "cpu")


def test_checked_build_compiles_and_is_selected_by_the_environment(monkeypatch):
    """The -DFLUX_DEBUG library builds (nvcc cross-compiles here), exports every
    declared symbol, and is the one the binding picks with FLUX_ATTN_DEBUG=1."""
    path = build.build_checked()
    checked = ctypes.CDLL(path)
    for name in _declared_symbols():
        assert hasattr(checked, name), name
    # a failed check's code reads as such; release codes are unchanged
    checked.flux_status_string.restype = ctypes.c_char_p
    assert b"checked" in checked.flux_status_string(-1005)
    assert checked.flux_status_string(-7) == b"a kernel gave up a bounded wait (device timeout)"
    monkeypatch.delenv("FLUX_ATTN_LIB", raising=False)
    monkeypatch.setenv("FLUX_ATTN_DEBUG", "1")
    assert binding.library_path() == build.CHECKED_LIB_PATH
    monkeypatch.setenv("FLUX_ATTN_DEBUG", "0")
    assert binding.library_path() == build.LIB_PATH

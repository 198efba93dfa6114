"""Python binding of libflux_attn.so (the C-ABI in include/flux_attn.h).

Argument marshalling only: torch supplies device memory and streams, every
step of the computation runs in the library's kernels. There is no fallback:
a missing library, a CPU tensor or a non-zero status raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

AXES_DIMS = (32, 32, 32, 32)
THETA = 2000.0

STATUS = {
    0: "FLUX_OK", -1: "FLUX_ERR_NULL", -2: "FLUX_ERR_SHAPE", -3: "FLUX_ERR_AXES",
    -4: "FLUX_ERR_ALIGN", -5: "FLUX_ERR_WORKSPACE", -6: "FLUX_ERR_CUDA",
    -7: "FLUX_ERR_DEVICE_TIMEOUT", -8: "FLUX_ERR_UNSUPPORTED", -9: "FLUX_ERR_ALIAS",
}

# every symbol include/flux_attn.h declares
EXPORTS = ("flux_rope_tables", "flux_rope_tables_packed", "flux_joint_rope_attention_workspace",
           "flux_joint_rope_attention_krot_bytes", "flux_joint_rope_attention_workspace_shared",
           "flux_joint_rope_attention", "flux_joint_rope_attention_tabled",
           "flux_joint_rope_attention_heads", "flux_joint_rope_attention_rows",
           "flux_joint_rope_attention_rows_workspace",
           "flux_joint_qknorm_rope_attention", "flux_joint_qknorm_rope_attention_tabled",
           "flux_joint_rope_attention_extract_workspace", "flux_joint_rope_attention_extract",
           "flux_joint_rope_attention_cached_workspace", "flux_joint_rope_attention_cached",
           "flux_joint_qknorm_rope_attention_extract", "flux_joint_qknorm_rope_attention_cached",
           "flux_qkv_mlp_proj", "flux_query_status", "flux_status_string")


class FluxError(RuntimeError):
    def __init__(self, fn: str, status: int, lib=None):
        msg = lib.flux_status_string(status).decode() if lib is not None else ""
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({msg})")
        self.status = status


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    """FLUX_ATTN_LIB if set; else the checked build when FLUX_ATTN_DEBUG=1
    (build it with ``python -m diffusion_transformer_joint_gb300.build
    --checked``); else the release build."""
    if "FLUX_ATTN_LIB" in os.environ:
        return os.environ["FLUX_ATTN_LIB"]
    if os.environ.get("FLUX_ATTN_DEBUG") == "1":
        return _build.CHECKED_LIB_PATH
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load (once) and return the ctypes handle; raises if the library is missing."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or library_path()
            if not os.path.exists(p):
                raise RuntimeError(f"CUDA library not built: {p} (run "
                                   "python -m diffusion_transformer_joint_gb300.build)")
            lib = ctypes.CDLL(p)
            V, I64, I32, SZ, D = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int,
                                  ctypes.c_size_t, ctypes.c_double)
            lib.flux_rope_tables.argtypes = [V, I64, V, I32, D, V, V, V]
            lib.flux_rope_tables.restype = I32
            lib.flux_rope_tables_packed.argtypes = [V, I64, V, I32, D, V, V]
            lib.flux_rope_tables_packed.restype = I32
            lib.flux_joint_rope_attention_workspace.argtypes = [I64, I32]
            lib.flux_joint_rope_attention_workspace.restype = SZ
            lib.flux_joint_rope_attention_krot_bytes.argtypes = [I32, I64, I32, I32]
            lib.flux_joint_rope_attention_krot_bytes.restype = SZ
            lib.flux_joint_rope_attention_workspace_shared.argtypes = [I32, I64, I32, I32]
            lib.flux_joint_rope_attention_workspace_shared.restype = SZ
            lib.flux_joint_rope_attention.argtypes = [V, V, V, V, I64, V, I64, I32, I32, I32,
                                                      V, I32, D, V, V, SZ, V]
            lib.flux_joint_rope_attention.restype = I32
            lib.flux_joint_rope_attention_tabled.argtypes = [V, V, V, V, I32, I64, I32, I32, V,
                                                             V, V, SZ, V]
            lib.flux_joint_rope_attention_heads.argtypes = [V, V, V, V, I64, V, I64, I32, I32,
                                                            I32, I32, I32, V, I32, D, V, V, SZ, V]
            lib.flux_joint_rope_attention_heads.restype = I32
            lib.flux_joint_rope_attention_rows.argtypes = [V, I64, I64, V, V, V, I64, V, I64, I32,
                                                           I32, I32, V, I32, D, V, V, SZ, V]
            lib.flux_joint_rope_attention_rows.restype = I32
            lib.flux_joint_rope_attention_rows_workspace.argtypes = [I32, I64, I64, I32, I32]
            lib.flux_joint_rope_attention_rows_workspace.restype = SZ
            lib.flux_joint_rope_attention_tabled.restype = I32
            F = ctypes.c_float
            lib.flux_joint_qknorm_rope_attention.argtypes = [
                V, V, V, V, I64, V, I64, I32, I32, I32, V, I32, D, V, V, V, V, F, V, V, SZ, V]
            lib.flux_joint_qknorm_rope_attention.restype = I32
            lib.flux_joint_qknorm_rope_attention_tabled.argtypes = [
                V, V, V, V, I32, I64, I32, I32, I64, V, V, V, V, F, V, V, V, SZ, V]
            lib.flux_joint_qknorm_rope_attention_tabled.restype = I32
            lib.flux_joint_rope_attention_extract_workspace.argtypes = [I32, I64, I64, I64, I32, I32]
            lib.flux_joint_rope_attention_extract_workspace.restype = SZ
            lib.flux_joint_rope_attention_extract.argtypes = [
                V, V, V, V, I64, V, I64, V, I64, I32, I32, I32, V, I32, D, V, V, V, V, SZ, V]
            lib.flux_joint_rope_attention_extract.restype = I32
            lib.flux_joint_rope_attention_cached_workspace.argtypes = [I32, I64, I64, I64, I32, I32]
            lib.flux_joint_rope_attention_cached_workspace.restype = SZ
            lib.flux_joint_rope_attention_cached.argtypes = [
                V, V, V, V, I64, V, I64, V, V, I64, I32, I32, I32, V, I32, D, V, V, SZ, V]
            lib.flux_joint_rope_attention_cached.restype = I32
            lib.flux_joint_qknorm_rope_attention_extract.argtypes = [
                V, V, V, V, I64, V, I64, V, I64, I32, I32, I32, V, I32, D, V, V, V, V, F, V, V, V, V,
                SZ, V]
            lib.flux_joint_qknorm_rope_attention_extract.restype = I32
            lib.flux_joint_qknorm_rope_attention_cached.argtypes = [
                V, V, V, V, I64, V, I64, V, V, I64, I32, I32, I32, V, I32, D, V, V, V, V, F, V, V,
                SZ, V]
            lib.flux_joint_qknorm_rope_attention_cached.restype = I32
            lib.flux_qkv_mlp_proj.argtypes = [V, V, I64, I32, I32, I32, I64, V, V, V, V, V, V]
            lib.flux_qkv_mlp_proj.restype = I32
            lib.flux_query_status.argtypes = [V, V]
            lib.flux_query_status.restype = I32
            lib.flux_status_string.argtypes = [I32]
            lib.flux_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def _axes_array(axes_dims):
    arr = (ctypes.c_int32 * len(axes_dims))(*[int(a) for a in axes_dims])
    return arr, len(axes_dims)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None and t.numel() > 0 else None


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _need_cuda(name, t, dtype):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (no CPU path exists)")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _need_shape(name, t, shape):
    """The C ABI takes pointers and sizes only: every tensor's shape is checked
    here, before a kernel could read or write past it."""
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _need_ids(name, ids, n_axes):
    if ids is not None and ids.numel() > 0 and (ids.dim() != 2 or int(ids.shape[1]) != n_axes):
        raise ValueError(f"{name} must be [tokens, {n_axes}], got {tuple(ids.shape)}")


def workspace_bytes(S: int, D: int = 128) -> int:
    """Smallest workspace of joint_rope_attention (status word + RoPE table)."""
    return int(load().flux_joint_rope_attention_workspace(int(S), int(D)))


def krot_bytes(B: int, S: int, H: int, D: int = 128) -> int:
    """Size of the rotated-K exchange buffer (0 for rejected shapes)."""
    return int(load().flux_joint_rope_attention_krot_bytes(int(B), int(S), int(H), int(D)))


def workspace_shared_bytes(B: int, S: int, H: int, D: int = 128) -> int:
    """Workspace size with which joint_rope_attention shares rotated K tiles."""
    return int(load().flux_joint_rope_attention_workspace_shared(int(B), int(S), int(H), int(D)))


def extract_workspace_bytes(B: int, S_txt: int, S_ref: int, S_img: int, H: int,
                            D: int = 128) -> int:
    """Workspace size of one attention_extract call (0: bad shape)."""
    return int(load().flux_joint_rope_attention_extract_workspace(int(B), int(S_txt), int(S_ref),
                                                                 int(S_img), int(H), int(D)))


def cached_workspace_bytes(B: int, S_txt: int, S_img: int, S_ref: int, H: int,
                           D: int = 128) -> int:
    """Workspace size of one attention_cached call (0: bad shape)."""
    return int(load().flux_joint_rope_attention_cached_workspace(int(B), int(S_txt), int(S_img),
                                                                int(S_ref), int(H), int(D)))


def rope_tables(ids, axes_dims=AXES_DIMS, theta=THETA, cos_out=None, sin_out=None, stream=None):
    """fp32 cos, sin [S, sum(axes_dims)/2] for int32 ids [S, n_axes] on the GPU."""
    import torch

    lib = load()
    _need_cuda("ids", ids, torch.int32)
    S, n_axes = ids.shape
    P = sum(int(a) for a in axes_dims) // 2
    if cos_out is None:
        cos_out = torch.empty((S, P), dtype=torch.float32, device=ids.device)
    if sin_out is None:
        sin_out = torch.empty((S, P), dtype=torch.float32, device=ids.device)
    for name, t in (("cos_out", cos_out), ("sin_out", sin_out)):
        _need_cuda(name, t, torch.float32)
        _need_shape(name, t, (S, P))
    axes, n = _axes_array(axes_dims)
    if n != n_axes:
        raise ValueError("ids' last dimension must equal len(axes_dims)")
    rc = lib.flux_rope_tables(_ptr(ids), S, axes, n, float(theta), _ptr(cos_out), _ptr(sin_out),
                              _stream_handle(stream))
    if rc != 0:
        raise FluxError("flux_rope_tables", rc, lib)
    return cos_out, sin_out


def rope_tables_packed(ids, axes_dims=AXES_DIMS, theta=THETA, out=None, stream=None):
    """Packed table [S, sum(axes_dims)/2] (int32 storage of uint32 words: fp16 cos
    in bits 0-15, fp16 sin in bits 16-31) for int32 ids [S, n_axes] on the GPU."""
    import torch

    lib = load()
    _need_cuda("ids", ids, torch.int32)
    S, n_axes = ids.shape
    P = sum(int(a) for a in axes_dims) // 2
    if out is None:
        out = torch.empty((S, P), dtype=torch.int32, device=ids.device)
    _need_cuda("out", out, torch.int32)
    _need_shape("out", out, (S, P))
    axes, n = _axes_array(axes_dims)
    if n != n_axes:
        raise ValueError("ids' last dimension must equal len(axes_dims)")
    rc = lib.flux_rope_tables_packed(_ptr(ids), S, axes, n, float(theta), _ptr(out),
                                     _stream_handle(stream))
    if rc != 0:
        raise FluxError("flux_rope_tables_packed", rc, lib)
    return out


def unpack_table(packed):
    """(cos, sin) fp32 tensors from a packed table (the fp16 halves, widened)."""
    import torch

    w = packed.contiguous()
    halves = w.view(torch.int16).view(torch.float16).reshape(*w.shape, 2)
    return halves[..., 0].float(), halves[..., 1].float()


def _norm_args(qk_norm, device, D=128):
    """(q_txt, k_txt, q_img, k_img, eps) -> four fp32 CUDA [D] tensors and eps
    (the kernels read D weights from each pointer)."""
    import torch

    if len(qk_norm) != 5:
        raise ValueError("qk_norm must be (q_norm_txt, k_norm_txt, q_norm_img, k_norm_img, eps)")
    *ws, eps = qk_norm
    names = ("q_norm_txt", "k_norm_txt", "q_norm_img", "k_norm_img")
    ts = [w if isinstance(w, torch.Tensor) else torch.as_tensor(w, dtype=torch.float32,
                                                                device=device) for w in ws]
    for name, w in zip(names, ts):
        _need_shape(name, w, (D,))
    for name, w in zip(names, ts):
        _need_cuda(name, w, torch.float32)
    return ts, float(eps)


def joint_rope_attention(q, k, v, txt_ids, img_ids, axes_dims=AXES_DIMS, theta=THETA, out=None,
                         workspace=None, stream=None, share_k=True, qk_norm=None):
    """softmax(RoPE(q) RoPE(k)^T / sqrt(D)) v over the joint sequence [txt ; img].

    q, k, v: bf16 CUDA [B, S, H, 128]; txt_ids [S_txt, n_axes], img_ids
    [S_img, n_axes] int32 CUDA (either may be None / empty). Returns ``out``.
    Without ``workspace`` one is allocated: with room for the rotated-K
    exchange buffer when ``share_k``, else the smallest one. ``qk_norm``:
    None, or (q_norm_txt, k_norm_txt, q_norm_img, k_norm_img, eps) with fp32
    [128] weights, for the QK RMS normalisation before RoPE.
    """
    import torch

    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(name, t, torch.bfloat16)
    B, S, H, D = q.shape
    _need_shape("k", k, q.shape)
    _need_shape("v", v, q.shape)
    S_txt = 0 if txt_ids is None else int(txt_ids.shape[0])
    S_img = 0 if img_ids is None else int(img_ids.shape[0])
    for name, t in (("txt_ids", txt_ids), ("img_ids", img_ids)):
        if t is not None and t.numel() > 0:
            _need_cuda(name, t, torch.int32)
            _need_ids(name, t, len(axes_dims))
    if S_txt + S_img != S:
        raise ValueError(f"the ids give {S_txt} + {S_img} tokens, q has {S}")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, torch.bfloat16)
        _need_shape("out", out, q.shape)
    if workspace is not None:
        _need_cuda("workspace", workspace, torch.uint8)
    if workspace is None:
        n = workspace_shared_bytes(B, S, H, D) if share_k else 0
        if n == 0:
            n = workspace_bytes(max(S, 1), D)
        workspace = torch.empty(max(n, 256), dtype=torch.uint8, device=q.device)
    axes, n = _axes_array(axes_dims)
    if qk_norm is None:
        rc = lib.flux_joint_rope_attention(
            _ptr(q), _ptr(k), _ptr(v), _ptr(txt_ids), S_txt, _ptr(img_ids), S_img, B, H, D, axes,
            n, float(theta), _ptr(out), _ptr(workspace), workspace.numel(), _stream_handle(stream))
        name = "flux_joint_rope_attention"
    else:
        ws, eps = _norm_args(qk_norm, q.device, D)
        rc = lib.flux_joint_qknorm_rope_attention(
            _ptr(q), _ptr(k), _ptr(v), _ptr(txt_ids), S_txt, _ptr(img_ids), S_img, B, H, D, axes,
            n, float(theta), *[_ptr(w) for w in ws], eps, _ptr(out), _ptr(workspace),
            workspace.numel(), _stream_handle(stream))
        name = "flux_joint_qknorm_rope_attention"
    if rc != 0:
        raise FluxError(name, rc, lib)
    return out


def _check_ids(txt_ids, img_ids, n_axes):
    import torch

    for name, t in (("txt_ids", txt_ids), ("img_ids", img_ids)):
        if t is not None and t.numel() > 0:
            _need_cuda(name, t, torch.int32)
            _need_ids(name, t, n_axes)
    return (0 if txt_ids is None else int(txt_ids.shape[0]),
            0 if img_ids is None else int(img_ids.shape[0]))


def joint_rope_attention_heads(q, k, v, txt_ids, img_ids, h0, n_heads, axes_dims=AXES_DIMS,
                               theta=THETA, out=None, workspace=None, stream=None, share_k=True):
    """joint_rope_attention over heads h0 .. h0 + n_heads - 1 of the [B, S, H, 128]
    tensors q, k, v (a tensor-parallel rank's heads); only those heads of
    ``out`` are written (it is allocated, and left uninitialised elsewhere,
    when None)."""
    import torch

    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(name, t, torch.bfloat16)
    B, S, H, D = q.shape
    _need_shape("k", k, q.shape)
    _need_shape("v", v, q.shape)
    S_txt, S_img = _check_ids(txt_ids, img_ids, len(axes_dims))
    if S_txt + S_img != S:
        raise ValueError(f"the ids give {S_txt} + {S_img} tokens, q has {S}")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, torch.bfloat16)
        _need_shape("out", out, q.shape)
    if workspace is None:
        n = workspace_shared_bytes(B, S, int(n_heads), D) if share_k else 0
        workspace = torch.empty(max(n or workspace_bytes(S, D), 256), dtype=torch.uint8,
                                device=q.device)
    else:
        _need_cuda("workspace", workspace, torch.uint8)
    axes, n = _axes_array(axes_dims)
    rc = lib.flux_joint_rope_attention_heads(
        _ptr(q), _ptr(k), _ptr(v), _ptr(txt_ids), S_txt, _ptr(img_ids), S_img, B, H, int(h0),
        int(n_heads), D, axes, n, float(theta), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream_handle(stream))
    if rc != 0:
        raise FluxError("flux_joint_rope_attention_heads", rc, lib)
    return out


def rows_workspace_bytes(B: int, S_q: int, S: int, H: int, D: int = 128) -> int:
    """Workspace of joint_rope_attention_rows with the exchange buffer."""
    return int(load().flux_joint_rope_attention_rows_workspace(int(B), int(S_q), int(S), int(H),
                                                               int(D)))


def joint_rope_attention_rows(q, q0, k, v, txt_ids, img_ids, axes_dims=AXES_DIMS, theta=THETA,
                              out=None, workspace=None, stream=None, share_k=True):
    """The attention of query tokens q0 .. q0 + S_q - 1 (q: bf16 [B, S_q, H, 128])
    over every token's key and value (k, v: [B, S, H, 128]); txt_ids / img_ids
    are the ids of the whole sequence. Returns out [B, S_q, H, 128]."""
    import torch

    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(name, t, torch.bfloat16)
    B, S_q, H, D = q.shape
    S = k.shape[1]
    _need_shape("k", k, (B, S, H, D))
    _need_shape("v", v, (B, S, H, D))
    S_txt, S_img = _check_ids(txt_ids, img_ids, len(axes_dims))
    if S_txt + S_img != S:
        raise ValueError(f"the ids give {S_txt} + {S_img} tokens, k has {S}")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, torch.bfloat16)
        _need_shape("out", out, q.shape)
    if workspace is None:
        n = rows_workspace_bytes(B, S_q, S, H, D) if share_k else 0
        workspace = torch.empty(max(n or workspace_bytes(S, D), 256), dtype=torch.uint8,
                                device=q.device)
    else:
        _need_cuda("workspace", workspace, torch.uint8)
    axes, n = _axes_array(axes_dims)
    rc = lib.flux_joint_rope_attention_rows(
        _ptr(q), int(q0), S_q, _ptr(k), _ptr(v), _ptr(txt_ids), S_txt, _ptr(img_ids), S_img, B,
        H, D, axes, n, float(theta), _ptr(out), _ptr(workspace), workspace.numel(),
        _stream_handle(stream))
    if rc != 0:
        raise FluxError("flux_joint_rope_attention_rows", rc, lib)
    return out


def joint_rope_attention_tabled(q, k, v, table, status, out=None, stream=None, krot=None,
                                qk_norm=None, s_txt=0):
    """Attention with a caller-built packed table (see rope_tables_packed); ``status``
    is a device int32 tensor of one element that the caller clears. ``krot``: a
    uint8 CUDA tensor of at least krot_bytes(B, S, H) bytes serving as the
    rotated-K exchange buffer; None allocates one, False runs without.
    ``qk_norm`` as for joint_rope_attention, with ``s_txt`` leading text tokens."""
    import torch

    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(name, t, torch.bfloat16)
    _need_cuda("table", table, torch.int32)
    _need_cuda("status", status, torch.int32)
    B, S, H, D = q.shape
    _need_shape("k", k, q.shape)
    _need_shape("v", v, q.shape)
    _need_shape("table", table, (S, D // 2))
    if status.numel() < 1:
        raise ValueError("status must hold one int32")
    if out is None:
        out = torch.empty_like(q)
    else:
        _need_cuda("out", out, torch.bfloat16)
        _need_shape("out", out, q.shape)
    if krot is None:
        krot = torch.empty(max(krot_bytes(B, S, H, D), 256), dtype=torch.uint8, device=q.device)
    if krot is False:
        kp, kn = None, 0
    else:
        _need_cuda("krot", krot, torch.uint8)
        kp, kn = _ptr(krot), krot.numel()
    if qk_norm is None:
        rc = lib.flux_joint_rope_attention_tabled(_ptr(q), _ptr(k), _ptr(v), _ptr(table), B, S, H,
                                                  D, _ptr(out), _ptr(status), kp, kn,
                                                  _stream_handle(stream))
        name = "flux_joint_rope_attention_tabled"
    else:
        ws, eps = _norm_args(qk_norm, q.device, D)
        rc = lib.flux_joint_qknorm_rope_attention_tabled(
            _ptr(q), _ptr(k), _ptr(v), _ptr(table), B, S, H, D, int(s_txt),
            *[_ptr(w) for w in ws], eps, _ptr(out), _ptr(status), kp, kn, _stream_handle(stream))
        name = "flux_joint_qknorm_rope_attention_tabled"
    if rc != 0:
        raise FluxError(name, rc, lib)
    return out


def _rows(ids):
    return 0 if ids is None else int(ids.shape[0])


def attention_extract(q, k, v, txt_ids, ref_ids, img_ids, axes_dims=AXES_DIMS, theta=THETA,
                      out=None, cache_k=None, cache_v=None, workspace=None, stream=None,
                      qk_norm=None):
    """Extract mode over tokens [txt ; ref ; img]: returns (out, cache_k, cache_v).
    ``qk_norm`` as for joint_rope_attention (reference tokens take the image
    weights; the cache then holds the normalised, rotated K)."""
    import torch

    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(name, t, torch.bfloat16)
    B, S, H, D = q.shape
    _need_shape("k", k, q.shape)
    _need_shape("v", v, q.shape)
    s_t, s_r, s_i = _rows(txt_ids), _rows(ref_ids), _rows(img_ids)
    for name, t in (("txt_ids", txt_ids), ("ref_ids", ref_ids), ("img_ids", img_ids)):
        if t is not None and t.numel() > 0:
            _need_cuda(name, t, torch.int32)
            _need_ids(name, t, len(axes_dims))
    if s_t + s_r + s_i != S:
        raise ValueError(f"the ids give {s_t} + {s_r} + {s_i} tokens, q has {S}")
    out = torch.empty_like(q) if out is None else out
    if cache_k is None:
        cache_k = torch.empty((B, s_r, H, D), dtype=torch.bfloat16, device=q.device)
    if cache_v is None:
        cache_v = torch.empty((B, s_r, H, D), dtype=torch.bfloat16, device=q.device)
    for name, t, shape in (("out", out, q.shape), ("cache_k", cache_k, (B, s_r, H, D)),
                           ("cache_v", cache_v, (B, s_r, H, D))):
        _need_cuda(name, t, torch.bfloat16)
        _need_shape(name, t, shape)
    if workspace is not None:
        _need_cuda("workspace", workspace, torch.uint8)
    if workspace is None:
        n = extract_workspace_bytes(B, s_t, s_r, s_i, H, D)
        workspace = torch.empty(max(int(n), 256), dtype=torch.uint8, device=q.device)
    axes, na = _axes_array(axes_dims)
    if qk_norm is None:
        name = "flux_joint_rope_attention_extract"
        rc = lib.flux_joint_rope_attention_extract(
            _ptr(q), _ptr(k), _ptr(v), _ptr(txt_ids), s_t, _ptr(ref_ids), s_r, _ptr(img_ids), s_i,
            B, H, D, axes, na, float(theta), _ptr(out), _ptr(cache_k), _ptr(cache_v),
            _ptr(workspace), workspace.numel(), _stream_handle(stream))
    else:
        name = "flux_joint_qknorm_rope_attention_extract"
        ws, eps = _norm_args(qk_norm, q.device, D)
        rc = lib.flux_joint_qknorm_rope_attention_extract(
            _ptr(q), _ptr(k), _ptr(v), _ptr(txt_ids), s_t, _ptr(ref_ids), s_r, _ptr(img_ids), s_i,
            B, H, D, axes, na, float(theta), *[_ptr(w) for w in ws], eps, _ptr(out),
            _ptr(cache_k), _ptr(cache_v), _ptr(workspace), workspace.numel(),
            _stream_handle(stream))
    if rc != 0:
        raise FluxError(name, rc, lib)
    return out, cache_k, cache_v


def attention_cached(q, k, v, txt_ids, img_ids, cache_k, cache_v, axes_dims=AXES_DIMS,
                     theta=THETA, out=None, workspace=None, stream=None, qk_norm=None):
    """Cached mode: queries [txt ; img] over keys [txt ; cache ; img]; returns out.
    ``qk_norm`` normalises q and the keys of k (the cache is used as stored)."""
    import torch

    lib = load()
    for name, t in (("q", q), ("k", k), ("v", v), ("cache_k", cache_k), ("cache_v", cache_v)):
        _need_cuda(name, t, torch.bfloat16)
    B, S, H, D = q.shape
    _need_shape("k", k, q.shape)
    _need_shape("v", v, q.shape)
    s_t, s_i, s_r = _rows(txt_ids), _rows(img_ids), int(cache_k.shape[1])
    _need_shape("cache_k", cache_k, (B, s_r, H, D))
    _need_shape("cache_v", cache_v, (B, s_r, H, D))
    for name, t in (("txt_ids", txt_ids), ("img_ids", img_ids)):
        if t is not None and t.numel() > 0:
            _need_cuda(name, t, torch.int32)
            _need_ids(name, t, len(axes_dims))
    if s_t + s_i != S:
        raise ValueError(f"the ids give {s_t} + {s_i} tokens, q has {S}")
    out = torch.empty_like(q) if out is None else out
    _need_cuda("out", out, torch.bfloat16)
    _need_shape("out", out, q.shape)
    if workspace is not None:
        _need_cuda("workspace", workspace, torch.uint8)
    if workspace is None:
        n = cached_workspace_bytes(B, s_t, s_i, s_r, H, D)
        workspace = torch.empty(max(int(n), 256), dtype=torch.uint8, device=q.device)
    axes, na = _axes_array(axes_dims)
    if qk_norm is None:
        name = "flux_joint_rope_attention_cached"
        rc = lib.flux_joint_rope_attention_cached(
            _ptr(q), _ptr(k), _ptr(v), _ptr(txt_ids), s_t, _ptr(img_ids), s_i, _ptr(cache_k),
            _ptr(cache_v), s_r, B, H, D, axes, na, float(theta), _ptr(out), _ptr(workspace),
            workspace.numel(), _stream_handle(stream))
    else:
        name = "flux_joint_qknorm_rope_attention_cached"
        ws, eps = _norm_args(qk_norm, q.device, D)
        rc = lib.flux_joint_qknorm_rope_attention_cached(
            _ptr(q), _ptr(k), _ptr(v), _ptr(txt_ids), s_t, _ptr(img_ids), s_i, _ptr(cache_k),
            _ptr(cache_v), s_r, B, H, D, axes, na, float(theta), *[_ptr(w) for w in ws], eps,
            _ptr(out), _ptr(workspace), workspace.numel(), _stream_handle(stream))
    if rc != 0:
        raise FluxError(name, rc, lib)
    return out


def qkv_mlp_proj(x, w, H, mlp=None, q=None, k=None, v=None, act=None, status=None,
                 stream=None):
    """Fused single-stream input projection: x [..., dim] and w [3 H 128 + 2 mlp, dim]
    bf16 -> (q, k, v [..., H, 128], act [..., mlp]); status (int32 [1], cleared
    here when allocated) receives a device timeout."""
    import torch

    lib = load()
    _need_cuda("x", x, torch.bfloat16)
    _need_cuda("w", w, torch.bfloat16)
    lead, dim = tuple(x.shape[:-1]), int(x.shape[-1])
    M = 1
    for n in lead:
        M *= int(n)
    inner = H * 128
    if mlp is None:
        mlp = (int(w.shape[0]) - 3 * inner) // 2
    if mlp < 0:
        raise ValueError(f"w has {int(w.shape[0])} rows, fewer than the {3 * inner} of q, k, v")
    if tuple(w.shape) != (3 * inner + 2 * mlp, dim):
        raise ValueError(f"w must be [{3 * inner + 2 * mlp}, {dim}], got {tuple(w.shape)}")
    dev = x.device
    q = torch.empty(lead + (H, 128), dtype=torch.bfloat16, device=dev) if q is None else q
    k = torch.empty(lead + (H, 128), dtype=torch.bfloat16, device=dev) if k is None else k
    v = torch.empty(lead + (H, 128), dtype=torch.bfloat16, device=dev) if v is None else v
    if act is None:
        act = torch.empty(lead + (mlp,), dtype=torch.bfloat16, device=dev)
    if status is None:
        status = torch.zeros(1, dtype=torch.int32, device=dev)
    for name, t in (("q", q), ("k", k), ("v", v), ("act", act)):
        _need_cuda(name, t, torch.bfloat16)
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_shape(name, t, lead + (H, 128))
    _need_shape("act", act, lead + (mlp,))
    _need_cuda("status", status, torch.int32)
    rc = lib.flux_qkv_mlp_proj(_ptr(x), _ptr(w), M, dim, int(H), 128, int(mlp), _ptr(q), _ptr(k),
                               _ptr(v), _ptr(act) if mlp > 0 else None, _ptr(status),
                               _stream_handle(stream))
    if rc != 0:
        raise FluxError("flux_qkv_mlp_proj", rc, lib)
    return q, k, v, act


def query_status(workspace, stream=None) -> int:
    """Synchronise and return the device status word of a call's workspace."""
    lib = load()
    return int(lib.flux_query_status(_ptr(workspace), _stream_handle(stream)))

"""Oracle: plain fp64 CPU restatement of the FLUX.2 joint RoPE attention.

TEST INFRASTRUCTURE ONLY. The test-suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` are the only
callers. The product path never imports this package, and this package
imports nothing from the product package.

The arithmetic lives in ``flux_oracle.c`` (compiled with gcc, no fast-math);
this file only builds it and marshals numpy arrays. The one step done here is
the concatenation of the text and image position ids into the joint sequence
[txt ; img] ("Diffusers 中 Flux2Transformer2DModel 全面解析", section
"前向传播输入输出约定": both id sets are 4-d (T, H, W, L) and the text and
image streams are attended jointly; "FLUX.2 [klein]" survey page, section
"模型架构": reference-image tokens are concatenated with the noisy tokens).

Pins (tests/test_oracle_pins.py): zero ids give the identity, rotations keep
norms, the post-RoPE dot product depends only on the id difference, the
per-axis frequencies match theta^(-2j/d_a) evaluated independently at high
precision, a complex-number brute force agrees, identical keys give the mean
of V, and the attention agrees with torch's float64 SDPA and with a naive
Python triple loop on tiny inputs. The optional QK RMS normalisation agrees
with torch's float64 rms_norm and with its closed-form mean square, and the
normalised attention with SDPA on inputs normalised and rotated separately.
The reference KV modes agree with SDPA under an explicit boolean mask
(extract) and over explicitly concatenated keys (cached), and a cache written
in extract mode reproduces extract's text and image rows in cached mode; with
the QK norm they equal the plain modes on inputs normalised by torch.
The fused single-stream projection places selected input channels exactly
where the split puts them (Q, K, V heads, gate and linear halves), agrees with
torch's float64 matmul and silu, and meets SiLU's closed forms.
No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "flux_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_default = None

GCC_FLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-fno-fast-math",
             "-ffp-contract=off"]


def compile_source(src: str, out: str) -> str:
    """gcc-compile an oracle C source into a shared library at ``out``."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *GCC_FLAGS, src, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile flux_oracle.c into oracle/_build/liboracle.so (gcc -O2, IEEE fp64)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stale = (not os.path.exists(_LIB_PATH)
             or os.path.getmtime(_LIB_PATH) < os.path.getmtime(SOURCE))
    if force or stale:
        compile_source(SOURCE, _LIB_PATH)
    return _LIB_PATH


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def joint_ids(txt_ids, img_ids) -> np.ndarray:
    """Position ids of the joint sequence: text tokens first, then image tokens."""
    parts = [np.asarray(x, dtype=np.int32).reshape(-1, np.asarray(x).shape[-1])
             for x in (txt_ids, img_ids) if x is not None and np.asarray(x).size > 0]
    return np.ascontiguousarray(np.concatenate(parts, axis=0), dtype=np.int32)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class Oracle:
    """The oracle's entry points bound to one compiled library."""

    def __init__(self, lib_path: str):
        lib = ctypes.CDLL(lib_path)
        P = ctypes.c_void_p
        lib.oracle_rope_tables.argtypes = [P, ctypes.c_int64, P, ctypes.c_int,
                                           ctypes.c_double, P, P]
        lib.oracle_rope_tables.restype = ctypes.c_int
        lib.oracle_rope_apply.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                          ctypes.c_int, P, P, P]
        lib.oracle_rope_apply.restype = None
        lib.oracle_joint_rope_attention.argtypes = [
            P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
            P, P, ctypes.c_int, ctypes.c_double, P, ctypes.c_int64, ctypes.c_int, P]
        lib.oracle_joint_rope_attention.restype = ctypes.c_int
        lib.oracle_rms_norm.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                        ctypes.c_int, P, ctypes.c_double, P]
        lib.oracle_rms_norm.restype = None
        lib.oracle_joint_qknorm_rope_attention.argtypes = [
            P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int,
            P, P, ctypes.c_int, ctypes.c_double, P, P, P, P, ctypes.c_int64, ctypes.c_double,
            P, ctypes.c_int64, ctypes.c_int, P]
        lib.oracle_joint_qknorm_rope_attention.restype = ctypes.c_int
        lib.oracle_attention_extract.argtypes = [
            P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
            ctypes.c_double, ctypes.c_int64, ctypes.c_int64, P, ctypes.c_int64, P, P, P]
        lib.oracle_attention_extract.restype = ctypes.c_int
        lib.oracle_attention_cached.argtypes = [
            P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
            ctypes.c_double, ctypes.c_int64, P, P, ctypes.c_int64, P, ctypes.c_int64, P]
        lib.oracle_attention_cached.restype = ctypes.c_int
        lib.oracle_qknorm_attention_extract.argtypes = [
            P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
            ctypes.c_double, ctypes.c_int64, ctypes.c_int64, P, P, P, P, ctypes.c_double, P,
            ctypes.c_int64, P, P, P]
        lib.oracle_qknorm_attention_extract.restype = ctypes.c_int
        lib.oracle_qknorm_attention_cached.argtypes = [
            P, P, P, ctypes.c_int, ctypes.c_int64, ctypes.c_int, ctypes.c_int, P, P, ctypes.c_int,
            ctypes.c_double, ctypes.c_int64, P, P, ctypes.c_int64, P, P, P, P, ctypes.c_double, P,
            ctypes.c_int64, P]
        lib.oracle_qknorm_attention_cached.restype = ctypes.c_int
        lib.oracle_qkv_mlp_proj.argtypes = [
            P, P, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int64, P,
            ctypes.c_int64, P, P, P, P]
        lib.oracle_qkv_mlp_proj.restype = ctypes.c_int
        self.lib = lib
        self.path = lib_path

    def rope_tables(self, ids, axes_dims=(32, 32, 32, 32), theta=2000.0):
        """cos, sin tables [S, sum(axes_dims)/2] in fp64 for ids [S, n_axes]."""
        ids = np.ascontiguousarray(ids, dtype=np.int32)
        axes = np.ascontiguousarray(axes_dims, dtype=np.int32)
        S, n_axes = ids.shape
        assert n_axes == axes.size
        P = int(axes.sum()) // 2
        c = np.empty((S, P), dtype=np.float64)
        s = np.empty((S, P), dtype=np.float64)
        rc = self.lib.oracle_rope_tables(_ptr(ids), S, _ptr(axes), n_axes, float(theta),
                                         _ptr(c), _ptr(s))
        if rc != 0:
            raise ValueError("oracle_rope_tables: every axis width must be positive and even")
        return c, s

    def rope_apply(self, x, cos_t, sin_t):
        """Rotate x [B, S, H, D] (fp64) with tables [S, D/2]."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        B, S, H, D = x.shape
        cos_t = np.ascontiguousarray(cos_t, dtype=np.float64)
        sin_t = np.ascontiguousarray(sin_t, dtype=np.float64)
        assert cos_t.shape == (S, D // 2) and sin_t.shape == (S, D // 2)
        y = np.empty_like(x)
        self.lib.oracle_rope_apply(_ptr(x), B, S, H, D, _ptr(cos_t), _ptr(sin_t), _ptr(y))
        return y

    def rms_norm(self, x, w, eps=1e-6):
        """RMS-normalise every head vector of x [B, S, H, D] with weights w [D] (fp64)."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        B, S, H, D = x.shape
        w = np.ascontiguousarray(w, dtype=np.float64)
        assert w.shape == (D,)
        y = np.empty_like(x)
        self.lib.oracle_rms_norm(_ptr(x), B, S, H, D, _ptr(w), float(eps), _ptr(y))
        return y

    def joint_rope_attention(self, q, k, v, txt_ids, img_ids, axes_dims=(32, 32, 32, 32),
                             theta=2000.0, rows=None, threads=None, qk_norm=None):
        """out[b, r, h, :] for the query tokens ``rows`` (all when None).

        q, k, v: [B, S, H, D] arrays (any float dtype; converted exactly to fp64).
        qk_norm: None, or (qw_txt, kw_txt, qw_img, kw_img, eps) with weights [D]:
        Q and K are RMS-normalised (text tokens with the text weights) before
        the rotation. Returns fp64 [B, len(rows), H, D].
        """
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        B, S, H, D = q.shape
        assert k.shape == q.shape and v.shape == q.shape
        ids = joint_ids(txt_ids, img_ids)
        assert ids.shape[0] == S, (ids.shape, S)
        axes = np.ascontiguousarray(axes_dims, dtype=np.int32)
        if rows is None:
            rows_arr = np.arange(S, dtype=np.int64)
        else:
            rows_arr = np.ascontiguousarray(rows, dtype=np.int64)
            assert rows_arr.size == 0 or (rows_arr.min() >= 0 and rows_arr.max() < S)
        out = np.zeros((B, rows_arr.size, H, D), dtype=np.float64)
        if rows_arr.size == 0:
            return out
        n_threads = int(threads) if threads else default_threads()
        if qk_norm is None:
            rc = self.lib.oracle_joint_rope_attention(
                _ptr(q), _ptr(k), _ptr(v), B, S, H, D, _ptr(ids), _ptr(axes), axes.size,
                float(theta), _ptr(rows_arr), rows_arr.size, n_threads, _ptr(out))
        else:
            *ws, eps = qk_norm
            ws = [np.ascontiguousarray(w, dtype=np.float64) for w in ws]
            assert all(w.shape == (D,) for w in ws)
            s_txt = 0 if txt_ids is None else int(np.asarray(txt_ids).reshape(-1, axes.size).shape[0])
            rc = self.lib.oracle_joint_qknorm_rope_attention(
                _ptr(q), _ptr(k), _ptr(v), B, S, H, D, _ptr(ids), _ptr(axes), axes.size,
                float(theta), *[_ptr(w) for w in ws], s_txt, float(eps), _ptr(rows_arr),
                rows_arr.size, n_threads, _ptr(out))
        if rc != 0:
            raise ValueError("oracle_joint_rope_attention: sum(axes_dims) must equal D, "
                             "sizes > 0")
        return out


    def attention_extract(self, q, k, v, txt_ids, ref_ids, img_ids, axes_dims=(32, 32, 32, 32),
                          theta=2000.0, rows=None, qk_norm=None):
        """Extract mode over tokens [txt ; ref ; img]: (out [B, len(rows) or S, H, D],
        cache_k, cache_v [B, S_ref, H, D]) in fp64."""
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        B, S, H, D = q.shape
        axes = np.ascontiguousarray(axes_dims, dtype=np.int32)
        n_t = 0 if txt_ids is None else np.asarray(txt_ids).reshape(-1, axes.size).shape[0]
        n_r = 0 if ref_ids is None else np.asarray(ref_ids).reshape(-1, axes.size).shape[0]
        ids = joint_ids(joint_ids(txt_ids, ref_ids) if n_t + n_r else None, img_ids)
        assert ids.shape[0] == S
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n_out = S if rows_arr is None else rows_arr.size
        out = np.empty((B, n_out, H, D))
        ck = np.empty((B, n_r, H, D))
        cv = np.empty((B, n_r, H, D))
        if qk_norm is None:
            rc = self.lib.oracle_attention_extract(
                _ptr(q), _ptr(k), _ptr(v), B, S, H, D, _ptr(ids), _ptr(axes), axes.size,
                float(theta), n_t, n_r, None if rows_arr is None else _ptr(rows_arr), n_out,
                _ptr(out), _ptr(ck), _ptr(cv))
        else:
            ws = [np.ascontiguousarray(w, dtype=np.float64) for w in qk_norm[:4]]
            rc = self.lib.oracle_qknorm_attention_extract(
                _ptr(q), _ptr(k), _ptr(v), B, S, H, D, _ptr(ids), _ptr(axes), axes.size,
                float(theta), n_t, n_r, *[_ptr(w) for w in ws], float(qk_norm[4]),
                None if rows_arr is None else _ptr(rows_arr), n_out, _ptr(out), _ptr(ck), _ptr(cv))
        if rc != 0:
            raise ValueError("oracle_attention_extract: bad arguments")
        return out, ck, cv

    def attention_cached(self, q, k, v, txt_ids, img_ids, cache_k, cache_v,
                         axes_dims=(32, 32, 32, 32), theta=2000.0, rows=None, qk_norm=None):
        """Cached mode: queries [txt ; img] over keys [txt ; cache ; img]; fp64 out."""
        q = np.ascontiguousarray(q, dtype=np.float64)
        k = np.ascontiguousarray(k, dtype=np.float64)
        v = np.ascontiguousarray(v, dtype=np.float64)
        ck = np.ascontiguousarray(cache_k, dtype=np.float64)
        cv = np.ascontiguousarray(cache_v, dtype=np.float64)
        B, S, H, D = q.shape
        axes = np.ascontiguousarray(axes_dims, dtype=np.int32)
        n_t = 0 if txt_ids is None else np.asarray(txt_ids).reshape(-1, axes.size).shape[0]
        ids = joint_ids(txt_ids, img_ids)
        assert ids.shape[0] == S and ck.shape == cv.shape and ck.shape[0] == B
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n_out = S if rows_arr is None else rows_arr.size
        out = np.empty((B, n_out, H, D))
        if qk_norm is None:
            rc = self.lib.oracle_attention_cached(
                _ptr(q), _ptr(k), _ptr(v), B, S, H, D, _ptr(ids), _ptr(axes), axes.size,
                float(theta), n_t, _ptr(ck), _ptr(cv), ck.shape[1],
                None if rows_arr is None else _ptr(rows_arr), n_out, _ptr(out))
        else:
            ws = [np.ascontiguousarray(w, dtype=np.float64) for w in qk_norm[:4]]
            rc = self.lib.oracle_qknorm_attention_cached(
                _ptr(q), _ptr(k), _ptr(v), B, S, H, D, _ptr(ids), _ptr(axes), axes.size,
                float(theta), n_t, _ptr(ck), _ptr(cv), ck.shape[1], *[_ptr(w) for w in ws],
                float(qk_norm[4]), None if rows_arr is None else _ptr(rows_arr), n_out, _ptr(out))
        if rc != 0:
            raise ValueError("oracle_attention_cached: bad arguments")
        return out


    def qkv_mlp_proj(self, x, w, H, D=128, mlp=None, rows=None):
        """The single-stream fused projection for x [M, dim] and w [3HD + 2 mlp, dim]:
        (q, k, v [n, H, D], act [n, mlp]) in fp64 for the rows (all M if None)."""
        x = np.ascontiguousarray(x, dtype=np.float64)
        w = np.ascontiguousarray(w, dtype=np.float64)
        M, dim = x.shape
        inner = H * D
        if mlp is None:
            mlp = (w.shape[0] - 3 * inner) // 2
        assert w.shape == (3 * inner + 2 * mlp, dim)
        rows_arr = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
        n = M if rows_arr is None else rows_arr.size
        q = np.empty((n, H, D))
        k = np.empty((n, H, D))
        v = np.empty((n, H, D))
        act = np.empty((n, mlp))
        rc = self.lib.oracle_qkv_mlp_proj(_ptr(x), _ptr(w), M, dim, H, D, mlp,
                                          None if rows_arr is None else _ptr(rows_arr), n,
                                          _ptr(q), _ptr(k), _ptr(v), _ptr(act))
        if rc != 0:
            raise ValueError("oracle_qkv_mlp_proj: bad arguments")
        return q, k, v, act


def default() -> Oracle:
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def rope_tables(ids, axes_dims=(32, 32, 32, 32), theta=2000.0):
    return default().rope_tables(ids, axes_dims, theta)


def rope_apply(x, cos_t, sin_t):
    return default().rope_apply(x, cos_t, sin_t)


def rms_norm(x, w, eps=1e-6):
    return default().rms_norm(x, w, eps)


def attention_extract(q, k, v, txt_ids, ref_ids, img_ids, axes_dims=(32, 32, 32, 32),
                      theta=2000.0, rows=None, qk_norm=None):
    return default().attention_extract(q, k, v, txt_ids, ref_ids, img_ids, axes_dims, theta, rows,
                                       qk_norm)


def attention_cached(q, k, v, txt_ids, img_ids, cache_k, cache_v, axes_dims=(32, 32, 32, 32),
                     theta=2000.0, rows=None, qk_norm=None):
    return default().attention_cached(q, k, v, txt_ids, img_ids, cache_k, cache_v, axes_dims,
                                      theta, rows, qk_norm)


def qkv_mlp_proj(x, w, H, D=128, mlp=None, rows=None):
    return default().qkv_mlp_proj(x, w, H, D, mlp, rows)


def joint_rope_attention(q, k, v, txt_ids, img_ids, axes_dims=(32, 32, 32, 32),
                         theta=2000.0, rows=None, threads=None, qk_norm=None):
    return default().joint_rope_attention(q, k, v, txt_ids, img_ids, axes_dims, theta,
                                          rows, threads, qk_norm)

"""Double-precision CPU oracle for head-major attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It shares no code with the CUDA path.

It restates, in plain f64 C (``vattn_oracle.c``), what the WGSL shader
"vision_attention_flash_sub_hpd_f16.wgsl" (rullama 0.1.0) computes:
``out[b, h, i, :] = softmax_j(q[b,h,i,:] . k[b,h,j,:]) @ v[b,h,:,:]`` with no
1/sqrt(head_dim) factor (q arrives pre-scaled), head-major layout
``[batch, n_heads, n_patches, head_dim]``.

``oracle.rope`` (plain NumPy, f64) restates the NeoX rotary embedding of the
WGSL kernel "rope_neox_backward.wgsl" (rullama 0.2.0), forward and inverse.

``oracle.conv1d`` (plain NumPy, f64) restates the depthwise conv1d
rolling-buffer step of the WGSL kernel "conv1d.wgsl" (cera 0.2.0).
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIB = None


def _lib():
    global _LIB
    if _LIB is None:
        path = _build.build()
        lib = ctypes.CDLL(path)
        f32p = ctypes.POINTER(ctypes.c_float)
        f64p = ctypes.POINTER(ctypes.c_double)
        i64 = ctypes.c_int64
        lib.vattn_oracle_forward.argtypes = [f32p, f32p, f32p, f64p, i64, i64,
                                             i64, i64, ctypes.c_int]
        lib.vattn_oracle_forward.restype = ctypes.c_int
        lib.vattn_oracle_rows.argtypes = [f32p, f32p, f32p, i64, i64, i64,
                                          ctypes.POINTER(ctypes.c_int64), i64,
                                          f64p, ctypes.c_int]
        lib.vattn_oracle_rows.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover - non-Linux
        return max(1, os.cpu_count() or 1)


def _as_f32(a: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"oracle inputs must be float32, got {a.dtype}")
    return a


def _ptr(a: np.ndarray, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def forward(q: np.ndarray, k: np.ndarray, v: np.ndarray,
            threads: int | None = None) -> np.ndarray:
    """Full oracle: q, k, v f32 ``[B, H, N, D]`` -> out f64 ``[B, H, N, D]``."""
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError(f"expected equal [B,H,N,D] shapes, got {q.shape}, "
                         f"{k.shape}, {v.shape}")
    B, H, N, D = q.shape
    out = np.zeros(q.shape, dtype=np.float64)
    rc = _lib().vattn_oracle_forward(_ptr(q, ctypes.c_float),
                                     _ptr(k, ctypes.c_float),
                                     _ptr(v, ctypes.c_float),
                                     _ptr(out, ctypes.c_double), B, H, N, D,
                                     threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"vattn_oracle_forward failed with code {rc}")
    return out


def rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, flat_rows,
         threads: int | None = None) -> np.ndarray:
    """Selected query rows.

    ``flat_rows`` holds indices ``(b*H + h)*N + i``; returns f64
    ``[len(flat_rows), D]`` with row r equal to ``out[b, h, i, :]``.
    """
    q, k, v = _as_f32(q), _as_f32(k), _as_f32(v)
    B, H, N, D = q.shape
    idx = np.ascontiguousarray(np.asarray(flat_rows, dtype=np.int64))
    out = np.zeros((idx.size, D), dtype=np.float64)
    rc = _lib().vattn_oracle_rows(_ptr(q, ctypes.c_float),
                                  _ptr(k, ctypes.c_float),
                                  _ptr(v, ctypes.c_float), B * H, N, D,
                                  _ptr(idx, ctypes.c_int64), idx.size,
                                  _ptr(out, ctypes.c_double),
                                  threads or default_threads())
    if rc != 0:
        raise RuntimeError(f"vattn_oracle_rows failed with code {rc}")
    return out

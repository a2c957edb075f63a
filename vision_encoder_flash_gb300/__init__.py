"""vision_encoder_flash_gb300 -- head-major vision attention on GB300 (sm_103a).

``forward(q, k, v)`` computes ``softmax(q @ k^T) @ v`` per (batch, head) for
f32 tensors of shape ``[batch, n_heads, n_patches, head_dim]`` (q already
scaled by the caller), through the C ABI of ``libvattn.so`` (include/vattn.h).
This module only marshals arguments: every step of the computation runs in
the library's CUDA kernel.  There is no CPU fallback; if the library is
missing or no GPU is present the calls raise.
"""
from __future__ import annotations

from ._lib import (VattnError, _check, conv1d_step_status, device_status, exported_symbols,
                   forward_accurate_status, forward_host_status,
                   forward_f16_raw, forward_f16io_status, forward_f32q_raw,
                   forward_noalloc_raw, forward_raw, forward_rope_status, lib_path,
                   load_library, rope_neox_status, status_string, version)

__all__ = ["forward", "forward_accurate", "conv1d_step", "forward_f16", "forward_f16io",
           "forward_f32q", "forward_rope", "rope_neox", "forward_raw",
           "forward_f16_raw", "forward_f32q_raw", "forward_noalloc_raw",
           "device_status", "VattnError", "load_library",
           "lib_path", "exported_symbols", "status_string", "version"]


def forward(q, k, v, out=None, stream=None):
    """out = softmax(q k^T) v for torch f32 tensors ``[B, H, N, D]``.

    CUDA tensors: runs on their device and on ``stream`` (default: the
    current torch stream); returns ``out`` without synchronising.

    CPU tensors: one call of the host-buffer entry point (vattn_forward_host)
    on the current CUDA device: chunks of heads are copied in, computed and
    copied back into ``out`` (or a new pinned tensor) on overlapping
    streams; the call synchronises ``stream`` before returning.  Pinned
    (page-locked) inputs let the copies overlap the kernels.
    """
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != torch.float32:
            raise TypeError(f"{name} must be float32, got {t.dtype}")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [batch, n_heads, n_patches, head_dim]")
    if not (q.shape == k.shape == v.shape):
        raise ValueError(f"shape mismatch: q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)}")
    if not (q.device == k.device == v.device):
        raise ValueError("q, k and v must be on the same device")

    if q.device.type == "cpu":
        for name, t in (("q", q), ("k", k), ("v", v)):
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous (head-major [B, H, N, D])")
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, pin_memory=True)
        if (out.device.type != "cpu" or out.dtype != torch.float32 or out.shape != q.shape
                or not out.is_contiguous()):
            raise ValueError("out must be a contiguous float32 CPU tensor of q's shape")
        dev = torch.device("cuda", torch.cuda.current_device())
        s = stream if stream is not None else torch.cuda.current_stream(dev)
        B, H, N, D = q.shape
        _check(forward_host_status(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H,
                                   N, D, s.cuda_stream))
        s.synchronize()
        return out

    if q.device.type != "cuda":
        raise ValueError(f"unsupported device {q.device}")
    if out is None:
        out = torch.empty_like(q, memory_format=torch.contiguous_format)
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    _launch(q, k, v, out, s)
    return out


def forward_f16(q, k, v, out=None, stream=None):
    """out (f32) = softmax(q k^T) v for CUDA float16 tensors ``[B, H, N, D]``,
    ``D`` a multiple of 8; the attention kernel reads the f16 tensors directly
    (no conversion pass).  Runs on ``stream`` (default: the current torch
    stream) and returns ``out`` without synchronising."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != torch.float16:
            raise TypeError(f"{name} must be float16, got {t.dtype}")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [batch, n_heads, n_patches, head_dim]")
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (head-major [B, H, N, D])")
    if not (q.shape == k.shape == v.shape) or not (q.device == k.device == v.device):
        raise ValueError("q, k and v must have one shape and one device")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.float32 or out.device != q.device \
            or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of q's shape and device")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    B, H, N, D = q.shape
    forward_f16_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N, D,
                    s.cuda_stream)
    return out


def forward_f32q(q, k, v, out=None, stream=None):
    """out (f32) = softmax(q k^T) v for a CUDA float32 ``q`` and float16 ``k``,
    ``v`` of one shape ``[B, H, N, D]`` (``D`` a multiple of 8 and at most 64,
    ``N`` > 128); the kernel rounds q to f16 itself.  Runs on ``stream``
    (default: the current torch stream) and returns ``out`` without
    synchronising."""
    import torch

    for name, t, dt in (("q", q, torch.float32), ("k", k, torch.float16), ("v", v, torch.float16)):
        if not isinstance(t, torch.Tensor):
            raise TypeError(f"{name} must be a torch.Tensor")
        if t.dtype != dt:
            raise TypeError(f"{name} must be {dt}, got {t.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dim() != 4:
            raise ValueError(f"{name} must be [batch, n_heads, n_patches, head_dim]")
        if t.device.type != "cuda":
            raise ValueError(f"{name} must be a CUDA tensor")
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (head-major [B, H, N, D])")
    if not (q.shape == k.shape == v.shape) or not (q.device == k.device == v.device):
        raise ValueError("q, k and v must have one shape and one device")
    if out is None:
        out = torch.empty(q.shape, dtype=torch.float32, device=q.device)
    if out.shape != q.shape or out.dtype != torch.float32 or out.device != q.device \
            or not out.is_contiguous():
        raise ValueError("out must be a contiguous float32 tensor of q's shape and device")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    B, H, N, D = q.shape
    forward_f32q_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N, D,
                     s.cuda_stream)
    return out


def forward_f16io(q, k, v, out=None, stream=None):
    """out (f16) = softmax(q k^T) v for CUDA float16 tensors ``[B, H, N, D]``
    (``D`` a multiple of 8): the output of ``forward_f16`` rounded to f16.
    Runs on ``stream`` (default: the current torch stream); no synchronisation."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if not isinstance(t, torch.Tensor) or t.dtype != torch.float16:
            raise TypeError(f"{name} must be a float16 torch.Tensor")
        if t.dim() != 4 or t.device.type != "cuda" or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA [batch, n_heads, n_patches, head_dim]")
    if not (q.shape == k.shape == v.shape) or not (q.device == k.device == v.device):
        raise ValueError("q, k and v must have one shape and one device")
    if out is None:
        out = torch.empty_like(q)
    if out.shape != q.shape or out.dtype != torch.float16 or out.device != q.device \
            or not out.is_contiguous():
        raise ValueError("out must be a contiguous float16 tensor of q's shape and device")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    B, H, N, D = q.shape
    _check(forward_f16io_status(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N,
                                D, s.cuda_stream))
    return out


def _cuda_f32(name, t):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _factors_ptr(factors, rope_dims, device):
    if factors is None:
        return 0
    _cuda_f32("factors", factors)
    if factors.device != device or factors.numel() < rope_dims // 2:
        raise ValueError("factors must hold rope_dims // 2 floats on the tensors' device")
    return factors.data_ptr()


def rope_neox(x, rope_dims, pos0=0, base=10000.0, factors=None, inverse=False, stream=None):
    """NeoX rotary embedding of a CUDA f32 tensor ``[B, H, N, D]`` in place
    (patch n at position ``pos0 + n``); ``inverse=True`` turns back.
    Returns ``x`` without synchronising."""
    import torch

    _cuda_f32("x", x)
    if x.dim() != 4:
        raise ValueError("x must be [batch, n_heads, n_patches, head_dim]")
    s = stream if stream is not None else torch.cuda.current_stream(x.device)
    B, H, N, D = x.shape
    _check(rope_neox_status(x.data_ptr(), B, H, N, D, rope_dims, pos0, float(base),
                            _factors_ptr(factors, rope_dims, x.device), bool(inverse),
                            s.cuda_stream))
    return x


def forward_rope(q, k, v, rope_dims, pos0=0, base=10000.0, factors=None, out=None, stream=None):
    """out = softmax(rope(q) rope(k)^T) v for CUDA f32 tensors ``[B, H, N, D]``,
    with the forward NeoX rotation of q and k (patch n at position ``pos0 + n``)
    fused into the f16 staging; q and k are not modified."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_f32(name, t)
        if t.dim() != 4:
            raise ValueError(f"{name} must be [batch, n_heads, n_patches, head_dim]")
    if not (q.shape == k.shape == v.shape) or not (q.device == k.device == v.device):
        raise ValueError("q, k and v must have one shape and one device")
    if out is None:
        out = torch.empty_like(q)
    _cuda_f32("out", out)
    if out.shape != q.shape or out.device != q.device:
        raise ValueError("out must match q in shape and device")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    B, H, N, D = q.shape
    _check(forward_rope_status(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N,
                               D, rope_dims, pos0, float(base),
                               _factors_ptr(factors, rope_dims, q.device), s.cuda_stream))
    return out


def forward_accurate(q, k, v, out=None, stream=None):
    """out = softmax(q k^T) v for CUDA f32 tensors ``[B, H, N, D]`` to about
    f32 accuracy: every operand is split into two f16 terms and each matrix
    product takes three tensor-core products.  Returns ``out`` without
    synchronising."""
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        _cuda_f32(name, t)
        if t.dim() != 4:
            raise ValueError(f"{name} must be [batch, n_heads, n_patches, head_dim]")
    if not (q.shape == k.shape == v.shape) or not (q.device == k.device == v.device):
        raise ValueError("q, k and v must have one shape and one device")
    if out is None:
        out = torch.empty_like(q)
    _cuda_f32("out", out)
    if out.shape != q.shape or out.device != q.device:
        raise ValueError("out must match q in shape and device")
    s = stream if stream is not None else torch.cuda.current_stream(q.device)
    B, H, N, D = q.shape
    _check(forward_accurate_status(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H,
                                   N, D, s.cuda_stream))
    return out


def conv1d_step(input, buffer, weight, out=None, stream=None):
    """One depthwise conv1d rolling-buffer step on CUDA f32 tensors.

    input ``[batch, hidden]`` (or ``[hidden]``), buffer ``[batch, d_conv,
    hidden]`` (or ``[d_conv, hidden]``, updated in place), weight
    ``[hidden, kernel_size]`` with ``kernel_size >= d_conv + 1``.  Returns
    ``out`` (shape of input) without synchronising."""
    import torch

    for name, t in (("input", input), ("buffer", buffer), ("weight", weight)):
        _cuda_f32(name, t)
    single = input.dim() == 1
    x = input.unsqueeze(0) if single else input
    buf = buffer.unsqueeze(0) if single else buffer
    if x.dim() != 2 or buf.dim() != 3 or weight.dim() != 2:
        raise ValueError("expected input [B, hidden], buffer [B, d_conv, hidden], weight [hidden, K]")
    B, hidden = x.shape
    d_conv = buf.shape[1]
    if tuple(buf.shape) != (B, d_conv, hidden) or weight.shape[0] != hidden:
        raise ValueError(f"shape mismatch: input {tuple(input.shape)}, buffer {tuple(buffer.shape)}, "
                         f"weight {tuple(weight.shape)}")
    if not (input.device == buffer.device == weight.device):
        raise ValueError("input, buffer and weight must be on one device")
    if out is None:
        out = torch.empty_like(input)
    _cuda_f32("out", out)
    if out.shape != input.shape or out.device != input.device:
        raise ValueError("out must match input in shape and device")
    s = stream if stream is not None else torch.cuda.current_stream(input.device)
    _check(conv1d_step_status(x.data_ptr(), buf.data_ptr(), weight.data_ptr(), out.data_ptr(), B,
                              hidden, weight.shape[1], d_conv, s.cuda_stream))
    return out


def _launch(q, k, v, out, stream):
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        if not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous (head-major [B, H, N, D])")
    if out.shape != q.shape or out.dtype != q.dtype or out.device != q.device:
        raise ValueError("out must match q in shape, dtype and device")
    B, H, N, D = q.shape
    forward_raw(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, H, N, D,
                stream.cuda_stream)

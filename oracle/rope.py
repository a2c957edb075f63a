"""Double-precision NeoX rotary embedding (RoPE) -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
use it; it shares no code with the CUDA path.

It restates the rotation of the WGSL kernel "rope_neox_backward.wgsl"
(rullama 0.2.0), whose header comment gives both directions:

* ``half = rope_dims // 2``; for every head and every ``i < half`` the pair
  ``(a, b) = (x[i], x[i + half])`` of that head is rotated by the angle
  ``theta_i = pos * base ** (-2 i / rope_dims)``, divided by ``factors[i]``
  when a factor table is given (the kernel's ``has_factors`` branch);
* forward: ``x[i] <- a cos - b sin``, ``x[i + half] <- a sin + b cos``;
* backward (inverse) rotates by ``-theta``:
  ``x[i] <- a cos + b sin``, ``x[i + half] <- -a sin + b cos``;
* dimensions ``>= 2 * half`` are left as they are.

The page rotates the heads of one token at one position ``pos``.  Here the
input is head-major ``[batch, n_heads, n_patches, head_dim]`` and patch ``n``
sits at position ``pos0 + n`` (with ``n_patches == 1`` and ``pos0 == pos``
this is exactly the page's kernel on ``[n_heads, head_dim]``).
"""
from __future__ import annotations

import numpy as np


def angles(n_patches: int, rope_dims: int, pos0: int, base: float,
           factors=None) -> np.ndarray:
    """theta[n, i] in f64 for patch n (position pos0 + n) and pair i."""
    half = rope_dims // 2
    theta = np.zeros((n_patches, half), dtype=np.float64)
    for i in range(half):
        inv_freq = float(base) ** (-2.0 * i / rope_dims)
        if factors is not None:
            inv_freq /= float(factors[i])
        for n in range(n_patches):
            theta[n, i] = (pos0 + n) * inv_freq
    return theta


def rope_neox(x: np.ndarray, rope_dims: int, pos0: int, base: float,
              factors=None, inverse: bool = False) -> np.ndarray:
    """Rotated copy (f64) of x ``[B, H, N, D]``; see the module docstring."""
    x = np.asarray(x, dtype=np.float64)
    if x.ndim != 4:
        raise ValueError(f"expected [B, H, N, D], got shape {x.shape}")
    B, H, N, D = x.shape
    if not 0 <= rope_dims <= D:
        raise ValueError(f"rope_dims {rope_dims} outside [0, {D}]")
    half = rope_dims // 2
    out = x.copy()
    if half == 0:
        return out
    theta = angles(N, rope_dims, pos0, base, factors)   # [N, half]
    c = np.cos(theta)[None, None, :, :]
    s = np.sin(theta)[None, None, :, :]
    a = x[..., :half]
    b = x[..., half:2 * half]
    if not inverse:
        out[..., :half] = a * c - b * s
        out[..., half:2 * half] = a * s + b * c
    else:
        out[..., :half] = a * c + b * s
        out[..., half:2 * half] = -a * s + b * c
    return out

"""Double-precision depthwise conv1d rolling-buffer step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU legs may
use it; it shares no code with the CUDA path.

It restates the WGSL kernel "conv1d.wgsl" (cera 0.2.0), one decode step of a
depthwise (per-channel) causal convolution whose past inputs live in a
rolling buffer.  From the page's header comment and bindings:

* ``input``  ``[hidden_size]``: this step's value of every channel;
* ``buffer`` ``[d_conv, hidden_size]``: slot ``k`` of channel ``ch`` at
  ``k * hidden_size + ch``, slot 0 the oldest;
* ``weight`` ``[hidden_size, kernel_size]``: channel ``ch``'s taps at
  ``ch * kernel_size + k``; tap ``k < d_conv`` weighs slot ``k`` and tap
  ``d_conv`` weighs the current input (so ``kernel_size >= d_conv + 1``);
* ``out[ch] = sum_{k < d_conv} buffer[k, ch] * weight[ch, k]
  + input[ch] * weight[ch, d_conv]``;
* then the buffer moves one slot towards the front (slot k takes slot
  k + 1) and the input goes into the last slot ``d_conv - 1``.

The page runs one sequence.  Here a leading ``batch`` axis may hold many
independent sequences, each with its own buffer; the weights are shared.
"""
from __future__ import annotations

import numpy as np


def conv1d_step(inp, buffer, weight):
    """One step; returns ``(out, new_buffer)`` in f64, inputs untouched.

    inp ``[hidden]`` or ``[batch, hidden]``; buffer ``[d_conv, hidden]`` or
    ``[batch, d_conv, hidden]``; weight ``[hidden, kernel_size]``.
    """
    x = np.asarray(inp, dtype=np.float64)
    buf = np.asarray(buffer, dtype=np.float64)
    w = np.asarray(weight, dtype=np.float64)
    single = x.ndim == 1
    if single:
        x = x[None]
        buf = buf[None]
    if x.ndim != 2 or buf.ndim != 3 or w.ndim != 2:
        raise ValueError("expected inp [B, hidden], buffer [B, d_conv, hidden], weight [hidden, K]")
    batch, hidden = x.shape
    d_conv = buf.shape[1]
    kernel_size = w.shape[1]
    if buf.shape != (batch, d_conv, hidden) or w.shape[0] != hidden:
        raise ValueError(f"shape mismatch: inp {x.shape}, buffer {buf.shape}, weight {w.shape}")
    if kernel_size < d_conv + 1:
        raise ValueError(f"kernel_size {kernel_size} < d_conv + 1 = {d_conv + 1}")

    out = np.zeros((batch, hidden), dtype=np.float64)
    for k in range(d_conv):                 # the rolling-buffer taps, oldest first
        out += buf[:, k, :] * w[None, :, k]
    out += x * w[None, :, d_conv]            # the current input's tap

    new_buf = buf.copy()
    for k in range(d_conv - 1):              # shift towards slot 0
        new_buf[:, k, :] = buf[:, k + 1, :]
    if d_conv > 0:
        new_buf[:, d_conv - 1, :] = x        # append this step's input
    if single:
        return out[0], new_buf[0]
    return out, new_buf

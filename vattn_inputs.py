"""Seeded synthetic inputs for the head-major attention workloads.

This module is shared by the oracle tests and the CUDA path's tests and
benchmark.  It holds none of the attention arithmetic: it only draws q, k, v.

Recipe (the workloads of the vision-attention shader: image patches, head-major
``[batch, n_heads, n_patches, head_dim]`` f32, q pre-scaled by the caller):

* ``numpy.random.Generator(PCG64(seed))``;
* draw, in this order and in float64: q, k, (per-head key offset), v, each
  ``standard_normal``;
* q is multiplied by ``1/sqrt(head_dim)`` in float64 (the caller's
  pre-scaling);
* the "peaked" workload adds to every key row of head h one offset vector
  ``offset[h]`` drawn from N(0, 2) (variance 2, standard deviation sqrt(2)),
  shared across the batch and across rows;
* every array is cast to float32 once, at the end.

The depthwise conv1d rolling-buffer step (page "conv1d.wgsl", cera 0.2.0)
has its own recipe, ``conv1d_inputs``: the same generator, drawing input
``[batch, hidden]``, buffer ``[batch, d_conv, hidden]`` (both
``standard_normal``) and weight ``[hidden, kernel_size]``
(``standard_normal / sqrt(d_conv + 1)``, so an output has unit variance), in
that order, cast to float32 at the end.  The page gives no sizes; the
benchmark workload ``CONV1D_WORKLOAD`` is a decode step of 8192 sequences
with 2048 channels and a 3-tap kernel (2 buffer slots): 403 MB moved per
step, three times the 129 MB L2.
"""
from __future__ import annotations

import dataclasses

import numpy as np

SEED_BASE = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    batch: int
    n_heads: int
    n_patches: int
    head_dim: int
    peaked: bool
    description: str

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index

    @property
    def shape(self):
        return (self.batch, self.n_heads, self.n_patches, self.head_dim)

    @property
    def flops(self) -> int:
        """4*B*H*N^2*D: two matrix products of 2*N*N*D per head."""
        return 4 * self.batch * self.n_heads * self.n_patches ** 2 * self.head_dim

    @property
    def name(self) -> str:
        b, h, n, d = self.shape
        return f"vit_attn_b{b}_h{h}_n{n}_d{d}" + ("_peaked" if self.peaked else "")


WORKLOADS = {
    1: Workload(1, 1, 2, 64, 32, False, "8x8 patches, tiny"),
    2: Workload(2, 1, 16, 256, 64, False, "16x16 patch grid"),
    3: Workload(3, 4, 16, 1024, 64, False, "32x32 patch grid"),
    4: Workload(4, 1, 16, 4100, 72, False,
                "ragged patch count, non-power-of-two head_dim"),
    5: Workload(5, 8, 16, 2304, 64, True,
                "48x48 patch grid, keys with a shared per-head offset"),
}


def make_inputs(batch: int, n_heads: int, n_patches: int, head_dim: int,
                seed: int, peaked: bool = False):
    """Return float32 ``(q, k, v)`` of shape ``[batch, n_heads, n_patches, head_dim]``."""
    shape = (batch, n_heads, n_patches, head_dim)
    rng = np.random.Generator(np.random.PCG64(seed))
    q = rng.standard_normal(shape)
    k = rng.standard_normal(shape)
    if peaked:
        offset = rng.standard_normal((n_heads, head_dim)) * np.sqrt(2.0)
        k = k + offset[None, :, None, :]
    v = rng.standard_normal(shape)
    if head_dim > 0:
        q = q * (1.0 / np.sqrt(head_dim))
    return (q.astype(np.float32), k.astype(np.float32), v.astype(np.float32))


def workload_inputs(index: int):
    w = WORKLOADS[index]
    return make_inputs(w.batch, w.n_heads, w.n_patches, w.head_dim, w.seed,
                       w.peaked)


CONV1D_WORKLOAD = dict(batch=8192, hidden=2048, kernel_size=3, d_conv=2, seed=SEED_BASE + 40)


def conv1d_workload_name(w=CONV1D_WORKLOAD) -> str:
    return f"conv1d_step_b{w['batch']}_h{w['hidden']}_k{w['kernel_size']}_dc{w['d_conv']}"


def conv1d_inputs(batch: int, hidden: int, kernel_size: int, d_conv: int, seed: int):
    """Return float32 ``(input, buffer, weight)`` for the conv1d step."""
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((batch, hidden))
    buf = rng.standard_normal((batch, d_conv, hidden))
    w = rng.standard_normal((hidden, kernel_size)) / np.sqrt(d_conv + 1)
    return x.astype(np.float32), buf.astype(np.float32), w.astype(np.float32)

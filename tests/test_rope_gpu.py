"""GPU parity of the NeoX rotary embedding (vattn_rope_neox) and of attention
with the rotation fused into the f16 staging (vattn_forward_rope), through
the C ABI, against the f64 oracles (oracle.rope, oracle.forward).

Tolerance of the rotation: the kernel computes theta, cos and sin in f32 as
the page "rope_neox_backward.wgsl" (rullama 0.2.0) does, so theta carries a
relative error of a few f32 ulps (absolute ~ theta_max * 2^-22) and cos/sin
and the two products a few ulps more: per element
|gpu - oracle| <= (theta_max * 2^-20 + 2^-19) * max|x| over its row pair.

Tolerance of the fused attention: the rotated q, k are rounded to f16 like
vattn_forward's inputs, so the acceptance bar of the attention parity tests
applies (max abs 3e-3, rel L2 1e-3; twice the rel-L2 bar for off-workload
shapes, as there), with the oracle run on q and k turned in f64.
"""
import numpy as np
import pytest

import oracle
from oracle import rope as orope
import vision_encoder_flash_gb300 as vef
from vattn_inputs import make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

MAX_ABS = 3e-3
MAX_REL_L2 = 1e-3


@pytest.fixture(scope="module")
def torch_dev():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need a CUDA device")
    from vision_encoder_flash_gb300 import build
    build.build()
    vef.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    return torch, dev


def gpu_rope(torch_dev, x, rope_dims, pos0, base, factors=None, inverse=False):
    torch, dev = torch_dev
    xd = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(dev)
    fd = None if factors is None else torch.from_numpy(np.asarray(factors, np.float32)).to(dev)
    vef.rope_neox(xd, rope_dims, pos0, base, factors=fd, inverse=inverse)
    torch.cuda.synchronize(dev)
    return xd.cpu().numpy()


def rope_bound(x, rope_dims, pos0, base, factors):
    n = x.shape[2]
    theta = orope.angles(n, rope_dims, pos0, base, factors)
    theta_max = float(np.abs(theta).max()) if theta.size else 0.0
    return (theta_max * 2.0 ** -20 + 2.0 ** -19) * float(np.abs(x).max())


ROPE_CASES = [
    # (shape, rope_dims, pos0, base, with factors)
    ((1, 8, 1, 64), 64, 17, 10000.0, False),     # the page's form: one token, all heads
    ((2, 3, 17, 64), 64, 0, 10000.0, False),
    ((2, 3, 17, 64), 62, 5, 10000.0, True),
    ((1, 4, 100, 72), 72, 1000, 10000.0, False),
    ((1, 2, 33, 128), 96, 4000, 500.0, True),
    ((2, 2, 5, 8), 7, 3, 10000.0, False),        # odd rope_dims: dim 6 stays
    ((1, 2, 9, 16), 2, 123456, 10000.0, False),  # one pair at large positions
    ((3, 1, 40, 40), 40, 77, 0.5, False),        # base < 1: frequencies grow
]


@pytest.mark.parametrize("shape,rope_dims,pos0,base,with_f", ROPE_CASES)
@pytest.mark.parametrize("inverse", [False, True])
def test_rope_matches_oracle(torch_dev, shape, rope_dims, pos0, base, with_f, inverse):
    x = make_inputs(*shape, seed=4000 + sum(shape) + rope_dims)[0] * 8.0
    factors = None
    if with_f:
        factors = np.random.default_rng(rope_dims).uniform(0.5, 4.0, rope_dims // 2).astype(np.float32)
    got = gpu_rope(torch_dev, x, rope_dims, pos0, base, factors, inverse)
    ref = orope.rope_neox(x, rope_dims, pos0, base, factors=factors, inverse=inverse)
    bound = rope_bound(x, rope_dims, pos0, base, factors)
    err = float(np.abs(got.astype(np.float64) - ref).max())
    assert err <= bound, f"max abs {err:.3e} > bound {bound:.3e}"
    half = rope_dims // 2
    np.testing.assert_array_equal(got[..., 2 * half:], x[..., 2 * half:])


def test_rope_round_trip(torch_dev):
    x = make_inputs(2, 4, 50, 64, seed=4100)[0]
    y = gpu_rope(torch_dev, x, 64, 200, 10000.0)
    back = gpu_rope(torch_dev, y, 64, 200, 10000.0, inverse=True)
    bound = 2 * rope_bound(x, 64, 200, 10000.0, None)
    assert float(np.abs(back - x).max()) <= bound


def test_rope_position_zero_and_empty_rotation_change_nothing(torch_dev):
    x = make_inputs(1, 2, 1, 32, seed=4200)[0]
    np.testing.assert_array_equal(gpu_rope(torch_dev, x, 32, 0, 10000.0), x)
    x = make_inputs(1, 2, 7, 32, seed=4201)[0]
    np.testing.assert_array_equal(gpu_rope(torch_dev, x, 1, 5, 10000.0), x)


def fused_reference(q, k, v, rope_dims, pos0, base, factors=None):
    qr = orope.rope_neox(q, rope_dims, pos0, base, factors=factors).astype(np.float32)
    kr = orope.rope_neox(k, rope_dims, pos0, base, factors=factors).astype(np.float32)
    return qr, kr


def run_fused(torch_dev, q, k, v, rope_dims, pos0, base, factors=None):
    torch, dev = torch_dev
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, v))
    q_keep, k_keep = qd.clone(), kd.clone()
    fd = None if factors is None else torch.from_numpy(np.asarray(factors, np.float32)).to(dev)
    out = vef.forward_rope(qd, kd, vd, rope_dims, pos0, base, factors=fd)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    assert torch.equal(qd, q_keep) and torch.equal(kd, k_keep), "q or k was modified"
    return out.cpu().numpy()


def assert_close(got, ref, what, rel_l2):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = got.astype(np.float64) - ref
    mx = float(np.abs(diff).max())
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    assert mx <= MAX_ABS and rel <= rel_l2, f"{what}: max abs {mx:.3e}, rel L2 {rel:.3e}"


FUSED_CASES = [
    ((1, 2, 64, 32), 32, 0, 10000.0, False),
    ((2, 3, 200, 40), 40, 11, 10000.0, True),
    ((1, 4, 257, 64), 64, 0, 10000.0, False),
    ((1, 4, 257, 64), 32, 100, 1000.0, False),   # partial rotation
    ((2, 2, 130, 72), 72, 3, 10000.0, False),
    ((1, 2, 300, 128), 128, 9, 10000.0, True),
    ((1, 2, 129, 20), 13, 0, 10000.0, False),    # odd rope_dims, head_dim % 8 != 0
]


@pytest.mark.parametrize("shape,rope_dims,pos0,base,with_f", FUSED_CASES)
def test_fused_rope_attention_matches_oracle(torch_dev, shape, rope_dims, pos0, base, with_f):
    q, k, v = make_inputs(*shape, seed=5000 + sum(shape) + rope_dims)
    factors = None
    if with_f:
        factors = np.random.default_rng(5 + rope_dims).uniform(0.5, 4.0, rope_dims // 2).astype(np.float32)
    got = run_fused(torch_dev, q, k, v, rope_dims, pos0, base, factors)
    qr, kr = fused_reference(q, k, v, rope_dims, pos0, base, factors)
    assert_close(got, oracle.forward(qr, kr, v), f"{shape} rope {rope_dims}", 2 * MAX_REL_L2)


def test_fused_rope_equals_rope_then_forward(torch_dev):
    """The fused pass and the two-step path (turn q and k in f32 on the GPU,
    then vattn_forward) agree to f16 rounding of the turned values."""
    torch, dev = torch_dev
    q, k, v = make_inputs(2, 4, 300, 64, seed=5100)
    fused = run_fused(torch_dev, q, k, v, 64, 7, 10000.0)
    qr = gpu_rope(torch_dev, q, 64, 7, 10000.0)
    kr = gpu_rope(torch_dev, k, 64, 7, 10000.0)
    two = vef.forward(*(torch.from_numpy(x).to(dev) for x in (qr, kr, v)))
    torch.cuda.synchronize(dev)
    assert_close(fused, two.cpu().numpy().astype(np.float64), "fused vs two-step", MAX_REL_L2)


@pytest.mark.parametrize("idx", [3, 4])
def test_fused_rope_on_workloads(torch_dev, idx):
    q, k, v = workload_inputs(idx)
    d = q.shape[-1]
    got = run_fused(torch_dev, q, k, v, d, 0, 10000.0)
    qr, kr = fused_reference(q, k, v, d, 0, 10000.0)
    assert_close(got, oracle.forward(qr, kr, v), f"workload {idx}", MAX_REL_L2)

"""GPU parity of vattn_forward_f16 (inputs already f16) through the C ABI.

Two checks per shape:

* against the f64 oracle evaluated on the same f16 values (converted to f32
  exactly): the only differences are the f16 rounding of the softmax weights
  P, f32 accumulation and the ex2 approximation, so
  |gpu - oracle| <= (2^-11 + n_patches * 2^-24) * max|v| + 1e-5 and
  rel L2 <= 5e-4 (the kernel-arithmetic bound of the f32-input tests);
* against vattn_forward on the f32 copies of the f16 inputs: its staging
  pass rounds them to f16 without change, so both calls run the same kernel
  on the same operands and must agree bit for bit.
"""
import numpy as np
import pytest

import oracle
import vision_encoder_flash_gb300 as vef
from vattn_inputs import make_inputs, workload_inputs

pytestmark = pytest.mark.gpu


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


def to_f16(x):
    return x.astype(np.float16)


def run_f16(torch_dev, q16, k16, v16):
    torch, dev = torch_dev
    out = vef.forward_f16(*(torch.from_numpy(x).to(dev) for x in (q16, k16, v16)))
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    return out.cpu().numpy()


def run_f32(torch_dev, q, k, v):
    torch, dev = torch_dev
    out = vef.forward(*(torch.from_numpy(x).to(dev) for x in (q, k, v)))
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    return out.cpu().numpy()


def assert_against_oracle(got, q16, k16, v16, rows=None, what=""):
    q, k, v = (x.astype(np.float32) for x in (q16, k16, v16))
    ref = oracle.forward(q, k, v) if rows is None else oracle.rows(q, k, v, rows)
    if rows is not None:
        got = got.reshape(-1, got.shape[-1])[rows]
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    n = q.shape[2]
    bound = (2.0 ** -11 + n * 2.0 ** -24) * float(np.abs(v).max()) + 1e-5
    diff = got.astype(np.float64) - ref
    mx = float(np.abs(diff).max())
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    assert mx <= bound and rel <= 5e-4, f"{what}: max abs {mx:.3e} (bound {bound:.3e}), rel L2 {rel:.3e}"


SHAPES = [
    (1, 2, 64, 32), (2, 3, 200, 40), (1, 16, 256, 64), (2, 2, 130, 72), (1, 2, 300, 128),
    (1, 1, 1, 8), (3, 1, 129, 8), (1, 4, 257, 64), (2, 2, 383, 96), (1, 1, 1000, 120),
]


@pytest.mark.parametrize("shape", SHAPES)
def test_f16_entry_matches_oracle_and_f32_entry(torch_dev, shape):
    q, k, v = make_inputs(*shape, seed=777 + sum(shape))
    q16, k16, v16 = to_f16(q), to_f16(k), to_f16(v)
    got = run_f16(torch_dev, q16, k16, v16)
    assert_against_oracle(got, q16, k16, v16, what=str(shape))
    same = run_f32(torch_dev, *(x.astype(np.float32) for x in (q16, k16, v16)))
    assert np.array_equal(got, same), f"{shape}: f16 entry differs from the f32 entry"


@pytest.mark.parametrize("idx", [3, 4, 5])
def test_f16_entry_on_workloads(torch_dev, idx):
    # every output element against the oracle on the f16 values
    q, k, v = workload_inputs(idx)
    q16, k16, v16 = to_f16(q), to_f16(k), to_f16(v)
    got = run_f16(torch_dev, q16, k16, v16)
    assert_against_oracle(got, q16, k16, v16, what=f"workload {idx}")


def test_f16_entry_on_a_side_stream(torch_dev):
    torch, dev = torch_dev
    q, k, v = make_inputs(1, 4, 333, 64, seed=99)
    q16, k16, v16 = (torch.from_numpy(to_f16(x)).to(dev) for x in (q, k, v))
    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        out = vef.forward_f16(q16, k16, v16, stream=s)
    s.synchronize()
    assert vef.device_status() == 0
    ref = run_f16(torch_dev, to_f16(q), to_f16(k), to_f16(v))
    assert np.array_equal(out.cpu().numpy(), ref)


def run_f16io(torch_dev, q16, k16, v16, out_offset=0):
    """vattn_forward_f16io; out_offset (in f16 elements) shifts the output
    inside a larger buffer to exercise an output that is only 2-byte aligned."""
    torch, dev = torch_dev
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q16, k16, v16))
    buf = torch.full((qd.numel() + out_offset,), float("nan"), dtype=torch.float16, device=dev)
    out = buf[out_offset:].view(qd.shape)
    if out_offset:
        B, H, N, D = qd.shape
        status = vef._lib.forward_f16io_status(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(),
                                               out.data_ptr(), B, H, N, D,
                                               torch.cuda.current_stream(dev).cuda_stream)
        assert status == 0
    else:
        vef.forward_f16io(qd, kd, vd, out=out)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    return out.cpu().numpy()


F16IO_SHAPES = [(1, 2, 64, 32), (2, 3, 200, 40), (1, 16, 256, 64), (2, 2, 130, 72),
                (1, 2, 300, 128), (3, 1, 129, 8), (1, 4, 257, 64)]


@pytest.mark.parametrize("shape", F16IO_SHAPES)
@pytest.mark.parametrize("out_offset", [0, 1])
def test_f16io_is_the_f16_entry_rounded_to_f16(torch_dev, shape, out_offset):
    """Bit for bit: the f16 output is the f32 output of vattn_forward_f16
    rounded to nearest even (numpy's float16 cast), for the bulk-store
    epilogue (head_dim <= 64, 16-byte aligned out) and the per-thread one."""
    q, k, v = make_inputs(*shape, seed=888 + sum(shape))
    q16, k16, v16 = to_f16(q), to_f16(k), to_f16(v)
    got = run_f16io(torch_dev, q16, k16, v16, out_offset)
    ref = run_f16(torch_dev, q16, k16, v16).astype(np.float16)
    assert np.array_equal(got.view(np.uint16), ref.view(np.uint16)), f"{shape}: differs"


def test_f16io_on_the_largest_workload(torch_dev):
    q, k, v = workload_inputs(5)
    q16, k16, v16 = to_f16(q), to_f16(k), to_f16(v)
    got = run_f16io(torch_dev, q16, k16, v16).astype(np.float32)
    n = q.shape[2]
    ref = oracle.forward(*(x.astype(np.float32) for x in (q16, k16, v16)))
    diff = got.astype(np.float64) - ref
    # f16 output rounding (2^-11 relative) on top of the kernel-arithmetic bound
    bound = (2.0 ** -10 + n * 2.0 ** -24) * float(np.abs(v16.astype(np.float32)).max()) + 1e-5
    assert float(np.abs(diff).max()) <= bound

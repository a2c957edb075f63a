"""GPU tests of the host-buffer entry point (vattn_forward_host), through the
C ABI: q, k, v in host memory, out written to host memory, heads cut into up
to eight chunks whose copies and kernels overlap.  The kernels per head are
those of vattn_forward, so the result must be bit-identical to it (with work
tiles uncut: vattn_forward cuts the tiles of a partial last round between two
blocks in large calls, the chunked host path never does); and it is
checked against the f64 oracle with the acceptance bar (max abs 3e-3, rel L2
1e-3; twice the rel-L2 bar off the seeded workloads, as elsewhere)."""
import numpy as np
import pytest

import oracle
import vision_encoder_flash_gb300 as vef
from vision_encoder_flash_gb300 import _lib
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


def device_forward(torch_dev, q, k, v):
    torch, dev = torch_dev
    out = vef.forward(*(torch.from_numpy(x).to(dev) for x in (q, k, v)))
    torch.cuda.synchronize(dev)
    return out.cpu().numpy()


def host_forward(torch_dev, q, k, v, pinned=True, stream=None):
    torch, dev = torch_dev
    ts = [torch.from_numpy(x) for x in (q, k, v)]
    if pinned:
        ts = [t.pin_memory() for t in ts]
    out = torch.empty(q.shape, dtype=torch.float32, pin_memory=pinned)
    s = stream if stream is not None else torch.cuda.current_stream(dev)
    B, H, N, D = q.shape
    st = _lib.forward_host_status(ts[0].data_ptr(), ts[1].data_ptr(), ts[2].data_ptr(),
                                  out.data_ptr(), B, H, N, D, s.cuda_stream)
    assert st == 0, vef.load_library().vattn_last_error_string().decode()
    s.synchronize()
    assert vef.device_status() == 0
    return out.numpy()


# batch*n_heads 1..17: one chunk, chunks of one head, chunks of two and
# three heads with a smaller last chunk (10 = 5 x 2; 17 = 5 x 3 + 2)
SHAPES = [(1, 1, 200, 64), (1, 3, 129, 72), (2, 3, 300, 40), (1, 5, 77, 17), (7, 1, 256, 128),
          (1, 4, 1, 8), (2, 5, 130, 64), (1, 17, 64, 32)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("pinned", [True, False])
def test_bit_identical_to_the_device_entry(torch_dev, shape, pinned):
    q, k, v = make_inputs(*shape, seed=8000 + sum(shape))
    got = host_forward(torch_dev, q, k, v, pinned=pinned)
    np.testing.assert_array_equal(got, device_forward(torch_dev, q, k, v))
    ref = oracle.forward(q, k, v)
    diff = got.astype(np.float64) - ref
    assert float(np.abs(diff).max()) <= 3e-3
    assert float(np.linalg.norm(diff) / np.linalg.norm(ref)) <= 2e-3


def test_workload_5_through_host_buffers(torch_dev):
    # the host path runs chunks of heads and never cuts a work tile between
    # two blocks; vattn_forward on the whole workload would cut the tiles of
    # its partial last round, so it is compared with cutting forbidden
    q, k, v = workload_inputs(5)
    got = host_forward(torch_dev, q, k, v)
    prev = _lib.set_split_tiles(False)
    try:
        ref = device_forward(torch_dev, q, k, v)
    finally:
        _lib.set_split_tiles(prev)
    np.testing.assert_array_equal(got, ref)


def test_side_stream_and_python_binding(torch_dev):
    torch, dev = torch_dev
    q, k, v = make_inputs(2, 4, 333, 64, seed=8100)
    side = torch.cuda.Stream(dev)
    a = host_forward(torch_dev, q, k, v, stream=side)
    b = vef.forward(*(torch.from_numpy(x).pin_memory() for x in (q, k, v)), stream=side).numpy()
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(a, device_forward(torch_dev, q, k, v))


def test_empty_problems(torch_dev):
    assert _lib.forward_host_status(0, 0, 0, 0, 0, 4, 16, 64, 0) == 0
    assert _lib.forward_host_status(0, 0, 0, 0, 2, 4, 0, 64, 0) == 0

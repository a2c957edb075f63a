"""On the GPU: the mode each call takes (vattn_forward_mode, which reads the
device's cooperative-launch support and the single kernel's occupancy), and
the fallback from the single cooperative kernel to the two-kernel mode when
the single kernel is forbidden (vattn_set_single_kernel(0), the same switch
as a device without cooperative launches): the results are bit-identical."""
import numpy as np
import pytest

import vision_encoder_flash_gb300 as vef
from vision_encoder_flash_gb300 import _lib
from vattn_inputs import make_inputs

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


def inputs(torch_dev, shape, seed):
    torch, dev = torch_dev
    return tuple(torch.from_numpy(x).to(dev) for x in make_inputs(*shape, seed=seed))


def mode_of(q, k, v, out):
    b, h, n, d = q.shape
    return _lib.forward_mode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), b, h, n, d)


def run(fn, q, k, v, out, stream):
    b, h, n, d = q.shape
    fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), b, h, n, d, stream.cuda_stream)


@pytest.mark.parametrize("shape,mode", [
    ((4, 16, 1024, 64), _lib.MODE_DIRECT),
    ((2, 16, 2304, 64), _lib.MODE_SINGLE_KERNEL),
    ((1, 16, 4100, 72), _lib.MODE_TWO_KERNELS),
])
def test_modes_on_this_device(torch_dev, shape, mode):
    q, k, v = inputs(torch_dev, shape, 71)
    out = torch_dev[0].empty_like(q)
    assert mode_of(q, k, v, out) == mode


@pytest.mark.parametrize("shape", [(2, 16, 2304, 64), (1, 3, 2500, 20), (1, 2, 300, 32)])
@pytest.mark.parametrize("entry", ["forward", "noalloc"])
def test_forbidden_single_kernel_falls_back_bit_identical(torch_dev, shape, entry):
    torch, dev = torch_dev
    fn = _lib.forward_raw if entry == "forward" else _lib.forward_noalloc_raw
    q, k, v = inputs(torch_dev, shape, 72)
    stream = torch.cuda.current_stream(dev)
    single = torch.full_like(q, float("nan"))
    assert mode_of(q, k, v, single) == _lib.MODE_SINGLE_KERNEL
    run(fn, q, k, v, single, stream)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    prev = _lib.set_single_kernel(False)
    try:
        two = torch.full_like(q, float("nan"))
        assert mode_of(q, k, v, two) == _lib.MODE_TWO_KERNELS
        run(fn, q, k, v, two, stream)
        torch.cuda.synchronize(dev)
        assert vef.device_status() == 0
    finally:
        _lib.set_single_kernel(prev)
    a, b = single.cpu().numpy(), two.cpu().numpy()
    assert np.all(np.isfinite(a))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))

"""vattn_forward_noalloc, the allocation-free entry point, through the C ABI.

It runs the same two kernels as vattn_forward but stages q, k and v in a fixed
device array of the library instead of a pool allocation, so its output must
match vattn_forward's within the parity tolerance (3e-3 max abs, 1e-3 rel
L2); with the same kernels on the same inputs it is in fact bit-identical.
Each case makes two noalloc calls in a row, the second on other inputs and
another shape, so that a call which read the previous call's staging would
show.  Every shape here takes a mode that stages through the fixed array
(the single cooperative kernel, whose flags and f16 k, v copies live there,
or the two-kernel mode, whose f16 q, k, v copies do): the direct f32 kernel
uses no scratch, so its shapes would prove nothing, and each case asserts
its mode.  This file is collected last and also passes run on its own in a
fresh process: it builds and loads the library itself.
"""
import numpy as np
import pytest

import vision_encoder_flash_gb300 as vef
from vision_encoder_flash_gb300 import _lib
from vattn_inputs import make_inputs

pytestmark = pytest.mark.gpu

MAX_ABS = 3e-3
MAX_REL_L2 = 1e-3
SCRATCH = 32 * 1024 * 1024  # VATTN_NOALLOC_MAX_SCRATCH_BYTES in include/vattn.h


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


def staged_bytes(b, h, n, d):
    region = (b * h * n * ((d + 15) // 16 * 16) * 2 + 255) // 256 * 256
    return 3 * region


def device_inputs(torch_dev, shape, seed):
    torch, dev = torch_dev
    q, k, v = make_inputs(*shape, seed=seed)
    return tuple(torch.from_numpy(x).to(dev) for x in (q, k, v))


SCRATCH_MODES = (_lib.MODE_SINGLE_KERNEL, _lib.MODE_TWO_KERNELS)


def assert_stages_through_scratch(q, k, v, out):
    b, h, n, d = q.shape
    mode = _lib.forward_mode(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), b, h, n, d)
    assert mode in SCRATCH_MODES, f"{tuple(q.shape)} takes mode {mode}, which uses no scratch"
    return mode


def call(fn, q, k, v, out, stream):
    b, h, n, d = q.shape
    fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), b, h, n, d, stream.cuda_stream)


def assert_close(got, ref, what):
    got = got.double().cpu().numpy()
    ref = ref.double().cpu().numpy()
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    diff = got - ref
    mx = float(np.abs(diff).max())
    rel = float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))
    assert mx <= MAX_ABS and rel <= MAX_REL_L2, f"{what}: max abs {mx:.3e}, rel L2 {rel:.3e}"
    assert np.array_equal(got, ref), f"{what}: not bit-identical to vattn_forward (max abs {mx:.3e})"


@pytest.mark.parametrize("first,second", [
    # single cooperative kernel (flags + f16 k, v in the array), then two
    # kernels on a head_dim that is not a multiple of 4 (f16 q, k, v there)
    ((1, 16, 2304, 64), (1, 3, 200, 38)),
    # two kernels: ragged tail at head_dim 72, then head_dim 128
    ((1, 16, 4100, 72), (2, 2, 130, 128)),
    # two kernels on one query tile (64 patches, head_dim not a multiple of
    # 4), then the single kernel at head_dim 20 with a ragged last key tile
    ((1, 2, 64, 30), (2, 8, 2500, 20)),
    # the single kernel with the last round's tiles cut by key range (the
    # default rule cuts 256 tiles of 32 key tiles on a 152-block grid): the
    # cut tiles' partial results in the second array; then a small call
    ((1, 16, 4096, 64), (1, 3, 200, 38)),
])
def test_noalloc_matches_forward_two_calls_in_a_row(torch_dev, first, second):
    torch, dev = torch_dev
    assert staged_bytes(*first) <= SCRATCH and staged_bytes(*second) <= SCRATCH
    stream = torch.cuda.current_stream(dev)
    ins = [device_inputs(torch_dev, first, 901), device_inputs(torch_dev, second, 902)]
    refs, outs = [], []
    for q, k, v in ins:
        ref = torch.empty_like(q)
        assert_stages_through_scratch(q, k, v, ref)
        call(_lib.forward_raw, q, k, v, ref, stream)
        refs.append(ref)
        outs.append(torch.full_like(q, float("nan")))
    torch.cuda.synchronize(dev)
    # two noalloc calls back to back on one stream, no synchronisation between
    for (q, k, v), out in zip(ins, outs):
        call(_lib.forward_noalloc_raw, q, k, v, out, stream)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    assert_close(outs[0], refs[0], f"first call {first}")
    assert_close(outs[1], refs[1], f"second call {second}")


def test_noalloc_largest_accepted_problem(torch_dev):
    """The largest single-head problem at head_dim 16 that fits the scratch."""
    torch, dev = torch_dev
    n = SCRATCH // 3 // 256 * 256 // (16 * 2)
    shape = (1, 1, n, 16)
    assert staged_bytes(*shape) <= SCRATCH < staged_bytes(1, 1, n + 1, 16)
    q, k, v = device_inputs(torch_dev, shape, 903)
    stream = torch.cuda.current_stream(dev)
    ref = torch.empty_like(q)
    assert_stages_through_scratch(q, k, v, ref)
    call(_lib.forward_raw, q, k, v, ref, stream)
    out = torch.full_like(q, float("nan"))
    call(_lib.forward_noalloc_raw, q, k, v, out, stream)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    assert_close(out, ref, f"{shape}")


def test_noalloc_rejects_a_problem_past_the_scratch(torch_dev):
    torch, dev = torch_dev
    n = SCRATCH // 3 // 256 * 256 // (16 * 2) + 1
    q, k, v = (torch.zeros(1, 1, n, 16, device=dev) for _ in range(3))
    out = torch.full_like(q, float("nan"))
    stream = torch.cuda.current_stream(dev)
    with pytest.raises(vef.VattnError) as err:
        call(_lib.forward_noalloc_raw, q, k, v, out, stream)
    assert err.value.status == 2
    assert "vattn_forward" in str(err.value)
    torch.cuda.synchronize(dev)
    assert torch.isnan(out).all(), "a rejected call wrote its output"
    # the regular entry point takes the same problem
    call(_lib.forward_raw, q, k, v, out, stream)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    assert torch.isfinite(out).all()


@pytest.mark.parametrize("shape", [(1, 16, 2304, 64), (1, 16, 4100, 72)])
def test_noalloc_does_not_take_device_memory(torch_dev, shape):
    """After a first call of a shape (which loads the code it needs), further
    calls leave the device's free memory unchanged: the single cooperative
    kernel and the two-kernel mode, both staging through the array."""
    torch, dev = torch_dev
    q, k, v = device_inputs(torch_dev, shape, 904)
    out = torch.empty_like(q)
    assert_stages_through_scratch(q, k, v, out)
    stream = torch.cuda.current_stream(dev)
    call(_lib.forward_noalloc_raw, q, k, v, out, stream)
    torch.cuda.synchronize(dev)
    free_before, _ = torch.cuda.mem_get_info(dev)
    for _ in range(3):
        call(_lib.forward_noalloc_raw, q, k, v, out, stream)
    torch.cuda.synchronize(dev)
    free_after, _ = torch.cuda.mem_get_info(dev)
    assert vef.device_status() == 0
    assert free_after == free_before


def test_noalloc_empty_problem_is_a_no_op(torch_dev):
    assert _lib.forward_noalloc_status(0, 0, 0, 0, 2, 4, 0, 64, 0) == 0
    assert _lib.forward_noalloc_status(0, 0, 0, 0, 0, 4, 10, 64, 0) == 0


def test_noalloc_workload_against_the_oracle(torch_dev, oracle_mod):
    """The seeded 16-head, 4100-patch, head_dim 72 workload (two kernels, its
    f16 copies filling most of the array) through the allocation-free entry,
    compared with the f64 oracle on every output element at the acceptance
    bar (max abs 3e-3, rel L2 1e-3)."""
    from vattn_inputs import workload_inputs
    torch, dev = torch_dev
    qn, kn, vn = workload_inputs(4)
    q, k, v = (torch.from_numpy(x).to(dev) for x in (qn, kn, vn))
    assert staged_bytes(*q.shape) <= SCRATCH
    out = torch.full_like(q, float("nan"))
    assert_stages_through_scratch(q, k, v, out)
    stream = torch.cuda.current_stream(dev)
    call(_lib.forward_noalloc_raw, q, k, v, out, stream)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    ref = oracle_mod.forward(qn, kn, vn)
    got = out.double().cpu().numpy()
    diff = got - ref
    mx = float(np.abs(diff).max())
    rel = float(np.linalg.norm(diff) / np.linalg.norm(ref))
    assert mx <= MAX_ABS and rel <= MAX_REL_L2, f"max abs {mx:.3e}, rel L2 {rel:.3e}"

"""GPU parity of the balanced schedule: work tiles cut by key range between
two thread blocks, the two parts merged by the log-sum-exp rule (the rescale
of (m, l, o) by the larger maximum that the shader applies per key tile).

Each shape below has more work tiles than the GPU has multiprocessors and a
partial last round, so vattn_forward, with cutting forced
(vattn_set_split_tiles(2); by default it cuts only where that pays), cuts
the tiles of the last round (or two) into one equal key range per block; every kernel mode is covered: the
direct f32 kernel, the single cooperative kernel, the two-kernel mode with
the f32-q attention kernel (q 4-byte aligned only) and with two query tiles
sharing one P buffer (head_dim 65..96), and one query tile per block
(head_dim 128).  Checks, on every output element:

* acceptance against the f64 oracle (max abs 3e-3, rel L2 twice 1e-3, as for
  the other shapes outside the seeded workloads);
* the kernel-arithmetic bound against the oracle on f16-rounded inputs;
* agreement with the same call with cutting forbidden
  (vattn_set_split_tiles(0)): the parts of a cut tile take their own maxima,
  so their f16 softmax weights round differently, within the same bound.

By default tiles are cut only where that pays: the pieces' extra prologues
and merges cost about the time of 5 to 10 key tiles per call, so only long
tiles (at least 16 key tiles) with a busiest block shorter by at least 7 key
tiles are cut (the rule is checked on the host in test_mode_rule.py)."""
import numpy as np
import pytest

import oracle
import vision_encoder_flash_gb300 as vef
from vision_encoder_flash_gb300 import _lib
from vattn_inputs import make_inputs

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


@pytest.fixture(autouse=True)
def cutting_forced(torch_dev):
    """By default tiles are cut only where it pays (long tiles, a clearly
    shorter busiest block); these tests cut wherever the schedule allows
    (vattn_set_split_tiles(2)), so that every kernel mode runs cut tiles,
    and restore the previous setting."""
    prev = _lib.set_split_tiles(2)
    yield
    _lib.set_split_tiles(prev)


def run(torch_dev, q, k, v, q_offset=0):
    """vattn_forward; q placed q_offset f32 elements past a 16-byte boundary."""
    torch, dev = torch_dev
    qd = torch.zeros(q.size + 4, device=dev)
    qd[q_offset:q_offset + q.size] = torch.from_numpy(q.ravel()).to(dev)
    kd, vd = (torch.from_numpy(x).to(dev) for x in (k, v))
    out = torch.full(q.shape, float("nan"), device=dev)
    b, h, n, d = q.shape
    qp = qd.data_ptr() + 4 * q_offset
    mode = _lib.forward_mode(qp, kd.data_ptr(), vd.data_ptr(), out.data_ptr(), b, h, n, d)
    vef.forward_raw(qp, kd.data_ptr(), vd.data_ptr(), out.data_ptr(), b, h, n, d,
                    torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    return out.cpu().numpy(), mode


def f16(x):
    return x.astype(np.float16).astype(np.float32)


# (shape, q offset in f32 elements, expected mode); the tile counts (work
# tiles of 256 query rows, or 128 at head_dim 128) are 160 to 720 against
# 152 multiprocessors
CUT = [
    ((1, 40, 1024, 64), 0, _lib.MODE_DIRECT),          # 160 tiles: every block cut, short pieces
    ((2, 80, 1000, 64), 0, _lib.MODE_DIRECT),          # 640 tiles: three whole rounds, then a cut tail
    ((1, 40, 2304, 64), 0, _lib.MODE_SINGLE_KERNEL),   # 360 tiles, 18 key tiles each
    ((1, 40, 2304, 64), 1, _lib.MODE_TWO_KERNELS),     # the same with q 4-byte aligned
    ((1, 20, 4100, 72), 0, _lib.MODE_TWO_KERNELS),     # shared P buffer, ragged last key tile
    ((1, 8, 2500, 128), 0, _lib.MODE_TWO_KERNELS),     # one query tile per block
    ((2, 30, 2100, 20), 0, _lib.MODE_SINGLE_KERNEL),   # head_dim 20, ragged tail
]


@pytest.mark.parametrize("shape,q_offset,mode", CUT)
def test_cut_schedule(torch_dev, shape, q_offset, mode):
    seed = 9100 + sum(shape) + q_offset
    q, k, v = make_inputs(*shape, seed=seed)
    got, got_mode = run(torch_dev, q, k, v, q_offset)
    assert got_mode == mode
    # every output element against the oracle
    sel = got.astype(np.float64)
    assert np.all(np.isfinite(sel))
    ref = oracle.forward(q, k, v)
    mx = float(np.abs(sel - ref).max())
    rel = float(np.linalg.norm(sel - ref) / np.linalg.norm(ref))
    assert mx <= MAX_ABS and rel <= 2 * MAX_REL_L2, f"{shape}: max abs {mx:.3e}, rel L2 {rel:.3e}"
    # kernel arithmetic against the oracle on the f16-rounded inputs
    ref16 = oracle.forward(f16(q), f16(k), f16(v))
    n = shape[2]
    bound = (2.0 ** -11 + n * 2.0 ** -24) * float(np.abs(f16(v)).max()) + 1e-5
    mx16 = float(np.abs(sel - ref16).max())
    rel16 = float(np.linalg.norm(sel - ref16) / np.linalg.norm(ref16))
    assert mx16 <= bound and rel16 <= 5e-4, f"{shape}: {mx16:.3e} (bound {bound:.3e}), {rel16:.3e}"
    # the same call without cut tiles
    prev = _lib.set_split_tiles(False)
    try:
        whole, _ = run(torch_dev, q, k, v, q_offset)
    finally:
        _lib.set_split_tiles(prev)
    diff = got.astype(np.float64) - whole
    assert float(np.abs(diff).max()) <= 2 * bound
    assert float(np.linalg.norm(diff) / np.linalg.norm(whole)) <= 5e-4


def test_cut_schedule_is_deterministic(torch_dev):
    q, k, v = make_inputs(1, 40, 2304, 64, seed=9200)
    a, _ = run(torch_dev, q, k, v)
    b, _ = run(torch_dev, q, k, v)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))


def test_forbidding_cuts_makes_rows_independent_of_the_batch(torch_dev):
    """With cutting forbidden a head's rows do not depend on the other heads
    of the call: one head alone and the same head inside a large call agree
    bit for bit."""
    q, k, v = make_inputs(1, 40, 2304, 64, seed=9300)
    prev = _lib.set_split_tiles(False)
    try:
        full, _ = run(torch_dev, q, k, v)
        one, _ = run(torch_dev, *(np.ascontiguousarray(x[:, 37:38]) for x in (q, k, v)))
    finally:
        _lib.set_split_tiles(prev)
    assert np.array_equal(full[:, 37:38].view(np.uint32), one.view(np.uint32))


@pytest.mark.parametrize("shape,mode", [
    ((2, 16, 4096, 64), _lib.MODE_SINGLE_KERNEL),   # 512 tiles of 32 key tiles
    ((4, 20, 2048, 64), _lib.MODE_SINGLE_KERNEL),   # 640 tiles of 16 key tiles
    ((1, 20, 2048, 64), _lib.MODE_DIRECT),          # 160 tiles of 16: 32 -> 17 per block
])
def test_default_rule_cuts_and_matches_the_oracle(torch_dev, shape, mode):
    """Shapes that the default setting itself cuts (vattn_set_split_tiles(1)),
    every output element against the oracle."""
    torch, dev = torch_dev
    prev = _lib.set_split_tiles(1)
    try:
        n_sm = torch.cuda.get_device_properties(dev).multi_processor_count
        assert _lib.cut_plan_for(*shape, n_sm)
        q, k, v = make_inputs(*shape, seed=9400 + shape[2])
        got, got_mode = run(torch_dev, q, k, v)
    finally:
        _lib.set_split_tiles(prev)
    assert got_mode == mode
    ref = oracle.forward(q, k, v)
    sel = got.astype(np.float64)
    assert np.all(np.isfinite(sel))
    mx = float(np.abs(sel - ref).max())
    rel = float(np.linalg.norm(sel - ref) / np.linalg.norm(ref))
    assert mx <= MAX_ABS and rel <= 2 * MAX_REL_L2, f"{shape}: max abs {mx:.3e}, rel L2 {rel:.3e}"

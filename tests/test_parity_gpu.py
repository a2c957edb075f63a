"""GPU parity: the CUDA path (through the C ABI) against the f64 oracle.

Two bars, both against the unmodified oracle:

* acceptance (the five seeded workloads and the extra cases): max
  |gpu - oracle| <= 3e-3 and ||gpu - oracle||_2 / ||oracle||_2 <= 1e-3 on the
  f32 inputs;
* kernel arithmetic: the oracle evaluated on the f16-rounded q, k, v (the
  shader vision_attention_flash_sub_hpd_f16, rullama 0.1.0, stages q, k and v
  in f16 workgroup storage) differs from the kernel only by the f16 rounding
  of the softmax weights P (at most 2^-11 relative per weight, so at most
  2^-11 * max|v| per output), f32 accumulation over n_patches terms and the
  ex2 approximation: |gpu - oracle16| <= (2^-11 + n_patches * 2^-24) * max|v|
  + 1e-5, and rel L2 <= 5e-4.

Shapes outside the seeded workloads (head_dim 1, tiny n_patches) can carry
more f16 staging error relative to their small outputs; there the acceptance
check uses twice the rel-L2 bar, the kernel-arithmetic check is unchanged.
"""
import numpy as np
import pytest

import oracle
import vision_encoder_flash_gb300 as vef
from vision_encoder_flash_gb300 import _lib
from vattn_inputs import WORKLOADS, make_inputs, workload_inputs

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


def run_gpu(torch_dev, q, k, v):
    torch, dev = torch_dev
    out = vef.forward(torch.from_numpy(q).to(dev), torch.from_numpy(k).to(dev),
                      torch.from_numpy(v).to(dev))
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    return out.cpu().numpy()


def errors(got, ref):
    got = got.astype(np.float64)
    diff = got - ref
    return float(np.abs(diff).max()), float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))


def assert_parity(got, ref, what="", rel_l2=MAX_REL_L2):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, rel = errors(got, ref)
    assert mx <= MAX_ABS and rel <= rel_l2, f"{what}: max abs {mx:.3e}, rel L2 {rel:.3e}"
    return mx, rel


def f16(x):
    return x.astype(np.float16).astype(np.float32)


def assert_kernel_arithmetic(got, q, k, v, rows=None, what=""):
    """GPU vs the oracle on f16-rounded inputs (see module docstring)."""
    q16, k16, v16 = f16(q), f16(k), f16(v)
    if rows is None:
        ref = oracle.forward(q16, k16, v16)
    else:
        ref = oracle.rows(q16, k16, v16, rows)
    n = q.shape[2]
    bound = (2.0 ** -11 + n * 2.0 ** -24) * float(np.abs(v16).max()) + 1e-5
    mx, rel = errors(got, ref)
    assert mx <= bound and rel <= 5e-4, \
        f"{what}: vs f16-input oracle max abs {mx:.3e} (bound {bound:.3e}), rel L2 {rel:.3e}"
    return mx, rel


# head_dim: 1..128 incl. non-multiples of 4 (plain-load variant), of 16 and
# of 64 (two column blocks); n_patches: 1, tile edges +-1 and several tiles.
SMALL = [(d, n) for d in (1, 3, 8, 16, 17, 32, 48, 64) for n in (1, 2, 127, 128, 129, 300)]
SMALL += [(d, n) for d in (72, 80, 96, 100, 127, 128) for n in (1, 128, 129, 385)]


@pytest.mark.parametrize("d,n", SMALL)
def test_small_shapes(torch_dev, d, n):
    q, k, v = make_inputs(2, 3, n, d, seed=1000 + 7 * d + n)
    got = run_gpu(torch_dev, q, k, v)
    assert_kernel_arithmetic(got, q, k, v, what=f"D={d} N={n}")
    assert_parity(got, oracle.forward(q, k, v), f"D={d} N={n}", rel_l2=2 * MAX_REL_L2)


# head_dim <= 64 with more than two query tiles: several thread blocks per
# head, ragged last block
PAIR = [(d, n) for d in (8, 20, 32, 48, 60, 64) for n in (257, 511, 512, 513, 1025)]


# head_dim 65..96 with more than one query tile: two query tiles that share
# one P buffer, two column blocks, several work tiles per head; n_patches
# with a whole number of key tiles (256), one key in the last one (257,
# 1025) and ragged ends
SHARED_P = [(d, n) for d in (65, 70, 80, 88, 96) for n in (129, 192, 256, 257, 511, 1025, 1057)]


@pytest.mark.parametrize("d,n", SHARED_P)
def test_shared_p_shapes(torch_dev, d, n):
    q, k, v = make_inputs(1, 3, n, d, seed=3500 + 11 * d + n)
    got = run_gpu(torch_dev, q, k, v)
    assert_kernel_arithmetic(got, q, k, v, what=f"shared P D={d} N={n}")
    assert_parity(got, oracle.forward(q, k, v), f"shared P D={d} N={n}", rel_l2=2 * MAX_REL_L2)


@pytest.mark.parametrize("d,n", PAIR)
def test_pair_shapes(torch_dev, d, n):
    q, k, v = make_inputs(1, 3, n, d, seed=3000 + 11 * d + n)
    got = run_gpu(torch_dev, q, k, v)
    assert_kernel_arithmetic(got, q, k, v, what=f"pair D={d} N={n}")
    assert_parity(got, oracle.forward(q, k, v), f"pair D={d} N={n}", rel_l2=2 * MAX_REL_L2)


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_workload_full(torch_dev, idx):
    q, k, v = workload_inputs(idx)
    got = run_gpu(torch_dev, q, k, v)
    mx, rel = assert_parity(got, oracle.forward(q, k, v), WORKLOADS[idx].name)
    assert_kernel_arithmetic(got, q, k, v, what=WORKLOADS[idx].name)
    print(f"{WORKLOADS[idx].name}: max abs {mx:.3e} rel L2 {rel:.3e}")


def test_workload_5_full(torch_dev):
    # full size, launch configuration of the benchmark, every output element
    # against the oracle (the multi-threaded f64 oracle takes a few seconds)
    q, k, v = workload_inputs(5)
    got = run_gpu(torch_dev, q, k, v)
    mx, rel = assert_parity(got, oracle.forward(q, k, v), WORKLOADS[5].name)
    assert_kernel_arithmetic(got, q, k, v, what=WORKLOADS[5].name)
    print(f"{WORKLOADS[5].name}: max abs {mx:.3e} rel L2 {rel:.3e}")


@pytest.mark.parametrize("D", [64, 80])
@pytest.mark.parametrize("order", ["increasing", "decreasing", "shuffled"])
def test_running_max_rescale_paths(torch_dev, order, D):
    # scores 40*j/512 (exact in f16): increasing order raises the row max by
    # 10 (14.4 in log2 units) on every key tile, forcing an O rescale each
    # time; head_dim 80 takes the shared-P kernel
    N = 1024
    j = np.arange(N)
    if order == "decreasing":
        j = j[::-1]
    elif order == "shuffled":
        j = np.random.Generator(np.random.PCG64(3)).permutation(N)
    q = np.zeros((1, 2, N, D), np.float32)
    q[..., 0] = 40.0
    q[:, 1, :, 0] = np.linspace(-40, 40, N, dtype=np.float32)  # second head: mixed signs
    k = np.zeros((1, 2, N, D), np.float32)
    k[..., 0] = (j / 512.0).astype(np.float32)
    v = make_inputs(1, 2, N, D, seed=77)[2]
    assert_parity(run_gpu(torch_dev, q, k, v), oracle.forward(q, k, v), order)


def test_single_patch_returns_v_rounded(torch_dev):
    q, k, v = make_inputs(1, 4, 1, 64, seed=11)
    got = run_gpu(torch_dev, q * 50, k, v)
    # P = 1 exactly after f16 rounding; l sums the unrounded exp2 of a ~1e-6
    # residual (s*log2e - round(s*log2e)), hence a relative error of ~1e-6
    np.testing.assert_allclose(got, v.astype(np.float16).astype(np.float32), rtol=1e-5, atol=0)


def test_identical_keys_give_mean(torch_dev):
    q, k, v = make_inputs(1, 2, 333, 64, seed=12)
    k[:] = k[:, :, :1]
    assert_parity(run_gpu(torch_dev, q, k, v),
                  np.broadcast_to(v.astype(np.float64).mean(axis=2, keepdims=True), q.shape), "mean")


def test_joint_permutation(torch_dev):
    # permuting the keys and values together leaves the output unchanged:
    # both orders against the oracle, and against each other
    q, k, v = make_inputs(1, 2, 700, 72, seed=13)
    perm = np.random.Generator(np.random.PCG64(13)).permutation(700)
    kp, vp = np.ascontiguousarray(k[:, :, perm]), np.ascontiguousarray(v[:, :, perm])
    a = run_gpu(torch_dev, q, k, v)
    b = run_gpu(torch_dev, q, kp, vp)
    ref = oracle.forward(q, k, v)
    assert_parity(a, ref, "original order", rel_l2=2 * MAX_REL_L2)
    assert_parity(b, ref, "permuted keys", rel_l2=2 * MAX_REL_L2)
    assert_kernel_arithmetic(b, q, kp, vp, what="permuted keys")
    assert_parity(b, a.astype(np.float64), "permutation")


def test_deterministic(torch_dev):
    q, k, v = make_inputs(2, 4, 513, 64, seed=14)
    a = run_gpu(torch_dev, q, k, v)
    b = run_gpu(torch_dev, q, k, v)
    np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("d,n", [(64, 200), (72, 129), (17, 130)])
def test_no_store_past_the_last_patch(torch_dev, d, n):
    # out is a view followed by sentinel memory: rows >= n must stay untouched
    torch, dev = torch_dev
    q, k, v = make_inputs(1, 1, n, d, seed=15)
    buf = torch.full((n * d + 4096,), 12345.0, device=dev)
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, v))
    vef.forward_raw(qd.data_ptr(), kd.data_ptr(), vd.data_ptr(), buf.data_ptr(), 1, 1, n, d,
                    torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize(dev)
    host = buf.cpu().numpy()
    assert np.all(host[n * d:] == 12345.0)
    assert_parity(host[:n * d].reshape(1, 1, n, d), oracle.forward(q, k, v), "sentinel")


def test_unaligned_pointers_take_the_plain_load_path(torch_dev):
    # 4-byte but not 16-byte aligned bases: TMA cannot be used
    torch, dev = torch_dev
    shape = (1, 2, 257, 64)
    q, k, v = make_inputs(*shape, seed=16)
    numel = q.size
    ts = []
    for x in (q, k, v):
        t = torch.zeros(numel + 1, device=dev)
        t[1:] = torch.from_numpy(x.ravel()).to(dev)
        ts.append(t)
    out = torch.zeros(numel + 1, device=dev)
    vef.forward_raw(ts[0].data_ptr() + 4, ts[1].data_ptr() + 4, ts[2].data_ptr() + 4,
                    out.data_ptr() + 4, *shape, torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize(dev)
    got = out[1:].cpu().numpy().reshape(shape)
    assert_parity(got, oracle.forward(q, k, v), "unaligned")


def test_side_stream_and_empty(torch_dev):
    torch, dev = torch_dev
    q, k, v = make_inputs(1, 2, 300, 32, seed=17)
    s = torch.cuda.Stream(dev)
    with torch.cuda.stream(s):
        qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, v))
        out = vef.forward(qd, kd, vd, stream=s)
    s.synchronize()
    assert_parity(out.cpu().numpy(), oracle.forward(q, k, v), "side stream")
    z = torch.zeros(0, 2, 5, 8, device=dev)
    assert vef.forward(z, z, z).shape == z.shape
    z = torch.zeros(1, 2, 0, 8, device=dev)
    assert vef.forward(z, z, z).shape == z.shape


def test_host_tensors_round_trip(torch_dev):
    torch, _ = torch_dev
    q, k, v = make_inputs(1, 2, 130, 64, seed=18)
    pin = lambda x: torch.from_numpy(x).pin_memory()
    out = vef.forward(pin(q), pin(k), pin(v))
    assert out.device.type == "cpu"
    assert_parity(out.numpy(), oracle.forward(q, k, v), "host tensors")


# The direct f32 path (one kernel that rounds q, k, v to f16 in shared
# memory): 128 < n_patches <= 2048 (past 1536 only for up to two rounds of
# work tiles), head_dim 33..64 and a multiple of 4, 16-byte aligned inputs.
# Ragged ends, the 2048 limit, and enough heads that every block takes
# several work tiles (40 heads x 4 query blocks > 152).
DIRECT = [(1, 3, n, d) for d in (36, 44, 52, 64) for n in (129, 255, 256, 257, 1000, 2048)]
DIRECT += [(2, 40, 1000, 64), (1, 160, 300, 40)]


def run_gpu_offset(torch_dev, q, k, v, offset_elems):
    """vattn_forward with every tensor starting offset_elems f32 past a
    fresh allocation (offset 1: 4-byte aligned only, which takes the
    two-kernel path)."""
    torch, dev = torch_dev
    numel = q.size
    ts = []
    for x in (q, k, v):
        t = torch.zeros(numel + 4, device=dev)
        t[offset_elems:offset_elems + numel] = torch.from_numpy(x.ravel()).to(dev)
        ts.append(t)
    out = torch.zeros(numel + 4, device=dev)
    vef.forward_raw(ts[0].data_ptr() + 4 * offset_elems, ts[1].data_ptr() + 4 * offset_elems,
                    ts[2].data_ptr() + 4 * offset_elems, out.data_ptr() + 4 * offset_elems,
                    *q.shape, torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    return out[offset_elems:offset_elems + numel].cpu().numpy().reshape(q.shape)


@pytest.mark.parametrize("shape", DIRECT)
def test_direct_f32_path(torch_dev, shape):
    q, k, v = make_inputs(*shape, seed=5000 + 13 * shape[3] + shape[2] + shape[1])
    got = run_gpu(torch_dev, q, k, v)
    # every output element against the oracle
    assert_kernel_arithmetic(got, q, k, v, what=f"direct {shape}")
    assert_parity(got, oracle.forward(q, k, v), f"direct {shape}", rel_l2=2 * MAX_REL_L2)


@pytest.mark.parametrize("shape", [(1, 3, 1000, 64), (2, 40, 1000, 64), (1, 2, 2048, 48),
                                   (1, 2, 129, 36)])
def test_direct_and_staged_paths_agree_bitwise(torch_dev, shape):
    # the same rounding (f32 -> f16, nearest even) and the same attention
    # kernel arithmetic on both paths: identical bits
    q, k, v = make_inputs(*shape, seed=5100 + shape[2])
    direct = run_gpu_offset(torch_dev, q, k, v, 4)   # 16-byte aligned: one kernel
    staged = run_gpu_offset(torch_dev, q, k, v, 1)   # 4-byte aligned: staging + attention
    assert np.array_equal(direct.view(np.uint32), staged.view(np.uint32))


@pytest.mark.parametrize("n", [2048, 2049])
def test_direct_path_limit(torch_dev, n):
    # one head: 2048 patches take the direct kernel, 2049 the single kernel
    q, k, v = make_inputs(1, 1, n, 64, seed=5200 + n)
    assert _lib.forward_mode_for(1, 1, n, 64, 1, 1, 1, 152) == (
        _lib.MODE_DIRECT if n == 2048 else _lib.MODE_SINGLE_KERNEL)
    got = run_gpu(torch_dev, q, k, v)
    assert_parity(got, oracle.forward(q, k, v), f"limit N={n}", rel_l2=2 * MAX_REL_L2)


def run_gpu_offsets(torch_dev, q, k, v, offsets):
    """vattn_forward with q, k, v (and out) starting offsets[i] f32 elements
    past fresh allocations."""
    torch, dev = torch_dev
    numel = q.size
    ptrs, keep = [], []
    for x, off in zip((q, k, v), offsets):
        t = torch.zeros(numel + 4, device=dev)
        t[off:off + numel] = torch.from_numpy(x.ravel()).to(dev)
        keep.append(t)
        ptrs.append(t.data_ptr() + 4 * off)
    out = torch.zeros(numel + 4, device=dev)
    vef.forward_raw(*ptrs, out.data_ptr() + 16, *q.shape, torch.cuda.current_stream(dev).cuda_stream)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    return out[4:4 + numel].cpu().numpy().reshape(q.shape)


# Shapes past the direct path's 2048 patches with head_dim <= 64 and a
# multiple of 4 (and head_dim 20 from 129 patches): with q, k, v 16-byte
# aligned, one cooperative kernel that writes the f16 copies of k and v
# itself and rounds q; ragged last key tiles, a grid smaller than the GPU
# (2 heads) and several rounds of work tiles per block (80 heads).
STAGED = [(1, 2, 2049, 64), (1, 2, 2300, 36), (1, 3, 2500, 20), (2, 40, 2176, 64)]


@pytest.mark.parametrize("shape", STAGED)
def test_single_kernel_staging_path(torch_dev, shape):
    q, k, v = make_inputs(*shape, seed=5300 + shape[2] + shape[3])
    got = run_gpu(torch_dev, q, k, v)
    # every output element against the oracle
    assert_kernel_arithmetic(got, q, k, v, what=f"q f32 {shape}")
    assert_parity(got, oracle.forward(q, k, v), f"q f32 {shape}", rel_l2=2 * MAX_REL_L2)


@pytest.mark.parametrize("shape", [(1, 2, 2049, 64), (2, 40, 2176, 64), (1, 3, 2500, 20)])
def test_single_kernel_and_two_kernel_modes_agree_bitwise(torch_dev, shape):
    # all 16-byte aligned: the single kernel (k, v staged inside, q rounded
    # in it); q 4-byte aligned only: staging of q, k, v then the attention
    # kernel; k 4-byte aligned only: staging of k, v then the attention
    # kernel that rounds q.  The same rounding every way: identical bits.
    q, k, v = make_inputs(*shape, seed=5400 + shape[2])
    a = run_gpu_offsets(torch_dev, q, k, v, (4, 4, 4))
    b = run_gpu_offsets(torch_dev, q, k, v, (1, 4, 4))
    c = run_gpu_offsets(torch_dev, q, k, v, (4, 1, 4))
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    assert np.array_equal(a.view(np.uint32), c.view(np.uint32))

"""GPU parity of the accurate mode (vattn_forward_accurate) against the f64
oracle, through the C ABI.

The shader vision_attention_flash_sub_hpd_f16 (rullama 0.1.0) names, in its
header comment, a "sub" sibling that keeps q, k, v and the scores in f32
workgroup storage.  The accurate mode reaches that accuracy on the tensor
cores: x = hi + lo with hi = f16(x), lo = f16(x - hi), three f16 products per
matrix product (the lo x lo terms dropped), f32 accumulation.

Error model, with u = 2^-24 (f32 unit roundoff):

* each operand is represented to |x - hi - lo| <= 4u|x| + 2^-25 (two f16
  roundings; the constant is the f16 subnormal floor of lo), and the dropped
  lo x lo term is below 4u|q_d||k_d|, so a score s = q.k carries about
  12u * sum_d |q_d k_d| from the split plus the f32 accumulation of 3D
  products, whose rounding errors add like a random walk:
  ~ sqrt(3D) u * sum_d |q_d k_d|.  For the seeded inputs (q ~ N(0, 1/D),
  k, v ~ N(0, 1)) sum_d |q_d k_d| ~ 0.64 sqrt(D), so a score is off by
  ~1e-6 at D = 64;
* the softmax weights (ex2 approximation, ~2u relative; f32 running sums)
  and their own hi + lo split add a few u relative;
* an output is a convex combination of v rows, so it moves by at most
  max|v - out| (~2 max|v|) times the score error;
* the accumulator O = sum_j p_j v_j takes one tensor-core product per 16
  keys, n_patches / 16 accumulations into f32.  If an accumulation does not
  round to nearest but truncates, it loses at most one f32 ulp of the
  running sum, 2u relative, and those losses share a sign, so they add up:
  at most (n_patches / 16) * 2u relative over the whole sum.  (Measured, the
  rel L2 error does grow linearly in n_patches, at about half that worst
  case: 4.5e-7, 1.3e-6, 3.9e-6, 1.5e-5 at n_patches 64, 256, 1024, 4100.)

The bars are max abs <= 5e-5 and rel L2 <= 1e-5 + (n_patches / 16) * 2u:
the score and weight model's few 1e-6 with a tenfold margin, plus the
worst-case truncation term of the O accumulation.  At n_patches <= 1024 that is under 2e-5, fifty times tighter than the
f16 path's acceptance bar (3e-3, 1e-3).  A second check pins the mode
against the f16 path itself: on the same inputs its rel L2 error is at least
ten times smaller.
"""
import numpy as np
import pytest

import oracle
import vision_encoder_flash_gb300 as vef
from vattn_inputs import WORKLOADS, make_inputs, workload_inputs

pytestmark = pytest.mark.gpu

MAX_ABS = 5e-5


def max_rel_l2(n_patches):
    return 1e-5 + n_patches / 16 * 2.0 ** -23


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


def run_accurate(torch_dev, q, k, v):
    torch, dev = torch_dev
    out = vef.forward_accurate(*(torch.from_numpy(x).to(dev) for x in (q, k, v)))
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    return out.cpu().numpy()


def run_f16_path(torch_dev, q, k, v):
    torch, dev = torch_dev
    out = vef.forward(*(torch.from_numpy(x).to(dev) for x in (q, k, v)))
    torch.cuda.synchronize(dev)
    return out.cpu().numpy()


def errors(got, ref):
    diff = got.astype(np.float64) - ref
    return float(np.abs(diff).max()), float(np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300))


def assert_accurate(got, ref, what, n_patches):
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    mx, rel = errors(got, ref)
    bar = max_rel_l2(n_patches)
    assert mx <= MAX_ABS and rel <= bar, \
        f"{what}: max abs {mx:.3e}, rel L2 {rel:.3e} (bar {bar:.3e})"
    return mx, rel


# head_dim 1..128: non-multiples of 4 and 8 (plain loads in the split
# staging), of 16 (zero-padded columns) and of 64 (two column blocks);
# n_patches 1, tile edges and a ragged tail over several key tiles
SMALL = [(d, n) for d in (1, 8, 17, 64) for n in (1, 127, 129, 300)]
SMALL += [(d, n) for d in (65, 72, 128) for n in (1, 128, 385)]


@pytest.mark.parametrize("d,n", SMALL)
def test_small_shapes(torch_dev, d, n):
    q, k, v = make_inputs(2, 3, n, d, seed=7000 + 7 * d + n)
    assert_accurate(run_accurate(torch_dev, q, k, v), oracle.forward(q, k, v), f"D={d} N={n}", n)


@pytest.mark.parametrize("idx", [1, 2, 3, 4])
def test_workload_full(torch_dev, idx):
    q, k, v = workload_inputs(idx)
    mx, rel = assert_accurate(run_accurate(torch_dev, q, k, v), oracle.forward(q, k, v),
                              WORKLOADS[idx].name, q.shape[2])
    print(f"{WORKLOADS[idx].name} accurate: max abs {mx:.3e} rel L2 {rel:.3e}")


def test_workload_5_full(torch_dev):
    q, k, v = workload_inputs(5)
    mx, rel = assert_accurate(run_accurate(torch_dev, q, k, v), oracle.forward(q, k, v),
                              WORKLOADS[5].name, q.shape[2])
    print(f"{WORKLOADS[5].name} accurate: max abs {mx:.3e} rel L2 {rel:.3e}")


@pytest.mark.parametrize("idx", [2, 4])
def test_far_more_accurate_than_the_f16_path(torch_dev, idx):
    q, k, v = workload_inputs(idx)
    ref = oracle.forward(q, k, v)
    _, rel_acc = errors(run_accurate(torch_dev, q, k, v), ref)
    _, rel_f16 = errors(run_f16_path(torch_dev, q, k, v), ref)
    assert rel_acc * 10 <= rel_f16, f"accurate {rel_acc:.3e} vs f16 path {rel_f16:.3e}"
    print(f"{WORKLOADS[idx].name}: rel L2 accurate {rel_acc:.3e}, f16 path {rel_f16:.3e}")


@pytest.mark.parametrize("order", ["increasing", "shuffled"])
def test_running_max_rescale_paths(torch_dev, order):
    # scores 40 j / 512 with the row max rising by 10 per key tile in the
    # increasing order (an O rescale on every tile); q, k are exact in f16,
    # so only the softmax-weight split and the f32 arithmetic remain
    N, D = 1024, 64
    j = np.arange(N)
    if order == "shuffled":
        j = np.random.Generator(np.random.PCG64(31)).permutation(N)
    q = np.zeros((1, 2, N, D), np.float32)
    q[..., 0] = 40.0
    q[:, 1, :, 0] = np.linspace(-40, 40, N, dtype=np.float32)
    k = np.zeros((1, 2, N, D), np.float32)
    k[..., 0] = (j / 512.0).astype(np.float32)
    v = make_inputs(1, 2, N, D, seed=78)[2]
    assert_accurate(run_accurate(torch_dev, q, k, v), oracle.forward(q, k, v), order, N)


def test_inputs_that_f16_cannot_hold(torch_dev):
    # q, k, v on a 2^-16 grid around 1 and with 20-bit significands: the f16
    # path loses the low bits of every operand, the accurate mode keeps them
    rng = np.random.Generator(np.random.PCG64(91))
    shape = (1, 2, 200, 64)
    q = (1.0 + rng.integers(0, 2 ** 20, shape) * 2.0 ** -20).astype(np.float32) / 8.0
    k = (rng.standard_normal(shape) * (1 + 2.0 ** -13)).astype(np.float32)
    v = (1000.0 + rng.integers(0, 2 ** 16, shape) * 2.0 ** -16).astype(np.float32)
    ref = oracle.forward(q, k, v)
    got = run_accurate(torch_dev, q, k, v)
    # outputs near 1000: hold the accurate mode to the same relative bar
    mx, rel = errors(got, ref)
    assert rel <= max_rel_l2(200) and mx <= MAX_ABS * 1000.0, f"max abs {mx:.3e}, rel L2 {rel:.3e}"


def test_unaligned_pointers_take_the_plain_load_path(torch_dev):
    torch, dev = torch_dev
    q, k, v = make_inputs(1, 2, 150, 64, seed=92)
    n = q.size
    bufs = []
    for x in (q, k, v):
        b = torch.zeros(n + 1, dtype=torch.float32, device=dev)
        b[1:] = torch.from_numpy(x.reshape(-1)).to(dev)
        bufs.append(b[1:].view(q.shape))  # 4-byte but not 16-byte aligned
    assert bufs[0].data_ptr() % 16 != 0
    out = vef.forward_accurate(*bufs)
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    assert_accurate(out.cpu().numpy(), oracle.forward(q, k, v), "unaligned", 150)


def test_deterministic_and_stream(torch_dev):
    torch, dev = torch_dev
    q, k, v = make_inputs(2, 4, 333, 72, seed=93)
    qd, kd, vd = (torch.from_numpy(x).to(dev) for x in (q, k, v))
    side = torch.cuda.Stream(dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        a = vef.forward_accurate(qd, kd, vd, stream=side)
        b = vef.forward_accurate(qd, kd, vd, stream=side)
    side.synchronize()
    assert vef.device_status() == 0
    assert torch.equal(a, b)
    assert_accurate(a.cpu().numpy(), oracle.forward(q, k, v), "side stream", 333)


def test_empty_problems(torch_dev):
    torch, dev = torch_dev
    for shape in ((0, 2, 5, 8), (1, 2, 0, 8)):
        x = torch.zeros(shape, device=dev)
        assert vef.forward_accurate(x, x, x).shape == shape

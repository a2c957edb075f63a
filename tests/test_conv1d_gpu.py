"""GPU parity of the depthwise conv1d rolling-buffer step (vattn_conv1d_step)
against the f64 oracle (oracle.conv1d), through the C ABI.

Bars:

* the updated buffer is bit-identical to the oracle's (the step only moves
  f32 values);
* each output is a chain of d_conv + 1 fused multiply-adds from 0, each
  rounding once in f32, so |gpu - oracle| <= gamma_n * sum_k |term_k| with
  n = d_conv + 1, gamma_n = n u / (1 - n u), u = 2^-24 (the classical bound
  for recursive summation of exact products; an FMA's product is exact).
"""
import numpy as np
import pytest

import vision_encoder_flash_gb300 as vef
from oracle import conv1d as oconv
from vattn_inputs import CONV1D_WORKLOAD, conv1d_inputs, conv1d_workload_name

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


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


def bound(x, buf, w):
    """gamma_{d_conv+1} * sum_k |term_k| per output, f64."""
    d_conv = buf.shape[-2]
    x64, b64, w64 = (a.astype(np.float64) for a in (x, buf, w))
    s = np.abs(x64 * w64[:, d_conv])
    for k in range(d_conv):
        s = s + np.abs(b64[..., k, :] * w64[:, k])
    n = d_conv + 1
    return n * U / (1 - n * U) * s


def check_step(got_out, got_buf, x, buf, w, what):
    ref_out, ref_buf = oconv.conv1d_step(x, buf, w)
    np.testing.assert_array_equal(got_buf.astype(np.float64), ref_buf, err_msg=f"{what}: buffer")
    err = np.abs(got_out.astype(np.float64) - ref_out)
    lim = bound(x, buf, w)
    bad = err > lim
    assert not bad.any(), f"{what}: {int(bad.sum())} outputs past the bound, worst {float((err - lim).max()):.3e}"


def gpu_step(torch_dev, x, buf, w):
    torch, dev = torch_dev
    xd, bd, wd = (torch.from_numpy(np.ascontiguousarray(a)).to(dev) for a in (x, buf, w))
    out = vef.conv1d_step(xd, bd, wd)
    torch.cuda.synchronize(dev)
    return out.cpu().numpy(), bd.cpu().numpy()


# (batch, hidden, kernel_size, d_conv): the 16-byte path (hidden % 4 == 0,
# d_conv <= 8) and the per-channel path (other hidden, d_conv > 8)
CASES = [
    (1, 1, 1, 0), (1, 8, 1, 0), (1, 5, 3, 2), (3, 4, 3, 2), (2, 64, 4, 3), (3, 256, 6, 3),
    (4, 96, 2, 1), (2, 40, 5, 4), (2, 48, 6, 5), (2, 32, 7, 6), (2, 36, 8, 7), (5, 4096, 9, 8),
    (7, 4099, 5, 4), (2, 128, 12, 11), (1, 2048, 3, 2), (300, 20, 3, 2),
]


@pytest.mark.parametrize("batch,hidden,kernel_size,d_conv", CASES)
def test_step_matches_oracle(torch_dev, batch, hidden, kernel_size, d_conv):
    x, buf, w = conv1d_inputs(batch, hidden, kernel_size, d_conv,
                              seed=9000 + batch + hidden + 13 * d_conv + kernel_size)
    out, nb = gpu_step(torch_dev, x, buf, w)
    check_step(out, nb, x, buf, w, f"B={batch} H={hidden} K={kernel_size} dc={d_conv}")


def test_the_pages_single_sequence_form(torch_dev):
    torch, dev = torch_dev
    x, buf, w = conv1d_inputs(1, 1024, 4, 3, seed=9100)
    xd = torch.from_numpy(x[0]).to(dev)              # [hidden]
    bd = torch.from_numpy(buf[0].copy()).to(dev)     # [d_conv, hidden]
    out = vef.conv1d_step(xd, bd, torch.from_numpy(w).to(dev))
    torch.cuda.synchronize(dev)
    assert out.shape == (1024,)
    check_step(out.cpu().numpy()[None], bd.cpu().numpy()[None], x, buf, w, "single sequence")


def test_many_steps_keep_the_buffer_exact(torch_dev):
    torch, dev = torch_dev
    B, H, K, DC, T = 6, 200, 4, 3, 16
    _, buf, w = conv1d_inputs(B, H, K, DC, seed=9200)
    xs = np.random.Generator(np.random.PCG64(9201)).standard_normal((T, B, H)).astype(np.float32)
    bd = torch.from_numpy(buf.copy()).to(dev)
    wd = torch.from_numpy(w).to(dev)
    ref_buf = buf.astype(np.float64)
    for t in range(T):
        out = vef.conv1d_step(torch.from_numpy(xs[t]).to(dev), bd, wd)
        torch.cuda.synchronize(dev)
        ref_out, new_ref = oconv.conv1d_step(xs[t], ref_buf, w)
        err = np.abs(out.cpu().numpy().astype(np.float64) - ref_out)
        assert (err <= bound(xs[t], ref_buf.astype(np.float32), w)).all(), f"step {t}"
        ref_buf = new_ref
        np.testing.assert_array_equal(bd.cpu().numpy().astype(np.float64), ref_buf)
    np.testing.assert_array_equal(bd.cpu().numpy(), xs[T - DC:].transpose(1, 0, 2))


def test_unaligned_pointers_take_the_per_channel_path(torch_dev):
    torch, dev = torch_dev
    B, H, K, DC = 3, 64, 4, 3
    x, buf, w = conv1d_inputs(B, H, K, DC, seed=9300)

    def shifted(a):
        t = torch.zeros(a.size + 1, dtype=torch.float32, device=dev)
        t[1:] = torch.from_numpy(a.reshape(-1)).to(dev)
        return t[1:].view(a.shape)

    xd, bd, wd = shifted(x), shifted(buf), shifted(w)
    od = shifted(np.zeros_like(x))
    assert xd.data_ptr() % 16 != 0
    vef.conv1d_step(xd, bd, wd, out=od)
    torch.cuda.synchronize(dev)
    check_step(od.cpu().numpy(), bd.cpu().numpy(), x, buf, w, "unaligned")


def test_no_buffer_slots_and_empty(torch_dev):
    torch, dev = torch_dev
    x, buf, w = conv1d_inputs(4, 16, 1, 0, seed=9400)
    out, nb = gpu_step(torch_dev, x, buf, w)
    np.testing.assert_array_equal(out, x * w[:, 0])  # one rounding of an exact product
    assert nb.shape == (4, 0, 16)
    e = torch.zeros(0, 16, device=dev)
    assert vef.conv1d_step(e, torch.zeros(0, 2, 16, device=dev), torch.zeros(16, 3, device=dev)).shape == (0, 16)


def test_workload_full(torch_dev):
    wl = CONV1D_WORKLOAD
    x, buf, w = conv1d_inputs(wl["batch"], wl["hidden"], wl["kernel_size"], wl["d_conv"], wl["seed"])
    out, nb = gpu_step(torch_dev, x, buf, w)
    check_step(out, nb, x, buf, w, conv1d_workload_name())

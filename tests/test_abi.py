"""The C-ABI library loads, exports every entry point of include/vattn.h, and
rejects bad arguments on the host before touching CUDA (no GPU needed)."""
import ctypes
import subprocess

import pytest

import vision_encoder_flash_gb300 as vef
from vision_encoder_flash_gb300 import _lib


@pytest.fixture(scope="module")
def lib():
    from vision_encoder_flash_gb300 import build
    build.build()
    return vef.load_library()


def test_exports_every_declared_symbol(lib):
    names = _lib.exported_symbols()
    assert set(names) == {"vattn_forward", "vattn_forward_f16", "vattn_forward_f16io",
                          "vattn_forward_f32q",
                          "vattn_forward_noalloc", "vattn_forward_accurate",
                          "vattn_conv1d_step", "vattn_forward_host",
                          "vattn_selftest_wait_timeout",
                          "vattn_rope_neox", "vattn_forward_rope",
                          "vattn_device_status", "vattn_status_string",
                          "vattn_last_error_string", "vattn_version",
                          "vattn_forward_mode", "vattn_forward_mode_for",
                          "vattn_set_single_kernel", "vattn_set_split_tiles", "vattn_cut_plan_for"}
    for name in names:
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.lib_path()], capture_output=True,
                         text=True, check=True).stdout
    for name in names:
        assert f" T {name}\n" in out, name


def test_library_does_not_link_the_driver():
    out = subprocess.run(["ldd", _lib.lib_path()], capture_output=True, text=True).stdout
    assert "libcuda.so" not in out


def test_status_strings(lib):
    assert vef.status_string(0) == "VATTN_OK"
    assert vef.status_string(5) == "VATTN_ERR_DEVICE_TIMEOUT"
    assert vef.version() == 100


FAKE = 0x10000  # never dereferenced: every case below fails before any CUDA call


@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, -1, 2, 3, 4), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, -3, 4), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 0), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 129), 2),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 4096), 2),
    ((0, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 4), 1),
    ((FAKE, FAKE, FAKE, 0, 1, 2, 3, 4), 1),
    ((FAKE + 2, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 4), 3),
    ((FAKE, FAKE, FAKE, FAKE + 4, 1, 2, 3, 4), 1),            # out overlaps q
    ((FAKE, FAKE, FAKE, FAKE, 1, 1, 2 ** 31, 4), 2),           # n_patches past 32 bits
])
def test_host_side_argument_errors(lib, args, status):
    assert _lib.forward_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""
    # the allocation-free entry point applies the same checks
    assert _lib.forward_noalloc_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""
    # and so does the accurate (split-f16) one
    assert _lib.forward_accurate_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""
    # and the host-buffer one
    assert _lib.forward_host_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""


@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, -1, 2, 3, 8), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 0), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 136), 2),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 12), 2),      # head_dim % 8 != 0
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 1), 2),
    ((0, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 8), 1),
    ((FAKE + 8, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 8), 3),  # f16 inputs need 16 bytes
    ((FAKE, FAKE, FAKE + 2, FAKE + 2 ** 30, 1, 2, 3, 8), 3),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30 + 2, 1, 2, 3, 8), 3),
    # out (f32, 2x the bytes) overlaps v: v's 96 bytes start 64 bytes after out
    ((FAKE + 2 ** 20, FAKE + 2 ** 21, FAKE + 64, FAKE, 1, 2, 3, 8), 1),
    ((FAKE, FAKE, FAKE, FAKE, 1, 1, 2 ** 31, 8), 2),
])
def test_f16_entry_host_side_argument_errors(lib, args, status):
    assert _lib.forward_f16_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""


@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, -1, 2, 200, 64), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 200, 0), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 200, 72), 2),    # head_dim > 64
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 200, 36), 2),    # head_dim % 8 != 0
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 128, 64), 2),    # one query tile
    ((0, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 200, 64), 1),
    ((FAKE + 8, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 200, 64), 3),  # q needs 16 bytes
    ((FAKE, FAKE + 2 ** 24 + 2, FAKE, FAKE + 2 ** 30, 1, 2, 200, 64), 3),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30 + 2, 1, 2, 200, 64), 3),
    ((FAKE, FAKE + 2 ** 24, FAKE + 2 ** 25, FAKE + 64, 1, 2, 200, 64), 1),  # out overlaps q
    ((FAKE, FAKE, FAKE, FAKE, 1, 1, 2 ** 31, 64), 2),
])
def test_f32q_entry_host_side_argument_errors(lib, args, status):
    assert _lib.forward_f32q_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""


@pytest.mark.parametrize("b,h,n", [(0, 4, 10), (2, 0, 10), (2, 4, 0)])
def test_f32q_entry_empty_problems_are_no_ops(lib, b, h, n):
    assert _lib.forward_f32q_status(0, 0, 0, 0, b, h, n, 64, 0) == 0


def test_f32q_binding_rejects_bad_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 2, 300, 64)
    kv = q.half()
    with pytest.raises(TypeError):
        vef.forward_f32q(kv, kv, kv)   # q must be float32
    with pytest.raises(TypeError):
        vef.forward_f32q(q, q, kv)     # k must be float16
    with pytest.raises(ValueError):
        vef.forward_f32q(q, kv, kv)    # CPU tensors


@pytest.mark.parametrize("b,h,n", [(0, 4, 10), (2, 0, 10), (2, 4, 0)])
def test_f16_entry_empty_problems_are_no_ops(lib, b, h, n):
    assert _lib.forward_f16_status(0, 0, 0, 0, b, h, n, 64, 0) == 0


def test_f16_binding_rejects_bad_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 2, 3, 8, dtype=torch.float16)
    with pytest.raises(TypeError):
        vef.forward_f16(q.float(), q, q)
    with pytest.raises(ValueError):
        vef.forward_f16(q, q, q)  # CPU tensors


# f16 staging of 1 x 1 x n x 16: 3 x round_up(n * 32, 256) bytes against the
# 32 MiB scratch (VATTN_NOALLOC_MAX_SCRATCH_BYTES)
NOALLOC_MAX_N16 = 32 * 1024 * 1024 // 3 // 256 * 256 // 32


@pytest.mark.parametrize("b,h,n,d", [
    (1, 1, NOALLOC_MAX_N16 + 1, 16),
    (8, 16, 2304, 64),
    (1, 64, 1024, 128),
])
def test_noalloc_rejects_problems_past_its_scratch_on_the_host(lib, b, h, n, d):
    assert _lib.forward_noalloc_status(FAKE, FAKE, FAKE, FAKE + 2 ** 40, b, h, n, d, 0) == 2
    text = lib.vattn_last_error_string().decode()
    assert "scratch" in text and "vattn_forward" in text


@pytest.mark.parametrize("b,h,n", [(0, 4, 10), (2, 0, 10), (2, 4, 0)])
def test_empty_problems_are_no_ops_even_with_null_pointers(lib, b, h, n):
    assert _lib.forward_status(0, 0, 0, 0, b, h, n, 64, 0) == 0
    assert _lib.forward_noalloc_status(0, 0, 0, 0, b, h, n, 64, 0) == 0
    assert _lib.forward_accurate_status(0, 0, 0, 0, b, h, n, 64, 0) == 0
    assert _lib.forward_host_status(0, 0, 0, 0, b, h, n, 64, 0) == 0


B4 = FAKE + 2 ** 24   # buffer
W4 = FAKE + 2 ** 28   # weight
O4 = FAKE + 2 ** 32   # output


@pytest.mark.parametrize("args,status", [
    ((FAKE, B4, W4, O4, -1, 8, 3, 2), 1),
    ((FAKE, B4, W4, O4, 1, -8, 3, 2), 1),
    ((FAKE, B4, W4, O4, 1, 8, 3, -1), 1),
    ((FAKE, B4, W4, O4, 1, 8, 2, 2), 1),          # kernel_size < d_conv + 1
    ((FAKE, B4, W4, O4, 1, 8, 0, 0), 1),          # kernel_size 0: no input tap
    ((0, B4, W4, O4, 1, 8, 3, 2), 1),
    ((FAKE, 0, W4, O4, 1, 8, 3, 2), 1),           # buffer needed when d_conv > 0
    ((FAKE, B4, 0, O4, 1, 8, 3, 2), 1),
    ((FAKE, B4, W4, 0, 1, 8, 3, 2), 1),
    ((FAKE + 2, B4, W4, O4, 1, 8, 3, 2), 3),
    ((FAKE, B4 + 1, W4, O4, 1, 8, 3, 2), 3),
    ((FAKE, B4, W4, FAKE + 16, 1, 8, 3, 2), 1),   # output overlaps input
    ((FAKE, B4, W4, B4 + 32, 1, 8, 3, 2), 1),     # output overlaps buffer
    ((FAKE, B4, W4, W4, 1, 8, 3, 2), 1),          # output overlaps weight
    ((FAKE, FAKE + 8, W4, O4, 1, 8, 3, 2), 1),    # buffer overlaps input
    ((FAKE, B4, B4 + 60, O4, 1, 8, 3, 2), 1),     # buffer (64 B) overlaps weight
    ((FAKE, B4, W4, O4, 1, 2 ** 31, 3, 2), 2),
    ((FAKE, B4, W4, O4, 2 ** 62, 2 ** 20, 3, 2), 2),
])
def test_conv1d_host_side_argument_errors(lib, args, status):
    assert _lib.conv1d_step_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""


@pytest.mark.parametrize("b,h", [(0, 16), (3, 0)])
def test_conv1d_empty_problems_are_no_ops(lib, b, h):
    assert _lib.conv1d_step_status(0, 0, 0, 0, b, h, 4, 3, 0) == 0


def test_conv1d_without_buffer_slots_needs_no_buffer(lib):
    # d_conv == 0 accepts a NULL buffer; this still fails later only for the
    # missing input, before any CUDA call
    assert _lib.conv1d_step_status(0, 0, W4, O4, 1, 8, 1, 0, 0) == 1
    assert "null" in lib.vattn_last_error_string().decode()


def test_python_binding_rejects_bad_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 2, 3, 4)
    with pytest.raises(TypeError):
        vef.forward(q.double(), q, q)
    with pytest.raises(ValueError):
        vef.forward(q, q[:, :1], q)
    with pytest.raises(ValueError):
        vef.forward(q[0], q[0], q[0])


def test_device_status_without_gpu_reports_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    code = ctypes.c_uint32(7)
    assert lib.vattn_device_status(ctypes.byref(code)) == 4
    assert code.value == 0


# vattn_rope_neox(x, B, H, N, D, rope_dims, pos0, base, factors, inverse)
@pytest.mark.parametrize("args,status", [
    ((FAKE, -1, 2, 3, 8, 8, 0, 1e4, 0, 0), 1),
    ((FAKE, 1, 2, 3, 0, 0, 0, 1e4, 0, 0), 1),           # head_dim 0
    ((FAKE, 1, 2, 3, 8, 10, 0, 1e4, 0, 0), 1),          # rope_dims > head_dim
    ((FAKE, 1, 2, 3, 8, -2, 0, 1e4, 0, 0), 1),
    ((FAKE, 1, 2, 3, 8, 8, 0, 0.0, 0, 0), 1),           # base must be > 0
    ((FAKE, 1, 2, 3, 8, 8, 0, -2.0, 0, 0), 1),
    ((FAKE, 1, 2, 3, 8, 8, 0, float("nan"), 0, 0), 1),
    ((FAKE, 1, 2, 3, 8, 8, 0, float("inf"), 0, 0), 1),
    ((FAKE, 1, 2, 3, 8, 8, -1, 1e4, 0, 0), 1),          # pos0 < 0
    ((FAKE, 1, 2, 3, 8, 8, 2 ** 24 - 2, 1e4, 0, 0), 2),  # last position past 2^24
    ((FAKE, 1, 2, 3, 8, 8, 0, 1e4, 0, 2), 1),           # inverse must be 0 or 1
    ((FAKE + 2, 1, 2, 3, 8, 8, 0, 1e4, 0, 0), 3),
    ((FAKE, 1, 2, 3, 8, 8, 0, 1e4, FAKE + 1, 0), 3),    # misaligned factors
    ((0, 1, 2, 3, 8, 8, 0, 1e4, 0, 0), 1),              # null x
])
def test_rope_host_side_argument_errors(lib, args, status):
    assert _lib.rope_neox_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""


@pytest.mark.parametrize("args", [
    (0, 0, 2, 3, 8, 8, 0, 1e4, 0, 0),       # no batch
    (0, 1, 2, 0, 8, 8, 0, 1e4, 0, 0),       # no patches
    (0, 1, 2, 3, 8, 0, 0, 1e4, 0, 0),       # rope_dims 0: nothing turns
    (0, 1, 2, 3, 8, 1, 0, 1e4, 0, 0),       # rope_dims 1: half = 0
])
def test_rope_no_ops_need_no_pointer(lib, args):
    assert _lib.rope_neox_status(*args, 0) == 0


# vattn_forward_rope(q, k, v, out, B, H, N, D, rope_dims, pos0, base, factors)
@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 8, 9, 0, 1e4, 0), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 8, 8, 0, -1.0, 0), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 8, 8, -5, 1e4, 0), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 136, 8, 0, 1e4, 0), 2),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 8, 8, 2 ** 24, 1e4, 0), 2),
    ((FAKE + 2, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 8, 8, 0, 1e4, 0), 3),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 8, 8, 0, 1e4, FAKE + 2), 3),
    ((FAKE, FAKE, FAKE, FAKE + 4, 1, 2, 3, 8, 8, 0, 1e4, 0), 1),   # out overlaps q
    ((FAKE, FAKE, FAKE, 0, 1, 2, 3, 8, 8, 0, 1e4, 0), 1),
])
def test_forward_rope_host_side_argument_errors(lib, args, status):
    assert _lib.forward_rope_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""


@pytest.mark.parametrize("args,status", [
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 12), 2),      # head_dim % 8 != 0
    ((FAKE + 8, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 8), 3),   # f16 inputs need 16 bytes
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30 + 1, 1, 2, 3, 8), 3),   # f16 out needs 2 bytes
    # f16 out (same bytes as an input) overlaps v: v starts 64 bytes after out
    ((FAKE + 2 ** 20, FAKE + 2 ** 21, FAKE + 64, FAKE, 1, 2, 3, 8), 1),
    ((FAKE, FAKE, FAKE, FAKE + 2 ** 30, 1, 2, 3, 136), 2),
])
def test_f16io_entry_host_side_argument_errors(lib, args, status):
    assert _lib.forward_f16io_status(*args, 0) == status
    assert lib.vattn_last_error_string().decode() != ""


def test_f16io_entry_out_may_sit_right_after_an_input(lib):
    """f16 out of 1 x 2 x 3 x 8 = 96 bytes starting where v's 96 bytes end is
    no overlap; the call gets past the host checks (no GPU: CUDA error 4)."""
    status = _lib.forward_f16io_status(FAKE, FAKE + 2 ** 20, FAKE + 2 ** 21,
                                       FAKE + 2 ** 21 + 96, 1, 2, 3, 8, 0)
    assert status in (0, 4)

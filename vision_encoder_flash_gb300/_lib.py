"""ctypes binding of libvattn.so: same entry points as include/vattn.h."""
from __future__ import annotations

import ctypes
import os
import re

_PKG = os.path.dirname(os.path.abspath(__file__))
_ROOT = os.path.dirname(_PKG)
HEADER = os.path.join(_ROOT, "include", "vattn.h")

_STATUS = {0: "VATTN_OK", 1: "VATTN_ERR_INVALID_ARG", 2: "VATTN_ERR_UNSUPPORTED",
           3: "VATTN_ERR_MISALIGNED", 4: "VATTN_ERR_CUDA", 5: "VATTN_ERR_DEVICE_TIMEOUT"}

_LIB = None


class VattnError(RuntimeError):
    def __init__(self, status: int, detail: str):
        self.status = status
        super().__init__(f"{_STATUS.get(status, status)}: {detail}")


def lib_path() -> str:
    return os.environ.get("VATTN_LIB", os.path.join(_PKG, "libvattn.so"))


def load_library():
    """Load libvattn.so (built by vision_encoder_flash_gb300/build.py); raises if absent."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = lib_path()
    if not os.path.exists(path):
        raise ImportError(f"{path} not found: build it with `python -c \"import __graft_entry__ as g; "
                          f"g.build()\"` (there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    vp, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.vattn_forward.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.vattn_forward.restype = ctypes.c_int
    f32 = ctypes.c_float
    lib.vattn_rope_neox.argtypes = [vp, i64, i64, i64, i64, i64, i64, f32, vp, ctypes.c_int, vp]
    lib.vattn_rope_neox.restype = ctypes.c_int
    lib.vattn_forward_rope.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f32, vp, vp]
    lib.vattn_forward_rope.restype = ctypes.c_int
    lib.vattn_forward_f16io.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.vattn_forward_f16io.restype = ctypes.c_int
    lib.vattn_forward_f16.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.vattn_forward_f16.restype = ctypes.c_int
    lib.vattn_forward_f32q.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.vattn_forward_f32q.restype = ctypes.c_int
    lib.vattn_forward_accurate.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.vattn_forward_accurate.restype = ctypes.c_int
    lib.vattn_conv1d_step.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.vattn_conv1d_step.restype = ctypes.c_int
    lib.vattn_forward_host.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.vattn_forward_host.restype = ctypes.c_int
    lib.vattn_forward_noalloc.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, vp]
    lib.vattn_forward_noalloc.restype = ctypes.c_int
    ip = ctypes.POINTER(ctypes.c_int)
    lib.vattn_forward_mode.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, ip]
    lib.vattn_forward_mode.restype = ctypes.c_int
    lib.vattn_forward_mode_for.argtypes = [i64, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ip]
    lib.vattn_forward_mode_for.restype = ctypes.c_int
    lib.vattn_set_single_kernel.argtypes = [ctypes.c_int]
    lib.vattn_set_single_kernel.restype = ctypes.c_int
    lib.vattn_set_split_tiles.argtypes = [ctypes.c_int]
    lib.vattn_set_split_tiles.restype = ctypes.c_int
    lib.vattn_cut_plan_for.argtypes = [i64, i64, i64, i64, ctypes.c_int, ctypes.POINTER(ctypes.c_int)]
    lib.vattn_cut_plan_for.restype = ctypes.c_int
    lib.vattn_selftest_wait_timeout.argtypes = [vp]
    lib.vattn_selftest_wait_timeout.restype = ctypes.c_int
    lib.vattn_device_status.argtypes = [ctypes.POINTER(ctypes.c_uint32)]
    lib.vattn_device_status.restype = ctypes.c_int
    lib.vattn_status_string.argtypes = [ctypes.c_int]
    lib.vattn_status_string.restype = ctypes.c_char_p
    lib.vattn_last_error_string.argtypes = []
    lib.vattn_last_error_string.restype = ctypes.c_char_p
    lib.vattn_version.argtypes = []
    lib.vattn_version.restype = ctypes.c_int
    _LIB = lib
    return lib


def _check(status: int):
    if status != 0:
        detail = load_library().vattn_last_error_string().decode(errors="replace")
        raise VattnError(status, detail)


def forward_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, batch: int, n_heads: int,
                n_patches: int, head_dim: int, stream: int = 0) -> None:
    """Direct call of vattn_forward with device addresses (ints) and a stream handle."""
    _check(load_library().vattn_forward(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches,
                                        head_dim, stream))


def forward_status(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches, head_dim,
                   stream=0) -> int:
    """Like forward_raw but returns the status code instead of raising."""
    return int(load_library().vattn_forward(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                            n_patches, head_dim, stream))


def forward_f16_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, batch: int, n_heads: int,
                    n_patches: int, head_dim: int, stream: int = 0) -> None:
    """Direct call of vattn_forward_f16: f16 q, k, v (device addresses), f32 out."""
    _check(load_library().vattn_forward_f16(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                            n_patches, head_dim, stream))


def forward_f16_status(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches, head_dim,
                       stream=0) -> int:
    """Like forward_f16_raw but returns the status code instead of raising."""
    return int(load_library().vattn_forward_f16(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                                n_patches, head_dim, stream))


def forward_f32q_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, batch: int, n_heads: int,
                     n_patches: int, head_dim: int, stream: int = 0) -> None:
    """Direct call of vattn_forward_f32q: f32 q, f16 k and v (device addresses), f32 out."""
    _check(load_library().vattn_forward_f32q(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                             n_patches, head_dim, stream))


def forward_f32q_status(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches, head_dim,
                        stream=0) -> int:
    """Like forward_f32q_raw but returns the status code instead of raising."""
    return int(load_library().vattn_forward_f32q(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                                 n_patches, head_dim, stream))


def forward_f16io_status(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches, head_dim,
                         stream=0) -> int:
    """vattn_forward_f16io with device addresses (f16 in, f16 out); returns the status."""
    return int(load_library().vattn_forward_f16io(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                                  n_patches, head_dim, stream))


def rope_neox_status(x_ptr, batch, n_heads, n_patches, head_dim, rope_dims, pos0, base,
                     factors_ptr, inverse, stream=0) -> int:
    """vattn_rope_neox with device addresses; returns the status code."""
    return int(load_library().vattn_rope_neox(x_ptr, batch, n_heads, n_patches, head_dim,
                                              rope_dims, pos0, base, factors_ptr, int(inverse),
                                              stream))


def forward_rope_status(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches, head_dim,
                        rope_dims, pos0, base, factors_ptr, stream=0) -> int:
    """vattn_forward_rope with device addresses; returns the status code."""
    return int(load_library().vattn_forward_rope(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                                 n_patches, head_dim, rope_dims, pos0, base,
                                                 factors_ptr, stream))


def forward_accurate_status(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches, head_dim,
                            stream=0) -> int:
    """vattn_forward_accurate (split-f16, about f32 accuracy) with device
    addresses; returns the status code."""
    return int(load_library().vattn_forward_accurate(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                                     n_patches, head_dim, stream))


def conv1d_step_status(input_ptr, buffer_ptr, weight_ptr, output_ptr, batch, hidden_size,
                       kernel_size, d_conv, stream=0) -> int:
    """vattn_conv1d_step with device addresses; returns the status code."""
    return int(load_library().vattn_conv1d_step(input_ptr, buffer_ptr, weight_ptr, output_ptr, batch,
                                                hidden_size, kernel_size, d_conv, stream))


def forward_host_status(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches, head_dim,
                        stream=0) -> int:
    """vattn_forward_host with HOST addresses (pipelined copies and kernels);
    returns the status code.  The result is ready once `stream` is synchronised."""
    return int(load_library().vattn_forward_host(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                                 n_patches, head_dim, stream))


def forward_noalloc_raw(q_ptr: int, k_ptr: int, v_ptr: int, out_ptr: int, batch: int,
                        n_heads: int, n_patches: int, head_dim: int, stream: int = 0) -> None:
    """Direct call of vattn_forward_noalloc: the allocation-free variant, for
    callers that may not allocate device memory while they run.  Its staging
    scratch is one fixed array per device, so calls that overlap in time race."""
    _check(load_library().vattn_forward_noalloc(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                                n_patches, head_dim, stream))


def forward_noalloc_status(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches, head_dim,
                           stream=0) -> int:
    """Like forward_noalloc_raw but returns the status code instead of raising."""
    return int(load_library().vattn_forward_noalloc(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                                    n_patches, head_dim, stream))


# vattn_mode values
MODE_NONE, MODE_DIRECT, MODE_SINGLE_KERNEL, MODE_TWO_KERNELS = 0, 1, 2, 3


def forward_mode(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads, n_patches, head_dim) -> int:
    """The kernel mode (MODE_*) vattn_forward takes for these device arguments
    on the current device (vattn_forward_mode); raises on argument errors."""
    mode = ctypes.c_int(-1)
    _check(load_library().vattn_forward_mode(q_ptr, k_ptr, v_ptr, out_ptr, batch, n_heads,
                                             n_patches, head_dim, ctypes.byref(mode)))
    return int(mode.value)


def forward_mode_for(batch, n_heads, n_patches, head_dim, aligned, cooperative_launch,
                     blocks_per_sm, n_sms) -> int:
    """The mode rule with the device facts passed in (vattn_forward_mode_for,
    no CUDA call; n_sms: the device's multiprocessors); raises on argument
    errors."""
    mode = ctypes.c_int(-1)
    _check(load_library().vattn_forward_mode_for(batch, n_heads, n_patches, head_dim, int(aligned),
                                                 int(cooperative_launch), int(blocks_per_sm),
                                                 int(n_sms), ctypes.byref(mode)))
    return int(mode.value)


def set_single_kernel(allow: bool) -> bool:
    """Allow or forbid the single cooperative kernel process-wide; returns the
    previous setting."""
    return bool(load_library().vattn_set_single_kernel(1 if allow else 0))


def set_split_tiles(allow) -> int:
    """Cut work tiles (balanced last round), process-wide: 0 / False never,
    1 / True where it pays (the default), 2 wherever it shortens the busiest
    block; returns the previous setting (0, 1 or 2)."""
    return int(load_library().vattn_set_split_tiles(int(allow)))


def cut_plan_for(batch: int, n_heads: int, n_patches: int, head_dim: int, n_blocks: int) -> bool:
    """Whether vattn_forward would cut work tiles for these sizes on a grid of
    n_blocks thread blocks, under the current setting (host only)."""
    cut = ctypes.c_int(0)
    _check(load_library().vattn_cut_plan_for(batch, n_heads, n_patches, head_dim, n_blocks,
                                              ctypes.byref(cut)))
    return cut.value != 0


def selftest_wait_timeout(stream: int = 0) -> None:
    """Launch the self-test kernel whose bounded wait runs out (about 2 s)."""
    _check(load_library().vattn_selftest_wait_timeout(stream))


def device_status() -> int:
    """Read-and-clear the kernel-side error word (synchronises the device)."""
    code = ctypes.c_uint32(0)
    status = load_library().vattn_device_status(ctypes.byref(code))
    if status not in (0, 5):
        _check(status)
    return int(code.value)


def status_string(status: int) -> str:
    return load_library().vattn_status_string(status).decode()


def version() -> int:
    return int(load_library().vattn_version())


def exported_symbols() -> list[str]:
    """Function names declared in include/vattn.h."""
    with open(HEADER) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(vattn_[a-z0-9_]+)\s*\(", text)))

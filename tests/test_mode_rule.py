"""The rule that picks vattn_forward's kernel mode, run on the host with the
device facts passed in (vattn_forward_mode_for: no GPU needed).

The single cooperative kernel (k and v staged inside it) is taken only where
the device supports cooperative launches and holds one of its blocks per
multiprocessor; any device that does not falls back to the two-kernel mode,
which gives the same bits.  The process-wide switch vattn_set_single_kernel
forbids the single kernel the same way."""
import pytest

import vision_encoder_flash_gb300 as vef
from vision_encoder_flash_gb300 import _lib

DIRECT, SINGLE, TWO = _lib.MODE_DIRECT, _lib.MODE_SINGLE_KERNEL, _lib.MODE_TWO_KERNELS


@pytest.fixture(scope="module")
def lib():
    from vision_encoder_flash_gb300 import build
    build.build()
    return vef.load_library()


@pytest.mark.parametrize("shape,aligned,mode", [
    ((8, 16, 2304, 64), 1, SINGLE),      # the benchmark workload
    ((8, 16, 2304, 64), 0, TWO),         # unaligned pointers: neither one-kernel mode
    ((4, 16, 1024, 64), 1, DIRECT),      # <= 1536 patches, head_dim 33..64
    ((8, 16, 1536, 64), 1, DIRECT),
    ((8, 16, 1537, 64), 1, SINGLE),      # 896 work tiles: more than two rounds of 152
    ((4, 16, 2048, 64), 1, SINGLE),      # 512 work tiles
    ((2, 19, 2048, 64), 1, DIRECT),      # 304 work tiles: two rounds
    ((2, 20, 2048, 64), 1, SINGLE),      # 320 work tiles
    ((1, 16, 2048, 64), 1, DIRECT),
    ((4, 16, 2049, 64), 1, SINGLE),
    ((1, 16, 4100, 72), 1, TWO),         # head_dim past 64
    ((1, 16, 4100, 62), 1, TWO),         # head_dim not a multiple of 4
    ((1, 2, 64, 32), 1, DIRECT),         # up to 128 patches: one launch, the direct kernel
    ((1, 2, 64, 30), 1, TWO),            # head_dim not a multiple of 4
    ((1, 2, 128, 64), 1, DIRECT),
    ((1, 2, 129, 32), 1, SINGLE),        # head_dim <= 32 takes the single kernel from 129 patches
    ((1, 16, 256, 64), 1, DIRECT),
    ((2, 2, 130, 128), 1, TWO),
])
def test_mode_rule_on_a_capable_device(lib, shape, aligned, mode):
    assert _lib.forward_mode_for(*shape, aligned, 1, 1, 152) == mode


@pytest.mark.parametrize("coop,blocks", [(0, 1), (1, 0), (0, 0)])
def test_single_kernel_needs_cooperative_launch_and_a_resident_block(lib, coop, blocks):
    # where the single kernel would run, a device without the facts gets two kernels
    assert _lib.forward_mode_for(8, 16, 2304, 64, 1, coop, blocks, 152) == TWO
    assert _lib.forward_mode_for(1, 2, 129, 32, 1, coop, blocks, 152) == TWO
    # the other modes do not depend on them
    assert _lib.forward_mode_for(4, 16, 1024, 64, 1, coop, blocks, 152) == DIRECT
    assert _lib.forward_mode_for(1, 16, 4100, 72, 1, coop, blocks, 152) == TWO
    # from 1537 to 2048 patches the direct kernel stands in for the single one
    assert _lib.forward_mode_for(4, 16, 2048, 64, 1, coop, blocks, 152) == DIRECT


def test_process_wide_switch(lib):
    prev = _lib.set_single_kernel(False)
    try:
        assert prev is True
        assert _lib.forward_mode_for(8, 16, 2304, 64, 1, 1, 1, 152) == TWO
        assert _lib.forward_mode_for(4, 16, 1024, 64, 1, 1, 1, 152) == DIRECT
    finally:
        assert _lib.set_single_kernel(True) is False
    assert _lib.forward_mode_for(8, 16, 2304, 64, 1, 1, 1, 152) == SINGLE


def test_rounds_follow_the_multiprocessor_count(lib):
    # 512 work tiles at 2048 patches: more than two rounds of 152 blocks, at
    # most two of 256
    assert _lib.forward_mode_for(4, 16, 2048, 64, 1, 1, 1, 152) == SINGLE
    assert _lib.forward_mode_for(4, 16, 2048, 64, 1, 1, 1, 256) == DIRECT
    # up to 1536 patches the direct kernel whatever the count
    assert _lib.forward_mode_for(64, 16, 1536, 64, 1, 1, 1, 8) == DIRECT
    with pytest.raises(vef.VattnError) as e:
        _lib.forward_mode_for(4, 16, 2048, 64, 1, 1, 1, 0)
    assert e.value.status == 1


def test_empty_and_invalid(lib):
    assert _lib.forward_mode_for(0, 16, 2304, 64, 1, 1, 1, 152) == _lib.MODE_NONE
    assert _lib.forward_mode_for(8, 16, 0, 64, 1, 1, 1, 152) == _lib.MODE_NONE
    with pytest.raises(vef.VattnError) as e:
        _lib.forward_mode_for(8, 16, 2304, 129, 1, 1, 1, 152)
    assert e.value.status == 2
    with pytest.raises(vef.VattnError) as e:
        _lib.forward_mode_for(8, -1, 2304, 64, 1, 1, 1, 152)
    assert e.value.status == 1


def test_device_query_checks_arguments_before_any_cuda_call(lib):
    fake = 0x10000
    with pytest.raises(vef.VattnError) as e:  # out overlaps q: rejected on the host
        _lib.forward_mode(fake, fake, fake, fake + 4, 1, 1, 2, 4)
    assert e.value.status == 1
    # an empty problem needs no device either
    assert _lib.forward_mode(fake, fake, fake, fake + 2 ** 30, 0, 1, 2, 4) == _lib.MODE_NONE


# The cut rule (vattn_set_split_tiles, vattn_cut_plan_for): on a 152-block
# grid, with the default setting, tiles are cut only where the measured
# saving exceeds the pieces' cost -- long tiles (>= 16 key tiles) and a
# busiest block shorter by >= 7 key tiles.
@pytest.mark.parametrize("shape,cut", [
    ((8, 16, 2304, 64), True),    # 1152 tiles of 18 key tiles: 144 -> 137 per block
    ((2, 16, 4096, 64), True),    # 512 tiles of 32: 128 -> 108
    ((1, 16, 4100, 72), False),   # 272 tiles of 33: saves 6
    ((4, 16, 1024, 64), False),   # tiles of 8 key tiles: too short
    ((2, 40, 2176, 64), False),   # 720 tiles of 17: saves 4
    ((1, 16, 2304, 64), False),   # 144 tiles: one round, nothing to balance
    ((2, 30, 2100, 20), True),    # 540 tiles of 17: 68 -> 61
])
def test_cut_rule_default(lib, shape, cut):
    prev = _lib.set_split_tiles(1)
    try:
        assert _lib.cut_plan_for(*shape, 152) == cut
    finally:
        _lib.set_split_tiles(prev)


def test_cut_rule_forced_and_forbidden(lib):
    prev = _lib.set_split_tiles(2)
    try:
        assert _lib.cut_plan_for(4, 16, 1024, 64, 152)       # forced: short tiles cut too
        assert not _lib.cut_plan_for(1, 16, 2304, 64, 152)   # nothing to balance
        assert _lib.set_split_tiles(0) == 2
        assert not _lib.cut_plan_for(8, 16, 2304, 64, 152)
        assert not _lib.cut_plan_for(2, 16, 4096, 64, 152)
        assert _lib.set_split_tiles(1) == 0
        assert _lib.cut_plan_for(8, 16, 2304, 64, 152)
    finally:
        _lib.set_split_tiles(prev)


def test_cut_rule_argument_errors(lib):
    with pytest.raises(vef.VattnError):
        _lib.cut_plan_for(8, 16, 2304, 64, 0)
    assert not _lib.cut_plan_for(0, 16, 2304, 64, 152)       # empty problem

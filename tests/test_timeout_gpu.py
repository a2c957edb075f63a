"""The kernels' failure detection on a GPU, without a fault: every wait in
the attention kernel is bounded, and one that runs out records a timeout in
the device status word.  vattn_selftest_wait_timeout runs that same bounded
wait on an mbarrier phase that nothing completes; the test checks the status
the host reads and that the device still computes afterwards."""
import numpy as np
import pytest

import oracle
import vision_encoder_flash_gb300 as vef
from vision_encoder_flash_gb300 import _lib
from vattn_inputs import make_inputs

pytestmark = pytest.mark.gpu


def test_a_wait_that_runs_out_is_reported_and_the_device_stays_usable():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("GPU tests need a CUDA device")
    from vision_encoder_flash_gb300 import build
    build.build()
    lib = vef.load_library()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    assert vef.device_status() == 0            # nothing pending before
    _lib.selftest_wait_timeout(torch.cuda.current_stream(dev).cuda_stream)
    assert vef.device_status() == 0x10F        # timeout bit + self-test site, then cleared
    assert "timed out" in lib.vattn_last_error_string().decode()
    assert vef.device_status() == 0
    q, k, v = make_inputs(1, 2, 200, 64, seed=9900)
    out = vef.forward(*(torch.from_numpy(x).to(dev) for x in (q, k, v)))
    torch.cuda.synchronize(dev)
    assert vef.device_status() == 0
    diff = out.cpu().numpy().astype(np.float64) - oracle.forward(q, k, v)
    assert float(np.abs(diff).max()) <= 3e-3

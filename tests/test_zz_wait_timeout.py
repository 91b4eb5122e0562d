"""The failure path of the bounded pipeline waits, on the GPU without a
fault: a wait on an mbarrier that nothing completes must give up by its own
bound (20 ms of global time for the timed wait, a fixed count of polls for
the polling wait), report MOE_STATUS_PIPE_TIMEOUT, and leave the context
usable for the next layer.  Collected after the other GPU tests."""
import time

import pytest
import torch

import oracle
import synth
from gpu_harness import DeviceLayer, check_full, require_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("sleep", [1, 0])
def test_wait_that_never_completes_reports_a_timeout(sleep):
    M = require_gpu()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    M.moe_selftest_wait_timeout(status, sleep)
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    assert int(status.item()) == M.MOE_STATUS_PIPE_TIMEOUT
    assert dt < 30.0, dt
    # the context still runs a layer, and the layer's own status is clean
    L = synth.config_layer(0)
    o = oracle.layer(L)
    dl = DeviceLayer(M, L)
    dl.run_layer()
    assert dl.status() == 0
    check_full(dl, o)

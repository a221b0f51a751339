"""Failure detection without a GPU fault: each bounded device wait the
library uses (the cooperative GroupNorm's acquire-poll on a unit counter and
the tensor-core kernels' mbarrier wait) is made to run out on an event that
never comes; the kernel records DPP_ERR_TIMEOUT, returns, and the context
stays usable for the next call."""
import time

import numpy as np
import pytest
import torch

import displaced_patch_parallelism_02_b300 as dpp
import oracle
import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kind", [0, 1], ids=["counter_wait", "mbarrier_wait"])
def test_bounded_wait_times_out_reports_and_recovers(cuda_device, kind):
    assert dpp.dpp_device_status() == dpp.DPP_OK  # reads and clears the status word
    scratch = torch.zeros(4, dtype=torch.int32, device="cuda")  # a counter nothing advances
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    dpp.dpp_wait_selftest(kind, scratch)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert dpp.dpp_device_status() == dpp.DPP_ERR_TIMEOUT
    assert dpp.dpp_device_status() == dpp.DPP_OK  # cleared by the read
    assert 0.5 < waited < 30.0
    # the context is still usable: a normal call runs and is right
    fresh = wl.normal((1, 8, 4, 16), 900, dtype="bf16").cuda()
    stale = wl.normal((1, 8, 4, 16), 901, dtype="bf16").cuda()
    dpp.dpp_refresh_stale(fresh, stale, 1, 8, 4 * 16 * 2, 2, 0b01)
    torch.cuda.synchronize()
    want = oracle.refresh_stale(fresh.double().cpu().numpy(),
                                wl.normal((1, 8, 4, 16), 901, dtype="bf16").double().numpy(),
                                2, 0b01)
    assert np.array_equal(stale.double().cpu().numpy(), want)
    assert dpp.dpp_device_status() == dpp.DPP_OK

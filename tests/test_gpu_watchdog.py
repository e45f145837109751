"""The failure path of every pipeline wait, exercised without faulting the GPU.

wan_watchdog_selftest enqueues a kernel whose only wait is on an mbarrier that nothing
arrives on.  The wait is the same bounded wait the GEMM and attention pipelines use: it
gives up after the limit, records a timeout in the device status word and returns.  The
host must then read WAN_ERR_TIMEOUT once, the word must be clear afterwards, and the
context must still compute correct results."""
import time

import numpy as np
import pytest
import torch

from oracle import wan_oracle as O
from tests.parity import assert_f32_close, to_dev, to_np

pytestmark = pytest.mark.gpu


def test_timeout_is_reported_once_and_context_stays_usable(wan):
    wan.wan_sync_status()                      # start from a clear status word
    t0 = time.time()
    wan.wan_watchdog_selftest(50)
    with pytest.raises(wan.WanError) as err:
        wan.wan_sync_status()
    assert err.value.status == wan.WAN_ERR_TIMEOUT
    assert time.time() - t0 < 10.0             # gave up after its limit, did not hang
    wan.wan_sync_status()                      # read-and-clear: no second report

    x = np.linspace(-1.0, 1.0, 1000).astype(np.float32)
    vc, vu = np.cos(x), np.sin(x)
    xd = to_dev(x, torch.float32)
    wan.wan_cfg_euler_step(xd, to_dev(vc, torch.float32), to_dev(vu, torch.float32), 5.0, -0.05)
    wan.wan_sync_status()
    assert_f32_close(to_np(xd), O.cfg_euler_step(x, vc, vu, 5.0, np.float32(-0.05)), "after timeout", tol=1e-6)


def test_selftest_rejects_out_of_range_limits(wan):
    assert wan.lib.wan_watchdog_selftest(0, None) == wan.WAN_ERR_INVALID_ARG
    assert wan.lib.wan_watchdog_selftest(5000, None) == wan.WAN_ERR_INVALID_ARG

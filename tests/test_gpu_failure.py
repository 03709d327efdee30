"""Failure detection on the GPU without a fault: a kernel whose mbarrier wait is
never satisfied gives up after a short limit, records FW_ERR_TIMEOUT in the
device error word and returns; the host reads it and the context stays usable."""
import time

import numpy as np
import pytest
import torch

from tests.parity import FW, O, assert_bits_equal, dev, host, synth

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_reports():
    FW.fw_check_device_errors()  # start from a clean error word
    t0 = time.perf_counter()
    FW.fw_selftest_bounded_wait(20000)  # 20 ms
    with pytest.raises(FW.FusedWinError, match="FW_ERR_TIMEOUT"):
        FW.fw_check_device_errors()
    assert time.perf_counter() - t0 < 10.0
    FW.fw_check_device_errors()  # the word was cleared by the read
    # the context still works
    x = synth.maxpool_inputs(1, 2, 16, 32, seed=1)["x"]
    assert_bits_equal(host(FW.fw_maxpool2d(dev(x), 4, 1, 1, 1)), O.maxpool2d(x, 4, 1, 1, 1))


def test_selftest_rejects_bad_limits():
    with pytest.raises(FW.FusedWinError, match="FW_ERR_PARAM"):
        FW.fw_selftest_bounded_wait(0)
    with pytest.raises(FW.FusedWinError, match="FW_ERR_PARAM"):
        FW.fw_selftest_bounded_wait(3_000_000)

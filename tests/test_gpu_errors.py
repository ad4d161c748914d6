"""The bounded-wait error path shared by every kernel: a barrier that nothing arrives on makes
the wait give up after its limit and record W4A16_ERR_TIMEOUT (8) in the device error word,
which the host reads and clears; the context stays usable for the next call."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import FP32_TOL, assert_close_rows, dev, host, lib

pytestmark = pytest.mark.gpu

W4A16_ERR_TIMEOUT = 8


@pytest.fixture(scope="module")
def w4():
    return lib()


def test_wait_that_completes_records_nothing(w4):
    assert w4.w4a16_device_error() == 0
    w4.w4a16_selftest_wait(True, 1000)
    assert w4.w4a16_device_error() == 0


def test_wait_that_runs_out_records_timeout_and_clears(w4):
    assert w4.w4a16_device_error() == 0
    w4.w4a16_selftest_wait(False, 2000)  # gives up after 2 ms
    assert w4.w4a16_device_error() == W4A16_ERR_TIMEOUT
    assert w4.w4a16_device_error() == 0  # read-and-clear


def test_context_usable_after_timeout(w4):
    w4.w4a16_selftest_wait(False, 1000)
    assert w4.w4a16_device_error() == W4A16_ERR_TIMEOUT
    M, K, N = 3, 256, 512
    x = synth.activations(M, K, seed=11)
    qo, so = oracle.quantize_w4a16(synth.weights(K, N, seed=11))
    y = w4.w4a16_gemm(dev(x), dev(qo), dev(so))
    assert_close_rows(host(y), oracle.gemm(x, qo, so), FP32_TOL, "gemm after a timeout")
    assert w4.w4a16_device_error() == 0


@pytest.mark.parametrize("limit_us", [0, 100001])
def test_limit_out_of_range_is_rejected(w4, limit_us):
    with pytest.raises(Exception):
        w4.w4a16_selftest_wait(False, limit_us)

"""The failure path on the GPU, without a fault: a bounded wait that nothing
completes gives up after its limit, sets its bit in the device error word and
lets the kernel return; the context stays usable and the word clears."""
import numpy as np
import pytest
import torch

import workloads
from helpers import host_bits, to_dev_e4m3, to_dev_f32

pytestmark = pytest.mark.gpu

SELFTEST_BIT = 1 << 13


def test_bounded_wait_times_out_and_reports(orc):
    import fp8_w8a8_scaled_gb300 as fp8
    fp8.clear_device_error()
    assert fp8.get_device_error() == 0
    fp8.selftest_bounded_wait(2000)          # 2 ms
    word = fp8.get_device_error()
    assert word & SELFTEST_BIT and word == SELFTEST_BIT
    fp8.clear_device_error()
    assert fp8.get_device_error() == 0
    # the context still runs the library's kernels correctly
    c = workloads.random_gemm(11, 4, 256, 512, 1)
    y = fp8.fp8_scaled_mm(to_dev_e4m3(c["A"]), to_dev_e4m3(c["B"]), to_dev_f32(c["sa"]), to_dev_f32(c["sb"]), 1)
    torch.cuda.synchronize()
    y64, _ = orc.scaled_mm(c["A"], c["B"], c["sa"], c["sb"], 1)
    yf = (host_bits(y).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.all(np.abs(yf - y64) <= 1e-2 * np.abs(y64) + 1e-3 * np.sqrt(512) * float(c["sa"][0]) *
                  c["sb"].astype(np.float64)[None, :] + (16 + 1) * 2.0 ** -23 * orc.gemm_acc_f64(
                      np.asarray(c["A"]) & 0x7F, np.asarray(c["B"]) & 0x7F) * float(c["sa"][0]) *
                  c["sb"].astype(np.float64)[None, :])
    assert fp8.get_device_error() == 0

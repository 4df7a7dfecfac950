"""Failure detection without a GPU fault: a bounded wait inside a kernel runs
out (an mbarrier nothing arrives on), the kernel records FP8LIN_ERR_TIMEOUT
in the device error word and exits; the host reads the status and the
context keeps working."""
import time

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import assert_gemm_close, bf16_to_f64, to_dev_u8

pytestmark = pytest.mark.gpu


def _small_gemm(fp8lin):
    rng = np.random.default_rng(0)
    A = rng.integers(0, 0x70, size=(128, 256), dtype=np.uint8)
    B = rng.integers(0, 0x70, size=(256, 256), dtype=np.uint8)
    one = torch.ones(1, device="cuda")
    y = torch.empty((128, 256), dtype=torch.bfloat16, device="cuda")
    fp8lin.fp8lin_fwd(to_dev_u8(A), one, to_dev_u8(B), one, y)
    torch.cuda.synchronize()
    assert_gemm_close(bf16_to_f64(y), oracle.gemm_rows(A, oracle.E4M3, B, oracle.E4M3, 1.0, 1.0), "after timeout")


def test_bounded_wait_times_out_and_context_survives(fp8lin):
    assert fp8lin.fp8lin_device_error() == 0            # clean start
    t0 = time.perf_counter()
    fp8lin.fp8lin_selftest_bounded_wait(20_000_000)     # 20 ms
    word = fp8lin.fp8lin_device_error()                 # synchronises
    dt = time.perf_counter() - t0
    assert word == 1 << 5                                # FP8LIN_ERR_TIMEOUT bit
    assert 0.015 < dt < 5.0                              # the wait ran out, bounded
    assert fp8lin.fp8lin_device_error() == 0            # read-and-clear
    _small_gemm(fp8lin)                                  # context still usable
    assert fp8lin.fp8lin_device_error() == 0


def test_selftest_rejects_out_of_range_limits(fp8lin):
    with pytest.raises(fp8lin.Fp8LinError):
        fp8lin.fp8lin_selftest_bounded_wait(10)
    with pytest.raises(fp8lin.Fp8LinError):
        fp8lin.fp8lin_selftest_bounded_wait(5_000_000_000)

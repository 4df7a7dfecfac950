"""Failure detection without a GPU fault: a bounded wait inside a kernel runs
out (an mbarrier nothing arrives on), the kernel records FP8LIN_ERR_TIMEOUT
in the device error word and exits; the host reads the status and the
context keeps working.

The GEMMs' own abort paths (per-tensor, fp32-block and power-of-two-block
scaled) run on the test library built with a fault injector
(libfp8lin_faultinj.so: the same GEMM source with a 20 ms wait limit, whose
producers can be told to withhold one slab's copies).  Nothing
is in flight on the withheld stage, so the MMA issuer's wait on it runs out;
the kernel raises its abort flag, lets every copy it did issue land, meets
the peer CTA at the cluster barrier, frees its tensor memory and returns."""
import ctypes
import time

import numpy as np
import pytest
import torch

import oracle
import workloads as wl
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


def _fault_library(fp8lin):
    lib = ctypes.CDLL(fp8lin._build.FAULT_LIB)
    for name in ("fp8lin_fwd", "fp8lin_fwd_block", "fp8lin_fwd_mx", "fp8lin_device_error"):
        fn = getattr(lib, name)
        fn.argtypes = fp8lin.SIGNATURES[name]
        fn.restype = ctypes.c_int
    lib.fp8lin_test_withhold_slab.argtypes = [ctypes.c_int]
    lib.fp8lin_test_withhold_slab.restype = ctypes.c_int
    return lib


def _operands(kind, M, N, K, seed):
    """Device operands of one forward GEMM of each kind, the entry point's
    arguments after the output, and the oracle's reference for given rows."""
    X = wl.generate((M, K), "normal", 1.0, seed, 0)
    W = wl.generate((N, K), "normal", 0.02, seed, 1)
    if kind == "tensor":
        rx, rw = oracle.quantize(X, oracle.E4M3), oracle.quantize(W, oracle.E4M3)
        args = [to_dev_u8(rx["q"]), torch.tensor([rx["inv_scale"]], device="cuda"), to_dev_u8(rw["q"]),
                torch.tensor([rw["inv_scale"]], device="cuda")]
        ref = lambda rows: oracle.fwd_ref(rx["q"], rx["inv_scale"], rw["q"], rw["inv_scale"], rows)
        return "fp8lin_fwd", args, ref
    if kind == "block":
        rx, rw = oracle.quantize_blocks(X, oracle.E4M3, 1, 128), oracle.quantize_blocks(W, oracle.E4M3, 128, 128)
        args = [to_dev_u8(rx["q"]), torch.from_numpy(np.ascontiguousarray(rx["inv_scale"].T)).cuda(),
                to_dev_u8(rw["q"]), torch.from_numpy(np.ascontiguousarray(rw["inv_scale"])).cuda()]
        ref = lambda rows: oracle.fwd_block_ref(rx["q"], rx["inv_scale"], rw["q"], rw["inv_scale"], rows)
        return "fp8lin_fwd_block", args, ref
    rx, rw = oracle.quantize_mx(X, oracle.E4M3, "cols"), oracle.quantize_mx(W, oracle.E4M3, "cols")
    atoms = lambda r, P: to_dev_u8(oracle.pack_sf(oracle.sf_by_operand_row(r["sf"], "cols"), P, K).reshape(-1))
    args = [to_dev_u8(rx["q"]), atoms(rx, M), to_dev_u8(rw["q"]), atoms(rw, N)]
    ref = lambda rows: oracle.fwd_mx_ref(rx["q"], rx["sf"], rw["q"], rw["sf"], rows)
    return "fp8lin_fwd_mx", args, ref


# (M, N, K, withheld slab): the first slab of every CTA pair's only tile, and
# a slab of the second tile of pairs that own two or three tiles (160 pair
# tiles), so completed tiles were already stored when the wait ran out.  The
# power-of-two block-scaled GEMM counts stages of two slabs (two per tile here).
@pytest.mark.parametrize("kind", ["tensor", "block", "mx"])
@pytest.mark.parametrize("M,N,K,slab", [(256, 1024, 512, 0), (256, 40960, 512, 5)])
def test_gemm_abort_path_on_a_withheld_slab(fp8lin, kind, M, N, K, slab):
    lib = _fault_library(fp8lin)
    if kind == "mx":
        slab = {0: 0, 5: 3}[slab]
    name, args, ref = _operands(kind, M, N, K, M + N + slab)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    word = ctypes.c_uint32(0)
    ptrs = [a.data_ptr() for a in args]
    gemm = lambda: getattr(lib, name)(ptrs[0], ptrs[1], ptrs[2], ptrs[3], y.data_ptr(), M, N, K, stream)

    assert lib.fp8lin_test_withhold_slab(slab) == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert gemm() == 0
    status = lib.fp8lin_device_error(stream, ctypes.byref(word))     # synchronises the stream
    dt = time.perf_counter() - t0
    assert status == 5 and word.value == 1 << 5                      # FP8LIN_ERR_TIMEOUT, recorded by the GEMM
    assert dt < 2.0                                                  # 20 ms waits: the kernel gave up and returned
    assert lib.fp8lin_device_error(stream, None) == 0                # read-and-clear

    # the next launch of the same kernel runs clean and matches the oracle
    assert lib.fp8lin_test_withhold_slab(-1) == 0
    y.fill_(float("nan"))
    assert gemm() == 0
    assert lib.fp8lin_device_error(stream, None) == 0
    rows = np.array([0, 1, M // 2, M - 1])
    assert_gemm_close(bf16_to_f64(y[torch.from_numpy(rows).cuda()]), ref(rows), f"{kind} after the abort")
    # the product library never saw a timeout
    assert fp8lin.fp8lin_device_error() == 0
    _small_gemm(fp8lin)

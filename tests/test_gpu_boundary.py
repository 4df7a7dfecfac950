"""The boundary's ownership rule on the device: no entry point allocates
device memory (every buffer is the caller's; the GEMMs' TMEM is on chip).
After one warm-up pass (module loading and the per-device set-up happen
there), repeated linear steps through every recipe leave the device's free
memory unchanged to the byte."""
import pytest
import torch

import workloads as wl
from gpu_helpers import to_dev_bf16

pytestmark = pytest.mark.gpu


def _linears(fp8lin, M, K, N):
    out = [fp8lin.Float8Linear(M, K, N, scaling="dynamic"),
           fp8lin.Float8Linear(M, K, N, scaling="dynamic", transpose=True),
           fp8lin.Float8Linear(M, K, N, scaling="delayed", history_len=4),
           fp8lin.Float8Linear(M, K, N, scaling="rowwise"),
           fp8lin.Float8Linear(M, K, N, scaling="block"),
           fp8lin.Float8Linear(M, K, N, scaling="mx"),
           fp8lin.Float8Linear(M, K, N, scaling="mx", mx_rule="ocp")]
    static = fp8lin.Float8Linear(M, K, N, scaling="static")
    for t8, s in ((static.x8, 64.0), (static.w8, 4096.0), (static.dy8, 65536.0)):
        t8.set_scale(s)
    return out + [static]


def test_entry_points_allocate_no_device_memory(fp8lin):
    M, K, N = 384, 512, 1040
    X = to_dev_bf16(wl.generate((M, K), "normal", 1.0, 71, wl.X))
    W = to_dev_bf16(wl.generate((N, K), "normal", 0.02, 71, wl.W))
    dY = to_dev_bf16(wl.generate((M, N), "normal", 1e-3, 71, wl.DY))
    lins = _linears(fp8lin, M, K, N)
    for _ in range(2):                     # warm-up: every kernel loaded, every attribute set
        for lin in lins:
            lin.step(X, W, dY)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        for lin in lins:
            lin.step(X, W, dY)
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    assert fp8lin.fp8lin_device_error() == 0
    assert free1 == free0, f"device memory changed by {free0 - free1} bytes across the calls"

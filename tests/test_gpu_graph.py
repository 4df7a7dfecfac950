"""The entry points inside a captured CUDA graph: a whole Float8 linear step
(memsets, amax, casts, three GEMMs) and the two-stream FFN schedule replay
with results bit-identical to eager execution."""
import numpy as np
import pytest
import torch

import workloads as wl
from gpu_helpers import to_dev_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("scaling", ["dynamic", "block", "mx"])
def test_linear_step_in_cuda_graph(fp8lin, scaling):
    M, K, N = 640, 384, 1296
    X = to_dev_bf16(wl.generate((M, K), "normal", 1.0, 31, 0))
    W = to_dev_bf16(wl.generate((N, K), "normal", 0.02, 31, 1))
    dY = to_dev_bf16(wl.generate((M, N), "normal", 1e-3, 31, 2))
    eager = fp8lin.Float8Linear(M, K, N, scaling=scaling)
    ref = [t.clone() for t in eager.step(X, W, dY)]

    lin = fp8lin.Float8Linear(M, K, N, scaling=scaling)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        lin.step(X, W, dY)                      # first use: per-device setup happens eagerly
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    for t in (lin.y, lin.dx, lin.dw):
        t.zero_()
    with torch.cuda.graph(g):
        lin.step(X, W, dY)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip((lin.y, lin.dx, lin.dw), ref):
            assert torch.equal(a, b)
    assert fp8lin.fp8lin_device_error() == 0


def test_two_stream_ffn_schedule_in_cuda_graph(fp8lin):
    import bench
    spec = bench.SPECS["tiny"]
    host = bench.host_inputs(spec, 0)
    dev = torch.device("cuda", 0)
    din = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(dev) for k, v in host.items()}
    step = bench.StepGraph(fp8lin, spec, dev, din)
    step.run()
    torch.cuda.synchronize()
    ref = [t.clone() for t in step.outputs()]
    for t in step.outputs():
        t.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=step.main):
        step.run()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(step.outputs(), ref):
        assert torch.equal(a, b)

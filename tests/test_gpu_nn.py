"""The autograd / nn.Module front end on the GPU: the same kernels as
Float8Linear.step, so every output and gradient is bit-identical to the
explicit nine-call step (itself checked against the oracle elsewhere)."""
import pytest
import torch

import workloads as wl
from gpu_helpers import to_dev_bf16

pytestmark = pytest.mark.gpu
SCALINGS = ["dynamic", "rowwise", "block", "mx", "mx_ocp"]


def _inputs(M, K, N, seed):
    X = wl.generate((M, K), "normal", 1.0, seed, wl.X, outlier_frac=1e-3)
    W = wl.generate((N, K), "normal", 0.02, seed, wl.W)
    dY = wl.generate((M, N), "normal", 1e-3, seed, wl.DY)
    return X, W, dY


@pytest.mark.parametrize("scaling", SCALINGS)
@pytest.mark.parametrize("lead", [(272,), (2, 136)])
def test_function_matches_the_explicit_step(fp8lin, scaling, lead):
    M, K, N = 272, 384, 528
    X, W, dY = _inputs(M, K, N, 31)
    x = to_dev_bf16(X).reshape(*lead, K).requires_grad_()
    w = torch.nn.Parameter(to_dev_bf16(W))
    y = fp8lin.Float8LinearFunction.apply(x, w, scaling)
    assert y.shape == (*lead, N) and y.dtype == torch.bfloat16
    y.backward(to_dev_bf16(dY).reshape(*lead, N))
    lin = (fp8lin.Float8Linear(M, K, N, scaling="mx", mx_rule="ocp") if scaling == "mx_ocp"
           else fp8lin.Float8Linear(M, K, N, scaling=scaling))
    y2, dx2, dw2 = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    assert torch.equal(y.reshape(M, N), y2)
    assert torch.equal(x.grad.reshape(M, K), dx2)
    assert torch.equal(w.grad, dw2)


def test_swapped_two_layer_model_matches_chained_steps(fp8lin):
    M, K, H, N = 256, 512, 768, 384
    X, W1, _ = _inputs(M, K, H, 41)
    _, W2, dY = _inputs(M, H, N, 42)
    model = torch.nn.Sequential(torch.nn.Linear(K, H, bias=False, dtype=torch.bfloat16, device="cuda"),
                                torch.nn.Linear(H, N, bias=False, dtype=torch.bfloat16, device="cuda"))
    with torch.no_grad():
        model[0].weight.copy_(to_dev_bf16(W1))
        model[1].weight.copy_(to_dev_bf16(W2))
    fp8lin.swap_linear_layers(model)
    assert all(isinstance(m, fp8lin.Float8LinearModule) for m in model)
    x = to_dev_bf16(X).requires_grad_()
    y = model(x)
    y.backward(to_dev_bf16(dY))
    l1, l2 = fp8lin.Float8Linear(M, K, H), fp8lin.Float8Linear(M, H, N)
    h = l1.forward(to_dev_bf16(X), to_dev_bf16(W1)).clone()
    y2 = l2.forward(h, to_dev_bf16(W2))
    dh, dw2 = l2.backward(to_dev_bf16(dY))
    dx, dw1 = l1.backward(dh.clone())
    torch.cuda.synchronize()
    assert torch.equal(y, y2)
    assert torch.equal(model[1].weight.grad, dw2) and torch.equal(model[0].weight.grad, dw1)
    assert torch.equal(x.grad, dx)


def test_weight_gradient_only_and_shape_errors(fp8lin):
    M, K, N = 128, 256, 128
    X, W, dY = _inputs(M, K, N, 51)
    x = to_dev_bf16(X)                                   # no gradient wanted for the input
    w = torch.nn.Parameter(to_dev_bf16(W))
    fp8lin.Float8LinearFunction.apply(x, w, "dynamic").backward(to_dev_bf16(dY))
    lin = fp8lin.Float8Linear(M, K, N)
    _, _, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    assert x.grad is None and torch.equal(w.grad, dw)
    with pytest.raises(fp8lin.Fp8LinError):              # M = 8 rows: not a multiple of 16
        fp8lin.Float8LinearFunction.apply(x[:8], w, "dynamic")
    with pytest.raises(ValueError):
        fp8lin.Float8LinearFunction.apply(x[:, :128], w, "dynamic")


@pytest.mark.parametrize("scaling", ["delayed", "static"])
def test_stateful_module_matches_the_explicit_step_over_steps(fp8lin, scaling):
    """Three training steps: the module's amax histories (or fixed scales)
    evolve exactly as Float8Linear's."""
    M, K, N = 256, 384, 512
    mod = fp8lin.Float8LinearModule(K, N, device="cuda", scaling=scaling, history_len=4)
    lin = fp8lin.Float8Linear(M, K, N, scaling=scaling, history_len=4)
    if scaling == "static":
        mod.set_static_scales(64.0, 8192.0, 2.0 ** 17)
        for t8, v in ((lin.x8, 64.0), (lin.w8, 8192.0), (lin.dy8, 2.0 ** 17)):
            t8.set_scale(v)
    for step in range(3):
        X, W, dY = _inputs(M, K, N, 60 + step)
        with torch.no_grad():
            mod.weight.copy_(to_dev_bf16(W))
        mod.weight.grad = None
        x = to_dev_bf16(X).requires_grad_()
        y = mod(x)
        y.backward(to_dev_bf16(dY))
        y2, dx2, dw2 = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
        torch.cuda.synchronize()
        assert torch.equal(y, y2) and torch.equal(x.grad, dx2) and torch.equal(mod.weight.grad, dw2), step
        if scaling == "delayed":
            for r, t8 in (("x", lin.x8), ("w", lin.w8), ("dy", lin.dy8)):
                assert torch.equal(getattr(mod, f"amax_history_{r}"), t8.history), (step, r)

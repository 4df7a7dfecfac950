"""The Float8 linear used for training: a two-layer bias-free MLP on a
synthetic regression task, trained from one initialisation once in bf16
(torch's own linears) and once with every linear swapped for a
Float8LinearModule.  The Float8 gradients have to train the model about as
well as the bf16 ones: the loss falls by the same order and ends close to
the bf16 run's.  No dataset is involved: inputs and targets are seeded
synthetic tensors, the target a fixed random non-linear map."""
import copy

import pytest
import torch

pytestmark = pytest.mark.gpu


def _task(seed=0, batch=512, d_in=256, d_out=256):
    g = torch.Generator(device="cuda").manual_seed(seed)
    a = torch.randn(d_in, d_out, device="cuda", generator=g) / d_in ** 0.5
    xs = [torch.randn(batch, d_in, device="cuda", generator=g) for _ in range(8)]
    return [(x.bfloat16(), torch.tanh(x @ a).bfloat16()) for x in xs]


def _train(model, data, steps=120, lr=0.5):
    opt = torch.optim.SGD(model.parameters(), lr=lr, momentum=0.9)
    losses = []
    for i in range(steps):
        x, y = data[i % len(data)]
        opt.zero_grad(set_to_none=True)
        loss = torch.nn.functional.mse_loss(model(x).float(), y.float())
        loss.backward()
        opt.step()
        losses.append(float(loss.detach()))
    return losses


@pytest.mark.parametrize("scaling", ["dynamic", "mx", "block", "delayed"])
def test_float8_mlp_trains_like_bf16(fp8lin, scaling):
    torch.manual_seed(0)
    ref = torch.nn.Sequential(torch.nn.Linear(256, 512, bias=False), torch.nn.GELU(),
                              torch.nn.Linear(512, 256, bias=False)).to("cuda", torch.bfloat16)
    f8 = fp8lin.swap_linear_layers(copy.deepcopy(ref), scaling=scaling)
    assert all(isinstance(f8[i], fp8lin.Float8LinearModule) for i in (0, 2))
    data = _task()
    l_ref = _train(ref, data)
    l_f8 = _train(f8, data)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    tail_ref = sum(l_ref[-8:]) / 8
    tail_f8 = sum(l_f8[-8:]) / 8
    assert tail_ref < 0.5 * l_ref[0]                       # the task is learnable in this budget
    assert tail_f8 < 0.5 * l_f8[0], (l_f8[0], tail_f8)     # so it is with Float8 gradients
    assert tail_f8 < 1.25 * tail_ref + 1e-3, (tail_f8, tail_ref)

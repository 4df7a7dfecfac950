"""The nn.Linear swap of the autograd front end (CPU: construction and module
surgery only, no kernel runs)."""
import pytest
import torch

import float8_linear_layers_gb300 as fl


def _lin(i, o, bias=False, dtype=torch.bfloat16):
    return torch.nn.Linear(i, o, bias=bias, dtype=dtype)


def test_swap_replaces_only_eligible_linears_and_shares_weights():
    eligible, biased, ragged, fp32 = _lin(64, 128), _lin(128, 48, bias=True), _lin(48, 40), _lin(48, 32, dtype=torch.float32)
    nested = _lin(32, 16)
    model = torch.nn.Sequential(eligible, torch.nn.ReLU(), biased, ragged, fp32, torch.nn.Sequential(nested))
    w0, w5 = eligible.weight, nested.weight
    out = fl.swap_linear_layers(model, scaling="block")
    assert out is model
    assert isinstance(model[0], fl.Float8LinearModule) and model[0].weight is w0 and model[0].scaling == "block"
    assert isinstance(model[5][0], fl.Float8LinearModule) and model[5][0].weight is w5
    assert model[2] is biased and model[3] is ragged and model[4] is fp32
    # the swapped weight is still the model's parameter (an optimizer keeps updating it)
    assert sum(p is w0 for p in model.parameters()) == 1


def test_swap_filter_and_a_bare_linear():
    model = torch.nn.Sequential(_lin(64, 64), _lin(64, 64))
    fl.swap_linear_layers(model, module_filter=lambda fqn, m: fqn != "1")
    assert isinstance(model[0], fl.Float8LinearModule) and type(model[1]) is torch.nn.Linear
    bare = _lin(32, 48)
    swapped = fl.swap_linear_layers(bare)
    assert isinstance(swapped, fl.Float8LinearModule) and swapped.weight is bare.weight
    assert (swapped.in_features, swapped.out_features) == (32, 48)


def test_module_and_function_arguments():
    m = fl.Float8LinearModule(32, 48)
    assert m.weight.dtype == torch.bfloat16 and tuple(m.weight.shape) == (48, 32)
    assert m.weight.abs().max() <= 1 / 32 ** 0.5 + 1e-6     # nn.Linear's kaiming-uniform bound
    with pytest.raises(ValueError):
        fl.Float8LinearModule(32, 48, bias=True)
    with pytest.raises(ValueError):
        fl.Float8LinearModule(32, 48, scaling="per-channel")
    with pytest.raises(ValueError):   # stateful scalings need the module that owns the state
        fl.Float8LinearFunction.apply(torch.zeros(16, 32, dtype=torch.bfloat16),
                                      torch.zeros(48, 32, dtype=torch.bfloat16), "delayed")
    with pytest.raises(ValueError):
        fl.Float8LinearModule.from_linear(_lin(32, 48, bias=True))
    with pytest.raises(TypeError):
        fl.Float8LinearModule.from_linear(_lin(32, 48, dtype=torch.float32))
    with pytest.raises(TypeError):   # dtype is checked before anything reaches the device
        fl.Float8LinearFunction.apply(torch.zeros(16, 32), torch.zeros(48, 32, dtype=torch.bfloat16), "dynamic")


def test_stateful_scalings_keep_their_state_in_module_buffers():
    d = fl.Float8LinearModule(32, 48, scaling="delayed", history_len=8)
    sd = d.state_dict()
    for r in ("x", "w", "dy"):
        assert tuple(sd[f"amax_history_{r}"].shape) == (8,) and float(sd[f"amax_history_{r}"].abs().sum()) == 0
    assert d.history_slot == {"x": 0, "w": 0, "dy": 0}
    s = fl.Float8LinearModule.from_linear(_lin(32, 48), scaling="static").set_static_scales(2.0, 64.0, 4096.0)
    assert [float(getattr(s, f"scale_{r}")) for r in ("x", "w", "dy")] == [2.0, 64.0, 4096.0]
    with pytest.raises(ValueError):
        d.set_static_scales(1.0, 1.0, 1.0)
    plain = fl.Float8LinearModule(32, 48)
    assert not [n for n, _ in plain.named_buffers()]


def test_history_slots_round_trip_through_a_state_dict():
    a = fl.Float8LinearModule(32, 48, scaling="delayed", history_len=4)
    a.history_slot["x"], a.history_seeded["x"] = 3, True
    a.amax_history_x.fill_(2.5)
    b = fl.Float8LinearModule(32, 48, scaling="delayed", history_len=4)
    b.load_state_dict(a.state_dict())
    assert b.history_slot["x"] == 3 and b.history_seeded["x"] and float(b.amax_history_x[0]) == 2.5

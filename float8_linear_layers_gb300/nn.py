"""Autograd and nn.Module front end of the Float8 linear layer.

The pages' only interface for the layer is a Float8 linear that takes the
place of nn.Linear and composes with autograd ("TorchTitan: a one-stop
PyTorch-native solution for production LLM pre-training", section 3.3,
"Mixed precision and Float8": Float8 applied selectively to linear layers,
composable with autograd).  This module is that swap:

* ``Float8LinearFunction`` -- forward: amax + cast of X and W, Y = X.W^T on
  the FP8 copies; backward: amax + cast of dY, dX = dY.W and dW = dY^T.X on
  the FP8 copies of X and W made in forward (only those are kept between the
  passes: "FP8 saves what is stored in FP8", "Lecture 9 exercises").  Every
  step runs in the library's kernels; this code only allocates outputs and
  marshals arguments.
* ``Float8LinearModule`` -- a bias-free nn.Linear replacement holding a bf16
  weight [out_features x in_features].
* ``swap_linear_layers`` -- replaces the eligible nn.Linear modules of a
  model in place.

Scalings: "dynamic" (default), "rowwise", "block", "mx" (power-of-two
block scales applied by the tensor cores) and "mx_ocp" (the same with the OCP
Microscaling scale rule) are stateless per call.
"delayed" and "static" keep per-tensor state across steps (the TorchTitan
page, section 3.3, names dynamic, delayed and static scaling): a Float8LinearModule
holds it as buffers, one per tensor role (X, W, dY) -- an amax history ring
with the slot the next cast records into, or a fixed scale -- and passes
itself to the function as the owner of that state.
"""
from __future__ import annotations

import math

import torch

from . import (E4M3, E5M2, Float8Tensor, fp8lin_dgrad, fp8lin_dgrad_block, fp8lin_dgrad_mn, fp8lin_dgrad_mx,
               fp8lin_dgrad_rowwise, fp8lin_fwd, fp8lin_fwd_block, fp8lin_fwd_mx, fp8lin_fwd_rowwise, fp8lin_wgrad,
               fp8lin_wgrad_block, fp8lin_wgrad_mn, fp8lin_wgrad_mx, fp8lin_wgrad_rowwise)

SCALINGS = ("dynamic", "rowwise", "block", "mx", "mx_ocp", "delayed", "static")
STATEFUL = ("delayed", "static")
ROLES = ("x", "w", "dy")


def _check_scaling(scaling: str) -> None:
    if scaling not in SCALINGS:
        raise ValueError(f"scaling must be one of {SCALINGS}, got {scaling!r}")


def _quantize(src: torch.Tensor, fmt: int, scaling: str, blocks: str, role: str, owner) -> Float8Tensor:
    """The FP8 copy of one operand for one call: a fresh Float8Tensor, wired
    to the owner's state for the stateful scalings."""
    rows, cols = src.shape
    if scaling in STATEFUL:
        if owner is None:
            raise ValueError(f"{scaling} scaling keeps state: call through a Float8LinearModule")
        t8 = Float8Tensor(rows, cols, fmt, src.device, scaling=scaling, transpose=False,
                          history_len=getattr(owner, f"amax_history_{role}").numel() if scaling == "delayed" else 1)
        if scaling == "delayed":
            t8.history = getattr(owner, f"amax_history_{role}")
            t8.slot, t8.seeded = owner.history_slot[role], owner.history_seeded[role]
        else:
            t8.scale = getattr(owner, f"scale_{role}")
        t8.quantize(src)
        if scaling == "delayed":
            owner.history_slot[role], owner.history_seeded[role] = t8.slot, True
        return t8
    if scaling == "mx_ocp":   # power-of-two blocks with the OCP Microscaling scale rule
        return Float8Tensor(rows, cols, fmt, src.device, scaling="mx", mx_rule="ocp").quantize(src)
    t8 = Float8Tensor(rows, cols, fmt, src.device, scaling=scaling, transpose=scaling == "rowwise", blocks=blocks)
    return t8.quantize(src)


def _fwd(x8: Float8Tensor, w8: Float8Tensor, y: torch.Tensor) -> None:
    if x8.scaling == "mx":
        fp8lin_fwd_mx(x8.q, x8.sf_row, w8.q, w8.sf_row, y)
    elif x8.scaling == "block":
        fp8lin_fwd_block(x8.q, x8.row_inv, w8.q, w8.tile_inv, y)
    elif x8.scaling == "rowwise":
        fp8lin_fwd_rowwise(x8.q, x8.row_inv, w8.q, w8.row_inv, y)
    else:
        fp8lin_fwd(x8.q, x8.inv_scale, w8.q, w8.inv_scale, y)


def _dgrad(d8: Float8Tensor, w8: Float8Tensor, dx: torch.Tensor) -> None:
    if d8.scaling == "mx":
        fp8lin_dgrad_mx(d8.q, d8.sf_row, w8.qc, w8.sf_col, dx)
    elif d8.scaling == "block":
        fp8lin_dgrad_block(d8.q, d8.row_inv, w8.q, w8.tile_inv, dx)
    elif d8.scaling == "rowwise":
        fp8lin_dgrad_rowwise(d8.q, d8.row_inv, w8.qT, w8.col_inv, dx)
    elif w8.qT is not None:
        fp8lin_dgrad(d8.q, d8.inv_scale, w8.qT, w8.inv_scale, dx)
    else:
        fp8lin_dgrad_mn(d8.q, d8.inv_scale, w8.q, w8.inv_scale, dx)


def _wgrad(d8: Float8Tensor, x8: Float8Tensor, dw: torch.Tensor) -> None:
    if d8.scaling == "mx":
        fp8lin_wgrad_mx(d8.qc, d8.sf_col, x8.qc, x8.sf_col, dw)
    elif d8.scaling == "block":
        fp8lin_wgrad_block(d8.qc, d8.col_inv, x8.qc, x8.col_inv, dw)
    elif d8.scaling == "rowwise":
        fp8lin_wgrad_rowwise(d8.qT, d8.col_inv, x8.qT, x8.col_inv, dw)
    elif x8.qT is not None:
        fp8lin_wgrad(d8.qT, d8.inv_scale, x8.qT, x8.inv_scale, dw)
    else:
        fp8lin_wgrad_mn(d8.q, d8.inv_scale, x8.q, x8.inv_scale, dw)


class Float8LinearFunction(torch.autograd.Function):
    """y = x . weight^T through the Float8 path; x [..., K] and weight [N x K]
    bf16 on one CUDA device, the product of x's leading sizes (M), K and N
    multiples of 16 (the library raises Fp8LinError otherwise)."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, weight: torch.Tensor, scaling: str = "dynamic", owner=None) -> torch.Tensor:
        _check_scaling(scaling)
        if scaling in STATEFUL and owner is None:
            raise ValueError(f"{scaling} scaling keeps state: call through a Float8LinearModule")
        for t, name in ((x, "input"), (weight, "weight")):
            if t.dtype != torch.bfloat16:
                raise TypeError(f"Float8LinearFunction: {name} must be bfloat16, got {t.dtype}")
        N, K = weight.shape
        if x.shape[-1] != K:
            raise ValueError(f"Float8LinearFunction: input has {x.shape[-1]} features, weight expects {K}")
        x2 = x.reshape(-1, K).contiguous()
        M = x2.shape[0]
        x8 = _quantize(x2, E4M3, scaling, "rowcol", "x", owner)
        w8 = _quantize(weight.contiguous(), E4M3, scaling, "tile", "w", owner)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
        _fwd(x8, w8, y)
        ctx.x8, ctx.w8, ctx.scaling, ctx.owner, ctx.x_shape = x8, w8, scaling, owner, x.shape
        return y.view(*x.shape[:-1], N)

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        x8, w8 = ctx.x8, ctx.w8
        M, K, N = x8.rows, x8.cols, w8.rows
        dy2 = dy.reshape(-1, N)
        if dy2.dtype != torch.bfloat16:
            raise TypeError(f"Float8LinearFunction: the output gradient must be bfloat16, got {dy2.dtype}")
        d8 = _quantize(dy2.contiguous(), E5M2, ctx.scaling, "rowcol", "dy", ctx.owner)
        dx = dw = None
        if ctx.needs_input_grad[0]:
            dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
            _dgrad(d8, w8, dx)
            dx = dx.view(ctx.x_shape)
        if ctx.needs_input_grad[1]:
            dw = torch.empty((N, K), dtype=torch.bfloat16, device=dy.device)
            _wgrad(d8, x8, dw)
        ctx.x8 = ctx.w8 = ctx.owner = None
        return dx, dw, None, None


class Float8LinearModule(torch.nn.Module):
    """Bias-free replacement for nn.Linear(in_features, out_features) whose
    forward and backward run through the Float8 path; the weight is a bf16
    parameter [out_features x in_features]."""

    def __init__(self, in_features: int, out_features: int, bias: bool = False, device=None,
                 scaling: str = "dynamic", history_len: int = 16):
        super().__init__()
        if bias:
            raise ValueError("Float8LinearModule has no bias (the Float8 linear path computes x . W^T only)")
        _check_scaling(scaling)
        self.in_features, self.out_features, self.scaling = in_features, out_features, scaling
        self.weight = torch.nn.Parameter(torch.empty((out_features, in_features), dtype=torch.bfloat16,
                                                     device=device))
        torch.nn.init.kaiming_uniform_(self.weight, a=math.sqrt(5))   # nn.Linear's initialisation
        self._init_state(history_len)

    def _init_state(self, history_len: int) -> None:
        """Buffers of the stateful scalings: per role an amax history ring
        (delayed) or a fixed scale, 1.0 until set_static_scales (static)."""
        dev = self.weight.device
        self.history_slot = {r: 0 for r in ROLES}
        self.history_seeded = {r: False for r in ROLES}
        for r in ROLES:
            if self.scaling == "delayed":
                self.register_buffer(f"amax_history_{r}", torch.zeros(history_len, dtype=torch.float32, device=dev))
            elif self.scaling == "static":
                self.register_buffer(f"scale_{r}", torch.ones(1, dtype=torch.float32, device=dev))

    def set_static_scales(self, x: float, w: float, dy: float) -> "Float8LinearModule":
        """The fixed scales of static scaling (q = sat_RNE(t * scale))."""
        if self.scaling != "static":
            raise ValueError("set_static_scales: the module does not use static scaling")
        for r, v in zip(ROLES, (x, w, dy)):
            getattr(self, f"scale_{r}").fill_(float(v))
        return self

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear, scaling: str = "dynamic",
                    history_len: int = 16) -> "Float8LinearModule":
        """Wrap an existing bias-free bf16 nn.Linear, sharing its weight parameter."""
        if linear.bias is not None:
            raise ValueError("from_linear: the linear has a bias")
        if linear.weight.dtype != torch.bfloat16:
            raise TypeError(f"from_linear: the weight must be bfloat16, got {linear.weight.dtype}")
        mod = cls.__new__(cls)
        torch.nn.Module.__init__(mod)
        _check_scaling(scaling)
        mod.in_features, mod.out_features, mod.scaling = linear.in_features, linear.out_features, scaling
        mod.weight = linear.weight
        mod._init_state(history_len)
        return mod

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return Float8LinearFunction.apply(x, self.weight, self.scaling, self)

    # the history slots travel with the history buffers in a state dict
    def get_extra_state(self):
        return {"history_slot": dict(self.history_slot), "history_seeded": dict(self.history_seeded)}

    def set_extra_state(self, state) -> None:
        self.history_slot = dict(state["history_slot"])
        self.history_seeded = dict(state["history_seeded"])

    def extra_repr(self) -> str:
        return f"in_features={self.in_features}, out_features={self.out_features}, scaling={self.scaling}"


def eligible(linear: torch.nn.Module) -> bool:
    """A module the swap replaces: a bias-free bf16 nn.Linear whose feature
    counts are multiples of 16."""
    return (type(linear) is torch.nn.Linear and linear.bias is None and linear.weight.dtype == torch.bfloat16
            and linear.in_features % 16 == 0 and linear.out_features % 16 == 0)


def swap_linear_layers(model: torch.nn.Module, scaling: str = "dynamic", module_filter=None,
                       history_len: int = 16) -> torch.nn.Module:
    """Replace, in place, every eligible nn.Linear of ``model`` (and ``model``
    itself if it is one) by a Float8LinearModule sharing its weight;
    ``module_filter(fqn, module)`` may exclude more.  Returns the model."""
    _check_scaling(scaling)

    def keep(fqn: str, mod: torch.nn.Module) -> bool:
        return eligible(mod) and (module_filter is None or module_filter(fqn, mod))

    if keep("", model):
        return Float8LinearModule.from_linear(model, scaling, history_len)
    for fqn, parent in list(model.named_modules()):
        for name, child in list(parent.named_children()):
            if keep(f"{fqn}.{name}" if fqn else name, child):
                setattr(parent, name, Float8LinearModule.from_linear(child, scaling, history_len))
    return model

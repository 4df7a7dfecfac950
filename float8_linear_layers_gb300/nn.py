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

Scalings: "dynamic" (default), "rowwise" and "block" are stateless per call.
Delayed and static scaling keep state across steps (an amax history, a fixed
scale): use ``Float8Linear`` / ``Float8Tensor`` for those.
"""
from __future__ import annotations

import math

import torch

from . import (E4M3, E5M2, Float8Tensor, fp8lin_dgrad, fp8lin_dgrad_block, fp8lin_dgrad_mn,
               fp8lin_dgrad_rowwise, fp8lin_fwd, fp8lin_fwd_block, fp8lin_fwd_rowwise, fp8lin_wgrad,
               fp8lin_wgrad_block, fp8lin_wgrad_mn, fp8lin_wgrad_rowwise)

SCALINGS = ("dynamic", "rowwise", "block")


def _check_scaling(scaling: str) -> None:
    if scaling not in SCALINGS:
        raise ValueError(f"Float8LinearFunction supports scaling in {SCALINGS}, got {scaling!r} "
                         "(delayed and static scaling keep state: use Float8Linear)")


def _fwd(x8: Float8Tensor, w8: Float8Tensor, y: torch.Tensor) -> None:
    if x8.scaling == "block":
        fp8lin_fwd_block(x8.q, x8.row_inv, w8.q, w8.tile_inv, y)
    elif x8.scaling == "rowwise":
        fp8lin_fwd_rowwise(x8.q, x8.row_inv, w8.q, w8.row_inv, y)
    else:
        fp8lin_fwd(x8.q, x8.inv_scale, w8.q, w8.inv_scale, y)


def _dgrad(d8: Float8Tensor, w8: Float8Tensor, dx: torch.Tensor) -> None:
    if d8.scaling == "block":
        fp8lin_dgrad_block(d8.q, d8.row_inv, w8.q, w8.tile_inv, dx)
    elif d8.scaling == "rowwise":
        fp8lin_dgrad_rowwise(d8.q, d8.row_inv, w8.qT, w8.col_inv, dx)
    elif w8.qT is not None:
        fp8lin_dgrad(d8.q, d8.inv_scale, w8.qT, w8.inv_scale, dx)
    else:
        fp8lin_dgrad_mn(d8.q, d8.inv_scale, w8.q, w8.inv_scale, dx)


def _wgrad(d8: Float8Tensor, x8: Float8Tensor, dw: torch.Tensor) -> None:
    if d8.scaling == "block":
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
    def forward(ctx, x: torch.Tensor, weight: torch.Tensor, scaling: str = "dynamic") -> torch.Tensor:
        _check_scaling(scaling)
        for t, name in ((x, "input"), (weight, "weight")):
            if t.dtype != torch.bfloat16:
                raise TypeError(f"Float8LinearFunction: {name} must be bfloat16, got {t.dtype}")
        N, K = weight.shape
        if x.shape[-1] != K:
            raise ValueError(f"Float8LinearFunction: input has {x.shape[-1]} features, weight expects {K}")
        x2 = x.reshape(-1, K).contiguous()
        M = x2.shape[0]
        transpose = scaling == "rowwise"
        x8 = Float8Tensor(M, K, E4M3, x.device, scaling=scaling, transpose=transpose, blocks="rowcol")
        w8 = Float8Tensor(N, K, E4M3, x.device, scaling=scaling, transpose=transpose, blocks="tile")
        x8.quantize(x2)
        w8.quantize(weight.contiguous())
        y = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
        _fwd(x8, w8, y)
        ctx.x8, ctx.w8, ctx.scaling, ctx.x_shape = x8, w8, scaling, x.shape
        return y.view(*x.shape[:-1], N)

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        x8, w8 = ctx.x8, ctx.w8
        M, K, N = x8.rows, x8.cols, w8.rows
        dy2 = dy.reshape(-1, N)
        if dy2.dtype != torch.bfloat16:
            raise TypeError(f"Float8LinearFunction: the output gradient must be bfloat16, got {dy2.dtype}")
        dy2 = dy2.contiguous()
        d8 = Float8Tensor(M, N, E5M2, dy.device, scaling=ctx.scaling, transpose=ctx.scaling == "rowwise",
                          blocks="rowcol")
        d8.quantize(dy2)
        dx = dw = None
        if ctx.needs_input_grad[0]:
            dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device)
            _dgrad(d8, w8, dx)
            dx = dx.view(ctx.x_shape)
        if ctx.needs_input_grad[1]:
            dw = torch.empty((N, K), dtype=torch.bfloat16, device=dy.device)
            _wgrad(d8, x8, dw)
        ctx.x8 = ctx.w8 = None
        return dx, dw, None


class Float8LinearModule(torch.nn.Module):
    """Bias-free replacement for nn.Linear(in_features, out_features) whose
    forward and backward run through the Float8 path; the weight is a bf16
    parameter [out_features x in_features]."""

    def __init__(self, in_features: int, out_features: int, bias: bool = False, device=None,
                 scaling: str = "dynamic"):
        super().__init__()
        if bias:
            raise ValueError("Float8LinearModule has no bias (the Float8 linear path computes x . W^T only)")
        _check_scaling(scaling)
        self.in_features, self.out_features, self.scaling = in_features, out_features, scaling
        self.weight = torch.nn.Parameter(torch.empty((out_features, in_features), dtype=torch.bfloat16,
                                                     device=device))
        torch.nn.init.kaiming_uniform_(self.weight, a=math.sqrt(5))   # nn.Linear's initialisation

    @classmethod
    def from_linear(cls, linear: torch.nn.Linear, scaling: str = "dynamic") -> "Float8LinearModule":
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
        return mod

    def forward(self, x: torch.Tensor) -> torch.Tensor:
        return Float8LinearFunction.apply(x, self.weight, self.scaling)

    def extra_repr(self) -> str:
        return f"in_features={self.in_features}, out_features={self.out_features}, scaling={self.scaling}"


def eligible(linear: torch.nn.Module) -> bool:
    """A module the swap replaces: a bias-free bf16 nn.Linear whose feature
    counts are multiples of 16."""
    return (type(linear) is torch.nn.Linear and linear.bias is None and linear.weight.dtype == torch.bfloat16
            and linear.in_features % 16 == 0 and linear.out_features % 16 == 0)


def swap_linear_layers(model: torch.nn.Module, scaling: str = "dynamic", module_filter=None) -> torch.nn.Module:
    """Replace, in place, every eligible nn.Linear of ``model`` (and ``model``
    itself if it is one) by a Float8LinearModule sharing its weight;
    ``module_filter(fqn, module)`` may exclude more.  Returns the model."""
    _check_scaling(scaling)

    def keep(fqn: str, mod: torch.nn.Module) -> bool:
        return eligible(mod) and (module_filter is None or module_filter(fqn, mod))

    if keep("", model):
        return Float8LinearModule.from_linear(model, scaling)
    for fqn, parent in list(model.named_modules()):
        for name, child in list(parent.named_children()):
            if keep(f"{fqn}.{name}" if fqn else name, child):
                setattr(parent, name, Float8LinearModule.from_linear(child, scaling))
    return model

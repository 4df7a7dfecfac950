"""Shared helpers for the gpu-marked parity tests (host <-> device marshalling
and the oracle comparisons).  Imports torch lazily so CPU-only collection
never touches CUDA."""
import numpy as np
import torch

import oracle

SENTINEL = 0xA5


def to_dev_bf16(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_dev_u8(codes: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(codes)).to(device)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def scalar_bits(t: torch.Tensor) -> int:
    return int(t.cpu().view(torch.int32).item()) & 0xFFFFFFFF


def f32_bits(v) -> int:
    return int(np.float32(v).view(np.uint32))


class Guarded:
    """A device buffer of `n` elements inside a larger one whose edges hold a
    sentinel, to catch writes outside the declared output."""

    def __init__(self, shape, dtype, device="cuda", pad=4096):
        n = int(np.prod(shape))
        esize = torch.empty((), dtype=dtype).element_size()
        self.pad = pad // esize
        self.raw = torch.empty(n + 2 * self.pad, dtype=dtype, device=device)
        self.raw.view(torch.uint8).fill_(SENTINEL)
        self.t = self.raw[self.pad: self.pad + n].view(shape)

    def intact(self) -> bool:
        b = self.raw.view(torch.uint8)
        nb = self.pad * self.raw.element_size()
        return bool((b[:nb] == SENTINEL).all()) and bool((b[-nb:] == SENTINEL).all())


def assert_gemm_close(got: np.ndarray, ref: np.ndarray, what: str, rms=None):
    if rms is None:
        rms = float(np.sqrt(np.mean(ref ** 2))) if ref.size else 0.0
    ok, worst = oracle.within_tolerance(got, ref, rms)
    if not ok:
        bound = 2.0 ** -7 * np.abs(ref) + 1e-3 * rms
        bad = np.argwhere(np.abs(got - ref) > bound)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} elements out of tolerance (worst err/bound "
                             f"{worst:.3g}); first at {i}: got {got[i]!r} ref {ref[i]!r}")
    return worst

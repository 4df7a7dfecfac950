"""Seeded synthetic inputs for the Float8 linear layer.

This module holds the workload table (shapes, value distributions, seeds) and
a counter-based generator of bf16 bit patterns.  It is shared by the tests,
the benchmark and the CPU oracle's callers, and it contains none of the
method's arithmetic: no FP8 format, no amax, no scale, no GEMM.

The shapes are those of the linear layers of Llama-3.1 8B / 70B / 405B
(tokens x in-features, out-features x in-features).  The pages use Llama 3.1
8B/70B/405B as the models on which Float8 training was measured ("TorchTitan:
a one-stop PyTorch-native solution for production LLM pre-training", section 7.3
"Sensitivity ranking" and section 5 "Architecture trade-offs"); no dataset,
tokenizer or trained weight is involved: only the shapes are used.

Generator (all steps are fixed so a reader can re-derive every bit):

* splitmix64 (Steele, Lea, Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014) as a counter-based generator: the stream key is
  splitmix64 of (seed << 32 | tensor id); draw j of element i is
  splitmix64(key + 2 i + j), j in {0, 1}.
* uniforms u = ((z >> 11) + 0.5) * 2^-53, strictly inside (0, 1);
* normals by Box-Muller, sqrt(-2 ln u0) * cos(2 pi u1) * std (one normal per
  pair of draws);
* Laplace(0, b) by the inverse CDF: t = u0 - 1/2, x = -b sgn(t) ln(1 - 2|t|);
* everything computed in binary64, rounded to binary32, then to bf16 with
  round-to-nearest-even on the bit pattern;
* outliers (70B case): floor(0.001 * M * K) distinct positions drawn with
  numpy's PCG64 generator seeded with the stream key; the value at each is
  replaced by bf16_RN(x * 100) (x * 100 is exact in binary32).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_GOLDEN = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_MASK = (1 << 64) - 1

# Tensor ids inside one workload's stream family.
X, W, DY, W3, DY3 = 0, 1, 2, 3, 4


def splitmix64_int(x: int) -> int:
    """splitmix64 mix of one 64-bit integer (Python ints)."""
    z = (x + _GOLDEN) & _MASK
    z = ((z ^ (z >> 30)) * _M1) & _MASK
    z = ((z ^ (z >> 27)) * _M2) & _MASK
    return z ^ (z >> 31)


def _splitmix64(x: np.ndarray) -> np.ndarray:
    z = x + np.uint64(_GOLDEN)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tensor_id: int) -> int:
    return splitmix64_int(((seed & 0xFFFFFFFF) << 32) | (tensor_id & 0xFFFFFFFF))


def _uniform(key: int, idx: np.ndarray, j: int) -> np.ndarray:
    ctr = np.uint64(key) + np.uint64(2) * idx + np.uint64(j)
    z = _splitmix64(ctr)
    return ((z >> np.uint64(11)).astype(np.float64) + 0.5) * (2.0 ** -53)


def f32_to_bf16_bits(f: np.ndarray) -> np.ndarray:
    """Round binary32 values to bf16 bit patterns (nearest, ties to even)."""
    b = np.ascontiguousarray(f, dtype=np.float32).view(np.uint32)
    b = b + np.uint32(0x7FFF) + ((b >> np.uint32(16)) & np.uint32(1))
    return (b >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def _fill_chunk(out: np.ndarray, lo: int, hi: int, key: int, dist: str, param: float) -> None:
    idx = np.arange(lo, hi, dtype=np.uint64)
    u0 = _uniform(key, idx, 0)
    u1 = _uniform(key, idx, 1)
    if dist == "normal":
        x = np.sqrt(-2.0 * np.log(u0)) * np.cos(2.0 * math.pi * u1) * param
    elif dist == "laplace":
        t = u0 - 0.5
        x = -param * np.sign(t) * np.log1p(-2.0 * np.abs(t))
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    out[lo:hi] = f32_to_bf16_bits(x.astype(np.float32))


_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_SO = os.path.join(_HERE, "_build", "libgen.so")
_lib = None
_DISTS = {"normal": 0, "laplace": 1}


def build(force: bool = False) -> str:
    """Compile gen.c with gcc (OpenMP) into workloads/_build/libgen.so."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
                    "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        lib.gen_bf16.restype = None
        lib.gen_bf16.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_uint64,
                                 ctypes.c_int, ctypes.c_double]
        _lib = lib
    return _lib


def generate_reference(n: int, dist: str, param: float, seed: int, tensor_id: int) -> np.ndarray:
    """The same stream as generate(), written in numpy (slow; small n only).
    Used to cross-check the C generator."""
    out = np.empty(n, dtype=np.uint16)
    _fill_chunk(out, 0, n, stream_key(seed, tensor_id), dist, param)
    return out


def generate(shape, dist: str, param: float, seed: int, tensor_id: int,
             outlier_frac: float = 0.0, outlier_mult: float = 100.0) -> np.ndarray:
    """bf16 bit patterns (uint16, C order) of one seeded synthetic tensor."""
    n = int(np.prod(shape))
    key = stream_key(seed, tensor_id)
    out = np.empty(n, dtype=np.uint16)
    if n:
        _load().gen_bf16(out.ctypes.data, n, key, _DISTS[dist], float(param))
    if outlier_frac > 0.0 and n > 0:
        count = int(math.floor(outlier_frac * n))
        rng = np.random.Generator(np.random.PCG64(key))
        pos = rng.choice(n, size=count, replace=False)
        vals = bf16_bits_to_f32(out[pos]) * np.float32(outlier_mult)
        out[pos] = f32_to_bf16_bits(vals)
    return out.reshape(shape)


@dataclass(frozen=True)
class Workload:
    """One linear layer: X [M x K], W [N x K], dY [M x N], all bf16."""
    name: str
    M: int
    K: int
    N: int
    x: tuple           # (distribution, parameter)
    w: tuple
    dy: tuple
    seed: int
    x_outlier_frac: float = 0.0
    note: str = ""
    tags: tuple = field(default_factory=tuple)

    @property
    def flops(self) -> int:
        """fwd + dgrad + wgrad: three GEMMs of 2 M N K flops each."""
        return 6 * self.M * self.N * self.K

    def make_x(self) -> np.ndarray:
        return generate((self.M, self.K), *self.x, seed=self.seed, tensor_id=X,
                        outlier_frac=self.x_outlier_frac)

    def make_w(self, tensor_id: int = W) -> np.ndarray:
        return generate((self.N, self.K), *self.w, seed=self.seed, tensor_id=tensor_id)

    def make_dy(self, tensor_id: int = DY) -> np.ndarray:
        return generate((self.M, self.N), *self.dy, seed=self.seed, tensor_id=tensor_id)


WORKLOADS = {
    "tiny": Workload("tiny", 256, 512, 1024, ("normal", 1.0), ("normal", 0.02),
                     ("normal", 1.0), seed=0),
    "llama3_8b_qkv": Workload("llama3_8b_qkv", 8192, 4096, 6144, ("normal", 1.0),
                              ("normal", 0.02), ("normal", 1e-3), seed=1,
                              note="Llama-3.1-8B fused QKV projection, 1 x 8192 tokens"),
    "llama3_8b_o": Workload("llama3_8b_o", 8192, 4096, 4096, ("normal", 1.0), ("normal", 0.02),
                            ("normal", 1e-3), seed=6,
                            note="Llama-3.1-8B attention output projection (used by the whole-block step)"),
    "llama3_8b_ffn_w13": Workload("llama3_8b_ffn_w13", 8192, 4096, 14336, ("normal", 1.0),
                                  ("normal", 0.02), ("normal", 1e-3), seed=2,
                                  note="Llama-3.1-8B SwiGLU FFN w1 (= w3 shape)"),
    "llama3_8b_ffn_w2": Workload("llama3_8b_ffn_w2", 8192, 14336, 4096, ("normal", 1.0),
                                 ("normal", 0.02), ("normal", 1e-3), seed=3,
                                 note="Llama-3.1-8B SwiGLU FFN w2"),
    "llama3_70b_ffn_w1": Workload("llama3_70b_ffn_w1", 16384, 8192, 28672, ("normal", 1.0),
                                  ("normal", 0.01), ("normal", 1e-3), seed=4,
                                  x_outlier_frac=1e-3,
                                  note="Llama-3.1-70B FFN w1, 2 x 8192 tokens, 0.1% x100 outliers in X"),
    "llama3_405b_ffn_w1": Workload("llama3_405b_ffn_w1", 8192, 16384, 53248, ("normal", 1.0),
                                   ("normal", 0.006), ("laplace", 1e-3), seed=5,
                                   note="Llama-3.1-405B FFN w1, dY Laplace"),
}

# The Llama-3.1-8B SwiGLU FFN as one training step: w1 and w3 read the same
# X [8192 x 4096] with their own weights (tensor ids W and W3) and output
# gradients (DY and DY3); w2 reads the hidden activation [8192 x 14336].
FFN_8B = ("llama3_8b_ffn_w13", "llama3_8b_ffn_w2")

"""The seeded input generator: C and numpy restatements agree, streams are
deterministic and distinct, and the value distributions are as stated."""
import numpy as np
import pytest

import workloads as wl


@pytest.mark.parametrize("dist,param", [("normal", 1.0), ("normal", 0.02), ("laplace", 1e-3)])
def test_c_generator_matches_numpy_restatement(dist, param):
    n = 50_000
    c = wl.generate((n,), dist, param, seed=4, tensor_id=2)
    r = wl.generate_reference(n, dist, param, seed=4, tensor_id=2)
    # both follow the same steps; libm last-ulp differences may flip a rare bf16 rounding
    assert (c == r).mean() >= 0.9999


def test_streams_deterministic_and_distinct():
    a = wl.generate((1000,), "normal", 1.0, 1, 0)
    b = wl.generate((1000,), "normal", 1.0, 1, 0)
    c = wl.generate((1000,), "normal", 1.0, 1, 1)
    d = wl.generate((1000,), "normal", 1.0, 2, 0)
    assert np.array_equal(a, b)
    assert (a != c).mean() > 0.9 and (a != d).mean() > 0.9


@pytest.mark.parametrize("dist,param,std", [("normal", 0.02, 0.02), ("laplace", 1e-3, np.sqrt(2) * 1e-3)])
def test_moments(dist, param, std):
    x = wl.bf16_bits_to_f32(wl.generate((400_000,), dist, param, 0, 0)).astype(np.float64)
    assert abs(x.mean()) < 5 * std / np.sqrt(x.size)
    assert abs(x.std() / std - 1) < 0.01


def test_outliers():
    w = wl.WORKLOADS["llama3_70b_ffn_w1"]
    shape = (256, 512)
    base = wl.generate(shape, "normal", 1.0, w.seed, wl.X)
    out = wl.generate(shape, "normal", 1.0, w.seed, wl.X, outlier_frac=1e-3)
    changed = base != out
    n = int(np.floor(1e-3 * base.size))
    # positions whose value is non-zero change; x100 of a bf16 value is exact in fp32
    assert changed.sum() <= n and changed.sum() >= n - 2
    bf = wl.bf16_bits_to_f32(base)[changed] * np.float32(100)
    assert np.array_equal(wl.f32_to_bf16_bits(bf), out[changed])


def test_bf16_rounding_ties_to_even():
    f = np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, 1.0 + 2.0 ** -9], dtype=np.float32)
    assert list(wl.f32_to_bf16_bits(f)) == [0x3F80, 0x3F82, 0x3F80]


def test_workload_table():
    w = wl.WORKLOADS["llama3_8b_ffn_w13"]
    assert (w.M, w.K, w.N) == (8192, 4096, 14336)
    assert w.flops == 6 * 8192 * 4096 * 14336
    for w in wl.WORKLOADS.values():
        assert w.M % 16 == 0 and w.K % 16 == 0 and w.N % 16 == 0

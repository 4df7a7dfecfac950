"""Pins for the oracle's amax, scale, cast-of-a-tensor and transpose (CPU).

* amax against numpy's max(|x|) in float64 and hand-built special cases;
* scale against a second route: the binary64 quotient rounded to binary32
  (division is correctly rounded through binary64, since 53 >= 2*24 + 2);
* the invariant that the element(s) at |amax| cast to +-448 exactly, on
  tensors drawn like every workload, for both formats;
* transpose against numpy's .T.
"""
import numpy as np
import pytest

import oracle
import workloads as wl

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def _bits(v):
    v = np.asarray(v, dtype=np.float32)
    b = (v.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(wl.bf16_bits_to_f32(b), v)
    return b


def test_amax_matches_numpy_on_random_tensors():
    for seed in range(5):
        x = wl.generate((333, 77), "normal", 10.0 ** (seed - 2), seed, 0)
        ref = np.max(np.abs(wl.bf16_bits_to_f32(x).astype(np.float64)))
        assert oracle.amax(x) == np.float32(ref)


def test_amax_special_cases():
    assert oracle.amax(np.zeros(0, np.uint16)) == 0.0
    assert oracle.amax(_bits([0.0, -0.0])) == 0.0
    assert oracle.amax(_bits([0.0, 0.0, -3.5, 0.0])) == 3.5          # single non-zero, negative
    assert oracle.amax(_bits([1.0, -2.0, 2.0])) == 2.0
    assert oracle.amax(np.array([0x0001], np.uint16)) == np.float32(2.0 ** -133)  # bf16 subnormal
    assert oracle.amax(_bits([1.0, np.inf, -5.0])) == np.inf
    # NaN lies above +Inf in totalOrder: amax is that NaN
    a = oracle.amax(np.array([0x3F80, 0x7F80, 0xFFC1], np.uint16))
    assert np.isnan(a) and np.float32(a).view(np.uint32) == np.uint32(0x7FC10000)


@pytest.mark.parametrize("amax", [1.0, 3.0, 5.34375, 0.004638671875, 2.0 ** -133, 0.0,
                                  1e-12, 7.0e30, 0.1, 123.0])
@pytest.mark.parametrize("fmt_max", [448.0, 57344.0])
def test_scale_second_route(amax, fmt_max):
    a32 = np.float32(amax)
    s, inv = oracle.scale(a32, fmt_max)
    floor = np.float32(1e-12)
    a_used = a32 if a32 >= floor else floor
    exp_s = np.float32(float(np.float32(fmt_max)) / float(a_used))
    exp_inv = np.float32(1.0 / float(exp_s))
    assert s == exp_s and inv == exp_inv


def test_scale_nan_propagates():
    # a NaN amax (any sign or payload) gives NaN scales, stored as the GPU's
    # one binary32 NaN, 0x7FFFFFFF
    for bits in (0x7FC00000, 0xFFC00000, 0x7F800001, 0x7FFF0000):
        s, inv = oracle.scale(np.array([bits], np.uint32).view(np.float32)[0], 448.0)
        assert np.float32(s).view(np.uint32) == 0x7FFFFFFF and np.float32(inv).view(np.uint32) == 0x7FFFFFFF
    assert np.float32(oracle.quantize_static(np.zeros((1, 16), np.uint16), 0, np.nan)["inv_scale"]).view(
        np.uint32) == 0x7FFFFFFF


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
@pytest.mark.parametrize("which", ["x", "w", "dy"])
def test_amax_element_casts_to_fmt_max(name, which):
    w = wl.WORKLOADS[name]
    dist = getattr(w, which)
    x = wl.generate((96, 160), *dist, seed=w.seed, tensor_id=11,
                    outlier_frac=w.x_outlier_frac if which == "x" else 0.0)
    fmt = E5M2 if which == "dy" else E4M3
    res = oracle.quantize(x, fmt)
    xf = wl.bf16_bits_to_f32(x)
    at = np.abs(xf) == res["amax"]
    assert at.any()
    code448 = {E4M3: 0x7E, E5M2: 0x5F}[fmt]
    assert np.all(res["q"][at & (xf > 0)] == code448)
    assert np.all(res["q"][at & (xf < 0)] == code448 | 0x80)
    # nothing else exceeds it
    dec = oracle.decode_table(fmt)[res["q"]]
    assert np.nanmax(np.abs(dec)) == 448.0


def test_all_zero_tensor_casts_to_zero_codes():
    x = _bits(np.zeros((16, 32)))
    res = oracle.quantize(x, E4M3)
    assert res["amax"] == 0.0 and np.all(res["q"] == 0)
    assert res["scale"] == np.float32(448.0 / float(np.float32(1e-12)))


def test_cast_is_elementwise_of_encode():
    x = wl.generate((64, 48), "normal", 1.0, 3, 0)
    s = np.float32(83.8)
    q = oracle.cast(x, E4M3, s)
    v = wl.bf16_bits_to_f32(x) * s
    assert np.array_equal(q, oracle.encode(E4M3, v))


def test_transpose_matches_numpy():
    rng = np.random.default_rng(1)
    q = rng.integers(0, 256, size=(48, 80), dtype=np.uint8)
    assert np.array_equal(oracle.transpose(q), q.T)


def test_dequantised_tensor_is_close_to_input():
    # the method's premise: x ~= dec(q) * inv_scale to within e4m3's half-ulp
    x = wl.generate((128, 128), "normal", 1.0, 9, 0)
    r = oracle.quantize(x, E4M3)
    xf = wl.bf16_bits_to_f32(x).astype(np.float64)
    back = oracle.decode_table(E4M3)[r["q"]] * float(r["inv_scale"])
    rel = np.abs(back - xf) / np.maximum(np.abs(xf), 2.0 ** -6 * float(r["inv_scale"]))
    assert rel.max() <= 2.0 ** -4 * 1.0001

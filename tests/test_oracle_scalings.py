"""Pins for the oracle's static and delayed scaling (CPU).

* history max against numpy's max over the other slots; NaN ordering;
* delayed scaling whose earlier slots hold this tensor's own amax is the
  dynamic recipe exactly (closed form);
* with a stale (smaller) history, exactly the elements with |x * scale| at or
  above the format's largest finite value saturate (a property computed
  independently with numpy);
* static scaling's inverse against the binary64 quotient rounded to binary32,
  its codes against the cast definition, its amax against numpy.
"""
import numpy as np
import pytest

import oracle
import workloads as wl

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def test_history_max_matches_numpy():
    rng = np.random.default_rng(2)
    for n in (2, 3, 16, 1000):
        h = rng.uniform(0, 10, n).astype(np.float32)
        for skip in (0, n // 2, n - 1):
            ref = np.max(np.delete(h, skip))
            assert oracle.history_max(h, skip) == ref


def test_history_max_special_cases():
    h = np.zeros(4, np.float32)
    assert oracle.history_max(h, 1) == 0.0
    h = np.array([1.0, 99.0, 2.0], np.float32)
    assert oracle.history_max(h, 1) == 2.0             # the skipped slot is left out
    h = np.array([1.0, np.inf, np.nan], np.float32)
    assert np.isnan(oracle.history_max(h, 0))          # NaN ranks above Inf
    assert oracle.history_max(h, 2) == np.inf


@pytest.mark.parametrize("fmt,dist", [(E4M3, ("normal", 1.0)), (E5M2, ("laplace", 1e-3))])
def test_delayed_with_own_amax_is_dynamic(fmt, dist):
    x = wl.generate((96, 160), *dist, seed=3, tensor_id=1)
    dyn = oracle.quantize(x, fmt)
    hist = np.zeros(8, np.float32)
    hist[[0, 3, 7]] = dyn["amax"]
    hist[5] = dyn["amax"] * np.float32(0.5)
    d = oracle.quantize_delayed(x, fmt, hist, slot=3)
    assert d["scale"] == dyn["scale"] and d["inv_scale"] == dyn["inv_scale"]
    assert np.array_equal(d["q"], dyn["q"]) and np.array_equal(d["qT"], dyn["qT"])
    assert d["history"][3] == dyn["amax"] and np.array_equal(np.delete(d["history"], 3), np.delete(hist, 3))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_delayed_with_stale_history_saturates_exactly_the_overflow(fmt):
    x = wl.generate((128, 128), "normal", 1.0, 5, 2)
    a = oracle.amax(x)
    hist = np.array([a * np.float32(0.5), 0.0, a * np.float32(0.25)], np.float32)
    d = oracle.quantize_delayed(x, fmt, hist, slot=1)
    s = d["scale"]
    assert s == np.float32(448.0) / (a * np.float32(0.5))
    v = np.abs(wl.bf16_bits_to_f32(x) * s)
    code = d["q"] & 0x7F
    if fmt == E4M3:
        # largest finite 448 (0x7E); its lower neighbour is 416, the midpoint
        # 432 ties to the even code 448: the top code holds exactly v >= 432,
        # and every v >= 448 (the overflow of the stale scale) is in it
        assert np.array_equal(code == 0x7E, v >= 432.0)
        assert (v >= 448.0).any()
    else:
        # e5m2 reaches 57344: the doubled amax only climbs to ~896, nothing saturates
        assert not (code == 0x7B).any() and v.max() < 1024
    assert d["history"][1] == a


def test_static_scaling():
    x = wl.generate((64, 80), "normal", 0.02, 7, 1)
    for s in (np.float32(1.0), np.float32(1000.0), np.float32(0.37), np.float32(2.0 ** 20)):
        r = oracle.quantize_static(x, E4M3, s)
        assert r["inv_scale"] == np.float32(1.0 / float(s))
        assert np.array_equal(r["q"], oracle.cast(x, E4M3, s))
        assert np.array_equal(r["qT"], r["q"].T)
        assert r["amax"] == np.float32(np.max(np.abs(wl.bf16_bits_to_f32(x))))

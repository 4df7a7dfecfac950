"""Pins for the oracle's scaled FP8 GEMMs (CPU).

* exact rational arithmetic (Python integers) on tiny shapes: FP8 values are
  integers times 2^-9 (e4m3) or 2^-16 (e5m2), so the true sum is an exact
  integer; the oracle's binary64 sum must equal it;
* a hand-worked 2x2 . 2x3 case (tests/golden/gemm_hand_case.txt);
* closed forms: one-hot rows copy a column of B, all-ones gives R;
* numpy's float64 matmul of the decoded operands (a library routine) for
  the three GEMMs of the linear, wired through the transposed copies exactly
  as the layer uses them: Y = X.W^T, dX = dY.W, dW = dY^T.X.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl
from conftest import GOLDEN

E4M3, E5M2 = oracle.E4M3, oracle.E5M2
FMTS = {"e4m3": E4M3, "e5m2": E5M2}


def _random_codes(rng, shape, fmt, limit=np.inf):
    """Random finite codes with |value| <= limit."""
    table = oracle.decode_table(fmt)
    ok = np.nonzero(np.isfinite(table) & (np.abs(table) <= limit))[0]
    return rng.choice(ok, size=shape).astype(np.uint8)


def _exact_value(fmt, code) -> Fraction:
    v = oracle.decode_table(fmt)[code]
    return Fraction(float(v))   # binary64 holds every FP8 value exactly


@pytest.mark.parametrize("fa,fb", [(E4M3, E4M3), (E5M2, E4M3), (E5M2, E5M2)])
@pytest.mark.parametrize("P,Q,R", [(1, 1, 1), (3, 5, 7), (8, 4, 33), (5, 9, 64)])
def test_exact_sum_on_tiny_shapes(fa, fb, P, Q, R):
    """Codes as the cast produces them (|v| <= 448): every product lies on a
    grid of 2^-25 (or coarser) below 2^18, so R <= 2^10 terms sum exactly in
    binary64 and the oracle must return the exact rational sum."""
    rng = np.random.default_rng(P * 100 + Q * 10 + R)
    A = _random_codes(rng, (P, R), fa, 448.0)
    B = _random_codes(rng, (Q, R), fb, 448.0)
    got = oracle.gemm_rows(A, fa, B, fb, 1.0, 1.0)
    for p in range(P):
        for q in range(Q):
            exact = sum(_exact_value(fa, A[p, k]) * _exact_value(fb, B[q, k]) for k in range(R))
            assert Fraction(got[p, q]) == exact


@pytest.mark.parametrize("R", [7, 64, 300])
def test_full_range_e5m2_within_recursive_summation_bound(R):
    """Over e5m2's whole range the products span more than 53 bits, so the
    binary64 sum is not exact; it must stay within the textbook bound for
    recursive summation, |err| <= (R - 1) u sum|a_k b_k| with u = 2^-53."""
    rng = np.random.default_rng(R)
    A = _random_codes(rng, (4, R), E5M2)
    B = _random_codes(rng, (5, R), E5M2)
    got = oracle.gemm_rows(A, E5M2, B, E5M2, 1.0, 1.0)
    for p in range(4):
        for q in range(5):
            terms = [_exact_value(E5M2, A[p, k]) * _exact_value(E5M2, B[q, k]) for k in range(R)]
            exact = sum(terms)
            bound = (R - 1) * Fraction(1, 2 ** 53) * sum(abs(t) for t in terms)
            assert abs(Fraction(got[p, q]) - exact) <= bound


def test_inverse_scales_applied_after_the_sum():
    rng = np.random.default_rng(3)
    A = _random_codes(rng, (4, 16), E4M3)
    B = _random_codes(rng, (6, 16), E5M2)
    ia, ib = np.float32(0.0119280135), np.float32(3.1e-6)
    got = oracle.gemm_rows(A, E4M3, B, E5M2, ia, ib)
    base = oracle.gemm_rows(A, E4M3, B, E5M2, 1.0, 1.0)
    exact = np.array([[float(Fraction(base[p, q]) * Fraction(float(ia)) * Fraction(float(ib)))
                       for q in range(6)] for p in range(4)])
    np.testing.assert_allclose(got, exact, rtol=4 * 2.0 ** -53, atol=0)


def test_golden_hand_case():
    mats, inv, C = {}, None, None
    with open(os.path.join(GOLDEN, "gemm_hand_case.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            t = line.split()
            if t[0] in ("A", "B"):
                r, c = int(t[2]), int(t[3])
                mats[(t[0], FMTS[t[1]])] = np.array([int(v, 16) for v in t[4:]], np.uint8).reshape(r, c)
            elif t[0] == "inv":
                inv = (float(t[1]), float(t[2]))
            elif t[0] == "C":
                r, c = int(t[1]), int(t[2])
                C = np.array([float(v) for v in t[3:]]).reshape(r, c)
    B = mats[("B", E4M3)]
    for fa in (E4M3, E5M2):
        got = oracle.gemm_rows(mats[("A", fa)], fa, B, E4M3, *inv)
        assert np.array_equal(got, C)


def test_one_hot_rows_copy_a_column():
    rng = np.random.default_rng(5)
    R, Q = 40, 24
    B = _random_codes(rng, (Q, R), E4M3)
    A = np.zeros((R, R), np.uint8)
    A[np.arange(R), np.arange(R)] = 0x38      # e4m3 1.0
    got = oracle.gemm_rows(A, E4M3, B, E4M3, 1.0, 1.0)
    assert np.array_equal(got, oracle.decode_table(E4M3)[B].T)


def test_all_ones():
    R = 4096
    A = np.full((2, R), 0x3C, np.uint8)        # e5m2 1.0
    B = np.full((3, R), 0x38, np.uint8)        # e4m3 1.0
    assert np.all(oracle.gemm_rows(A, E5M2, B, E4M3, 1.0, 1.0) == R)


def test_row_selection():
    rng = np.random.default_rng(11)
    A = _random_codes(rng, (20, 32), E4M3)
    B = _random_codes(rng, (8, 32), E4M3)
    full = oracle.gemm_rows(A, E4M3, B, E4M3, 0.5, 0.25)
    rows = np.array([19, 0, 7, 7])
    assert np.array_equal(oracle.gemm_rows(A, E4M3, B, E4M3, 0.5, 0.25, rows), full[rows])


def test_three_gemms_of_the_linear_match_numpy_matmul():
    """Wiring of fwd / dgrad / wgrad through the transposed copies."""
    M, K, N = 48, 80, 64
    X = wl.generate((M, K), "normal", 1.0, 21, 0)
    W = wl.generate((N, K), "normal", 0.02, 21, 1)
    dY = wl.generate((M, N), "normal", 1e-3, 21, 2)
    qx = oracle.quantize(X, E4M3)
    qw = oracle.quantize(W, E4M3)
    qd = oracle.quantize(dY, E5M2)
    d4, d5 = oracle.decode_table(E4M3), oracle.decode_table(E5M2)
    Xd = d4[qx["q"]] * float(qx["inv_scale"])
    Wd = d4[qw["q"]] * float(qw["inv_scale"])
    Dd = d5[qd["q"]] * float(qd["inv_scale"])

    Y = oracle.fwd_ref(qx["q"], qx["inv_scale"], qw["q"], qw["inv_scale"])
    dX = oracle.dgrad_ref(qd["q"], qd["inv_scale"], qw["qT"], qw["inv_scale"])
    dW = oracle.wgrad_ref(qd["qT"], qd["inv_scale"], qx["qT"], qx["inv_scale"])
    for got, ref in ((Y, Xd @ Wd.T), (dX, Dd @ Wd), (dW, Dd.T @ Xd)):
        # different summation orders: allow binary64 rounding relative to the
        # output's scale (a cancelled sum has a large relative error)
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13 * np.abs(ref).max())
    assert Y.shape == (M, N) and dX.shape == (M, K) and dW.shape == (N, K)

    # and the FP8 result approximates the bf16 product (the method's point)
    Xf = wl.bf16_bits_to_f32(X).astype(np.float64)
    Wf = wl.bf16_bits_to_f32(W).astype(np.float64)
    Df = wl.bf16_bits_to_f32(dY).astype(np.float64)
    for got, true in ((Y, Xf @ Wf.T), (dX, Df @ Wf), (dW, Df.T @ Xf)):
        rel = np.linalg.norm(got - true) / np.linalg.norm(true)
        assert rel < 0.08


def test_tolerance_helper():
    ref = np.array([1.0, -2.0, 0.0])
    rms = float(np.sqrt(np.mean(ref ** 2)))
    ok, _ = oracle.within_tolerance(ref * (1 + 2.0 ** -8), ref, rms)
    assert ok
    ok, _ = oracle.within_tolerance(ref * (1 + 2.0 ** -6), ref, rms)
    assert not ok

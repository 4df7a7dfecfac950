"""Pins for the oracle's power-of-two block scaling (CPU).

* the exponent rule against an exact rational check of its definition
  (2^e the largest power of two with max(amax, 1e-12) 2^e <= fmt_max) on
  thousands of random and edge-case amax values and several fmt_max, plus
  hand-worked cases (448 -> e = 0, 449 -> e = -1, 1 -> e = 8, ...);
* a block whose amax is fmt_max / 2^e casts exactly like per-tensor scaling
  with that scale (pinned elsewhere), so the cast wiring is tied to the
  pinned per-tensor cast;
* in every block the largest magnitude lands in the top binade below
  fmt_max and nothing saturates (the defining property of the rule);
* 32 x 1 blocks of x are 1 x 32 blocks of x^T;
* the GEMM refs against numpy's float64 matmul of the dequantised operands
  (exact: the inverse scales are powers of two), and one small case against
  exact rationals, so a transposed operand or a scale taken from the wrong
  block shows;
* the scale-atom layout: a bijection from (operand row, block) to atom
  bytes with every other byte 127, and a few offsets worked by hand.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def _rule_holds(amax: float, fmt_max: float, byte: int) -> bool:
    """The definition, in exact rationals: e = 127 - byte is the largest
    integer with a * 2^e <= fmt_max (a = max(amax, 1e-12f)), clamped."""
    a = Fraction(max(float(np.float32(amax)), float(np.float32(1e-12))))
    f = Fraction(float(np.float32(fmt_max)))
    e = 127 - byte
    two = Fraction(2)
    if e == 127:
        return a * two ** 127 <= f
    if e == -127:
        return a * two ** -126 > f
    return a * two ** e <= f < a * two ** (e + 1)


@pytest.mark.parametrize("fmt_max", [448.0, 57344.0, 1.0, 3.0, 1e-20, 1e30])
def test_exponent_rule_against_its_definition(fmt_max):
    rng = np.random.default_rng(7)
    with np.errstate(over="ignore"):
        amax = _amax_cases(rng, fmt_max)
    amax = amax[np.isfinite(amax)]
    got = oracle.pow2_scale_bytes(amax, fmt_max)
    for a, b in zip(amax, got):
        assert _rule_holds(float(a), fmt_max, int(b)), (a, b)


def _amax_cases(rng, fmt_max):
    return np.concatenate([
        np.ldexp(rng.uniform(1.0, 2.0, 3000), rng.integers(-60, 60, 3000)).astype(np.float32),
        np.float32(fmt_max) * np.ldexp(1.0, np.arange(-40, 41)).astype(np.float32),   # exact powers
        np.nextafter(np.float32(fmt_max) * np.ldexp(1.0, np.arange(-5, 6)).astype(np.float32), np.float32(np.inf)),
        np.array([0.0, 1e-13, 1e-12, 3.3895314e38], np.float32),
    ]).astype(np.float32)


def test_exponent_rule_hand_cases():
    # (amax, fmt_max) -> e = 127 - byte, worked by hand:
    # 448 * 2^0 <= 448; 449 > 448 so 2^-1; 224 * 2 = 448; 1 * 256 <= 448 < 512;
    # 0 floors to 1e-12 and 1e-12 * 2^48 = 281.5 <= 448 < 563; 57344 (e5m2 max) at 448: 2^-7
    cases = [(448.0, 448.0, 0), (449.0, 448.0, -1), (224.0, 448.0, 1), (1.0, 448.0, 8), (0.0, 448.0, 48),
             (57344.0, 448.0, -7), (57344.0, 57344.0, 0), (1.0, 57344.0, 15), (0.75, 1.0, 0), (1.5, 1.0, -1)]
    for a, f, e in cases:
        assert int(oracle.pow2_scale_bytes(np.array([a], np.float32), f)[0]) == 127 - e, (a, f, e)
    nonfinite = oracle.pow2_scale_bytes(np.array([np.inf, np.nan], np.float32), 448.0)
    assert nonfinite.tolist() == [255, 255]


def test_scale_values_are_exact_powers_of_two():
    b = np.arange(0, 255, dtype=np.uint8)
    s, inv = oracle.pow2_scale(b), oracle.pow2_inverse(b)
    for byte, sv, iv in zip(b, s, inv):
        assert Fraction(float(sv)) == Fraction(2) ** (127 - int(byte))
        assert Fraction(float(iv)) == Fraction(2) ** (int(byte) - 127)
    assert np.isnan(oracle.pow2_scale(np.array([255], np.uint8))[0])


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_block_at_a_power_of_two_amax_is_per_tensor_scaling(fmt):
    # one 1 x 32 block whose amax is 448 / 8: the power-of-two scale is 8,
    # exactly per-tensor scaling's 448 / amax, so the codes must agree
    x = wl.generate((1, 32), "normal", 1.0, 21, fmt)
    xf = wl.bf16_bits_to_f32(x).astype(np.float32)
    k = int(np.argmax(np.abs(xf)))
    xf[0, k] = np.float32(56.0) * np.sign(xf[0, k])
    x = wl.f32_to_bf16_bits(xf)
    m = oracle.quantize_mx(x, fmt, "cols")
    t = oracle.quantize(x, fmt)
    assert float(t["scale"]) == 8.0 and float(m["scale"][0, 0]) == 8.0
    assert np.array_equal(m["q"], t["q"])


@pytest.mark.parametrize("along", ["cols", "rows"])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_block_amax_top_binade_and_no_saturation(along, fmt):
    x = wl.generate((96, 80), "normal", 1.0, 22, 0)          # ragged: 80 = 2.5 blocks of 32
    m = oracle.quantize_mx(x, fmt, along)
    xf = np.abs(wl.bf16_bits_to_f32(x).astype(np.float64))
    dec = np.abs(oracle.decode_table(fmt))
    br, bc = (1, 32) if along == "cols" else (32, 1)
    assert m["amax"].shape == ((96 + br - 1) // br, (80 + bc - 1) // bc)
    for i in range(m["amax"].shape[0]):
        for j in range(m["amax"].shape[1]):
            blk = xf[br * i:br * (i + 1), bc * j:bc * (j + 1)]
            assert m["amax"][i, j] == blk.max()
            s = float(m["scale"][i, j])
            top = blk.max() * s
            assert 224.0 < top <= 448.0          # the largest magnitude lands in [448/2, 448]
            qb = m["q"][br * i:br * (i + 1), bc * j:bc * (j + 1)]
            # nothing saturates: every code is within half a step of x * s
            assert np.all(dec[qb] <= 448.0)
            assert np.all(np.abs(dec[qb] - blk * s) <= 2.0 ** -3 * np.maximum(blk * s, 2.0 ** -6))


def test_column_blocks_are_row_blocks_of_the_transpose():
    x = wl.generate((112, 48), "laplace", 1e-3, 23, 2)
    c = oracle.quantize_mx(x, E5M2, "rows")
    r = oracle.quantize_mx(np.ascontiguousarray(x.T), E5M2, "cols")
    assert np.array_equal(c["sf"], r["sf"].T)
    assert np.array_equal(c["q"], r["q"].T)


def _exact(code, fmt):
    return Fraction(float(oracle.decode_table(fmt)[code]))


def test_mx_gemm_against_exact_rationals():
    rng = np.random.default_rng(24)
    M, N, K = 3, 4, 80                                      # three contraction blocks, the last one short
    X = wl.generate((M, K), "normal", 1.0, 24, wl.X)
    W = wl.generate((N, K), "normal", 0.02, 24, wl.W)
    xk = oracle.quantize_mx(X, E4M3, "cols")
    wk = oracle.quantize_mx(W, E4M3, "cols")
    got = oracle.fwd_mx_ref(xk["q"], xk["sf"], wk["q"], wk["sf"])
    for m in range(M):
        for n in range(N):
            total = Fraction(0)
            for k in range(K):
                j = k // 32
                total += (_exact(xk["q"][m, k], E4M3) * Fraction(2) ** (int(xk["sf"][m, j]) - 127) *
                          _exact(wk["q"][n, k], E4M3) * Fraction(2) ** (int(wk["sf"][n, j]) - 127))
            assert abs(Fraction(got[m, n]) - total) <= abs(total) * Fraction(1, 2 ** 50)
    del rng


def test_mx_recipe_gemms_against_numpy():
    M, K, N = 136, 264, 200
    X = wl.generate((M, K), "normal", 1.0, 25, wl.X)
    W = wl.generate((N, K), "normal", 0.02, 25, wl.W)
    dY = wl.generate((M, N), "normal", 1e-3, 25, wl.DY)
    r = oracle.quantize_mx_recipe(X, W, dY)
    d4, d5 = oracle.decode_table(E4M3), oracle.decode_table(E5M2)

    def deq(t, dec, along):
        inv = oracle.pow2_inverse(t["sf"]).astype(np.float64)
        inv = np.repeat(inv, 32, axis=1 if along == "cols" else 0)
        return dec[t["q"]] * inv[:t["q"].shape[0], :t["q"].shape[1]]

    xk, xm = deq(r["x_k"], d4, "cols"), deq(r["x_m"], d4, "rows")
    wk, wn = deq(r["w_k"], d4, "cols"), deq(r["w_n"], d4, "rows")
    dyn, dym = deq(r["dy_n"], d5, "cols"), deq(r["dy_m"], d5, "rows")
    y = oracle.fwd_mx_ref(r["x_k"]["q"], r["x_k"]["sf"], r["w_k"]["q"], r["w_k"]["sf"])
    dx = oracle.dgrad_mx_ref(r["dy_n"]["q"], r["dy_n"]["sf"], r["w_n"]["q"], r["w_n"]["sf"])
    dw = oracle.wgrad_mx_ref(r["dy_m"]["q"], r["dy_m"]["sf"], r["x_m"]["q"], r["x_m"]["sf"])
    for got, want in ((y, xk @ wk.T), (dx, dyn @ wn), (dw, dym.T @ xm)):
        assert got.shape == want.shape
        assert np.max(np.abs(got - want)) <= 1e-12 * np.abs(want).max()
    # the dequantised copies approximate the bf16 originals to FP8 precision
    xf = wl.bf16_bits_to_f32(X).astype(np.float64)
    assert np.max(np.abs(xk - xf)) <= 2.0 ** -4 * np.abs(xf).max()
    assert np.max(np.abs(xm - xf)) <= 2.0 ** -4 * np.abs(xf).max()


@pytest.mark.parametrize("P,K", [(128, 128), (200, 80), (16, 16), (384, 272)])
def test_scale_atom_layout(P, K):
    nj = (K + 31) // 32
    rng = np.random.default_rng(P * 1000 + K)
    sf = rng.integers(0, 127, size=(P, nj), dtype=np.uint8)      # never 127, so every placed byte is visible
    atoms = oracle.pack_sf(sf, P, K)
    assert atoms.shape == ((K + 127) // 128, (P + 127) // 128, 512)
    assert np.array_equal(oracle.unpack_sf(atoms, P, K), sf)
    # a bijection onto P * nj bytes; everything else is the padding value 127
    assert int(np.count_nonzero(atoms != 127)) == P * nj
    # offsets worked by hand: row 0 block 0 -> byte 0 of atom (0, 0); row 33
    # block 1 -> 16 * 1 + 4 * 1 + 1 = 21; row 127 block 3 -> 16 * 31 + 4 * 3 + 3 = 511
    assert atoms[0, 0, 0] == sf[0, 0]
    if P > 33 and nj > 1:
        assert atoms[0, 0, 21] == sf[33, 1]
    if P >= 128 and nj >= 4:
        assert atoms[0, 0, 511] == sf[127, 3]
    if P > 130 and nj > 5:
        # row 130 (second row block), block 5 (second contraction block): atom (1, 1), 16 * 2 + 0 + 1
        assert atoms[1, 1, 33] == sf[130, 5]


# ---------------------------------------------------------------- OCP rule

@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_ocp_rule_against_its_definition(fmt):
    """byte = 127 + floor(log2 amax) - emax (8 for e4m3, 15 for e5m2), with
    floor(log2 amax) checked in exact rationals: 2^f <= amax < 2^(f + 1)."""
    emax = 8 if fmt == E4M3 else 15
    rng = np.random.default_rng(9)
    amax = np.concatenate([np.ldexp(rng.uniform(1.0, 2.0, 3000), rng.integers(-140, 128, 3000)),
                           np.ldexp(1.0, np.arange(-140, 128))]).astype(np.float32)
    amax = amax[np.isfinite(amax) & (amax > 0)]
    got = oracle.ocp_scale_bytes(amax, fmt)
    for a, b in zip(amax, got):
        fa = Fraction(float(a))
        f = int(b) - 127 + emax
        if b == 0:
            assert fa < Fraction(2) ** (emax - 126), a
        elif b == 254:
            assert fa >= Fraction(2) ** (127 + emax), a
        else:
            assert Fraction(2) ** f <= fa < Fraction(2) ** (f + 1), (a, b)


def test_ocp_rule_hand_cases():
    cases = [(448.0, E4M3, 127), (500.0, E4M3, 127), (1.0, E4M3, 119), (0.0, E4M3, 0),
             (57344.0, E4M3, 134), (448.0, E5M2, 120), (57344.0, E5M2, 127), (65000.0, E5M2, 127)]
    for a, fmt, want in cases:
        assert int(oracle.ocp_scale_bytes(np.array([a], np.float32), fmt)[0]) == want, (a, fmt)
    assert oracle.ocp_scale_bytes(np.array([np.inf, np.nan], np.float32), E4M3).tolist() == [255, 255]


@pytest.mark.parametrize("fmt,fmt_max", [(E4M3, 448.0), (E5M2, 57344.0)])
def test_ocp_rule_is_the_floor_rule_or_one_binade_above(fmt, fmt_max):
    """With fmt_max the format's own maximum (1.75 x 2^emax) the OCP scale is
    the no-saturation rule's scale, or twice it exactly when the block's
    amax scaled into [2^emax, 2^(emax+1)) exceeds fmt_max (and then that
    block's top values saturate)."""
    rng = np.random.default_rng(10)
    amax = np.ldexp(rng.uniform(1.0, 2.0, 5000), rng.integers(-20, 20, 5000)).astype(np.float32)
    fl = oracle.pow2_scale_bytes(amax, fmt_max).astype(int)
    oc = oracle.ocp_scale_bytes(amax, fmt).astype(int)
    mant = np.frexp(amax.astype(np.float64))[0] * 2.0          # amax = mant * 2^f, mant in [1, 2)
    assert np.array_equal(fl - oc, (mant > 1.75).astype(int))


@pytest.mark.parametrize("along", ["cols", "rows"])
def test_ocp_quantize_saturates_only_the_top_of_the_top_binade(along):
    x = wl.generate((96, 80), "normal", 1.0, 26, 0)
    m = oracle.quantize_mx(x, E4M3, along, rule="ocp")
    xf = np.abs(wl.bf16_bits_to_f32(x).astype(np.float64))
    dec = np.abs(oracle.decode_table(E4M3))
    br, bc = (1, 32) if along == "cols" else (32, 1)
    for i in range(m["amax"].shape[0]):
        for j in range(m["amax"].shape[1]):
            blk = xf[br * i:br * (i + 1), bc * j:bc * (j + 1)] * float(m["scale"][i, j])
            assert 256.0 <= blk.max() < 512.0                 # the top magnitude in [2^8, 2^9)
            qb = dec[m["q"][br * i:br * (i + 1), bc * j:bc * (j + 1)]]
            sat = blk > 448.0
            assert np.all(qb[sat] == 448.0)                   # above the format's maximum: saturated
            assert np.all(np.abs(qb[~sat] - blk[~sat]) <= 2.0 ** -4 * np.maximum(blk[~sat], 2.0 ** -6))


def test_ocp_block_of_subnormals_hand_codes():
    """Under the OCP rule a block whose amax is a bf16 subnormal gets the
    scale byte 0 (X = 2^-127, the elements multiplied by 2^127), so its codes
    are not zero: 2^-133 -> 2^-6, 3 * 2^-133 -> 1.5 * 2^-5 and the largest
    bf16 subnormal 127 * 2^-133 -> 1.984375, which rounds to 2 in e4m3 (the
    halfway point is 1.9375) and in e5m2 (halfway 1.875).  Codes from the
    formats' fields: e4m3 = sign | exponent + 7 (4 bits) | 3 mantissa bits,
    e5m2 = sign | exponent + 15 (5 bits) | 2 mantissa bits."""
    x = np.zeros((1, 32), np.uint16)
    x[0, 0], x[0, 1], x[0, 2], x[0, 3] = 0x0001, 0x0003, 0x8001, 0x007F
    want = {E4M3: [0x08, 0x14, 0x88, 0x40], E5M2: [0x24, 0x2A, 0xA4, 0x40]}
    for fmt in (E4M3, E5M2):
        m = oracle.quantize_mx(x, fmt, "cols", rule="ocp")
        assert int(m["sf"][0, 0]) == 0, fmt
        assert m["q"][0, :4].tolist() == want[fmt], fmt
        assert (m["q"][0, 4:] == 0).all()
    # the floor rule floors amax at 1e-12 instead: these elements cast to zero
    m = oracle.quantize_mx(x, E4M3, "cols")
    assert set(m["q"][0].tolist()) <= {0x00, 0x80}

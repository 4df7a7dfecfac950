"""Pins for the oracle's FP8 decode / encode (CPU only).

The oracle's encoder is integer manipulation of binary32 fields; it is pinned
here against things other than itself:

* the published code points of e4m3 / e5m2 (hand-worked, tests/golden);
* torch's own float8 dtypes (a library routine) for decoding all 256 codes
  and for round-to-nearest-even of in-range values;
* an exhaustive brute-force nearest search over the decoded code table, with
  ties to the even code and saturation, over all 65,536 bf16 patterns times
  a set of scales, for both formats.
"""
import os

import numpy as np
import pytest
import torch

import oracle
from conftest import GOLDEN

E4M3, E5M2 = oracle.E4M3, oracle.E5M2
FMTS = {"e4m3": E4M3, "e5m2": E5M2}
TORCH_DT = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


def _parse_num(tok: str) -> float:
    t = tok.strip()
    if "0x" in t.lower() and "p" in t.lower():
        return float.fromhex(t)
    return float(t)


def test_decode_published_code_points():
    d4 = oracle.decode_table(E4M3)
    d5 = oracle.decode_table(E5M2)
    # e4m3 (fn): bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN
    assert d4[0x00] == 0.0 and np.signbit(d4[0x80])
    assert d4[0x01] == 2.0 ** -9 and d4[0x07] == 7 * 2.0 ** -9
    assert d4[0x08] == 2.0 ** -6 and d4[0x38] == 1.0
    assert d4[0x7E] == 448.0 and d4[0xFE] == -448.0
    assert np.isnan(d4[0x7F]) and np.isnan(d4[0xFF])
    assert np.isfinite(d4[[c for c in range(256) if c & 0x7F != 0x7F]]).all()
    # e5m2: bias 15, 2 mantissa bits, exponent 31 = Inf / NaN
    assert d5[0x01] == 2.0 ** -16 and d5[0x04] == 2.0 ** -14 and d5[0x3C] == 1.0
    assert d5[0x7B] == 57344.0 and d5[0x7C] == np.inf and d5[0xFC] == -np.inf
    assert all(np.isnan(d5[c]) for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_matches_torch_float8(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(TORCH_DT[fmt]).to(torch.float64).numpy()
    ours = oracle.decode_table(fmt)
    nan = np.isnan(ref)
    assert np.array_equal(nan, np.isnan(ours))
    assert np.array_equal(ref[~nan], ours[~nan])
    assert np.array_equal(np.signbit(ref[~nan]), np.signbit(ours[~nan]))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_monotone_and_symmetric(fmt):
    d = oracle.decode_table(fmt)
    maxc = 0x7E if fmt == E4M3 else 0x7B
    pos = d[: maxc + 1]
    assert np.all(np.diff(pos) > 0)
    assert np.array_equal(d[0x80: 0x80 + maxc + 1], -pos)


def _brute_force_codes(fmt: int, v: np.ndarray) -> np.ndarray:
    """Nearest finite code of the same sign by exhaustive search; ties go to
    the even code; NaN in gives a NaN code."""
    table = oracle.decode_table(fmt)
    finite = np.isfinite(table)
    codes = np.arange(256)
    out = np.empty(v.shape, dtype=np.uint8)
    vd = v.astype(np.float64)
    sign = np.signbit(vd)
    for s in (False, True):
        cand = codes[finite & (np.signbit(table) == s)]
        cv = table[cand]
        sel = (sign == s) & ~np.isnan(vd)
        vv = vd[sel]
        # beyond 4x the largest finite value every distance is dominated by
        # |v| in binary64; the nearest finite code there is the largest one,
        # so clamp (exactly) to keep the distances distinct
        big = 4.0 * np.nanmax(np.abs(cv))
        vv = np.clip(vv, -big, big)
        dist = np.abs(vv[:, None] - cv[None, :])
        best = dist.min(axis=1, keepdims=True)
        tie = dist == best
        n_tie = tie.sum(axis=1)
        pick = np.argmax(tie, axis=1)
        two = n_tie == 2
        if two.any():
            idx = np.nonzero(two)[0]
            pair = np.array([np.nonzero(tie[i])[0] for i in idx])
            even = np.where(cand[pair[:, 0]] % 2 == 0, pair[:, 0], pair[:, 1])
            pick[idx] = even
        assert n_tie.max() <= 2
        out[sel] = cand[pick]
    out[np.isnan(vd)] = 0x7F
    return out


ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)
SCALES = [1.0, 2.0 ** -8, 2.0 ** 8, np.float32(448.0) / np.float32(3.0),
          np.float32(448.0) / np.float32(5.34375), np.float32(448.0) / np.float32(0.004638671875),
          np.float32(57344.0) / np.float32(7.0), 1.0e-30, 3.0e30]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("scale", SCALES)
def test_cast_exhaustive_vs_brute_force(fmt, scale):
    s = np.float32(scale)
    x = (ALL_BF16.astype(np.uint32) << 16).view(np.float32)
    with np.errstate(over="ignore", invalid="ignore"):
        v = x * s                                   # one binary32 RN multiply
    got = oracle.cast(ALL_BF16, fmt, s)
    nan = np.isnan(v)
    exp = _brute_force_codes(fmt, np.where(nan, 0, v).astype(np.float32))
    # NaN inputs (either sign, any payload) give the one NaN code the GPU's
    # conversion emits, 0x7F, in both formats
    assert nan.sum() == 2 * 127 and (got[nan] == 0x7F).all()
    assert np.array_equal(got[~nan], exp[~nan]), \
        f"first mismatch at bf16 0x{int(ALL_BF16[~nan][got[~nan] != exp[~nan]][0]):04x}"


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_rne_in_range(fmt):
    rng = np.random.default_rng(7)
    maxv = 448.0 if fmt == E4M3 else 57344.0
    allbf = (ALL_BF16.astype(np.uint32) << 16).view(np.float32)
    allbf = allbf[np.isfinite(allbf)].astype(np.float64)
    v = np.concatenate([
        rng.uniform(-maxv, maxv, 20000),
        rng.standard_normal(20000) * 2.0 ** rng.integers(-20, 10, 20000),
        allbf,
    ]).astype(np.float32)
    v = v[np.abs(v) <= maxv]
    ref = torch.from_numpy(v).to(TORCH_DT[fmt]).view(torch.uint8).numpy()
    got = oracle.encode(fmt, v)
    assert np.array_equal(got, ref)


def _golden_cast_rows():
    rows = []
    with open(os.path.join(GOLDEN, "cast_hand_cases.txt")) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            fmt, fmt_max, amax, x, code = line.split()[:5]
            # x is a number, or "bf16:0x...." for a bit pattern (the NaNs)
            xv = int(x[5:], 16) if x.startswith("bf16:") else _parse_num(x)
            rows.append((FMTS[fmt], _parse_num(fmt_max), _parse_num(amax), xv, int(code, 16)))
    return rows


@pytest.mark.parametrize("fmt,fmt_max,amax,x,code", _golden_cast_rows())
def test_golden_hand_cases(fmt, fmt_max, amax, x, code):
    if isinstance(x, int):
        bits = np.array([x], dtype=np.uint16)
    else:
        xb = np.array([x], dtype=np.float32)
        bits = (xb.view(np.uint32) >> 16).astype(np.uint16)
        assert (bits.astype(np.uint32) << 16).view(np.float32)[0] == xb[0], "golden x not bf16-exact"
    s, _ = oracle.scale(amax, fmt_max)
    q = oracle.cast(bits, fmt, s)
    assert int(q[0]) == code, f"got 0x{int(q[0]):02x}"

"""Pins for the oracle's block scaling (CPU).

* a block covering the whole tensor is per-tensor scaling, and one-row
  blocks are row-wise scaling (both already pinned);
* every 128 x 128 block of a ragged matrix is per-tensor scaling of that
  sub-matrix on its own;
* 128 x 1 blocks of x are 1 x 128 blocks of x^T;
* block amax against numpy, and in every block the element at the block's
  amax casts to +-448 exactly;
* the block-scaled GEMM with one contraction block is the row-scaled GEMM
  (pinned), and with several blocks it matches an exact rational brute
  force whose scales differ per row and per block, so a wrong block index,
  a dropped block or a transposed operand shows;
* the fwd / dgrad / wgrad wiring of the block recipe against numpy's
  float64 matmul of the block-dequantised operands.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
import workloads as wl

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def _same(a, b):
    return np.array_equal(np.asarray(a).view(np.uint32), np.asarray(b).view(np.uint32))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_whole_tensor_block_is_per_tensor_scaling(fmt):
    x = wl.generate((72, 200), "normal", 1.0, 11, fmt)
    b = oracle.quantize_blocks(x, fmt, 72, 200)
    t = oracle.quantize(x, fmt)
    assert b["amax"].shape == (1, 1)
    assert _same(b["amax"][0, 0], np.float32(t["amax"]))
    assert _same(b["scale"][0, 0], np.float32(t["scale"]))
    assert _same(b["inv_scale"][0, 0], np.float32(t["inv_scale"]))
    assert np.array_equal(b["q"], t["q"])


def test_one_row_blocks_are_row_wise_scaling():
    x = wl.generate((40, 136), "laplace", 1e-3, 12, 2)
    b = oracle.quantize_blocks(x, E5M2, 1, 136)
    r = oracle.quantize_rowwise(x, E5M2)
    assert _same(b["scale"][:, 0], r["row_scale"]) and _same(b["inv_scale"][:, 0], r["row_inv"])
    assert np.array_equal(b["q"], r["q"])


def test_each_block_is_its_own_per_tensor_cast():
    x = wl.generate((300, 260), "normal", 1.0, 13, 0)       # 3 x 3 blocks, the last row and column short
    b = oracle.quantize_blocks(x, E4M3, 128, 128)
    assert b["amax"].shape == (3, 3)
    for i in range(3):
        for j in range(3):
            sub = np.ascontiguousarray(x[128 * i:128 * (i + 1), 128 * j:128 * (j + 1)])
            t = oracle.quantize(sub, E4M3)
            assert _same(b["inv_scale"][i, j], np.float32(t["inv_scale"]))
            assert np.array_equal(b["q"][128 * i:128 * (i + 1), 128 * j:128 * (j + 1)], t["q"])


def test_column_blocks_are_row_blocks_of_the_transpose():
    x = wl.generate((264, 96), "normal", 1.0, 14, 0)
    c = oracle.quantize_blocks(x, E4M3, 128, 1)
    r = oracle.quantize_blocks(np.ascontiguousarray(x.T), E4M3, 1, 128)
    assert _same(c["inv_scale"], r["inv_scale"].T)
    assert np.array_equal(c["q"], r["q"].T)


@pytest.mark.parametrize("br,bc", [(1, 128), (128, 1), (128, 128), (64, 32)])
def test_block_amax_and_the_amax_invariant(br, bc):
    x = wl.generate((200, 300), "normal", 1.0, 15, 1)
    xf = np.abs(wl.bf16_bits_to_f32(x)).astype(np.float32)
    b = oracle.quantize_blocks(x, E4M3, br, bc)
    dec = oracle.decode_table(E4M3)
    for i in range(b["amax"].shape[0]):
        for j in range(b["amax"].shape[1]):
            blk = xf[br * i:br * (i + 1), bc * j:bc * (j + 1)]
            assert b["amax"][i, j] == blk.max()
            qb = b["q"][br * i:br * (i + 1), bc * j:bc * (j + 1)]
            at_max = blk == blk.max()
            assert np.all(np.abs(dec[qb[at_max]]) == 448.0)


def test_single_block_gemm_is_the_row_scaled_gemm():
    A = np.random.default_rng(1).integers(0, 0x7E, size=(9, 96), dtype=np.uint8)
    B = np.random.default_rng(2).integers(0, 0x7B, size=(7, 96), dtype=np.uint8)
    ia = np.random.default_rng(3).uniform(1e-3, 1e-1, size=9).astype(np.float32)
    ib = np.random.default_rng(4).uniform(1e-3, 1e-1, size=7).astype(np.float32)
    got = oracle.gemm_blocks(A, E4M3, B, E5M2, ia[:, None], ib[:, None])
    want = oracle.gemm_rows_vec(A, E4M3, B, E5M2, ia, ib)
    assert np.array_equal(got, want)


def _exact(code, fmt):
    return Fraction(float(oracle.decode_table(fmt)[code]))


def test_multi_block_gemm_against_exact_rationals():
    rng = np.random.default_rng(5)
    P, Q, R = 5, 4, 300                                   # three contraction blocks, the last one short
    # finite codes of moderate magnitude: no NaN, no saturation
    A = rng.integers(0x08, 0x70, size=(P, R), dtype=np.uint8) | (rng.integers(0, 2, size=(P, R)) << 7).astype(np.uint8)
    B = rng.integers(0x04, 0x68, size=(Q, R), dtype=np.uint8) | (rng.integers(0, 2, size=(Q, R)) << 7).astype(np.uint8)
    nb = 3
    ia = (2.0 ** rng.integers(-9, 3, size=(P, nb))).astype(np.float32)    # per row and block, all different
    ib = (2.0 ** rng.integers(-9, 3, size=(Q, nb))).astype(np.float32)
    got = oracle.gemm_blocks(A, E4M3, B, E5M2, ia, ib)
    for p in range(P):
        for q in range(Q):
            total = Fraction(0)
            for j in range(nb):
                part = sum(_exact(A[p, k], E4M3) * _exact(B[q, k], E5M2) for k in range(128 * j, min(R, 128 * (j + 1))))
                total += part * Fraction(float(ia[p, j])) * Fraction(float(ib[q, j]))
            assert abs(Fraction(got[p, q]) - total) <= abs(total) * Fraction(1, 2 ** 50) + Fraction(1, 2 ** 80)


def test_block_recipe_gemms_against_numpy():
    M, K, N = 136, 264, 200
    X = wl.generate((M, K), "normal", 1.0, 16, wl.X)
    W = wl.generate((N, K), "normal", 0.02, 16, wl.W)
    dY = wl.generate((M, N), "normal", 1e-3, 16, wl.DY)
    r = oracle.quantize_block_recipe(X, W, dY)
    d4, d5 = oracle.decode_table(E4M3), oracle.decode_table(E5M2)

    def deq(t, dec, br, bc):
        inv = np.repeat(np.repeat(t["inv_scale"].astype(np.float64), br, axis=0), bc, axis=1)
        return dec[t["q"]] * inv[:t["q"].shape[0], :t["q"].shape[1]]

    xk, xm = deq(r["x_k"], d4, 1, 128), deq(r["x_m"], d4, 128, 1)
    w = deq(r["w"], d4, 128, 128)
    dyn, dym = deq(r["dy_n"], d5, 1, 128), deq(r["dy_m"], d5, 128, 1)
    y = oracle.fwd_block_ref(r["x_k"]["q"], r["x_k"]["inv_scale"], r["w"]["q"], r["w"]["inv_scale"])
    dx = oracle.dgrad_block_ref(r["dy_n"]["q"], r["dy_n"]["inv_scale"], r["w"]["q"], r["w"]["inv_scale"])
    dw = oracle.wgrad_block_ref(r["dy_m"]["q"], r["dy_m"]["inv_scale"], r["x_m"]["q"], r["x_m"]["inv_scale"])
    for got, want in ((y, xk @ w.T), (dx, dyn @ w), (dw, dym.T @ xm)):
        assert got.shape == want.shape
        scale = np.abs(want).max()
        assert np.max(np.abs(got - want)) <= 1e-12 * scale
    # the dequantised operands approximate the bf16 originals to FP8 precision
    xf = wl.bf16_bits_to_f32(X).astype(np.float64)
    assert np.max(np.abs(xk - xf)) <= 2.0 ** -4 * np.abs(xf).max()

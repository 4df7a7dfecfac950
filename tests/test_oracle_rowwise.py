"""Pins for the oracle's row-wise (per-block) scaling (CPU).

* row / column amax against numpy;
* a matrix whose rows all share one amax casts exactly like per-tensor
  scaling (closed form);
* in every row of q (and of qT) the element at that row's amax casts to
  +-448 (the per-block form of the amax invariant);
* the vector-scaled GEMM against numpy's float64 matmul of the dequantised
  operands, wired for fwd / dgrad / wgrad; with constant scale vectors it
  equals the per-tensor GEMM.
"""
import numpy as np
import pytest

import oracle
import workloads as wl

E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def test_row_and_col_amax_match_numpy():
    x = wl.generate((48, 80), "normal", 1.0, 2, 0)
    xf = np.abs(wl.bf16_bits_to_f32(x))
    assert np.array_equal(oracle.amax_rows(x), xf.max(axis=1))
    assert np.array_equal(oracle.amax_cols(x), xf.max(axis=0))


def test_equal_row_amax_reduces_to_per_tensor():
    x = wl.generate((32, 64), "normal", 1.0, 3, 0).copy()
    x[:, 0] = 0x4080  # every row holds 4.0, the largest magnitude in it
    xf = np.abs(wl.bf16_bits_to_f32(x))
    assert np.all(xf.max(axis=1) == 4.0)
    r = oracle.quantize_rowwise(x, E4M3)
    t = oracle.quantize(x, E4M3)
    assert np.all(r["row_scale"] == t["scale"]) and np.array_equal(r["q"], t["q"])


@pytest.mark.parametrize("fmt,dist", [(E4M3, ("normal", 1.0)), (E5M2, ("laplace", 1e-3))])
def test_per_row_amax_invariant(fmt, dist):
    x = wl.generate((64, 96), *dist, seed=4, tensor_id=1)
    r = oracle.quantize_rowwise(x, fmt)
    xf = wl.bf16_bits_to_f32(x)
    code448 = {E4M3: 0x7E, E5M2: 0x5F}[fmt]
    for q, mat in ((r["q"], xf), (r["qT"], xf.T)):
        at = np.abs(mat) == np.abs(mat).max(axis=1, keepdims=True)
        assert np.all((q[at] & 0x7F) == code448)


def test_vector_scaled_gemms_match_numpy():
    M, K, N = 48, 80, 64
    X = wl.generate((M, K), "normal", 1.0, 5, 0)
    W = wl.generate((N, K), "normal", 0.02, 5, 1)
    D = wl.generate((M, N), "normal", 1e-3, 5, 2)
    rx, rw, rd = (oracle.quantize_rowwise(X, E4M3), oracle.quantize_rowwise(W, E4M3),
                  oracle.quantize_rowwise(D, E5M2))
    d4, d5 = oracle.decode_table(E4M3), oracle.decode_table(E5M2)
    # dequantised copies, each with the scales of its own rows
    Xq = d4[rx["q"]] * rx["row_inv"][:, None]       # X,  rows m
    XqT = d4[rx["qT"]] * rx["col_inv"][:, None]     # X^T, rows k
    Wq = d4[rw["q"]] * rw["row_inv"][:, None]       # W,  rows n
    WqT = d4[rw["qT"]] * rw["col_inv"][:, None]     # W^T, rows k
    Dq = d5[rd["q"]] * rd["row_inv"][:, None]       # dY, rows m
    DqT = d5[rd["qT"]] * rd["col_inv"][:, None]     # dY^T, rows n
    Y = oracle.gemm_rows_vec(rx["q"], E4M3, rw["q"], E4M3, rx["row_inv"], rw["row_inv"])
    dX = oracle.gemm_rows_vec(rd["q"], E5M2, rw["qT"], E4M3, rd["row_inv"], rw["col_inv"])
    dW = oracle.gemm_rows_vec(rd["qT"], E5M2, rx["qT"], E4M3, rd["col_inv"], rx["col_inv"])
    for got, ref in ((Y, Xq @ Wq.T), (dX, Dq @ WqT.T), (dW, DqT @ XqT.T)):
        np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13 * np.abs(ref).max())
    Xf, Wf, Df = (wl.bf16_bits_to_f32(t).astype(np.float64) for t in (X, W, D))
    for got, true in ((Y, Xf @ Wf.T), (dX, Df @ Wf), (dW, Df.T @ Xf)):
        assert np.linalg.norm(got - true) / np.linalg.norm(true) < 0.06


def test_constant_vectors_equal_per_tensor_gemm():
    rng = np.random.default_rng(9)
    A = rng.integers(0, 0x7E, size=(16, 48), dtype=np.uint8)
    B = rng.integers(0, 0x7E, size=(24, 48), dtype=np.uint8)
    ia, ib = np.float32(0.125), np.float32(3.0)
    v = oracle.gemm_rows_vec(A, E4M3, B, E4M3, np.full(16, ia, np.float32), np.full(24, ib, np.float32))
    assert np.array_equal(v, oracle.gemm_rows(A, E4M3, B, E4M3, ia, ib))

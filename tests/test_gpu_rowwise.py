"""Row-wise (per-block) scaling on the GPU against the oracle: row / column
amax, inverse-scale vectors and every FP8 byte bit-exact; the vector-scaled
GEMMs within the GEMM tolerance; whole linear steps."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import Guarded, assert_gemm_close, bf16_to_f64, to_dev_bf16, to_dev_u8

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def _bits(t):
    return t.cpu().numpy().view(np.uint32)


@pytest.mark.parametrize("shape", [(16, 16), (144, 272), (384, 1040), (1040, 384), (2048, 4096)])
@pytest.mark.parametrize("fmt,dist", [(E4M3, ("normal", 1.0)), (E5M2, ("laplace", 1e-3))])
def test_rowwise_cast_bit_exact(fp8lin, shape, fmt, dist):
    rows, cols = shape
    x = wl.generate(shape, *dist, seed=rows + cols, tensor_id=3, outlier_frac=1e-3)
    xd = to_dev_bf16(x)
    ra = torch.full((rows,), -1.0, device="cuda")
    ca = torch.full((cols,), -1.0, device="cuda")
    ri = torch.zeros(rows, device="cuda")
    ci = torch.zeros(cols, device="cuda")
    q = Guarded((rows, cols), torch.uint8)
    qT = Guarded((cols, rows), torch.uint8)
    fp8lin.fp8lin_amax_rowcol(xd, ra, ca)
    fp8lin.fp8lin_cast_transpose_rowwise(xd, fmt, ra, ca, ri, ci, q.t, qT.t)
    ref = oracle.quantize_rowwise(x, fmt)
    assert np.array_equal(_bits(ra), ref["row_amax"].view(np.uint32))
    assert np.array_equal(_bits(ca), ref["col_amax"].view(np.uint32))
    assert np.array_equal(_bits(ri), ref["row_inv"].view(np.uint32))
    assert np.array_equal(_bits(ci), ref["col_inv"].view(np.uint32))
    assert np.array_equal(q.t.cpu().numpy(), ref["q"])
    assert np.array_equal(qT.t.cpu().numpy(), ref["qT"])
    assert q.intact() and qT.intact()


@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (144, 272, 208), (384, 1040, 4112), (2048, 2048, 2048)])
@pytest.mark.parametrize("which", ["fwd", "dgrad", "wgrad"])
def test_rowwise_gemm_matches_oracle(fp8lin, M, N, K, which):
    P, Q, R = {"fwd": (M, N, K), "dgrad": (M, K, N), "wgrad": (N, K, M)}[which]
    fa = E4M3 if which == "fwd" else E5M2
    a = oracle.quantize_rowwise(wl.generate((P, R), "normal", 1.0, P, 1), fa)
    b = oracle.quantize_rowwise(wl.generate((Q, R), "normal", 0.02, Q, 2), E4M3)
    out = Guarded((P, Q), torch.bfloat16)
    fn = getattr(fp8lin, f"fp8lin_{which}_rowwise")
    ia, ib = torch.from_numpy(a["row_inv"]).cuda(), torch.from_numpy(b["row_inv"]).cuda()
    fn(to_dev_u8(a["q"]), ia, to_dev_u8(b["q"]), ib, out.t)
    torch.cuda.synchronize()
    ref = oracle.gemm_rows_vec(a["q"], fa, b["q"], E4M3, a["row_inv"], b["row_inv"])
    assert_gemm_close(bf16_to_f64(out.t), ref, f"{which} rowwise {M}x{N}x{K}")
    assert out.intact()


@pytest.mark.parametrize("M,K,N", [(256, 512, 1024), (144, 208, 272)])
def test_rowwise_linear_step(fp8lin, M, K, N):
    X = wl.generate((M, K), "normal", 1.0, 6, wl.X, outlier_frac=1e-3)
    W = wl.generate((N, K), "normal", 0.02, 6, wl.W)
    dY = wl.generate((M, N), "normal", 1e-3, 6, wl.DY)
    lin = fp8lin.Float8Linear(M, K, N, scaling="rowwise")
    y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    rx, rw, rd = oracle.quantize_rowwise(X, E4M3), oracle.quantize_rowwise(W, E4M3), oracle.quantize_rowwise(dY, E5M2)
    for t8, r in ((lin.x8, rx), (lin.w8, rw), (lin.dy8, rd)):
        assert np.array_equal(t8.q.cpu().numpy(), r["q"]) and np.array_equal(t8.qT.cpu().numpy(), r["qT"])
    assert_gemm_close(bf16_to_f64(y), oracle.gemm_rows_vec(rx["q"], E4M3, rw["q"], E4M3, rx["row_inv"], rw["row_inv"]), "Y")
    assert_gemm_close(bf16_to_f64(dx), oracle.gemm_rows_vec(rd["q"], E5M2, rw["qT"], E4M3, rd["row_inv"], rw["col_inv"]), "dX")
    assert_gemm_close(bf16_to_f64(dw), oracle.gemm_rows_vec(rd["qT"], E5M2, rx["qT"], E4M3, rd["col_inv"], rx["col_inv"]), "dW")


def _rows(n, seed, count=40):
    rng = np.random.default_rng(seed)
    pick = rng.choice(n, size=min(n, count - 2), replace=False)
    return np.unique(np.concatenate([[0, n - 1], pick])).astype(np.int64)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_rowwise_workload_step_matches_oracle(fp8lin, name):
    """Every configuration at full size: row and column inverse scales and
    every byte of both FP8 copies of X, W and dY bit-exact; Y, dX, dW on
    sampled rows."""
    w = wl.WORKLOADS[name]
    X, W, dY = w.make_x(), w.make_w(), w.make_dy()
    lin = fp8lin.Float8Linear(w.M, w.K, w.N, scaling="rowwise")
    y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    rx, rw, rd = oracle.quantize_rowwise(X, E4M3), oracle.quantize_rowwise(W, E4M3), oracle.quantize_rowwise(dY, E5M2)
    for key, t8, r in (("X", lin.x8, rx), ("W", lin.w8, rw), ("dY", lin.dy8, rd)):
        assert np.array_equal(_bits(t8.row_inv), r["row_inv"].view(np.uint32)), f"{name} {key} row scales"
        assert np.array_equal(_bits(t8.col_inv), r["col_inv"].view(np.uint32)), f"{name} {key} column scales"
        assert np.array_equal(t8.q.cpu().numpy(), r["q"]), f"{name} {key} q"
        assert np.array_equal(t8.qT.cpu().numpy(), r["qT"]), f"{name} {key} qT"
    rm, rn = _rows(w.M, w.seed), _rows(w.N, w.seed + 1)
    pick = lambda t, rows: bf16_to_f64(t[torch.from_numpy(rows).cuda()])
    assert_gemm_close(pick(y, rm), oracle.gemm_rows_vec(rx["q"], E4M3, rw["q"], E4M3, rx["row_inv"], rw["row_inv"], rm),
                      f"{name} Y")
    assert_gemm_close(pick(dx, rm), oracle.gemm_rows_vec(rd["q"], E5M2, rw["qT"], E4M3, rd["row_inv"], rw["col_inv"],
                                                         rm), f"{name} dX")
    assert_gemm_close(pick(dw, rn), oracle.gemm_rows_vec(rd["qT"], E5M2, rx["qT"], E4M3, rd["col_inv"], rx["col_inv"],
                                                         rn), f"{name} dW")


def _fuzz_shapes(n=20, seed=77):
    rng = np.random.default_rng(seed)
    return [(int(16 * rng.integers(1, 129)), int(16 * rng.integers(1, 129))) for _ in range(n)]


@pytest.mark.parametrize("rows,cols", _fuzz_shapes() + [(128, 128 * 9), (256, 128 * 5 + 16), (16, 128 * 4)])
def test_rowcol_amax_fuzz_shapes(fp8lin, rows, cols):
    """Row and column amax on seeded random shapes (up to 2048 x 2048) and
    shapes whose tile count per row is not a multiple of the kernel's strip
    of four tiles: bit-exact against the oracle, each mode alone too."""
    x = wl.generate((rows, cols), "normal", 1.0, rows * 5 + cols, 3, outlier_frac=1e-3)
    xd = to_dev_bf16(x)
    ra = torch.full((rows,), -1.0, device="cuda")
    ca = torch.full((cols,), -1.0, device="cuda")
    fp8lin.fp8lin_amax_rowcol(xd, ra, ca)
    torch.cuda.synchronize()
    assert np.array_equal(_bits(ra), oracle.amax_rows(x).view(np.uint32))
    assert np.array_equal(_bits(ca), oracle.amax_cols(x).view(np.uint32))
    ra2 = torch.full((rows,), -1.0, device="cuda")
    ca2 = torch.full((cols,), -1.0, device="cuda")
    fp8lin.fp8lin_amax_rowcol(xd, ra2, None)
    fp8lin.fp8lin_amax_rowcol(xd, None, ca2)
    torch.cuda.synchronize()
    assert torch.equal(ra2, ra) and torch.equal(ca2, ca)

"""Block scaling on the GPU against the oracle: the one-pass block cast
(1 x 128, 128 x 1 and 128 x 128 blocks) with every FP8 byte and every
inverse scale bit-exact."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import Guarded, assert_gemm_close, bf16_to_f64, to_dev_bf16

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2
KINDS = {"row": (1, 128), "col": (128, 1), "tile": (128, 128)}


def _blocks(rows, cols, kind):
    br, bc = KINDS[kind]
    n = ((rows + br - 1) // br, (cols + bc - 1) // bc)
    return n[::-1] if kind == "row" else n   # row-block scales are stored block-major


def _layout(kind, inv):
    """The oracle's [block rows x block columns] scales in the library's layout."""
    return np.ascontiguousarray(inv.T) if kind == "row" else inv


@pytest.mark.parametrize("shape", [(16, 16), (144, 272), (384, 1040), (1040, 384), (2048, 4096)])
@pytest.mark.parametrize("fmt,dist", [(E4M3, ("normal", 1.0)), (E5M2, ("laplace", 1e-3))])
@pytest.mark.parametrize("kinds", [("row", "col"), ("tile",), ("row",), ("col",), ("row", "col", "tile")])
def test_block_cast_bit_exact(fp8lin, shape, fmt, dist, kinds):
    rows, cols = shape
    x = wl.generate(shape, *dist, seed=rows * 3 + cols, tensor_id=5, outlier_frac=1e-3)
    xd = to_dev_bf16(x)
    q, inv = {}, {}
    for k in kinds:
        q[k] = Guarded((rows, cols), torch.uint8)
        inv[k] = Guarded(_blocks(rows, cols, k), torch.float32)
    args = {}
    for k in ("row", "col", "tile"):
        args["q_" + k] = q[k].t if k in q else None
        args["inv_" + k] = inv[k].t if k in inv else None
    fp8lin.fp8lin_cast_blockwise(xd, fmt, **args)
    torch.cuda.synchronize()
    for k in kinds:
        ref = oracle.quantize_blocks(x, fmt, *KINDS[k])
        assert np.array_equal(inv[k].t.cpu().numpy().view(np.uint32), _layout(k, ref["inv_scale"]).view(np.uint32)), k
        assert np.array_equal(q[k].t.cpu().numpy(), ref["q"]), k
        assert q[k].intact() and inv[k].intact(), k


def test_block_cast_zero_tensor_and_arguments(fp8lin):
    x = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    q = torch.full((128, 256), 0xFF, dtype=torch.uint8, device="cuda")
    inv = torch.zeros((2, 128), dtype=torch.float32, device="cuda")
    fp8lin.fp8lin_cast_blockwise(x, E4M3, q_row=q, inv_row=inv)
    torch.cuda.synchronize()
    ref = oracle.quantize_blocks(np.zeros((128, 256), np.uint16), E4M3, 1, 128)
    assert (q == 0).all() and np.array_equal(inv.cpu().numpy().view(np.uint32), ref["inv_scale"].T.copy().view(np.uint32))
    with pytest.raises(fp8lin.Fp8LinError):
        fp8lin.fp8lin_cast_blockwise(x, E4M3, q_row=q)            # a copy without its scales
    with pytest.raises(fp8lin.Fp8LinError):
        fp8lin.fp8lin_cast_blockwise(x, E4M3)                     # nothing asked for


# (M, N, K): ragged pair tiles in every direction, a contraction shorter than
# one block, 16-row and 16-column outputs (one pair tile mostly past the edge)
GEMM_SHAPES = [(128, 128, 128), (144, 272, 208), (384, 1040, 4112), (1040, 400, 96), (2048, 2048, 2048),
               (16, 16, 16), (16, 528, 144), (272, 16, 400)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("which", ["fwd", "dgrad", "wgrad"])
def test_block_gemm_matches_oracle(fp8lin, M, N, K, which):
    X = wl.generate((M, K), "normal", 1.0, M + 1, wl.X, outlier_frac=1e-3)
    W = wl.generate((N, K), "normal", 0.02, N + 2, wl.W)
    dY = wl.generate((M, N), "laplace", 1e-3, K + 3, wl.DY)
    r = oracle.quantize_block_recipe(X, W, dY)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
    if which == "fwd":
        out, args = Guarded((M, N), torch.bfloat16), (r["x_k"], r["w"])
        ref = oracle.fwd_block_ref(r["x_k"]["q"], r["x_k"]["inv_scale"], r["w"]["q"], r["w"]["inv_scale"])
    elif which == "dgrad":
        out, args = Guarded((M, K), torch.bfloat16), (r["dy_n"], r["w"])
        ref = oracle.dgrad_block_ref(r["dy_n"]["q"], r["dy_n"]["inv_scale"], r["w"]["q"], r["w"]["inv_scale"])
    else:
        out, args = Guarded((N, K), torch.bfloat16), (r["dy_m"], r["x_m"])
        ref = oracle.wgrad_block_ref(r["dy_m"]["q"], r["dy_m"]["inv_scale"], r["x_m"]["q"], r["x_m"]["inv_scale"])
    out.t.fill_(float("nan"))
    a, b = args
    ia = a["inv_scale"].T if which in ("fwd", "dgrad") else a["inv_scale"]   # row-block scales block-major
    getattr(fp8lin, f"fp8lin_{which}_block")(dev(a["q"]), dev(ia), dev(b["q"]), dev(b["inv_scale"]), out.t)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    assert_gemm_close(bf16_to_f64(out.t), ref, f"{which} block {M}x{N}x{K}")
    assert out.intact()


def _check_block_copies(name, lin, r):
    got = {"x_k": (lin.x8.q, lin.x8.row_inv.t()), "x_m": (lin.x8.qc, lin.x8.col_inv),
           "w": (lin.w8.q, lin.w8.tile_inv), "dy_n": (lin.dy8.q, lin.dy8.row_inv.t()),
           "dy_m": (lin.dy8.qc, lin.dy8.col_inv)}
    for key, (q, inv) in got.items():
        assert np.array_equal(inv.contiguous().cpu().numpy().view(np.uint32), r[key]["inv_scale"].view(np.uint32)), \
            f"{name} {key}"
        assert np.array_equal(q.cpu().numpy(), r[key]["q"]), f"{name} {key}"


@pytest.mark.parametrize("M,K,N", [(256, 512, 1024), (144, 208, 272), (640, 384, 1296)])
def test_block_linear_step_matches_oracle(fp8lin, M, K, N):
    X = wl.generate((M, K), "normal", 1.0, 21, wl.X, outlier_frac=1e-3)
    W = wl.generate((N, K), "normal", 0.02, 21, wl.W)
    dY = wl.generate((M, N), "normal", 1e-3, 21, wl.DY)
    lin = fp8lin.Float8Linear(M, K, N, scaling="block")
    y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    r = oracle.quantize_block_recipe(X, W, dY)
    _check_block_copies(f"{M}x{K}x{N}", lin, r)
    assert_gemm_close(bf16_to_f64(y), oracle.fwd_block_ref(r["x_k"]["q"], r["x_k"]["inv_scale"], r["w"]["q"],
                                                           r["w"]["inv_scale"]), "Y")
    assert_gemm_close(bf16_to_f64(dx), oracle.dgrad_block_ref(r["dy_n"]["q"], r["dy_n"]["inv_scale"], r["w"]["q"],
                                                              r["w"]["inv_scale"]), "dX")
    assert_gemm_close(bf16_to_f64(dw), oracle.wgrad_block_ref(r["dy_m"]["q"], r["dy_m"]["inv_scale"], r["x_m"]["q"],
                                                              r["x_m"]["inv_scale"]), "dW")


def _rows(n, seed, count=40):
    rng = np.random.default_rng(seed)
    pick = rng.choice(n, size=min(n, count - 2), replace=False)
    return np.unique(np.concatenate([[0, n - 1], pick])).astype(np.int64)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_block_workload_step_matches_oracle(fp8lin, name):
    """Every configuration at full size: every FP8 byte and inverse scale of
    the five block-scaled copies bit-exact; Y, dX, dW on sampled rows."""
    w = wl.WORKLOADS[name]
    X, W, dY = w.make_x(), w.make_w(), w.make_dy()
    lin = fp8lin.Float8Linear(w.M, w.K, w.N, scaling="block")
    y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    r = oracle.quantize_block_recipe(X, W, dY)
    _check_block_copies(name, lin, r)
    rm, rn = _rows(w.M, w.seed), _rows(w.N, w.seed + 1)
    pick = lambda t, rows: bf16_to_f64(t[torch.from_numpy(rows).cuda()])
    assert_gemm_close(pick(y, rm), oracle.fwd_block_ref(r["x_k"]["q"], r["x_k"]["inv_scale"], r["w"]["q"],
                                                        r["w"]["inv_scale"], rm), f"{name} Y")
    assert_gemm_close(pick(dx, rm), oracle.dgrad_block_ref(r["dy_n"]["q"], r["dy_n"]["inv_scale"], r["w"]["q"],
                                                           r["w"]["inv_scale"], rm), f"{name} dX")
    assert_gemm_close(pick(dw, rn), oracle.wgrad_block_ref(r["dy_m"]["q"], r["dy_m"]["inv_scale"], r["x_m"]["q"],
                                                           r["x_m"]["inv_scale"], rn), f"{name} dW")

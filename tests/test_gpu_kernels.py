"""Parity of each CUDA kernel with the CPU oracle, through the C ABI, on
seeded inputs that span several tiles and ragged tails, plus edge cases.

Bar: amax, scale, inverse scale and every FP8 byte bit-exact; GEMM outputs
within |y - ref| <= 2^-7 |ref| + 1e-3 rms(ref) elementwise.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import (Guarded, assert_gemm_close, bf16_to_f64, f32_bits, scalar_bits,
                         to_dev_bf16, to_dev_u8)

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2


# ------------------------------------------------------------------ amax

@pytest.mark.parametrize("n", [1, 7, 8, 9, 1000, 4096 * 3 + 5, 1 << 20, (1 << 22) + 24])
def test_amax_bit_exact(fp8lin, n):
    x = wl.generate((n,), "normal", 1.0, 17, n % 1000)
    amax = torch.full((1,), -1.0, device="cuda")
    fp8lin.fp8lin_amax(to_dev_bf16(x), amax)
    assert scalar_bits(amax) == f32_bits(oracle.amax(x))


def test_amax_empty_and_special_values(fp8lin):
    amax = torch.full((1,), 7.0, device="cuda")
    fp8lin.fp8lin_amax(torch.empty(0, dtype=torch.bfloat16, device="cuda"), amax)
    assert amax.item() == 0.0
    cases = [
        np.array([0x0000, 0x8000] * 20, np.uint16),                       # +-0
        np.array([0x0001, 0x8003, 0x0002] * 11, np.uint16),               # bf16 subnormals
        np.array([0x3F80] * 100 + [0xC2C8] + [0x3F80] * 37, np.uint16),   # single negative extreme
        np.array([0x3F80, 0x7F80, 0xC000] * 9, np.uint16),                # +Inf
        np.array([0x3F80, 0x7F80, 0xFFC1, 0x7FC0] * 9, np.uint16),        # NaNs above Inf
    ]
    for x in cases:
        fp8lin.fp8lin_amax(to_dev_bf16(x), amax)
        assert scalar_bits(amax) == f32_bits(oracle.amax(x))


def test_amax_every_bf16_pattern(fp8lin):
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = x[(x & 0x7FFF) < 0x7F80]
    amax = torch.zeros(1, device="cuda")
    for arr in (finite, x):
        fp8lin.fp8lin_amax(to_dev_bf16(arr), amax)
        assert scalar_bits(amax) == f32_bits(oracle.amax(arr))


# ------------------------------------------------------------------ cast

CAST_SHAPES = [(16, 16), (128, 128), (144, 272), (256, 512), (384, 1040), (1040, 384), (2048, 4096)]


def _run_cast(fp8lin, x_bits, fmt, fmt_max=448.0, want_q=True, want_qT=True):
    rows, cols = x_bits.shape
    x = to_dev_bf16(x_bits)
    amax = torch.zeros(1, device="cuda")
    scale = torch.full((1,), -1.0, device="cuda")
    inv = torch.full((1,), -1.0, device="cuda")
    q = Guarded((rows, cols), torch.uint8) if want_q else None
    qT = Guarded((cols, rows), torch.uint8) if want_qT else None
    fp8lin.fp8lin_amax(x, amax)
    fp8lin.fp8lin_cast_transpose(x, fmt, amax, scale, inv, q.t if q else None, qT.t if qT else None,
                                 fmt_max)
    torch.cuda.synchronize()
    return amax, scale, inv, q, qT


@pytest.mark.parametrize("shape", CAST_SHAPES)
@pytest.mark.parametrize("fmt,dist", [(E4M3, ("normal", 1.0)), (E4M3, ("normal", 0.02)),
                                      (E5M2, ("normal", 1e-3)), (E5M2, ("laplace", 1e-3))])
def test_cast_transpose_bit_exact(fp8lin, shape, fmt, dist):
    x = wl.generate(shape, *dist, seed=shape[0] + shape[1], tensor_id=fmt)
    amax, scale, inv, q, qT = _run_cast(fp8lin, x, fmt)
    ref = oracle.quantize(x, fmt)
    assert scalar_bits(amax) == f32_bits(ref["amax"])
    assert scalar_bits(scale) == f32_bits(ref["scale"])
    assert scalar_bits(inv) == f32_bits(ref["inv_scale"])
    assert np.array_equal(q.t.cpu().numpy(), ref["q"])
    assert np.array_equal(qT.t.cpu().numpy(), ref["qT"])
    assert q.intact() and qT.intact()


@pytest.mark.parametrize("fmt,fmt_max", [(E4M3, 448.0), (E5M2, 448.0), (E5M2, 57344.0)])
def test_cast_every_bf16_pattern(fp8lin, fmt, fmt_max):
    """All 65,536 bf16 patterns as one 256 x 256 tensor, cast with the scale
    from a fixed amax (so the scale is not dominated by NaN/Inf)."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    xd = to_dev_bf16(x)
    for amax_value in (448.0, 3.0, 1e-3, 5.0e4):
        amax = torch.tensor([amax_value], dtype=torch.float32, device="cuda")
        scale = torch.zeros(1, device="cuda")
        inv = torch.zeros(1, device="cuda")
        q = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
        qT = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
        fp8lin.fp8lin_cast_transpose(xd, fmt, amax, scale, inv, q, qT, fmt_max)
        s, i = oracle.scale(np.float32(amax_value), fmt_max)
        assert scalar_bits(scale) == f32_bits(s) and scalar_bits(inv) == f32_bits(i)
        ref = oracle.cast(x, fmt, s)
        got = q.cpu().numpy()
        assert np.array_equal(got, ref)                     # NaNs included: every NaN casts to 0x7F
        assert np.array_equal(qT.cpu().numpy(), got.T)


def test_cast_zero_tensor_and_one_sided_outputs(fp8lin):
    x = np.zeros((64, 96), np.uint16)
    x[3, 5] = 0x8000  # -0
    amax, scale, inv, q, qT = _run_cast(fp8lin, x, E4M3)
    ref = oracle.quantize(x, E4M3)
    assert amax.item() == 0.0 and scalar_bits(scale) == f32_bits(ref["scale"])
    assert np.array_equal(q.t.cpu().numpy(), ref["q"]) and q.t.cpu().numpy()[3, 5] == 0x80
    y = wl.generate((160, 208), "normal", 1.0, 5, 0)
    ref = oracle.quantize(y, E5M2)
    _, _, _, q, qT = _run_cast(fp8lin, y, E5M2, want_qT=False)
    assert qT is None and np.array_equal(q.t.cpu().numpy(), ref["q"]) and q.intact()
    _, _, _, q, qT = _run_cast(fp8lin, y, E5M2, want_q=False)
    assert q is None and np.array_equal(qT.t.cpu().numpy(), ref["qT"]) and qT.intact()


def test_cast_empty_matrix_still_publishes_scale(fp8lin):
    x = torch.empty((0, 32), dtype=torch.bfloat16, device="cuda")
    amax = torch.tensor([2.0], device="cuda")
    scale = torch.zeros(1, device="cuda")
    inv = torch.zeros(1, device="cuda")
    fp8lin.fp8lin_cast_transpose(x, E4M3, amax, scale, inv, None, None)
    assert scale.item() == 224.0 and scalar_bits(inv) == f32_bits(oracle.scale(2.0)[1])


def test_cast_amax_invariant(fp8lin):
    x = wl.generate((512, 384), "normal", 1.0, 8, 0, outlier_frac=1e-3)
    _, _, _, q, _ = _run_cast(fp8lin, x, E4M3)
    xf = wl.bf16_bits_to_f32(x)
    at = np.abs(xf) == np.abs(xf).max()
    qq = q.t.cpu().numpy()
    assert np.all((qq[at] & 0x7F) == 0x7E)


# ------------------------------------------------------------------ GEMMs

def _codes(shape, fmt, seed):
    """FP8 operands as the oracle's cast makes them from seeded bf16 input."""
    dist = ("normal", 1.0) if fmt == E4M3 else ("laplace", 1e-3)
    x = wl.generate(shape, *dist, seed=seed, tensor_id=7)
    r = oracle.quantize(x, fmt)
    return r["q"], r["inv_scale"]


GEMM_SHAPES = [(16, 16, 16), (128, 256, 128), (256, 1024, 512), (144, 272, 208),
               (384, 1040, 4112), (1040, 400, 96), (2048, 2048, 2048)]


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("which", ["fwd", "dgrad", "wgrad"])
def test_gemm_matches_oracle(fp8lin, M, N, K, which):
    seed = M * 7 + N * 3 + K
    if which == "fwd":      # Y[M,N] = Xq[M,K] . Wq[N,K]^T
        P, Q, R, fa = M, N, K, E4M3
    elif which == "dgrad":  # dX[M,K] = dYq[M,N] . WqT[K,N]^T
        P, Q, R, fa = M, K, N, E5M2
    else:                   # dW[N,K] = dYqT[N,M] . XqT[K,M]^T
        P, Q, R, fa = N, K, M, E5M2
    A, ia = _codes((P, R), fa, seed)
    B, ib = _codes((Q, R), E4M3, seed + 1)
    out = Guarded((P, Q), torch.bfloat16)
    out.t.fill_(float("nan"))
    a, b = to_dev_u8(A), to_dev_u8(B)
    sa = torch.tensor([ia], dtype=torch.float32, device="cuda")
    sb = torch.tensor([ib], dtype=torch.float32, device="cuda")
    getattr(fp8lin, "fp8lin_" + which)(a, sa, b, sb, out.t)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    ref = oracle.gemm_rows(A, fa, B, E4M3, ia, ib)
    assert_gemm_close(bf16_to_f64(out.t), ref, f"{which} {M}x{N}x{K}")
    assert out.intact()


def test_gemm_empty_dimensions(fp8lin):
    z = torch.zeros(1, device="cuda")
    y = torch.full((32, 48), 3.0, dtype=torch.bfloat16, device="cuda")
    e = torch.empty((32, 0), dtype=torch.uint8, device="cuda")
    f = torch.empty((48, 0), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_fwd(e, z, f, z, y)          # K = 0: Y = 0
    assert (y == 0).all()
    y0 = torch.empty((0, 48), dtype=torch.bfloat16, device="cuda")
    fp8lin.fp8lin_fwd(torch.empty((0, 32), dtype=torch.uint8, device="cuda"), z,
                      torch.empty((48, 32), dtype=torch.uint8, device="cuda"), z, y0)
    torch.cuda.synchronize()


def test_gemm_closed_forms(fp8lin):
    # one-hot rows of A pick columns of B; all-ones gives K
    K, N = 256, 272
    A = np.zeros((K, K), np.uint8)
    A[np.arange(K), np.arange(K)] = 0x38  # e4m3 1.0
    B, _ = _codes((N, K), E4M3, 99)
    one = torch.ones(1, device="cuda")
    y = torch.empty((K, N), dtype=torch.bfloat16, device="cuda")
    fp8lin.fp8lin_fwd(to_dev_u8(A), one, to_dev_u8(B), one, y)
    exp = oracle.decode_table(E4M3)[B].T
    assert np.array_equal(bf16_to_f64(y), exp)
    ones_a = torch.full((128, 4096), 0x3C, dtype=torch.uint8, device="cuda")  # e5m2 1.0
    ones_b = torch.full((256, 4096), 0x38, dtype=torch.uint8, device="cuda")  # e4m3 1.0
    y = torch.empty((128, 256), dtype=torch.bfloat16, device="cuda")
    fp8lin.fp8lin_dgrad(ones_a, one, ones_b, one, y)
    assert (y.float() == 4096.0).all()


# -------------------------------------------------------------- sequence

@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
def test_gemm_mn_operands_match_transposed_copies(fp8lin, M, N, K):
    """dgrad / wgrad reading the row-major copies MN-major: the oracle's
    product, and bit for bit what the K-major GEMMs give on the transposed
    copies of the same bytes."""
    seed = M * 5 + N * 11 + K
    dyq, idy = _codes((M, N), E5M2, seed)
    wq, iw = _codes((N, K), E4M3, seed + 1)
    xq, ix = _codes((M, K), E4M3, seed + 2)
    d_dyq, d_wq, d_xq = to_dev_u8(dyq), to_dev_u8(wq), to_dev_u8(xq)
    sdy, sw, sx = (torch.tensor([v], dtype=torch.float32, device="cuda") for v in (idy, iw, ix))
    dx_mn, dw_mn = Guarded((M, K), torch.bfloat16), Guarded((N, K), torch.bfloat16)
    dx_mn.t.fill_(float("nan"))
    dw_mn.t.fill_(float("nan"))
    fp8lin.fp8lin_dgrad_mn(d_dyq, sdy, d_wq, sw, dx_mn.t)
    fp8lin.fp8lin_wgrad_mn(d_dyq, sdy, d_xq, sx, dw_mn.t)
    dx_t = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw_t = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    fp8lin.fp8lin_dgrad(d_dyq, sdy, to_dev_u8(np.ascontiguousarray(wq.T)), sw, dx_t)
    fp8lin.fp8lin_wgrad(to_dev_u8(np.ascontiguousarray(dyq.T)), sdy, to_dev_u8(np.ascontiguousarray(xq.T)), sx, dw_t)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    assert dx_mn.intact() and dw_mn.intact()
    assert torch.equal(dx_mn.t.view(torch.int16), dx_t.view(torch.int16))
    assert torch.equal(dw_mn.t.view(torch.int16), dw_t.view(torch.int16))
    assert_gemm_close(bf16_to_f64(dx_mn.t), oracle.dgrad_ref(dyq, idy, np.ascontiguousarray(wq.T), iw),
                      f"dgrad_mn {M}x{N}x{K}")
    assert_gemm_close(bf16_to_f64(dw_mn.t), oracle.wgrad_ref(np.ascontiguousarray(dyq.T), idy,
                                                             np.ascontiguousarray(xq.T), ix), f"wgrad_mn {M}x{N}x{K}")


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("M,K,N", [(256, 512, 1024), (144, 208, 272), (640, 384, 1296)])
def test_float8_linear_step_matches_oracle(fp8lin, M, K, N, transpose):
    X = wl.generate((M, K), "normal", 1.0, 3, wl.X)
    W = wl.generate((N, K), "normal", 0.02, 3, wl.W)
    dY = wl.generate((M, N), "normal", 1e-3, 3, wl.DY)
    lin = fp8lin.Float8Linear(M, K, N, transpose=transpose)
    y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    ox, ow, od = oracle.quantize(X, E4M3), oracle.quantize(W, E4M3), oracle.quantize(dY, E5M2)
    for t8, r in ((lin.x8, ox), (lin.w8, ow), (lin.dy8, od)):
        assert scalar_bits(t8.amax) == f32_bits(r["amax"])
        assert scalar_bits(t8.scale) == f32_bits(r["scale"])
        assert scalar_bits(t8.inv_scale) == f32_bits(r["inv_scale"])
        assert np.array_equal(t8.q.cpu().numpy(), r["q"])
        if transpose:
            assert np.array_equal(t8.qT.cpu().numpy(), r["qT"])
        else:
            assert t8.qT is None
    assert_gemm_close(bf16_to_f64(y), oracle.fwd_ref(ox["q"], ox["inv_scale"], ow["q"], ow["inv_scale"]), "Y")
    assert_gemm_close(bf16_to_f64(dx), oracle.dgrad_ref(od["q"], od["inv_scale"], ow["qT"], ow["inv_scale"]), "dX")
    assert_gemm_close(bf16_to_f64(dw), oracle.wgrad_ref(od["qT"], od["inv_scale"], ox["qT"], ox["inv_scale"]), "dW")


def test_repeated_calls_and_streams(fp8lin):
    """Same inputs on a side stream, twice: identical results."""
    M, K, N = 256, 512, 1024
    X = to_dev_bf16(wl.generate((M, K), "normal", 1.0, 4, 0))
    W = to_dev_bf16(wl.generate((N, K), "normal", 0.02, 4, 1))
    dY = to_dev_bf16(wl.generate((M, N), "normal", 1e-3, 4, 2))
    a = fp8lin.Float8Linear(M, K, N)
    ra = [t.clone() for t in a.step(X, W, dY)]
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    b = fp8lin.Float8Linear(M, K, N)
    with torch.cuda.stream(s):
        b.step(X, W, dY, stream=s)
        rb = [t.clone() for t in b.step(X, W, dY, stream=s)]
    torch.cuda.synchronize()
    for u, v in zip(ra, rb):
        assert torch.equal(u, v)


@pytest.mark.parametrize("shape", [(16, 16), (144, 272), (1040, 384), (2048, 4096), (8192, 4096)])
@pytest.mark.parametrize("fmt,dist", [(E4M3, ("normal", 1.0)), (E5M2, ("laplace", 1e-3))])
@pytest.mark.parametrize("want_qT", [False, True])
def test_one_call_quantize_matches_amax_then_cast(fp8lin, shape, fmt, dist, want_qT):
    """fp8lin_quantize (amax + cast in one call, tuned for running alone):
    amax, scale, inverse scale and every FP8 byte bit-exact against the
    oracle, and the same bytes as fp8lin_amax followed by
    fp8lin_cast_transpose.  8192 x 4096 (67 MB) is larger than the part the
    amax pass keeps in L2, so the cast reads both kept and evicted rows."""
    rows, cols = shape
    x = wl.generate(shape, *dist, seed=rows * 3 + cols, tensor_id=9, outlier_frac=1e-3)
    xd = to_dev_bf16(x)
    amax = torch.full((1,), -1.0, device="cuda")
    scale = torch.full((1,), -1.0, device="cuda")
    inv = torch.full((1,), -1.0, device="cuda")
    q = Guarded((rows, cols), torch.uint8)
    qT = Guarded((cols, rows), torch.uint8) if want_qT else None
    fp8lin.fp8lin_quantize(xd, fmt, amax, scale, inv, q.t, qT.t if qT else None)
    a2, s2, i2, q2, qT2 = _run_cast(fp8lin, x, fmt, want_qT=want_qT)
    torch.cuda.synchronize()
    ref = oracle.quantize(x, fmt)
    assert scalar_bits(amax) == f32_bits(ref["amax"]) == scalar_bits(a2)
    assert scalar_bits(scale) == f32_bits(ref["scale"]) == scalar_bits(s2)
    assert scalar_bits(inv) == f32_bits(ref["inv_scale"]) == scalar_bits(i2)
    assert np.array_equal(q.t.cpu().numpy(), ref["q"]) and torch.equal(q.t, q2.t) and q.intact()
    if want_qT:
        assert np.array_equal(qT.t.cpu().numpy(), ref["qT"]) and torch.equal(qT.t, qT2.t) and qT.intact()


@pytest.mark.parametrize("fmt_max", [448.0, 57344.0, 1.0e5])
def test_one_call_quantize_fmt_max_and_separate_slots(fp8lin, fmt_max):
    """fp8lin_quantize with amax, scale and inverse scale in separate
    allocations (each slot cleared on its own), and with fmt_max above
    65504 (taken by the two-kernel path): same bytes as the oracle."""
    x = wl.generate((1040, 2048), "laplace", 1e-3, seed=77, tensor_id=2)
    amax, scale, inv = (torch.full((4,), 7.0, device="cuda")[:1] for _ in range(3))
    q = Guarded((1040, 2048), torch.uint8)
    fp8lin.fp8lin_quantize(to_dev_bf16(x), E5M2, amax, scale, inv, q.t, None, fmt_max)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    ref = oracle.quantize(x, E5M2, fmt_max)
    assert scalar_bits(amax) == f32_bits(ref["amax"]) and scalar_bits(scale) == f32_bits(ref["scale"])
    assert scalar_bits(inv) == f32_bits(ref["inv_scale"])
    assert np.array_equal(q.t.cpu().numpy(), ref["q"]) and q.intact()


# 786432 elements (98304 16-byte vectors, 1.5 MB of bf16) is the largest
# tensor the one-cluster path stages in shared memory; 784 x 1024 is the
# whole-GPU grid's.
@pytest.mark.parametrize("shape", [(16, 16), (32, 16), (16, 48), (768, 1024), (784, 1024)])
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_one_call_quantize_small_tensor_edges(fp8lin, shape, fmt):
    """The one-cluster path of small tensors writes all three slots itself
    (no clearing first): slots holding NaN or garbage beforehand, slices
    that do not split evenly over the cluster's CTAs, the largest tensor it
    takes and the smallest the grid takes, each bit-exact against the oracle
    and against fp8lin_amax + fp8lin_cast_transpose."""
    rows, cols = shape
    x = wl.generate(shape, "laplace", 0.5, seed=rows + 7 * cols + fmt, tensor_id=3, outlier_frac=1e-3)
    slots = torch.tensor([float("nan"), -1.0, 12345.0], device="cuda")
    q = Guarded(shape, torch.uint8)
    fp8lin.fp8lin_quantize(to_dev_bf16(x), fmt, slots[0:1], slots[1:2], slots[2:3], q.t, None)
    a2, s2, i2, q2, _ = _run_cast(fp8lin, x, fmt, want_qT=False)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    ref = oracle.quantize(x, fmt)
    assert scalar_bits(slots[0:1]) == f32_bits(ref["amax"]) == scalar_bits(a2)
    assert scalar_bits(slots[1:2]) == f32_bits(ref["scale"]) == scalar_bits(s2)
    assert scalar_bits(slots[2:3]) == f32_bits(ref["inv_scale"]) == scalar_bits(i2)
    assert np.array_equal(q.t.cpu().numpy(), ref["q"]) and torch.equal(q.t, q2.t) and q.intact()


def test_one_call_quantize_small_zero_and_alternating_sizes(fp8lin):
    """An all-zero small tensor publishes amax 0 and the floor scale; small
    and large tensors alternating on the same slots (the grid path clears
    them, the cluster path overwrites them) each match the oracle."""
    slots = torch.full((3,), 9.0, device="cuda")
    z = np.zeros((64, 128), dtype=np.uint16)
    q = torch.empty((64, 128), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_quantize(to_dev_bf16(z), E4M3, slots[0:1], slots[1:2], slots[2:3], q, None)
    torch.cuda.synchronize()
    assert slots[0].item() == 0.0 and scalar_bits(slots[1:2]) == f32_bits(oracle.scale(np.float32(0.0))[0])
    assert (q == 0).all()
    for i, shape in enumerate([(128, 256), (2048, 1024), (256, 128), (1024, 2048), (16, 16)]):
        x = wl.generate(shape, "normal", (1.0, 0.02, 3.0, 0.5, 7.0)[i], seed=90 + i, tensor_id=1)
        q = torch.empty(shape, dtype=torch.uint8, device="cuda")
        fp8lin.fp8lin_quantize(to_dev_bf16(x), E4M3, slots[0:1], slots[1:2], slots[2:3], q, None)
        torch.cuda.synchronize()
        ref = oracle.quantize(x, E4M3)
        assert scalar_bits(slots[0:1]) == f32_bits(ref["amax"])
        assert scalar_bits(slots[1:2]) == f32_bits(ref["scale"])
        assert scalar_bits(slots[2:3]) == f32_bits(ref["inv_scale"])
        assert np.array_equal(q.cpu().numpy(), ref["q"])
    assert fp8lin.fp8lin_device_error() == 0


# batches on both one-launch paths: up to 786432 elements in all one cluster
# of eight CTAs, beyond that the whole-GPU grid; empty members inside
BATCHES = [
    [(16, 16)],
    [(256, 512), (1024, 512)],          # the 1024 x 512 linear's X and W: one cluster
    [(256, 1024), (32, 16), (16, 48)],  # slices cut across three tensors
    [(768, 1024), (16, 16)],            # just past the cluster's 1.5 MB: the grid
    [(1040, 384), (2048, 4096), (0, 64), (16, 48)],
    [(8192, 4096), (14336, 4096)],      # the 8B FFN's X and W1
]


@pytest.mark.parametrize("shapes", BATCHES, ids=lambda b: "+".join(f"{r}x{c}" for r, c in b))
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_batched_quantize_matches_each_tensor_alone(fp8lin, shapes, fmt):
    """fp8lin_quantize_batch: every tensor's amax, scale, inverse scale and
    FP8 bytes bit-exact against the oracle and against fp8lin_quantize on
    that tensor alone, with every slot holding garbage beforehand."""
    xs = [wl.generate(sh, "laplace" if fmt == E5M2 else "normal", 1e-3 if fmt == E5M2 else 1.0,
                      seed=31 * k + sh[0] + sh[1], tensor_id=k, outlier_frac=1e-3) if sh[0] * sh[1] else
          np.zeros(sh, dtype=np.uint16) for k, sh in enumerate(shapes)]
    slots = [torch.tensor([float("nan"), -3.0, 7.5], device="cuda") for _ in shapes]
    qs = [Guarded(sh, torch.uint8) for sh in shapes]
    fp8lin.fp8lin_quantize_batch([(to_dev_bf16(x), sl[0:1], sl[1:2], sl[2:3], q.t) for x, sl, q in zip(xs, slots, qs)],
                                 fmt)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    for x, sl, q in zip(xs, slots, qs):
        ref = oracle.quantize(x, fmt)
        alone = torch.zeros(3, device="cuda")
        q1 = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
        fp8lin.fp8lin_quantize(to_dev_bf16(x), fmt, alone[0:1], alone[1:2], alone[2:3], q1, None)
        torch.cuda.synchronize()
        assert scalar_bits(sl[0:1]) == f32_bits(ref["amax"]) == scalar_bits(alone[0:1])
        assert scalar_bits(sl[1:2]) == f32_bits(ref["scale"]) == scalar_bits(alone[1:2])
        assert scalar_bits(sl[2:3]) == f32_bits(ref["inv_scale"]) == scalar_bits(alone[2:3])
        assert np.array_equal(q.t.cpu().numpy(), ref["q"]) and torch.equal(q.t, q1) and q.intact()


@pytest.mark.parametrize("shapes", [[(8192, 4096)], [(2048, 4096), (8192, 4096)], [(256, 512), (1024, 512)]],
                         ids=["grid", "grid-batch", "cluster-batch"])
def test_quantize_max_in_either_half_of_a_packed_pair(fp8lin, shapes):
    """Each CTA folds the magnitudes of element pairs (an even and an odd
    element share one 32-bit word): the largest |x| sits in the first
    element of the tensor, an even one, in the part of a slice read before
    the staged tail, while larger values than the rest sit in odd elements
    of every slice's tail.  A fold that compared whole words instead of
    each half would report the odd elements' 0.5."""
    xs = []
    for rows, cols in shapes:
        x = np.zeros((rows, cols), dtype=np.uint16)
        flat = x.reshape(-1)
        flat[1::16] = 0x3F00            # 0.5 in odd elements everywhere, tails included
        flat[0] = 0x4080                # 4.0: the first (even) element
        flat[-7] = 0xBF80               # -1.0 near the end, odd element
        xs.append(x)
    slots = [torch.zeros(3, device="cuda") for _ in xs]
    qs = [torch.empty(x.shape, dtype=torch.uint8, device="cuda") for x in xs]
    fp8lin.fp8lin_quantize_batch([(to_dev_bf16(x), sl[0:1], sl[1:2], sl[2:3], q) for x, sl, q in zip(xs, slots, qs)],
                                 E4M3)
    torch.cuda.synchronize()
    for x, sl, q in zip(xs, slots, qs):
        ref = oracle.quantize(x, E4M3)
        assert sl[0].item() == 4.0 and scalar_bits(sl[0:1]) == f32_bits(ref["amax"])
        assert np.array_equal(q.cpu().numpy(), ref["q"])


def test_batched_quantize_nan_empty_and_fallback(fp8lin):
    """A NaN in one tensor of a batch leaves the others' scales alone; a
    batch of empty tensors publishes the floor scales; fmt_max above 65504
    casts each tensor through amax + cast, with the same results as the
    oracle."""
    x_nan = wl.generate((256, 256), "normal", 1.0, seed=5, tensor_id=0)
    x_nan[17, 33] = 0x7FC1
    x_ok = wl.generate((512, 256), "normal", 0.02, seed=6, tensor_id=1)
    for shapes_x in ([x_nan, x_ok], [x_nan, wl.generate((2048, 1024), "normal", 0.02, seed=7, tensor_id=2)]):
        slots = [torch.zeros(3, device="cuda") for _ in shapes_x]
        qs = [torch.empty(x.shape, dtype=torch.uint8, device="cuda") for x in shapes_x]
        fp8lin.fp8lin_quantize_batch([(to_dev_bf16(x), sl[0:1], sl[1:2], sl[2:3], q)
                                      for x, sl, q in zip(shapes_x, slots, qs)], E4M3)
        torch.cuda.synchronize()
        for x, sl, q in zip(shapes_x, slots, qs):
            ref = oracle.quantize(x, E4M3)
            assert scalar_bits(sl[0:1]) == f32_bits(ref["amax"])
            assert scalar_bits(sl[1:2]) == f32_bits(ref["scale"])
            assert np.array_equal(q.cpu().numpy(), ref["q"])
    empties = [torch.full((3,), 5.0, device="cuda") for _ in range(2)]
    e = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    fp8lin.fp8lin_quantize_batch([(e, sl[0:1], sl[1:2], sl[2:3], torch.empty((0, 64), dtype=torch.uint8,
                                                                             device="cuda")) for sl in empties], E4M3)
    torch.cuda.synchronize()
    for sl in empties:
        assert sl[0].item() == 0.0 and scalar_bits(sl[1:2]) == f32_bits(oracle.scale(np.float32(0.0))[0])
    xs = [wl.generate((1040, 2048), "laplace", 1e-3, seed=77 + k, tensor_id=k) for k in range(2)]
    slots = [torch.zeros(3, device="cuda") for _ in xs]
    qs = [torch.empty(x.shape, dtype=torch.uint8, device="cuda") for x in xs]
    fp8lin.fp8lin_quantize_batch([(to_dev_bf16(x), sl[0:1], sl[1:2], sl[2:3], q) for x, sl, q in zip(xs, slots, qs)],
                                 E5M2, 1.0e5)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    for x, sl, q in zip(xs, slots, qs):
        ref = oracle.quantize(x, E5M2, 1.0e5)
        assert scalar_bits(sl[1:2]) == f32_bits(ref["scale"]) and np.array_equal(q.cpu().numpy(), ref["q"])


def test_one_call_quantize_repeated_and_empty(fp8lin):
    """Back-to-back calls reuse the same slots (each call clears them before
    its grid counts itself in); an empty matrix publishes the floor scale."""
    xs = [wl.generate((2048, 1024), "normal", sd, seed=80 + i, tensor_id=0) for i, sd in enumerate((1.0, 0.02, 3.0))]
    slots = torch.zeros(3, device="cuda")
    q = torch.empty((2048, 1024), dtype=torch.uint8, device="cuda")
    for x in xs:
        fp8lin.fp8lin_quantize(to_dev_bf16(x), E4M3, slots[0:1], slots[1:2], slots[2:3], q, None)
        torch.cuda.synchronize()
        ref = oracle.quantize(x, E4M3)
        assert scalar_bits(slots[1:2]) == f32_bits(ref["scale"])
        assert np.array_equal(q.cpu().numpy(), ref["q"])
    e = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    fp8lin.fp8lin_quantize(e, E4M3, slots[0:1], slots[1:2], slots[2:3], torch.empty((0, 64), dtype=torch.uint8,
                                                                                     device="cuda"), None)
    torch.cuda.synchronize()
    assert slots[0].item() == 0.0 and scalar_bits(slots[1:2]) == f32_bits(oracle.scale(np.float32(0.0))[0])
    assert fp8lin.fp8lin_device_error() == 0

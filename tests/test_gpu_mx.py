"""Power-of-two block scaling on the GPU against the oracle: the one-pass cast
(1 x 32 and 32 x 1 blocks) with every FP8 byte and every scale byte of the
atoms bit-exact, and the three block-scaled GEMMs (scales applied by the
tensor cores) within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import Guarded, assert_gemm_close, bf16_to_f64, to_dev_bf16

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2


def _atoms(P, K):
    return ((P + 127) // 128) * ((K + 127) // 128) * 512


def _ref_atoms(ref, along, rows, cols):
    P, K = (rows, cols) if along == "cols" else (cols, rows)
    return oracle.pack_sf(oracle.sf_by_operand_row(ref["sf"], along), P, K).reshape(-1)


@pytest.mark.parametrize("shape", [(16, 16), (48, 80), (144, 272), (384, 1040), (1040, 384), (2048, 4096)])
@pytest.mark.parametrize("fmt,dist", [(E4M3, ("normal", 1.0)), (E5M2, ("laplace", 1e-3))])
@pytest.mark.parametrize("kinds", [("row", "col"), ("row",), ("col",)])
def test_mx_cast_bit_exact(fp8lin, shape, fmt, dist, kinds):
    rows, cols = shape
    x = wl.generate(shape, *dist, seed=rows * 7 + cols, tensor_id=6, outlier_frac=1e-3)
    xd = to_dev_bf16(x)
    bufs = {}
    for k in kinds:
        P, K = (rows, cols) if k == "row" else (cols, rows)
        bufs[k] = (Guarded((rows, cols), torch.uint8), Guarded((_atoms(P, K),), torch.uint8))
    args = {}
    for k in ("row", "col"):
        args["q_" + k] = bufs[k][0].t if k in bufs else None
        args["sf_" + k] = bufs[k][1].t if k in bufs else None
    fp8lin.fp8lin_cast_mx(xd, fmt, **args)
    torch.cuda.synchronize()
    for k in kinds:
        along = "cols" if k == "row" else "rows"
        ref = oracle.quantize_mx(x, fmt, along)
        q, sf = bufs[k]
        assert np.array_equal(sf.t.cpu().numpy(), _ref_atoms(ref, along, rows, cols)), k
        assert np.array_equal(q.t.cpu().numpy(), ref["q"]), k
        assert q.intact() and sf.intact(), k


def test_mx_cast_zero_tensor_and_arguments(fp8lin):
    x = torch.zeros((128, 256), dtype=torch.bfloat16, device="cuda")
    q = torch.full((128, 256), 0xFF, dtype=torch.uint8, device="cuda")
    sf = torch.zeros((_atoms(128, 256),), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_cast_mx(x, E4M3, q_row=q, sf_row=sf)
    torch.cuda.synchronize()
    ref = oracle.quantize_mx(np.zeros((128, 256), np.uint16), E4M3, "cols")
    assert (q == 0).all()
    assert np.array_equal(sf.cpu().numpy(), _ref_atoms(ref, "cols", 128, 256))
    assert int(sf[0].item()) == 127 - 48                 # amax floored at 1e-12: scale 2^48
    with pytest.raises(fp8lin.Fp8LinError):
        fp8lin.fp8lin_cast_mx(x, E4M3, q_row=q)          # a copy without its scales
    with pytest.raises(fp8lin.Fp8LinError):
        fp8lin.fp8lin_cast_mx(x, E4M3)                   # nothing asked for


def test_mx_cast_fmt_max_e5m2_range(fp8lin):
    # the alternative reading of the e5m2 numerator (its own maximum, 57344)
    x = wl.generate((256, 384), "laplace", 1e-3, 31, 2)
    q = torch.empty((256, 384), dtype=torch.uint8, device="cuda")
    sf = torch.empty((_atoms(256, 384),), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_cast_mx(to_dev_bf16(x), E5M2, q_row=q, sf_row=sf, fmt_max=57344.0)
    torch.cuda.synchronize()
    ref = oracle.quantize_mx(x, E5M2, "cols", 57344.0)
    assert np.array_equal(sf.cpu().numpy(), _ref_atoms(ref, "cols", 256, 384))
    assert np.array_equal(q.cpu().numpy(), ref["q"])


# (M, N, K): ragged pair tiles in every direction, a contraction shorter than
# one slab and not a multiple of 32, 16-row and 16-column outputs, an odd
# number of 128-row blocks of B
GEMM_SHAPES = [(128, 128, 128), (144, 272, 208), (384, 1040, 4112), (1040, 400, 96), (2048, 2048, 2048),
               (16, 16, 16), (16, 528, 144), (272, 16, 400), (256, 384, 48)]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


@pytest.mark.parametrize("M,N,K", GEMM_SHAPES)
@pytest.mark.parametrize("which", ["fwd", "dgrad", "wgrad"])
def test_mx_gemm_matches_oracle(fp8lin, M, N, K, which):
    X = wl.generate((M, K), "normal", 1.0, M + 1, wl.X, outlier_frac=1e-3)
    W = wl.generate((N, K), "normal", 0.02, N + 2, wl.W)
    dY = wl.generate((M, N), "laplace", 1e-3, K + 3, wl.DY)
    r = oracle.quantize_mx_recipe(X, W, dY)
    if which == "fwd":
        out, (a, b) = Guarded((M, N), torch.bfloat16), (r["x_k"], r["w_k"])
        ref = oracle.fwd_mx_ref(a["q"], a["sf"], b["q"], b["sf"])
    elif which == "dgrad":
        out, (a, b) = Guarded((M, K), torch.bfloat16), (r["dy_n"], r["w_n"])
        ref = oracle.dgrad_mx_ref(a["q"], a["sf"], b["q"], b["sf"])
    else:
        out, (a, b) = Guarded((N, K), torch.bfloat16), (r["dy_m"], r["x_m"])
        ref = oracle.wgrad_mx_ref(a["q"], a["sf"], b["q"], b["sf"])
    out.t.fill_(float("nan"))
    getattr(fp8lin, f"fp8lin_{which}_mx")(_dev(a["q"]), _dev(a["atoms"].reshape(-1)), _dev(b["q"]),
                                         _dev(b["atoms"].reshape(-1)), out.t)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    assert_gemm_close(bf16_to_f64(out.t), ref, f"{which} mx {M}x{N}x{K}")
    assert out.intact()


def test_mx_gemm_scales_per_run_reach_the_output(fp8lin):
    # Every 32-run of the contraction carries its own power of two: with
    # codes of 1.0 and scales 2^-(j % 7) per run j of row m, Y[m][n] is a
    # plain sum of powers of two, which a scale taken from the wrong run or
    # row changes.
    M, N, K = 256, 256, 512
    one = 0x38                                              # e4m3 1.0
    a = np.full((M, K), one, np.uint8)
    b = np.full((N, K), one, np.uint8)
    nj = K // 32
    sfa = (127 + ((np.arange(M)[:, None] + np.arange(nj)[None, :]) % 7)).astype(np.uint8)   # 2^-0 .. 2^-6
    sfb = (127 + (np.arange(N)[:, None] % 3) + 0 * np.arange(nj)[None, :]).astype(np.uint8)
    ref = oracle.gemm_blocks(a, E4M3, b, E4M3, oracle.pow2_inverse(sfa), oracle.pow2_inverse(sfb), 32)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8lin.fp8lin_fwd_mx(_dev(a), _dev(oracle.pack_sf(sfa, M, K).reshape(-1)), _dev(b),
                         _dev(oracle.pack_sf(sfb, N, K).reshape(-1)), y)
    torch.cuda.synchronize()
    got = bf16_to_f64(y)
    # the fp32 sum is exact (multiples of 2^-3 below 2^10); the kernel rounds it once to bf16
    want = wl.bf16_bits_to_f32(wl.f32_to_bf16_bits(ref.astype(np.float32))).astype(np.float64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("M,K,N", [(256, 512, 1024), (144, 208, 272), (640, 384, 1296)])
def test_mx_cast_then_gemms_match_oracle(fp8lin, M, K, N):
    """The recipe end to end on the device: cast every copy, then the three GEMMs."""
    X = wl.generate((M, K), "normal", 1.0, 41, wl.X, outlier_frac=1e-3)
    W = wl.generate((N, K), "normal", 0.02, 41, wl.W)
    dY = wl.generate((M, N), "normal", 1e-3, 41, wl.DY)
    r = oracle.quantize_mx_recipe(X, W, dY)
    dev = {}
    for name, bits, fmt in (("x", X, E4M3), ("w", W, E4M3), ("dy", dY, E5M2)):
        rows, cols = bits.shape
        qr = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
        qc = torch.empty_like(qr)
        sr = torch.empty((_atoms(rows, cols),), dtype=torch.uint8, device="cuda")
        sc = torch.empty((_atoms(cols, rows),), dtype=torch.uint8, device="cuda")
        fp8lin.fp8lin_cast_mx(to_dev_bf16(bits), fmt, q_row=qr, sf_row=sr, q_col=qc, sf_col=sc)
        dev[name] = (qr, sr, qc, sc)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    fp8lin.fp8lin_fwd_mx(dev["x"][0], dev["x"][1], dev["w"][0], dev["w"][1], y)
    fp8lin.fp8lin_dgrad_mx(dev["dy"][0], dev["dy"][1], dev["w"][2], dev["w"][3], dx)
    fp8lin.fp8lin_wgrad_mx(dev["dy"][2], dev["dy"][3], dev["x"][2], dev["x"][3], dw)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    for key, (q, atoms) in (("x_k", dev["x"][0:2]), ("x_m", dev["x"][2:4]), ("w_k", dev["w"][0:2]),
                            ("w_n", dev["w"][2:4]), ("dy_n", dev["dy"][0:2]), ("dy_m", dev["dy"][2:4])):
        assert np.array_equal(q.cpu().numpy(), r[key]["q"]), key
        assert np.array_equal(atoms.cpu().numpy(), r[key]["atoms"].reshape(-1)), key
    assert_gemm_close(bf16_to_f64(y), oracle.fwd_mx_ref(r["x_k"]["q"], r["x_k"]["sf"], r["w_k"]["q"],
                                                        r["w_k"]["sf"]), "fwd")
    assert_gemm_close(bf16_to_f64(dx), oracle.dgrad_mx_ref(r["dy_n"]["q"], r["dy_n"]["sf"], r["w_n"]["q"],
                                                           r["w_n"]["sf"]), "dgrad")
    assert_gemm_close(bf16_to_f64(dw), oracle.wgrad_mx_ref(r["dy_m"]["q"], r["dy_m"]["sf"], r["x_m"]["q"],
                                                           r["x_m"]["sf"]), "wgrad")


def _rows(n, seed, count=40):
    rng = np.random.default_rng(seed)
    pick = rng.choice(n, size=min(n, count - 2), replace=False)
    return np.unique(np.concatenate([[0, n - 1], pick])).astype(np.int64)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_mx_workload_step_matches_oracle(fp8lin, name):
    """Every configuration at full size through Float8Linear: every FP8 byte
    and every scale byte of the six copies bit-exact; Y, dX, dW on sampled
    rows (the first, the last and 38 seeded others)."""
    w = wl.WORKLOADS[name]
    X, W, dY = w.make_x(), w.make_w(), w.make_dy()
    lin = fp8lin.Float8Linear(w.M, w.K, w.N, scaling="mx")
    y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    r = oracle.quantize_mx_recipe(X, W, dY)
    got = {"x_k": (lin.x8.q, lin.x8.sf_row), "x_m": (lin.x8.qc, lin.x8.sf_col),
           "w_k": (lin.w8.q, lin.w8.sf_row), "w_n": (lin.w8.qc, lin.w8.sf_col),
           "dy_n": (lin.dy8.q, lin.dy8.sf_row), "dy_m": (lin.dy8.qc, lin.dy8.sf_col)}
    for key, (q, atoms) in got.items():
        assert np.array_equal(atoms.cpu().numpy(), r[key]["atoms"].reshape(-1)), f"{name} {key} scales"
        assert np.array_equal(q.cpu().numpy(), r[key]["q"]), f"{name} {key} codes"
    rm, rn = _rows(w.M, w.seed), _rows(w.N, w.seed + 1)
    pick = lambda t, rows: bf16_to_f64(t[torch.from_numpy(rows).cuda()])
    assert_gemm_close(pick(y, rm), oracle.fwd_mx_ref(r["x_k"]["q"], r["x_k"]["sf"], r["w_k"]["q"], r["w_k"]["sf"],
                                                     rm), f"{name} Y")
    assert_gemm_close(pick(dx, rm), oracle.dgrad_mx_ref(r["dy_n"]["q"], r["dy_n"]["sf"], r["w_n"]["q"],
                                                        r["w_n"]["sf"], rm), f"{name} dX")
    assert_gemm_close(pick(dw, rn), oracle.wgrad_mx_ref(r["dy_m"]["q"], r["dy_m"]["sf"], r["x_m"]["q"],
                                                        r["x_m"]["sf"], rn), f"{name} dW")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx_cast_special_values(fp8lin, fmt):
    """NaN, +-Inf, signed zeros, bf16 subnormals and the largest bf16 in
    chosen blocks: a block whose amax is NaN or infinite gets the scale byte
    0xFF (its codes come out NaN); the other blocks are unaffected."""
    rows, cols = 128, 256
    x = wl.generate((rows, cols), "normal", 1.0, 51, 0)
    x[0, 5] = 0x7FC0            # NaN in row block (0, 0)
    x[40, 100] = 0xFF80         # -Inf in row block (40, 3)
    x[70, 200] = 0x7F7F         # largest finite bf16
    x[3, 33:64] = 0x8000        # -0 across a run
    x[90, 130:140] = 0x0001     # bf16 subnormals
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    qc = torch.empty_like(q)
    sr = torch.empty((_atoms(rows, cols),), dtype=torch.uint8, device="cuda")
    sc = torch.empty((_atoms(cols, rows),), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_cast_mx(to_dev_bf16(x), fmt, q_row=q, sf_row=sr, q_col=qc, sf_col=sc)
    torch.cuda.synchronize()
    table = oracle.decode_table(fmt)
    for along, got_q, got_sf in (("cols", q, sr), ("rows", qc, sc)):
        ref = oracle.quantize_mx(x, fmt, along)
        assert np.array_equal(got_sf.cpu().numpy(), _ref_atoms(ref, along, rows, cols)), along
        assert (ref["sf"] == 0xFF).sum() == 2                 # the NaN and the Inf blocks
        got = got_q.cpu().numpy()
        nan_ref = np.isnan(table[ref["q"]])
        assert nan_ref.sum() == 64                            # every element of those two blocks
        assert np.array_equal(got, ref["q"]), along           # NaN codes included (0x7F)


def _fuzz_shapes(n=24, seed=2024):
    rng = np.random.default_rng(seed)
    return [tuple(int(16 * rng.integers(1, 66)) for _ in range(3)) for _ in range(n)]


@pytest.mark.parametrize("M,K,N", _fuzz_shapes())
def test_mx_fuzz_shapes(fp8lin, M, K, N):
    """Seeded random shapes (multiples of 16 from 16 to 1040): the device
    casts of X, W, dY and the three GEMMs on them against the oracle."""
    X = wl.generate((M, K), "normal", 1.0, M + K, wl.X)
    W = wl.generate((N, K), "normal", 0.02, N + K, wl.W)
    dY = wl.generate((M, N), "laplace", 1e-3, M + N, wl.DY)
    lin = fp8lin.Float8Linear(M, K, N, scaling="mx")
    y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    r = oracle.quantize_mx_recipe(X, W, dY)
    for key, (q, atoms) in (("x_k", (lin.x8.q, lin.x8.sf_row)), ("w_n", (lin.w8.qc, lin.w8.sf_col)),
                            ("dy_m", (lin.dy8.qc, lin.dy8.sf_col))):
        assert np.array_equal(q.cpu().numpy(), r[key]["q"]), key
        assert np.array_equal(atoms.cpu().numpy(), r[key]["atoms"].reshape(-1)), key
    assert_gemm_close(bf16_to_f64(y), oracle.fwd_mx_ref(r["x_k"]["q"], r["x_k"]["sf"], r["w_k"]["q"],
                                                        r["w_k"]["sf"]), f"Y {M}x{K}x{N}")
    assert_gemm_close(bf16_to_f64(dx), oracle.dgrad_mx_ref(r["dy_n"]["q"], r["dy_n"]["sf"], r["w_n"]["q"],
                                                           r["w_n"]["sf"]), f"dX {M}x{K}x{N}")
    assert_gemm_close(bf16_to_f64(dw), oracle.wgrad_mx_ref(r["dy_m"]["q"], r["dy_m"]["sf"], r["x_m"]["q"],
                                                           r["x_m"]["sf"]), f"dW {M}x{K}x{N}")


# ------------------------------------------------------- OCP scale rule

@pytest.mark.parametrize("shape", [(16, 16), (48, 80), (384, 1040), (2048, 4096)])
@pytest.mark.parametrize("fmt,dist", [(E4M3, ("normal", 1.0)), (E5M2, ("laplace", 1e-3))])
def test_mx_ocp_cast_bit_exact(fp8lin, shape, fmt, dist):
    """fp8lin_cast_mx_ocp: the OCP Microscaling rule, every code and scale
    byte bit-exact (the top binade above the format's maximum saturates)."""
    rows, cols = shape
    x = wl.generate(shape, *dist, seed=rows * 11 + cols, tensor_id=7, outlier_frac=1e-3)
    q, qc = Guarded((rows, cols), torch.uint8), Guarded((rows, cols), torch.uint8)
    sr, sc = Guarded((_atoms(rows, cols),), torch.uint8), Guarded((_atoms(cols, rows),), torch.uint8)
    fp8lin.fp8lin_cast_mx(to_dev_bf16(x), fmt, q_row=q.t, sf_row=sr.t, q_col=qc.t, sf_col=sc.t, rule="ocp")
    torch.cuda.synchronize()
    for along, gq, gs in (("cols", q, sr), ("rows", qc, sc)):
        ref = oracle.quantize_mx(x, fmt, along, rule="ocp")
        assert np.array_equal(gs.t.cpu().numpy(), _ref_atoms(ref, along, rows, cols)), along
        assert np.array_equal(gq.t.cpu().numpy(), ref["q"]), along
        assert gq.intact() and gs.intact()


def test_mx_ocp_cast_zero_and_special_blocks(fp8lin):
    rows, cols = 64, 128
    x = wl.generate((rows, cols), "normal", 1.0, 52, 0)
    x[0:32, 0] = 0                                            # an all-zero 32 x 1 block: scale byte 0
    x[33, 0:32] = 0                                           # an all-zero 1 x 32 block
    x[5, 70] = 0x7F80                                         # +Inf
    x[40, 100] = 0x0003                                       # a bf16 subnormal
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    qc = torch.empty_like(q)
    sr = torch.empty((_atoms(rows, cols),), dtype=torch.uint8, device="cuda")
    sc = torch.empty((_atoms(cols, rows),), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_cast_mx(to_dev_bf16(x), E4M3, q_row=q, sf_row=sr, q_col=qc, sf_col=sc, rule="ocp")
    torch.cuda.synchronize()
    for along, gq, gs in (("cols", q, sr), ("rows", qc, sc)):
        ref = oracle.quantize_mx(x, E4M3, along, rule="ocp")
        assert np.array_equal(gs.cpu().numpy(), _ref_atoms(ref, along, rows, cols)), along
        assert (ref["sf"] == 0).sum() >= 1 and (ref["sf"] == 0xFF).sum() == 1
        assert np.array_equal(gq.cpu().numpy(), ref["q"]), along   # NaN codes included (0x7F)


@pytest.mark.parametrize("M,K,N", [(256, 512, 1024), (144, 208, 272)])
def test_mx_ocp_linear_step_matches_oracle(fp8lin, M, K, N):
    """Copies cast with the OCP rule feed the same block-scaled GEMMs."""
    X = wl.generate((M, K), "normal", 1.0, 61, wl.X, outlier_frac=1e-3)
    W = wl.generate((N, K), "normal", 0.02, 61, wl.W)
    dY = wl.generate((M, N), "normal", 1e-3, 61, wl.DY)
    lin = fp8lin.Float8Linear(M, K, N, scaling="mx", mx_rule="ocp")
    y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    r = oracle.quantize_mx_recipe(X, W, dY, rule="ocp")
    assert np.array_equal(lin.x8.q.cpu().numpy(), r["x_k"]["q"])
    assert np.array_equal(lin.dy8.sf_col.cpu().numpy(), r["dy_m"]["atoms"].reshape(-1))
    assert_gemm_close(bf16_to_f64(y), oracle.fwd_mx_ref(r["x_k"]["q"], r["x_k"]["sf"], r["w_k"]["q"],
                                                        r["w_k"]["sf"]), "Y")
    assert_gemm_close(bf16_to_f64(dx), oracle.dgrad_mx_ref(r["dy_n"]["q"], r["dy_n"]["sf"], r["w_n"]["q"],
                                                           r["w_n"]["sf"]), "dX")
    assert_gemm_close(bf16_to_f64(dw), oracle.wgrad_mx_ref(r["dy_m"]["q"], r["dy_m"]["sf"], r["x_m"]["q"],
                                                           r["x_m"]["sf"]), "dW")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_mx_ocp_cast_blocks_of_subnormals(fp8lin, fmt):
    """A 1 x 32 and a 32 x 1 block of bf16 subnormals (signs mixed) under the
    OCP rule: scale byte 0, the elements multiplied by 2^127 into normal FP8
    codes.  The kernel's products take the subnormals as they are (no flush
    to zero); both copies bit-exact against the oracle."""
    rows, cols = 128, 128
    x = wl.generate((rows, cols), "normal", 1.0, 53, 0)
    sub = np.array([0x0001, 0x0003, 0x8001, 0x007F, 0x0040, 0x8055, 0x0000, 0x8000] * 4, np.uint16)
    x[10, 32:64] = sub                 # a 1 x 32 block of the row copy
    x[64:96, 7] = sub                  # a 32 x 1 block of the column copy
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    qc = torch.empty_like(q)
    sr = torch.empty((_atoms(rows, cols),), dtype=torch.uint8, device="cuda")
    sc = torch.empty((_atoms(cols, rows),), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_cast_mx(to_dev_bf16(x), fmt, q_row=q, sf_row=sr, q_col=qc, sf_col=sc, rule="ocp")
    torch.cuda.synchronize()
    for along, got_q, got_sf in (("cols", q, sr), ("rows", qc, sc)):
        ref = oracle.quantize_mx(x, fmt, along, rule="ocp")
        blk = ref["sf"][10, 1] if along == "cols" else ref["sf"][2, 7]
        assert blk == 0, along
        assert np.array_equal(got_sf.cpu().numpy(), _ref_atoms(ref, along, rows, cols)), along
        assert np.array_equal(got_q.cpu().numpy(), ref["q"]), along

"""Static and delayed scaling on the GPU against the oracle, bit-exact:
scale, inverse scale, recorded amax / history and every FP8 byte."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import Guarded, f32_bits, scalar_bits, to_dev_bf16

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2
SHAPES = [(16, 16), (144, 272), (384, 1040), (2048, 4096)]


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("scale_value", [1.0, 97.25, 2.0 ** 20])
def test_static_scaling_bit_exact(fp8lin, shape, fmt, scale_value):
    x = wl.generate(shape, "normal", 0.5, shape[0], fmt)
    scale = torch.tensor([scale_value], dtype=torch.float32, device="cuda")
    inv = torch.zeros(1, device="cuda")
    amax = torch.full((1,), -1.0, device="cuda")
    q = Guarded(shape, torch.uint8)
    qT = Guarded(shape[::-1], torch.uint8)
    fp8lin.fp8lin_cast_transpose_static(to_dev_bf16(x), fmt, scale, inv, q.t, qT.t, amax)
    ref = oracle.quantize_static(x, fmt, scale_value)
    assert scalar_bits(inv) == f32_bits(ref["inv_scale"])
    assert scalar_bits(amax) == f32_bits(ref["amax"])
    assert scalar_bits(scale) == f32_bits(np.float32(scale_value))
    assert np.array_equal(q.t.cpu().numpy(), ref["q"]) and np.array_equal(qT.t.cpu().numpy(), ref["qT"])
    assert q.intact() and qT.intact()


@pytest.mark.parametrize("shape", SHAPES)
@pytest.mark.parametrize("fmt,fmt_max", [(E4M3, 448.0), (E5M2, 448.0), (E5M2, 57344.0)])
def test_delayed_scaling_bit_exact(fp8lin, shape, fmt, fmt_max):
    x = wl.generate(shape, "normal", 1.0, 11, fmt)
    a = oracle.amax(x)
    hist = np.array([a * np.float32(0.75), 3.0, 0.0, a * np.float32(0.5), 0.25], np.float32)
    for slot in (1, 4):
        h = torch.from_numpy(hist.copy()).cuda()
        scale = torch.zeros(1, device="cuda")
        inv = torch.zeros(1, device="cuda")
        q = torch.empty(shape, dtype=torch.uint8, device="cuda")
        qT = torch.empty(shape[::-1], dtype=torch.uint8, device="cuda")
        fp8lin.fp8lin_cast_transpose_delayed(to_dev_bf16(x), fmt, h, slot, scale, inv, q, qT, fmt_max)
        ref = oracle.quantize_delayed(x, fmt, hist, slot, fmt_max)
        assert scalar_bits(scale) == f32_bits(ref["scale"]) and scalar_bits(inv) == f32_bits(ref["inv_scale"])
        assert np.array_equal(h.cpu().numpy().view(np.uint32), ref["history"].view(np.uint32))
        assert np.array_equal(q.cpu().numpy(), ref["q"]) and np.array_equal(qT.cpu().numpy(), ref["qT"])


def test_delayed_ring_over_steps_matches_oracle(fp8lin):
    """Several steps of a Float8Tensor with delayed scaling: seed, ring
    rotation and the recorded statistics all follow the oracle."""
    shape, H = (256, 384), 4
    t8 = fp8lin.Float8Tensor(*shape, E4M3, "cuda", scaling="delayed", history_len=H)
    hist = np.zeros(H, np.float32)
    slot = 0
    for step in range(6):
        x = wl.generate(shape, "normal", 1.0 + step, 20 + step, 0)
        if step == 0:
            hist[(slot - 1) % H] = oracle.amax(x)        # the seed amax pass
        ref = oracle.quantize_delayed(x, E4M3, hist, slot)
        t8.quantize(to_dev_bf16(x))
        assert scalar_bits(t8.scale) == f32_bits(ref["scale"]), f"step {step}"
        assert np.array_equal(t8.q.cpu().numpy(), ref["q"]), f"step {step}"
        hist, slot = ref["history"], (slot + 1) % H
        assert np.array_equal(t8.history.cpu().numpy(), hist)


def test_delayed_argument_checks(fp8lin):
    x = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    one = torch.zeros(1, device="cuda")
    with pytest.raises(fp8lin.Fp8LinError):   # history of one slot
        fp8lin.fp8lin_cast_transpose_delayed(x, E4M3, torch.zeros(1, device="cuda"), 0, one, one, None, None)
    with pytest.raises(fp8lin.Fp8LinError):   # slot out of range
        fp8lin.fp8lin_cast_transpose_delayed(x, E4M3, torch.zeros(4, device="cuda"), 4, one, one, None, None)


@pytest.mark.parametrize("transpose", [False, True])
@pytest.mark.parametrize("scaling", ["delayed", "static"])
def test_float8_linear_step_with_other_scalings(fp8lin, scaling, transpose):
    """A whole linear step under delayed / static scaling against the oracle."""
    from gpu_helpers import assert_gemm_close, bf16_to_f64
    M, K, N = 256, 512, 1024
    X = wl.generate((M, K), "normal", 1.0, 8, wl.X)
    W = wl.generate((N, K), "normal", 0.02, 8, wl.W)
    dY = wl.generate((M, N), "normal", 1e-3, 8, wl.DY)
    lin = fp8lin.Float8Linear(M, K, N, scaling=scaling, transpose=transpose)
    if scaling == "static":
        for t8, s in ((lin.x8, 64.0), (lin.w8, 8192.0), (lin.dy8, 65536.0)):
            t8.set_scale(s)
    y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
    torch.cuda.synchronize()
    if scaling == "static":
        rx, rw, rd = (oracle.quantize_static(X, E4M3, 64.0), oracle.quantize_static(W, E4M3, 8192.0),
                      oracle.quantize_static(dY, E5M2, 65536.0))
    else:
        def seeded(bits, fmt):
            h = np.zeros(16, np.float32)
            h[15] = oracle.amax(bits)
            return oracle.quantize_delayed(bits, fmt, h, 0)
        rx, rw, rd = seeded(X, E4M3), seeded(W, E4M3), seeded(dY, E5M2)
    for t8, r in ((lin.x8, rx), (lin.w8, rw), (lin.dy8, rd)):
        assert scalar_bits(t8.inv_scale) == f32_bits(r["inv_scale"])
        assert np.array_equal(t8.q.cpu().numpy(), r["q"])
        assert (t8.qT is None) if not transpose else np.array_equal(t8.qT.cpu().numpy(), r["qT"])
    assert_gemm_close(bf16_to_f64(y), oracle.fwd_ref(rx["q"], rx["inv_scale"], rw["q"], rw["inv_scale"]), "Y")
    assert_gemm_close(bf16_to_f64(dx), oracle.dgrad_ref(rd["q"], rd["inv_scale"], rw["qT"], rw["inv_scale"]), "dX")
    assert_gemm_close(bf16_to_f64(dw), oracle.wgrad_ref(rd["qT"], rd["inv_scale"], rx["qT"], rx["inv_scale"]), "dW")


def _times_two(bits):
    """x * 2 in bf16, exactly (bf16 -> f32 -> *2 -> the top 16 bits)."""
    f = wl.bf16_bits_to_f32(bits) * np.float32(2.0)
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def _rows(n, seed, count=24):
    rng = np.random.default_rng(seed)
    pick = rng.choice(n, size=min(n, count - 2), replace=False)
    return np.unique(np.concatenate([[0, n - 1], pick])).astype(np.int64)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_delayed_workload_two_steps_match_oracle(fp8lin, name):
    """Every configuration at full size, two steps of delayed scaling: the
    second step's tensors are the first's times two, so its scales come from
    the first step's recorded amax and the upper half of every tensor
    saturates.  Scales, histories and every FP8 byte bit-exact; Y, dX, dW on
    sampled rows of the second step."""
    from gpu_helpers import assert_gemm_close, bf16_to_f64
    w = wl.WORKLOADS[name]
    H = 4
    lin = fp8lin.Float8Linear(w.M, w.K, w.N, scaling="delayed", history_len=H)
    steps = [(w.make_x(), w.make_w(), w.make_dy())]
    steps.append(tuple(_times_two(t) for t in steps[0]))
    hist = {k: np.zeros(H, np.float32) for k in "xwd"}
    for step, (X, W, dY) in enumerate(steps):
        y, dx, dw = lin.step(to_dev_bf16(X), to_dev_bf16(W), to_dev_bf16(dY))
        torch.cuda.synchronize()
        assert fp8lin.fp8lin_device_error() == 0
        refs = {}
        for k, bits, fmt in (("x", X, E4M3), ("w", W, E4M3), ("d", dY, E5M2)):
            if step == 0:
                hist[k][(0 - 1) % H] = oracle.amax(bits)      # the seed amax pass
            refs[k] = oracle.quantize_delayed(bits, fmt, hist[k], step)
            hist[k] = refs[k]["history"]
        for k, t8 in (("x", lin.x8), ("w", lin.w8), ("d", lin.dy8)):
            r = refs[k]
            assert scalar_bits(t8.inv_scale) == f32_bits(r["inv_scale"]), (name, step, k)
            assert np.array_equal(t8.history.cpu().numpy().view(np.uint32), r["history"].view(np.uint32)), (name, step, k)
            assert np.array_equal(t8.q.cpu().numpy(), r["q"]), (name, step, k)
    rx, rw, rd = refs["x"], refs["w"], refs["d"]
    rm, rn = _rows(w.M, w.seed), _rows(w.N, w.seed + 1)
    pick = lambda t, rows: bf16_to_f64(t[torch.from_numpy(rows).cuda()])
    assert_gemm_close(pick(y, rm), oracle.fwd_ref(rx["q"], rx["inv_scale"], rw["q"], rw["inv_scale"], rm), f"{name} Y")
    assert_gemm_close(pick(dx, rm), oracle.dgrad_ref(rd["q"], rd["inv_scale"], rw["qT"], rw["inv_scale"], rm), f"{name} dX")
    assert_gemm_close(pick(dw, rn), oracle.wgrad_ref(rd["qT"], rd["inv_scale"], rx["qT"], rx["inv_scale"], rn), f"{name} dW")

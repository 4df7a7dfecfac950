"""NaN inputs through every cast on the GPU, compared with the oracle byte for
byte: the per-tensor cast (every bf16 pattern, NaNs of both signs and every
payload included), the row-wise cast, the fp32 block casts (1 x 128,
128 x 1, 128 x 128) and the power-of-two block casts (both scale rules).
A NaN anywhere in a row, column or block makes that statistic NaN, so the
whole row, column or block casts through a NaN scale; the FP8 bytes, the
scale bytes and the binary32 scales must all equal the oracle's."""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import to_dev_bf16

pytestmark = pytest.mark.gpu
E4M3, E5M2 = oracle.E4M3, oracle.E5M2
NAN_INPUTS = (0x7FC0, 0xFFC0, 0x7F81, 0xFFFF, 0x7FFF, 0xFF81)   # quiet and signalling payloads, both signs


def _nan_matrix(rows, cols, seed):
    x = wl.generate((rows, cols), "normal", 1.0, seed, 0)
    rng = np.random.default_rng(seed)
    for k, v in enumerate(NAN_INPUTS):
        x[rng.integers(rows), rng.integers(cols)] = v
    x[rows - 1, cols - 1] = 0xFF80                                 # -Inf as well
    return x


def _same_bytes(got, ref, x_in, what):
    """Byte-for-byte equality; on failure, list the distinct (input, got, oracle) triples."""
    got, ref = np.asarray(got), np.asarray(ref)
    if np.array_equal(got, ref):
        return
    bad = np.argwhere(got != ref)
    seen = {}
    for i in bad[:4096]:
        i = tuple(i)
        key = (int(x_in[i]) if x_in is not None else None, int(got[i]), int(ref[i]))
        seen[key] = seen.get(key, 0) + 1
    lines = ", ".join(f"in {k[0]:#06x} got {k[1]:#04x} oracle {k[2]:#04x} (x{n})" if k[0] is not None else
                      f"got {k[1]:#04x} oracle {k[2]:#04x} (x{n})" for k, n in sorted(seen.items()))
    raise AssertionError(f"{what}: {len(bad)} bytes differ: {lines}")


def _same_f32(got, ref, what):
    """Bit-for-bit equality of binary32 values (NaN payloads and signs included)."""
    g = np.asarray(got, dtype=np.float32).reshape(-1).view(np.uint32)
    r = np.asarray(ref, dtype=np.float32).reshape(-1).view(np.uint32)
    assert g.shape == r.shape, f"{what}: {g.shape} values, oracle {r.shape}"
    if not np.array_equal(g, r):
        i = np.flatnonzero(g != r)[:8]
        pairs = ", ".join(f"[{j}] got {int(g[j]):#010x} oracle {int(r[j]):#010x}" for j in i)
        raise AssertionError(f"{what}: {int((g != r).sum())} binary32 values differ: {pairs}")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_per_tensor_cast_every_bf16_pattern_bytes(fp8lin, fmt):
    """All 65,536 bf16 patterns (254 NaNs among them) at a fixed scale."""
    x = np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(256, 256)
    amax = torch.tensor([3.0], dtype=torch.float32, device="cuda")
    scale, inv = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    q = torch.empty((256, 256), dtype=torch.uint8, device="cuda")
    qT = torch.empty_like(q)
    fp8lin.fp8lin_cast_transpose(to_dev_bf16(x), fmt, amax, scale, inv, q, qT)
    torch.cuda.synchronize()
    s, _ = oracle.scale(np.float32(3.0))
    ref = oracle.cast(x, fmt, s)
    _same_bytes(q.cpu().numpy(), ref, x, "q")
    _same_bytes(qT.cpu().numpy(), ref.T, x.T, "qT")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_per_tensor_nan_amax(fp8lin, fmt):
    """A NaN in the tensor: amax, scale and inverse scale NaN, every code NaN."""
    x = _nan_matrix(64, 96, 71)
    xd = to_dev_bf16(x)
    amax = torch.zeros(1, device="cuda")
    scale, inv = torch.zeros(1, device="cuda"), torch.zeros(1, device="cuda")
    q = torch.empty((64, 96), dtype=torch.uint8, device="cuda")
    qT = torch.empty((96, 64), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_amax(xd, amax)
    fp8lin.fp8lin_cast_transpose(xd, fmt, amax, scale, inv, q, qT)
    torch.cuda.synchronize()
    ref = oracle.quantize(x, fmt)
    _same_f32(amax.cpu().numpy(), ref["amax"], "amax")
    _same_f32(scale.cpu().numpy(), ref["scale"], "scale")
    _same_f32(inv.cpu().numpy(), ref["inv_scale"], "inv_scale")
    _same_bytes(q.cpu().numpy(), ref["q"], x, "q")
    _same_bytes(qT.cpu().numpy(), ref["qT"], x.T, "qT")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_rowwise_cast_nan_rows_and_columns(fp8lin, fmt):
    rows, cols = 144, 272
    x = _nan_matrix(rows, cols, 72)
    xd = to_dev_bf16(x)
    ra, ca = torch.zeros(rows, device="cuda"), torch.zeros(cols, device="cuda")
    ri, ci = torch.zeros(rows, device="cuda"), torch.zeros(cols, device="cuda")
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    qT = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_amax_rowcol(xd, ra, ca)
    fp8lin.fp8lin_cast_transpose_rowwise(xd, fmt, ra, ca, ri, ci, q, qT)
    torch.cuda.synchronize()
    ref = oracle.quantize_rowwise(x, fmt)
    _same_f32(ra.cpu().numpy(), ref["row_amax"], "row amax")
    _same_f32(ca.cpu().numpy(), ref["col_amax"], "column amax")
    _same_f32(ri.cpu().numpy(), ref["row_inv"], "row inverse scales")
    _same_f32(ci.cpu().numpy(), ref["col_inv"], "column inverse scales")
    _same_bytes(q.cpu().numpy(), ref["q"], x, "q")
    _same_bytes(qT.cpu().numpy(), ref["qT"], x.T, "qT")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_block_cast_nan_blocks(fp8lin, fmt):
    rows, cols = 256, 384
    x = _nan_matrix(rows, cols, 73)
    nr, nc = rows // 128, cols // 128
    q = {k: torch.empty((rows, cols), dtype=torch.uint8, device="cuda") for k in ("row", "col", "tile")}
    inv = {"row": torch.zeros((nc, rows), device="cuda"), "col": torch.zeros((nr, cols), device="cuda"),
           "tile": torch.zeros((nr, nc), device="cuda")}
    fp8lin.fp8lin_cast_blockwise(to_dev_bf16(x), fmt, q_row=q["row"], inv_row=inv["row"], q_col=q["col"],
                                 inv_col=inv["col"], q_tile=q["tile"], inv_tile=inv["tile"])
    torch.cuda.synchronize()
    for k, (br, bc) in (("row", (1, 128)), ("col", (128, 1)), ("tile", (128, 128))):
        ref = oracle.quantize_blocks(x, fmt, br, bc)
        got_inv = inv[k].cpu().numpy()
        _same_f32(got_inv.T if k == "row" else got_inv, ref["inv_scale"], f"{k} inverse scales")
        _same_bytes(q[k].cpu().numpy(), ref["q"], x, f"{k} q")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("rule", ["floor", "ocp"])
def test_mx_cast_nan_blocks(fp8lin, fmt, rule):
    rows, cols = 128, 256
    x = _nan_matrix(rows, cols, 74)
    atoms = lambda P, K: ((P + 127) // 128) * ((K + 127) // 128) * 512
    q, qc = (torch.empty((rows, cols), dtype=torch.uint8, device="cuda") for _ in range(2))
    sr = torch.empty((atoms(rows, cols),), dtype=torch.uint8, device="cuda")
    sc = torch.empty((atoms(cols, rows),), dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_cast_mx(to_dev_bf16(x), fmt, q_row=q, sf_row=sr, q_col=qc, sf_col=sc, rule=rule)
    torch.cuda.synchronize()
    for along, gq, gs in (("cols", q, sr), ("rows", qc, sc)):
        ref = oracle.quantize_mx(x, fmt, along, rule=rule)
        P, K = (rows, cols) if along == "cols" else (cols, rows)
        ref_atoms = oracle.pack_sf(oracle.sf_by_operand_row(ref["sf"], along), P, K).reshape(-1)
        _same_bytes(gs.cpu().numpy(), ref_atoms, None, f"{along} scale atoms")
        _same_bytes(gq.cpu().numpy(), ref["q"], x, f"{along} q")


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
@pytest.mark.parametrize("shape", [(512, 384), (1024, 1024)])
def test_one_call_quantize_with_nan(fp8lin, fmt, shape):
    """The one-launch dynamic cast (fp8lin_quantize, no transposed copy) on a
    tensor holding NaNs: amax, scale and inverse scale NaN exactly as the
    oracle's, every code 0x7F.  512 x 384 takes the one-cluster path of small
    tensors, 1024 x 1024 the whole-GPU grid."""
    x = _nan_matrix(*shape, 75)
    slots = torch.zeros(3, device="cuda")
    q = torch.empty(shape, dtype=torch.uint8, device="cuda")
    fp8lin.fp8lin_quantize(to_dev_bf16(x), fmt, slots[0:1], slots[1:2], slots[2:3], q, None)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    ref = oracle.quantize(x, fmt)
    _same_f32(slots[0:1].cpu().numpy(), ref["amax"], "amax")
    _same_f32(slots[1:2].cpu().numpy(), ref["scale"], "scale")
    _same_f32(slots[2:3].cpu().numpy(), ref["inv_scale"], "inv_scale")
    _same_bytes(q.cpu().numpy(), ref["q"], x, "q")

"""CPU oracle for the Float8 linear layer with dynamic per-tensor scaling.

TEST INFRASTRUCTURE ONLY.  The oracle is a plain, slow, obviously correct CPU
statement of what the hot path computes.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it;
the product package never does, and it never imports the product package.

Every function states the passage it follows.  Page titles used below:

* [TT]  "TorchTitan: a one-stop PyTorch-native solution for production LLM
  pre-training" (zenmind.me paper analysis), section 3.3 "Memory and compute
  optimisations", bullet "Mixed precision and Float8" -- Float8 is a derived
  dtype for linear layers with dynamic/delayed/static per-tensor scaling,
  composable with autograd.
* [L9]  "Lecture 9 exercises" (juanwang-buaa tutorials), the answer on fp16
  loss scaling versus FP8 scaling -- one scale factor per tensor (or per block).

Where the pages are silent the reading taken is stated on the function.  The
arithmetic lives in ``fp8_oracle.c`` (plain C, built with gcc by ``build()``);
this module only marshals numpy arrays.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against something other than itself (brute force,
exact integer arithmetic, closed forms, library routines, hand-worked cases in
``tests/golden/``).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 0
E5M2 = 1
FMT_MAX = 448.0          # numerator of the scale for all three tensors
AMAX_FLOOR = 1e-12       # amax floor before the division

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libfp8oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile fp8_oracle.c into a shared library with gcc; return its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if not force and os.path.exists(_SO) and os.path.getmtime(_SO) >= os.path.getmtime(_SRC):
        return _SO
    tmp = _SO + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared",
           "-ffp-contract=off", "-fno-fast-math", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _SO)
    return _SO


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, f32, u8p, f32p = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_void_p
        lib.orc_fp8_decode.restype = ctypes.c_double
        lib.orc_fp8_decode.argtypes = [ctypes.c_int, ctypes.c_uint8]
        lib.orc_fp8_encode.restype = ctypes.c_uint8
        lib.orc_fp8_encode.argtypes = [ctypes.c_int, f32]
        lib.orc_encode_f32.restype = None
        lib.orc_encode_f32.argtypes = [ctypes.c_void_p, i64, ctypes.c_int, u8p]
        lib.orc_amax_bf16.restype = f32
        lib.orc_amax_bf16.argtypes = [ctypes.c_void_p, i64]
        lib.orc_scale.restype = None
        lib.orc_scale.argtypes = [f32, f32, f32p, f32p]
        lib.orc_cast_bf16.restype = None
        lib.orc_cast_bf16.argtypes = [ctypes.c_void_p, i64, ctypes.c_int, f32, u8p]
        lib.orc_transpose_u8.restype = None
        lib.orc_transpose_u8.argtypes = [u8p, i64, i64, u8p]
        lib.orc_gemm_rows.restype = None
        lib.orc_gemm_rows.argtypes = [u8p, ctypes.c_int, u8p, ctypes.c_int, i64, i64, i64,
                                      f32, f32, ctypes.c_void_p, i64, ctypes.c_void_p]
        lib.orc_reciprocal.restype = f32
        lib.orc_reciprocal.argtypes = [f32]
        lib.orc_history_max.restype = f32
        lib.orc_history_max.argtypes = [ctypes.c_void_p, i64, i64]
        lib.orc_amax_rows_bf16.restype = None
        lib.orc_amax_rows_bf16.argtypes = [ctypes.c_void_p, i64, i64, ctypes.c_void_p]
        lib.orc_amax_cols_bf16.restype = None
        lib.orc_amax_cols_bf16.argtypes = [ctypes.c_void_p, i64, i64, ctypes.c_void_p]
        lib.orc_cast_rows_bf16.restype = None
        lib.orc_cast_rows_bf16.argtypes = [ctypes.c_void_p, i64, i64, ctypes.c_int, ctypes.c_void_p, u8p]
        lib.orc_gemm_rows_vec.restype = None
        lib.orc_gemm_rows_vec.argtypes = [u8p, ctypes.c_int, u8p, ctypes.c_int, i64, i64, i64,
                                          ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, i64, ctypes.c_void_p]
        lib.orc_scales.restype = None
        lib.orc_scales.argtypes = [ctypes.c_void_p, i64, f32, ctypes.c_void_p, ctypes.c_void_p]
        lib.orc_amax_blocks_bf16.restype = None
        lib.orc_amax_blocks_bf16.argtypes = [ctypes.c_void_p, i64, i64, i64, i64, ctypes.c_void_p]
        lib.orc_cast_blocks_bf16.restype = None
        lib.orc_cast_blocks_bf16.argtypes = [ctypes.c_void_p, i64, i64, i64, i64, ctypes.c_int, ctypes.c_void_p,
                                             u8p]
        lib.orc_gemm_blocks.restype = None
        lib.orc_gemm_blocks.argtypes = [u8p, ctypes.c_int, u8p, ctypes.c_int, i64, i64, i64, i64,
                                        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, i64, ctypes.c_void_p]
        lib.orc_pow2_scale_byte.restype = ctypes.c_uint8
        lib.orc_pow2_scale_byte.argtypes = [f32, f32]
        lib.orc_pow2_scale_bytes.restype = None
        lib.orc_pow2_scale_bytes.argtypes = [ctypes.c_void_p, i64, f32, ctypes.c_void_p]
        lib.orc_ocp_scale_byte.restype = ctypes.c_uint8
        lib.orc_ocp_scale_byte.argtypes = [f32, ctypes.c_int]
        lib.orc_ocp_scale_bytes.restype = None
        lib.orc_ocp_scale_bytes.argtypes = [ctypes.c_void_p, i64, ctypes.c_int, ctypes.c_void_p]
        lib.orc_num_threads.restype = ctypes.c_int
        lib.orc_num_threads.argtypes = []
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle takes C-contiguous arrays"
    return a.ctypes.data


def num_threads() -> int:
    """Host threads the oracle's parallel loops use (OpenMP)."""
    return int(_load().orc_num_threads())


# ---------------------------------------------------------------- formats

def decode_table(fmt: int) -> np.ndarray:
    """Value of each of the 256 FP8 codes (float64) from the sign/exponent/
    mantissa definition of e4m3 (fn variant) or e5m2.  The pages name only
    the "derived dtype" [TT]; the two formats are the reading stated in the
    design notes."""
    lib = _load()
    return np.array([lib.orc_fp8_decode(fmt, c) for c in range(256)], dtype=np.float64)


def encode(fmt: int, v) -> np.ndarray:
    """Saturating round-to-nearest-even of fp32 values into FP8 codes."""
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float32))
    q = np.empty(v.shape, dtype=np.uint8)
    _load().orc_encode_f32(_ptr(v), v.size, fmt, _ptr(q))
    return q


# ---------------------------------------------------------- scaling steps

def amax(x_bits: np.ndarray) -> np.float32:
    """amax = max |x| over the whole bf16 tensor: dynamic per-tensor scaling
    takes one statistic per tensor per step [TT], [L9]."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    return np.float32(_load().orc_amax_bf16(_ptr(x_bits), x_bits.size))


def scale(amax_value: float, fmt_max: float = FMT_MAX):
    """(scale, inv_scale) = (fmt_max / max(amax, 1e-12), 1 / scale) in fp32.

    The pages give one factor per tensor [L9]; fmt_max = 448 for all three
    tensors and the 1e-12 floor are the readings stated in the design notes."""
    s = ctypes.c_float()
    inv = ctypes.c_float()
    _load().orc_scale(float(np.float32(amax_value)), float(np.float32(fmt_max)),
                      ctypes.addressof(s), ctypes.addressof(inv))
    return np.float32(s.value), np.float32(inv.value)


def cast(x_bits: np.ndarray, fmt: int, scale_value: float) -> np.ndarray:
    """q = sat_RNE_fp8(fp32(x) * scale), element by element (derived dtype
    [TT]); the fp32 product is rounded once, then once more into FP8."""
    x_bits = np.ascontiguousarray(x_bits, dtype=np.uint16)
    q = np.empty(x_bits.shape, dtype=np.uint8)
    _load().orc_cast_bf16(_ptr(x_bits), x_bits.size, fmt, float(np.float32(scale_value)), _ptr(q))
    return q


def transpose(q: np.ndarray) -> np.ndarray:
    """qT[c][r] = q[r][c]: the copy whose contiguous index is the other one."""
    q = np.ascontiguousarray(q, dtype=np.uint8)
    rows, cols = q.shape
    qT = np.empty((cols, rows), dtype=np.uint8)
    _load().orc_transpose_u8(_ptr(q), rows, cols, _ptr(qT))
    return qT


def quantize(x_bits: np.ndarray, fmt: int, fmt_max: float = FMT_MAX) -> dict:
    """The whole per-tensor scaling of one bf16 matrix: amax, scale, the FP8
    copy and its transpose."""
    a = amax(x_bits)
    s, inv = scale(a, fmt_max)
    q = cast(x_bits, fmt, s)
    return {"amax": a, "scale": s, "inv_scale": inv, "q": q, "qT": transpose(q)}


def quantize_static(x_bits: np.ndarray, fmt: int, scale_value: float) -> dict:
    """Static scaling [TT]: the caller fixes the scale; the inverse scale is
    1/scale in fp32; the tensor's amax is reported alongside."""
    s = np.float32(scale_value)
    inv = np.float32(_load().orc_reciprocal(float(s)))
    q = cast(x_bits, fmt, s)
    return {"amax": amax(x_bits), "scale": s, "inv_scale": inv, "q": q, "qT": transpose(q)}


def history_max(history: np.ndarray, skip: int) -> np.float32:
    """Largest amax in the history, leaving out the slot being written."""
    h = np.ascontiguousarray(history, dtype=np.float32)
    return np.float32(_load().orc_history_max(_ptr(h), h.size, int(skip)))


def quantize_delayed(x_bits: np.ndarray, fmt: int, history: np.ndarray, slot: int,
                     fmt_max: float = FMT_MAX) -> dict:
    """Delayed scaling: the scale comes from the previous steps' statistics
    ([TT] "delayed"; [L9]: delayed scaling uses the previous step's
    statistics).  Reading taken (the pages give no history rule): a ring of
    amax values; scale = fmt_max / max(max over the ring except `slot`,
    1e-12); this tensor's amax is then stored at `slot`."""
    s, inv = scale(history_max(history, slot), fmt_max)
    q = cast(x_bits, fmt, s)
    new_hist = np.array(history, dtype=np.float32, copy=True)
    new_hist[slot] = amax(x_bits)
    return {"scale": s, "inv_scale": inv, "q": q, "qT": transpose(q), "history": new_hist}


def amax_rows(x_bits: np.ndarray) -> np.ndarray:
    """amax of every row of a bf16 matrix (row-wise scaling's statistic)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    out = np.empty(x.shape[0], dtype=np.float32)
    _load().orc_amax_rows_bf16(_ptr(x), x.shape[0], x.shape[1], _ptr(out))
    return out


def amax_cols(x_bits: np.ndarray) -> np.ndarray:
    """amax of every column of a bf16 matrix."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    out = np.empty(x.shape[1], dtype=np.float32)
    _load().orc_amax_cols_bf16(_ptr(x), x.shape[0], x.shape[1], _ptr(out))
    return out


def scales(amax_values: np.ndarray, fmt_max: float = FMT_MAX):
    """scale() applied to every entry of an amax vector."""
    pairs = [scale(a, fmt_max) for a in np.asarray(amax_values, dtype=np.float32)]
    s = np.array([p[0] for p in pairs], dtype=np.float32)
    inv = np.array([p[1] for p in pairs], dtype=np.float32)
    return s, inv


def cast_rows(x_bits: np.ndarray, fmt: int, row_scales: np.ndarray) -> np.ndarray:
    """q[r][c] = sat_RNE(fp32(x[r][c]) * scale[r])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    sc = np.ascontiguousarray(row_scales, dtype=np.float32)
    assert sc.size == x.shape[0]
    q = np.empty(x.shape, dtype=np.uint8)
    _load().orc_cast_rows_bf16(_ptr(x), x.shape[0], x.shape[1], fmt, _ptr(sc), _ptr(q))
    return q


def quantize_rowwise(x_bits: np.ndarray, fmt: int, fmt_max: float = FMT_MAX) -> dict:
    """Per-block scaling with one block per row of each GEMM operand ([L9]:
    one factor per tensor, or even per block).  Reading taken: a block must
    not vary along the GEMM's contraction (the scale then factors out of the
    sum and is applied after it), so the row-major copy q takes one scale per
    row of x and the transposed copy qT one scale per row of x^T, i.e. per
    column of x; each copy is cast from the bf16 source with its own scales."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    ar, ac = amax_rows(x), amax_cols(x)
    sr, ir = scales(ar, fmt_max)
    sc, ic = scales(ac, fmt_max)
    q = cast_rows(x, fmt, sr)
    qT = cast_rows(np.ascontiguousarray(x.T), fmt, sc)
    return {"row_amax": ar, "col_amax": ac, "row_scale": sr, "row_inv": ir, "col_scale": sc, "col_inv": ic,
            "q": q, "qT": qT}


def gemm_rows_vec(A: np.ndarray, fa: int, B: np.ndarray, fb: int, inv_a: np.ndarray, inv_b: np.ndarray,
                  rows=None) -> np.ndarray:
    """C = (dec(A) . dec(B)^T)[p][q] * inv_a[p] * inv_b[q] in float64, for the
    listed rows of C: the GEMM with row-wise (per-block) scales."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    P, R = A.shape
    Q, R2 = B.shape
    assert R == R2
    ia = np.ascontiguousarray(inv_a, dtype=np.float32)
    ib = np.ascontiguousarray(inv_b, dtype=np.float32)
    assert ia.size == P and ib.size == Q
    if rows is None:
        rows = np.arange(P, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, Q), dtype=np.float64)
    _load().orc_gemm_rows_vec(_ptr(A), fa, _ptr(B), fb, P, Q, R, _ptr(ia), _ptr(ib), _ptr(rows), rows.size,
                              _ptr(out))
    return out


# ------------------------------------------------------------ block scaling

BLOCK = 128  # contraction block of the block recipe: 1 x 128 and 128 x 128 blocks


def scales_array(amax_values: np.ndarray, fmt_max: float = FMT_MAX):
    """scale() of every entry of an amax array (any shape), in C."""
    a = np.ascontiguousarray(amax_values, dtype=np.float32)
    s = np.empty_like(a)
    inv = np.empty_like(a)
    _load().orc_scales(_ptr(a), a.size, float(np.float32(fmt_max)), _ptr(s), _ptr(inv))
    return s, inv


def amax_blocks(x_bits: np.ndarray, br: int, bc: int) -> np.ndarray:
    """amax of every br x bc block of a bf16 matrix ([ceil(rows/br) x ceil(cols/bc)];
    edge blocks are cut short)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    rows, cols = x.shape
    out = np.empty(((rows + br - 1) // br, (cols + bc - 1) // bc), dtype=np.float32)
    _load().orc_amax_blocks_bf16(_ptr(x), rows, cols, br, bc, _ptr(out))
    return out


def cast_blocks(x_bits: np.ndarray, fmt: int, br: int, bc: int, block_scales: np.ndarray) -> np.ndarray:
    """q[r][c] = sat_RNE(fp32(x[r][c]) * scale[r // br][c // bc])."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    sc = np.ascontiguousarray(block_scales, dtype=np.float32)
    rows, cols = x.shape
    assert sc.shape == ((rows + br - 1) // br, (cols + bc - 1) // bc)
    q = np.empty(x.shape, dtype=np.uint8)
    _load().orc_cast_blocks_bf16(_ptr(x), rows, cols, br, bc, fmt, _ptr(sc), _ptr(q))
    return q


def quantize_blocks(x_bits: np.ndarray, fmt: int, br: int, bc: int, fmt_max: float = FMT_MAX) -> dict:
    """Block scaling ([L9]: one factor per tensor, "or even per block"): the
    per-tensor recipe applied to every br x bc block of x on its own --
    amax of the block, scale = fmt_max / max(amax, 1e-12), saturating RNE
    cast of the block's elements.  Returns amax, scale and inv_scale as
    [blocks down x blocks across] arrays and q (row-major, like x)."""
    a = amax_blocks(x_bits, br, bc)
    s, inv = scales_array(a, fmt_max)
    return {"amax": a, "scale": s, "inv_scale": inv, "q": cast_blocks(x_bits, fmt, br, bc, s)}


def gemm_blocks(A: np.ndarray, fa: int, B: np.ndarray, fb: int, inv_a: np.ndarray, inv_b: np.ndarray,
                rb: int = BLOCK, rows=None) -> np.ndarray:
    """C[p][q] = sum_j (sum_{k in block j} dec(A[p][k]) dec(B[q][k])) * inv_a[p][j] * inv_b[q][j]
    in float64: the GEMM with block scales along the contraction (blocks of
    rb indices).  A [P x R] and B [Q x R] codes, contraction contiguous;
    inv_a [P x nb], inv_b [Q x nb] with nb = ceil(R / rb)."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    P, R = A.shape
    Q, R2 = B.shape
    assert R == R2
    nb = (R + rb - 1) // rb
    ia = np.ascontiguousarray(inv_a, dtype=np.float32)
    ib = np.ascontiguousarray(inv_b, dtype=np.float32)
    assert ia.shape == (P, nb) and ib.shape == (Q, nb)
    if rows is None:
        rows = np.arange(P, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.empty((rows.size, Q), dtype=np.float64)
    _load().orc_gemm_blocks(_ptr(A), fa, _ptr(B), fb, P, Q, R, rb, _ptr(ia), _ptr(ib), _ptr(rows), rows.size,
                            _ptr(out))
    return out


def quantize_block_recipe(x_bits, w_bits, dy_bits, fmt_max: float = FMT_MAX) -> dict:
    """The FP8 copies of one linear under block scaling, each with its blocks
    along the contraction of the GEMM that reads it (reading in the design
    notes): X in 1 x 128 blocks (forward, contraction K) and 128 x 1 blocks
    (weight gradient, contraction M); W in 128 x 128 blocks (forward and
    input gradient); dY in 1 x 128 blocks (input gradient, contraction N)
    and 128 x 1 blocks (weight gradient)."""
    return {"x_k": quantize_blocks(x_bits, E4M3, 1, BLOCK, fmt_max),
            "x_m": quantize_blocks(x_bits, E4M3, BLOCK, 1, fmt_max),
            "w": quantize_blocks(w_bits, E4M3, BLOCK, BLOCK, fmt_max),
            "dy_n": quantize_blocks(dy_bits, E5M2, 1, BLOCK, fmt_max),
            "dy_m": quantize_blocks(dy_bits, E5M2, BLOCK, 1, fmt_max)}


def _rows_of(block_inv: np.ndarray, n: int) -> np.ndarray:
    """[nbr x nb] block inverse scales of 128-row blocks -> one row per operand row ([n x nb])."""
    return np.ascontiguousarray(np.repeat(block_inv, BLOCK, axis=0)[:n])


def fwd_block_ref(xq_k, ix_k, wq, iw, rows=None):
    """Y = X . W^T with X in 1 x 128 and W in 128 x 128 blocks (contraction K)."""
    return gemm_blocks(xq_k, E4M3, wq, E4M3, ix_k, _rows_of(iw, wq.shape[0]), BLOCK, rows)


def dgrad_block_ref(dyq_n, idy_n, wq, iw, rows=None):
    """dX = dY . W with dY in 1 x 128 and W in 128 x 128 blocks (contraction N):
    B = W^T, whose row k takes the scales of W's block column k // 128."""
    wqT = np.ascontiguousarray(np.asarray(wq).T)
    return gemm_blocks(dyq_n, E5M2, wqT, E4M3, idy_n, _rows_of(np.asarray(iw).T, wqT.shape[0]), BLOCK, rows)


def wgrad_block_ref(dyq_m, idy_m, xq_m, ix_m, rows=None):
    """dW = dY^T . X with dY and X in 128 x 1 blocks (contraction M):
    A = dY^T with row n scaled by idy_m[:, n], B = X^T with row k by ix_m[:, k]."""
    dyqT = np.ascontiguousarray(np.asarray(dyq_m).T)
    xqT = np.ascontiguousarray(np.asarray(xq_m).T)
    return gemm_blocks(dyqT, E5M2, xqT, E4M3, np.ascontiguousarray(np.asarray(idy_m).T),
                       np.ascontiguousarray(np.asarray(ix_m).T), BLOCK, rows)


# ------------------------------------------- power-of-two block scaling

MX_BLOCK = 32    # contraction elements per power-of-two scale (the tensor cores' block-scaled MMA)
SF_ATOM = 512    # bytes of one scale atom: 128 operand rows x 128 contraction elements


def pow2_scale_bytes(amax_values: np.ndarray, fmt_max: float = FMT_MAX) -> np.ndarray:
    """Power-of-two block scales ([L9]: one factor per block), in C: for each
    amax the byte 127 - e with 2^e the largest power of two such that
    max(amax, 1e-12) * 2^e <= fmt_max (clamped to -127 <= e <= 127), i.e. the
    unsigned-exponent code of the inverse scale 2^-e; 0xFF for a NaN or
    infinite amax.  Same shape as the input."""
    a = np.ascontiguousarray(amax_values, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    _load().orc_pow2_scale_bytes(_ptr(a), a.size, float(np.float32(fmt_max)), _ptr(out))
    return out


def pow2_scale(sf: np.ndarray) -> np.ndarray:
    """The scale 2^e of scale byte 127 - e (float32, exact); NaN for 0xFF."""
    b = np.asarray(sf, dtype=np.int64)
    s = np.ldexp(np.float64(1.0), (127 - b).astype(np.int32)).astype(np.float32)
    return np.where(b == 0xFF, np.float32(np.nan), s).astype(np.float32)


def pow2_inverse(sf: np.ndarray) -> np.ndarray:
    """The inverse scale 2^-e of scale byte 127 - e (float32, exact)."""
    b = np.asarray(sf, dtype=np.int64)
    s = np.ldexp(np.float64(1.0), (b - 127).astype(np.int32)).astype(np.float32)
    return np.where(b == 0xFF, np.float32(np.nan), s).astype(np.float32)


def ocp_scale_bytes(amax_values: np.ndarray, fmt: int) -> np.ndarray:
    """The OCP Microscaling rule, in C: byte 127 + floor(log2 amax) - emax_elem
    (emax_elem 8 for e4m3, 15 for e5m2), i.e. the code of the shared scale
    X = 2^(floor(log2 amax) - emax_elem) by which the elements are divided;
    0 for a zero amax, 0xFF for a NaN or infinite one; clamped to 0 .. 254."""
    a = np.ascontiguousarray(amax_values, dtype=np.float32)
    out = np.empty(a.shape, dtype=np.uint8)
    _load().orc_ocp_scale_bytes(_ptr(a), a.size, int(fmt), _ptr(out))
    return out


def quantize_mx(x_bits: np.ndarray, fmt: int, along: str, fmt_max: float = FMT_MAX, rule: str = "floor") -> dict:
    """Block scaling with power-of-two scales: x cut into 1 x 32 blocks
    (along="cols": each row's runs of 32 columns) or 32 x 1 blocks
    (along="rows": each column's runs of 32 rows), blocks at the edge cut
    short; each block's amax, its scale 2^e and the saturating
    round-to-nearest-even cast of fp32(x) * 2^e (the product is exact).
    rule="floor": 2^e the largest power of two with amax * 2^e <= fmt_max
    (pow2_scale_bytes); rule="ocp": the OCP Microscaling rule
    (ocp_scale_bytes; fmt_max unused).  Returns amax and sf ([ceil(rows/32) x
    cols] or [rows x ceil(cols/32)], like the blocks), scale = 2^e and q
    (row-major, like x)."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    br, bc = (1, MX_BLOCK) if along == "cols" else (MX_BLOCK, 1)
    a = amax_blocks(x, br, bc)
    sf = pow2_scale_bytes(a, fmt_max) if rule == "floor" else ocp_scale_bytes(a, fmt)
    s = pow2_scale(sf)
    return {"amax": a, "sf": sf, "scale": s, "q": cast_blocks(x, fmt, br, bc, s)}


def sf_by_operand_row(sf: np.ndarray, along: str) -> np.ndarray:
    """Scale bytes indexed [operand row p][contraction block j] for the GEMM
    that reads the copy: a row copy (along="cols") is read with its rows as
    operand rows; a column copy (along="rows") with its columns."""
    return np.ascontiguousarray(sf if along == "cols" else np.asarray(sf).T)


def pack_sf(sf_pj: np.ndarray, P: int, K: int) -> np.ndarray:
    """Scale bytes [P x ceil(K/32)] (operand row p, 32-long contraction block
    j) laid out as the tensor cores read them: atoms of 512 bytes, one per
    128 operand rows x 128 contraction elements, atom (kb, pb) at index
    kb * ceil(P/128) + pb; inside an atom, row p and block j at byte
    16 (p % 32) + 4 ((p % 128) // 32) + j % 4.  Entries past P or past the
    last block hold 127 (scale 1).  Returns uint8 [ceil(K/128) x ceil(P/128) x 512].
    Pure data layout, no arithmetic."""
    sf_pj = np.asarray(sf_pj, dtype=np.uint8)
    nj = (K + MX_BLOCK - 1) // MX_BLOCK
    assert sf_pj.shape == (P, nj)
    npb, nkb = (P + 127) // 128, (K + 127) // 128
    out = np.full((nkb, npb, SF_ATOM), 127, dtype=np.uint8)
    p = np.arange(P)[:, None]
    j = np.arange(nj)[None, :]
    off = 16 * (p % 32) + 4 * ((p % 128) // 32) + j % 4
    out[(j // 4) + 0 * p, (p // 128) + 0 * j, off] = sf_pj
    return out


def unpack_sf(atoms: np.ndarray, P: int, K: int) -> np.ndarray:
    """Inverse of pack_sf: the [P x ceil(K/32)] scale bytes held in the atoms."""
    atoms = np.asarray(atoms, dtype=np.uint8).reshape((K + 127) // 128, (P + 127) // 128, SF_ATOM)
    nj = (K + MX_BLOCK - 1) // MX_BLOCK
    p = np.arange(P)[:, None]
    j = np.arange(nj)[None, :]
    return atoms[(j // 4) + 0 * p, (p // 128) + 0 * j, 16 * (p % 32) + 4 * ((p % 128) // 32) + j % 4]


def quantize_mx_recipe(x_bits, w_bits, dy_bits, fmt_max: float = FMT_MAX, rule: str = "floor") -> dict:
    """The FP8 copies of one linear under power-of-two block scaling, each
    with its 32-long blocks along the contraction of the GEMM that reads it:
    X in 1 x 32 (forward, contraction K) and 32 x 1 (weight gradient,
    contraction M); W in 1 x 32 (forward) and 32 x 1 (input gradient,
    contraction N); dY in 1 x 32 (input gradient) and 32 x 1 (weight
    gradient).  Each entry also carries its scales packed as pack_sf lays
    them out ("atoms") for the GEMM that reads it.  rule as for quantize_mx."""
    out = {}
    for name, bits, fmt, along in (("x_k", x_bits, E4M3, "cols"), ("x_m", x_bits, E4M3, "rows"),
                                   ("w_k", w_bits, E4M3, "cols"), ("w_n", w_bits, E4M3, "rows"),
                                   ("dy_n", dy_bits, E5M2, "cols"), ("dy_m", dy_bits, E5M2, "rows")):
        d = quantize_mx(bits, fmt, along, fmt_max, rule)
        rows, cols = np.asarray(bits).shape
        P, K = (rows, cols) if along == "cols" else (cols, rows)
        d["atoms"] = pack_sf(sf_by_operand_row(d["sf"], along), P, K)
        out[name] = d
    return out


def fwd_mx_ref(xq_k, sf_x_k, wq_k, sf_w_k, rows=None):
    """Y = X . W^T with X and W in 1 x 32 power-of-two blocks along K: the
    block GEMM with 32-long contraction blocks and inverse scales 2^-e."""
    return gemm_blocks(xq_k, E4M3, wq_k, E4M3, pow2_inverse(sf_x_k), pow2_inverse(sf_w_k), MX_BLOCK, rows)


def dgrad_mx_ref(dyq_n, sf_dy_n, wq_n, sf_w_n, rows=None):
    """dX = dY . W with dY in 1 x 32 blocks along N and W in 32 x 1 blocks
    along N: B = W^T, whose row k takes W's column-k block scales."""
    wqT = np.ascontiguousarray(np.asarray(wq_n).T)
    return gemm_blocks(dyq_n, E5M2, wqT, E4M3, pow2_inverse(sf_dy_n),
                       pow2_inverse(sf_by_operand_row(sf_w_n, "rows")), MX_BLOCK, rows)


def wgrad_mx_ref(dyq_m, sf_dy_m, xq_m, sf_x_m, rows=None):
    """dW = dY^T . X with dY and X in 32 x 1 blocks along M."""
    dyqT = np.ascontiguousarray(np.asarray(dyq_m).T)
    xqT = np.ascontiguousarray(np.asarray(xq_m).T)
    return gemm_blocks(dyqT, E5M2, xqT, E4M3, pow2_inverse(sf_by_operand_row(sf_dy_m, "rows")),
                       pow2_inverse(sf_by_operand_row(sf_x_m, "rows")), MX_BLOCK, rows)


# ------------------------------------------------------------------ GEMMs

def gemm_rows(A: np.ndarray, fa: int, B: np.ndarray, fb: int,
              inv_a: float, inv_b: float, rows=None) -> np.ndarray:
    """C = (dec(A) . dec(B)^T) * inv_a * inv_b in float64 for the listed rows
    of C (all rows when ``rows`` is None).  A is [P x R] codes and B is
    [Q x R] codes, both with the contraction index contiguous."""
    A = np.ascontiguousarray(A, dtype=np.uint8)
    B = np.ascontiguousarray(B, dtype=np.uint8)
    P, R = A.shape
    Q, R2 = B.shape
    assert R == R2, "contraction lengths differ"
    if rows is None:
        rows = np.arange(P, dtype=np.int64)
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    assert rows.size == 0 or (rows.min() >= 0 and rows.max() < P)
    out = np.empty((rows.size, Q), dtype=np.float64)
    _load().orc_gemm_rows(_ptr(A), fa, _ptr(B), fb, P, Q, R,
                          float(np.float32(inv_a)), float(np.float32(inv_b)),
                          _ptr(rows), rows.size, _ptr(out))
    return out


def fwd_ref(xq, inv_x, wq, inv_w, rows=None):
    """Y = X . W^T of the Float8 linear (forward), e4m3 x e4m3 [TT]."""
    return gemm_rows(xq, E4M3, wq, E4M3, inv_x, inv_w, rows)


def dgrad_ref(dyq, inv_dy, wqT, inv_w, rows=None):
    """dX = dY . W (input gradient through autograd [TT]), e5m2 x e4m3."""
    return gemm_rows(dyq, E5M2, wqT, E4M3, inv_dy, inv_w, rows)


def wgrad_ref(dyqT, inv_dy, xqT, inv_x, rows=None):
    """dW = dY^T . X (weight gradient through autograd [TT]), e5m2 x e4m3."""
    return gemm_rows(dyqT, E5M2, xqT, E4M3, inv_dy, inv_x, rows)


def within_tolerance(y: np.ndarray, ref: np.ndarray, rms_ref: float):
    """Elementwise GEMM bar: |y - ref| <= 2^-7 |ref| + 1e-3 rms(ref).
    Returns (ok, worst ratio of error to the allowed bound)."""
    y = np.asarray(y, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    bound = 2.0 ** -7 * np.abs(ref) + 1e-3 * rms_ref
    err = np.abs(y - ref)
    ratio = float(np.max(err / np.maximum(bound, np.finfo(np.float64).tiny))) if err.size else 0.0
    return bool(np.all(err <= bound)), ratio

"""Python binding of libfp8lin: the Float8 linear layer hot path on one GB300.

Argument marshalling only.  Every step of the path (amax, scale, cast,
transpose, the three GEMMs) runs in the library's own CUDA kernels; PyTorch
provides device memory and streams.  There is no fallback: importing this
module fails when the library has not been built.

The names mirror the C ABI in include/fp8lin.h:

    fp8lin_amax(x, amax)
    fp8lin_cast_transpose(x, fmt, amax, scale, inv_scale, q, qT, fmt_max=448.0)
    fp8lin_fwd(xq, inv_x, wq, inv_w, y)
    fp8lin_dgrad(dyq, inv_dy, wqT, inv_w, dx)
    fp8lin_wgrad(dyqT, inv_dy, xqT, inv_x, dw)

Each takes an optional ``stream`` (a torch.cuda.Stream; default: the current
stream) and raises Fp8LinError on a non-OK status.  ``Float8Linear`` below
sequences the nine calls of one linear's forward and backward pass.

Source of the method: "TorchTitan: a one-stop PyTorch-native solution for
production LLM pre-training" (zenmind.me analysis), section 3.3, bullet
"Mixed precision and Float8" (Float8 linear layers with dynamic per-tensor
scaling, composable with autograd); "Lecture 9 exercises", the answer on FP8
scaling (one factor per tensor; only what is stored in FP8 is saved).
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import _build

E4M3 = 0
E5M2 = 1
FMT_MAX = 448.0

_STATUS = {0: "FP8LIN_OK", 1: "FP8LIN_ERR_INVALID_ARG", 2: "FP8LIN_ERR_MISALIGNED",
           3: "FP8LIN_ERR_UNSUPPORTED_SHAPE", 4: "FP8LIN_ERR_CUDA", 5: "FP8LIN_ERR_TIMEOUT",
           6: "FP8LIN_ERR_UNSUPPORTED_DEVICE"}

# Every entry point declared in include/fp8lin.h.
ENTRY_POINTS = ("fp8lin_amax", "fp8lin_cast_transpose", "fp8lin_quantize", "fp8lin_quantize_batch",
                "fp8lin_cast_transpose_static",
                "fp8lin_cast_transpose_delayed", "fp8lin_amax_rowcol", "fp8lin_cast_transpose_rowwise",
                "fp8lin_fwd", "fp8lin_dgrad", "fp8lin_wgrad", "fp8lin_dgrad_mn", "fp8lin_wgrad_mn",
                "fp8lin_cast_blockwise", "fp8lin_fwd_block", "fp8lin_dgrad_block", "fp8lin_wgrad_block",
                "fp8lin_fwd_rowwise", "fp8lin_dgrad_rowwise", "fp8lin_wgrad_rowwise",
                "fp8lin_cast_mx", "fp8lin_cast_mx_ocp", "fp8lin_fwd_mx", "fp8lin_dgrad_mx", "fp8lin_wgrad_mx",
                "fp8lin_status_str", "fp8lin_device_error", "fp8lin_selftest_bounded_wait")


class Fp8LinError(RuntimeError):
    def __init__(self, call: str, status: int):
        self.status = status
        super().__init__(f"{call}: {_STATUS.get(status, status)}: {status_str(status)}")


def _load_library() -> ctypes.CDLL:
    path = _build.LIB
    if not os.path.exists(path):
        raise ImportError(f"libfp8lin is not built ({path} missing): run "
                          "`python -c 'import __graft_entry__ as g; g.build()'` first")
    lib = ctypes.CDLL(path)
    missing = set(ENTRY_POINTS) - set(SIGNATURES) - {"fp8lin_status_str"}
    if missing:
        # ctypes would pass undeclared 64-bit pointers as 32-bit ints
        raise ImportError(f"no ctypes signature for {sorted(missing)}")
    for name, args in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.fp8lin_status_str.argtypes = [ctypes.c_int]
    lib.fp8lin_status_str.restype = ctypes.c_char_p
    return lib


# Argument types of every entry point, in the order include/fp8lin.h declares
# them (pointers and cudaStream_t as c_void_p).
_vp, _i64, _f32, _ci = ctypes.c_void_p, ctypes.c_int64, ctypes.c_float, ctypes.c_int
SIGNATURES = {
    "fp8lin_amax": [_vp, _i64, _vp, _vp],
    "fp8lin_cast_transpose": [_vp, _i64, _i64, _ci, _f32, _vp, _vp, _vp, _vp, _vp, _vp],
    "fp8lin_quantize": [_vp, _i64, _i64, _ci, _f32, _vp, _vp, _vp, _vp, _vp, _vp],
    "fp8lin_quantize_batch": [_vp, _ci, _ci, _f32, _vp],
    "fp8lin_cast_transpose_static": [_vp, _i64, _i64, _ci, _vp, _vp, _vp, _vp, _vp, _vp],
    "fp8lin_cast_transpose_delayed": [_vp, _i64, _i64, _ci, _f32, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp],
    "fp8lin_amax_rowcol": [_vp, _i64, _i64, _vp, _vp, _vp],
    "fp8lin_cast_transpose_rowwise": [_vp, _i64, _i64, _ci, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "fp8lin_cast_blockwise": [_vp, _i64, _i64, _ci, _f32, _vp, _vp, _vp, _vp, _vp, _vp, _vp],
    "fp8lin_fwd_block": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_dgrad_block": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_wgrad_block": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_fwd_rowwise": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_dgrad_rowwise": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_wgrad_rowwise": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_fwd": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_dgrad": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_wgrad": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_dgrad_mn": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_wgrad_mn": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_cast_mx": [_vp, _i64, _i64, _ci, _f32, _vp, _vp, _vp, _vp, _vp],
    "fp8lin_cast_mx_ocp": [_vp, _i64, _i64, _ci, _vp, _vp, _vp, _vp, _vp],
    "fp8lin_fwd_mx": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_dgrad_mx": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_wgrad_mx": [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _vp],
    "fp8lin_device_error": [_vp, _vp],
    "fp8lin_selftest_bounded_wait": [ctypes.c_uint64, _vp],
}


_lib = _load_library()
LIBRARY_PATH = _build.LIB


def library() -> ctypes.CDLL:
    return _lib


def status_str(status: int) -> str:
    return _lib.fp8lin_status_str(int(status)).decode()


def _stream(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _ptr(t) -> int:
    return 0 if t is None else int(t.data_ptr())


def _check(call: str, status: int) -> None:
    if status != 0:
        raise Fp8LinError(call, status)


def _dev(t: torch.Tensor, name: str, dtype=None) -> None:
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")


# ------------------------------------------------------------ entry points

def fp8lin_amax(x: torch.Tensor, amax: torch.Tensor, stream=None) -> None:
    """amax[0] = max |x| over the whole bf16 tensor x."""
    _dev(x, "x", torch.bfloat16)
    _dev(amax, "amax", torch.float32)
    _check("fp8lin_amax", _lib.fp8lin_amax(_ptr(x), x.numel(), _ptr(amax), _stream(stream)))


def fp8lin_cast_transpose(x: torch.Tensor, fmt: int, amax: torch.Tensor, scale: torch.Tensor,
                          inv_scale: torch.Tensor, q: torch.Tensor | None, qT: torch.Tensor | None,
                          fmt_max: float = FMT_MAX, stream=None) -> None:
    """scale = fmt_max / amax; q = sat_RNE(x * scale) [rows x cols]; qT = q^T."""
    _dev(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be a 2-D [rows x cols] matrix")
    for t, n in ((amax, "amax"), (scale, "scale"), (inv_scale, "inv_scale")):
        _dev(t, n, torch.float32)
    _dev(q, "q")
    _dev(qT, "qT")
    rows, cols = x.shape
    _check("fp8lin_cast_transpose",
           _lib.fp8lin_cast_transpose(_ptr(x), rows, cols, int(fmt), float(fmt_max), _ptr(amax),
                                      _ptr(scale), _ptr(inv_scale), _ptr(q), _ptr(qT),
                                      _stream(stream)))


def fp8lin_quantize(x: torch.Tensor, fmt: int, amax: torch.Tensor, scale: torch.Tensor, inv_scale: torch.Tensor,
                    q: torch.Tensor | None, qT: torch.Tensor | None, fmt_max: float = FMT_MAX,
                    stream=None) -> None:
    """fp8lin_amax + fp8lin_cast_transpose in one call, for a cast with nothing beside it."""
    _dev(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be a 2-D [rows x cols] matrix")
    for t, n in ((amax, "amax"), (scale, "scale"), (inv_scale, "inv_scale")):
        _dev(t, n, torch.float32)
    _dev(q, "q")
    _dev(qT, "qT")
    rows, cols = x.shape
    _check("fp8lin_quantize",
           _lib.fp8lin_quantize(_ptr(x), rows, cols, int(fmt), float(fmt_max), _ptr(amax), _ptr(scale),
                                _ptr(inv_scale), _ptr(q), _ptr(qT), _stream(stream)))


MAX_QUANTIZE_BATCH = 4   # FP8LIN_MAX_QUANTIZE_BATCH


class _QuantizeItem(ctypes.Structure):
    """fp8lin_quantize_item of include/fp8lin.h."""
    _fields_ = [("x", ctypes.c_void_p), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64),
                ("amax", ctypes.c_void_p), ("scale", ctypes.c_void_p), ("inv_scale", ctypes.c_void_p),
                ("q", ctypes.c_void_p)]


def fp8lin_quantize_batch(items, fmt: int, fmt_max: float = FMT_MAX, stream=None) -> None:
    """fp8lin_quantize for up to MAX_QUANTIZE_BATCH tensors of one format in
    one launch; items: (x, amax, scale, inv_scale, q) per tensor, each with
    slots of its own."""
    items = list(items)
    if not 1 <= len(items) <= MAX_QUANTIZE_BATCH:
        raise ValueError(f"1 to {MAX_QUANTIZE_BATCH} tensors per call")
    arr = (_QuantizeItem * len(items))()
    for k, (x, amax, scale, inv_scale, q) in enumerate(items):
        _dev(x, "x", torch.bfloat16)
        if x.dim() != 2:
            raise ValueError("x must be a 2-D [rows x cols] matrix")
        for t, n in ((amax, "amax"), (scale, "scale"), (inv_scale, "inv_scale")):
            _dev(t, n, torch.float32)
        _dev(q, "q")
        if q is not None and tuple(q.shape) != tuple(x.shape):
            raise ValueError("q must have x's shape")
        arr[k] = _QuantizeItem(_ptr(x), x.shape[0], x.shape[1], _ptr(amax), _ptr(scale), _ptr(inv_scale), _ptr(q))
    _check("fp8lin_quantize_batch", _lib.fp8lin_quantize_batch(ctypes.addressof(arr), len(items), int(fmt),
                                                               float(fmt_max), _stream(stream)))


def fp8lin_cast_transpose_static(x: torch.Tensor, fmt: int, scale: torch.Tensor, inv_scale: torch.Tensor,
                                 q: torch.Tensor | None, qT: torch.Tensor | None,
                                 amax: torch.Tensor | None = None, stream=None) -> None:
    """Static scaling: q = sat_RNE(x * scale) with a caller-fixed scale;
    inv_scale = 1/scale; amax (optional) receives max |x|."""
    _dev(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be a 2-D [rows x cols] matrix")
    for t, n in ((scale, "scale"), (inv_scale, "inv_scale"), (amax, "amax")):
        _dev(t, n, torch.float32)
    _dev(q, "q")
    _dev(qT, "qT")
    rows, cols = x.shape
    _check("fp8lin_cast_transpose_static",
           _lib.fp8lin_cast_transpose_static(_ptr(x), rows, cols, int(fmt), _ptr(scale), _ptr(inv_scale),
                                             _ptr(q), _ptr(qT), _ptr(amax), _stream(stream)))


def fp8lin_cast_transpose_delayed(x: torch.Tensor, fmt: int, amax_history: torch.Tensor, slot: int,
                                  scale: torch.Tensor, inv_scale: torch.Tensor, q: torch.Tensor | None,
                                  qT: torch.Tensor | None, fmt_max: float = FMT_MAX, stream=None) -> None:
    """Delayed scaling: scale from the amax history (all slots but `slot`);
    the cast records max |x| into amax_history[slot]."""
    _dev(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be a 2-D [rows x cols] matrix")
    for t, n in ((amax_history, "amax_history"), (scale, "scale"), (inv_scale, "inv_scale")):
        _dev(t, n, torch.float32)
    _dev(q, "q")
    _dev(qT, "qT")
    rows, cols = x.shape
    _check("fp8lin_cast_transpose_delayed",
           _lib.fp8lin_cast_transpose_delayed(_ptr(x), rows, cols, int(fmt), float(fmt_max), _ptr(amax_history),
                                              amax_history.numel(), int(slot), _ptr(scale), _ptr(inv_scale),
                                              _ptr(q), _ptr(qT), _stream(stream)))


def fp8lin_cast_blockwise(x: torch.Tensor, fmt: int, q_row=None, inv_row=None, q_col=None, inv_col=None,
                          q_tile=None, inv_tile=None, fmt_max: float = FMT_MAX, stream=None) -> None:
    """Block scaling in one pass: q_row / inv_row (1 x 128 blocks, inv_row [ceil(cols/128) x rows]), q_col / inv_col
    (128 x 1 blocks), q_tile / inv_tile (128 x 128 blocks); any subset of the pairs."""
    _dev(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be a 2-D [rows x cols] matrix")
    for t, n in ((q_row, "q_row"), (q_col, "q_col"), (q_tile, "q_tile")):
        _dev(t, n)
    for t, n in ((inv_row, "inv_row"), (inv_col, "inv_col"), (inv_tile, "inv_tile")):
        _dev(t, n, torch.float32)
    rows, cols = x.shape
    _check("fp8lin_cast_blockwise",
           _lib.fp8lin_cast_blockwise(_ptr(x), rows, cols, int(fmt), float(fmt_max), _ptr(q_row), _ptr(inv_row),
                                      _ptr(q_col), _ptr(inv_col), _ptr(q_tile), _ptr(inv_tile), _stream(stream)))


def fp8lin_amax_rowcol(x: torch.Tensor, row_amax: torch.Tensor | None, col_amax: torch.Tensor | None,
                       stream=None) -> None:
    """row_amax[r] = max |x[r, :]|, col_amax[c] = max |x[:, c]| (either may be None)."""
    _dev(x, "x", torch.bfloat16)
    _dev(row_amax, "row_amax", torch.float32)
    _dev(col_amax, "col_amax", torch.float32)
    rows, cols = x.shape
    _check("fp8lin_amax_rowcol", _lib.fp8lin_amax_rowcol(_ptr(x), rows, cols, _ptr(row_amax), _ptr(col_amax),
                                                         _stream(stream)))


def fp8lin_cast_transpose_rowwise(x: torch.Tensor, fmt: int, row_amax, col_amax, row_inv_scale, col_inv_scale,
                                  q, qT, fmt_max: float = FMT_MAX, stream=None) -> None:
    """q with one scale per row, qT with one scale per column of x."""
    _dev(x, "x", torch.bfloat16)
    for t, n in ((row_amax, "row_amax"), (col_amax, "col_amax"), (row_inv_scale, "row_inv_scale"),
                 (col_inv_scale, "col_inv_scale")):
        _dev(t, n, torch.float32)
    _dev(q, "q")
    _dev(qT, "qT")
    rows, cols = x.shape
    _check("fp8lin_cast_transpose_rowwise",
           _lib.fp8lin_cast_transpose_rowwise(_ptr(x), rows, cols, int(fmt), float(fmt_max), _ptr(row_amax),
                                              _ptr(col_amax), _ptr(row_inv_scale), _ptr(col_inv_scale),
                                              _ptr(q), _ptr(qT), _stream(stream)))


def _gemm_call(name, a, sa, b, sb, c, M, N, K, stream):
    for t, n in ((a, "a"), (b, "b"), (sa, "inv_a"), (sb, "inv_b"), (c, "out")):
        _dev(t, n)
    _check(name, getattr(_lib, name)(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(c), M, N, K, _stream(stream)))


def _blocks(n: int) -> int:
    return (n + 127) // 128


def _block_gemm(name, a, ia, b, ib, out, M, N, K, ia_shape, ib_shape, out_shape, stream):
    for t, n in ((a, "a"), (b, "b"), (out, "out")):
        _dev(t, n)
    for t, n, shape in ((ia, "inv_a", ia_shape), (ib, "inv_b", ib_shape)):
        _dev(t, n, torch.float32)
        if tuple(t.shape) != shape:
            raise ValueError(f"{name}: {n} must be {shape}, got {tuple(t.shape)}")
    if tuple(out.shape) != out_shape or out.dtype != torch.bfloat16:
        raise ValueError(f"{name}: output must be bf16 {out_shape}")
    _check(name, getattr(_lib, name)(_ptr(a), _ptr(ia), _ptr(b), _ptr(ib), _ptr(out), M, N, K, _stream(stream)))


def fp8lin_fwd_block(xq, inv_x, wq, inv_w, y, stream=None) -> None:
    """Y = sum_j (Xq . Wq^T)_j * inv_x[j][m] * inv_w[n/128][j]: Xq in 1 x 128 and Wq in 128 x 128 blocks."""
    M, K = xq.shape
    N = wq.shape[0]
    _block_gemm("fp8lin_fwd_block", xq, inv_x, wq, inv_w, y, M, N, K, (_blocks(K), M), (_blocks(N), _blocks(K)),
                (M, N), stream)


def fp8lin_dgrad_block(dyq, inv_dy, wq, inv_w, dx, stream=None) -> None:
    """dX = sum_j (dYq . Wq)_j * inv_dy[j][m] * inv_w[j][k/128]: dYq in 1 x 128 and Wq in 128 x 128 blocks."""
    M, N = dyq.shape
    K = wq.shape[1]
    _block_gemm("fp8lin_dgrad_block", dyq, inv_dy, wq, inv_w, dx, M, N, K, (_blocks(N), M),
                (_blocks(N), _blocks(K)), (M, K), stream)


def fp8lin_wgrad_block(dyq, inv_dy, xq, inv_x, dw, stream=None) -> None:
    """dW = sum_j (dYq^T . Xq)_j * inv_dy[j][n] * inv_x[j][k]: dYq and Xq in 128 x 1 blocks."""
    M, N = dyq.shape
    K = xq.shape[1]
    _block_gemm("fp8lin_wgrad_block", dyq, inv_dy, xq, inv_x, dw, M, N, K, (_blocks(M), N), (_blocks(M), K),
                (N, K), stream)


def sf_atom_bytes(P: int, K: int) -> int:
    """Bytes of the power-of-two scale atoms of a copy read with P operand rows
    and a contraction of K: ceil(P/128) * ceil(K/128) * 512."""
    return _blocks(P) * _blocks(K) * 512


def fp8lin_cast_mx(x: torch.Tensor, fmt: int, q_row=None, sf_row=None, q_col=None, sf_col=None,
                   fmt_max: float = FMT_MAX, stream=None, rule: str = "floor") -> None:
    """Power-of-two block scaling in one pass: q_row / sf_row (1 x 32 blocks; sf_row holds
    sf_atom_bytes(rows, cols) bytes), q_col / sf_col (32 x 1 blocks; sf_atom_bytes(cols, rows)).
    rule="floor": the largest power of two not above fmt_max / amax (fp8lin_cast_mx);
    rule="ocp": the OCP Microscaling rule (fp8lin_cast_mx_ocp; fmt_max unused)."""
    if rule not in ("floor", "ocp"):
        raise ValueError(f"unknown rule {rule!r}")
    _dev(x, "x", torch.bfloat16)
    if x.dim() != 2:
        raise ValueError("x must be a 2-D [rows x cols] matrix")
    rows, cols = x.shape
    for q, sf, n, nbytes in ((q_row, sf_row, "row", sf_atom_bytes(rows, cols)),
                             (q_col, sf_col, "col", sf_atom_bytes(cols, rows))):
        _dev(q, "q_" + n, torch.uint8)
        _dev(sf, "sf_" + n, torch.uint8)
        if q is not None and tuple(q.shape) != (rows, cols):
            raise ValueError(f"q_{n} must be [{rows} x {cols}]")
        if sf is not None and sf.numel() != nbytes:
            raise ValueError(f"sf_{n} must hold {nbytes} bytes, got {sf.numel()}")
    if rule == "ocp":
        _check("fp8lin_cast_mx_ocp", _lib.fp8lin_cast_mx_ocp(_ptr(x), rows, cols, int(fmt), _ptr(q_row), _ptr(sf_row),
                                                             _ptr(q_col), _ptr(sf_col), _stream(stream)))
        return
    _check("fp8lin_cast_mx", _lib.fp8lin_cast_mx(_ptr(x), rows, cols, int(fmt), float(fmt_max), _ptr(q_row),
                                                 _ptr(sf_row), _ptr(q_col), _ptr(sf_col), _stream(stream)))


def _mx_gemm(name, a, sa, b, sb, out, M, N, K, sa_bytes, sb_bytes, out_shape, stream):
    for t, n in ((a, "a"), (b, "b"), (sa, "sf_a"), (sb, "sf_b"), (out, "out")):
        _dev(t, n)
    for t, n, nbytes in ((sa, "sf_a", sa_bytes), (sb, "sf_b", sb_bytes)):
        if t.numel() * t.element_size() != nbytes:
            raise ValueError(f"{name}: {n} must hold {nbytes} bytes")
    if tuple(out.shape) != out_shape or out.dtype != torch.bfloat16:
        raise ValueError(f"{name}: output must be bf16 {out_shape}")
    _check(name, getattr(_lib, name)(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), _ptr(out), M, N, K, _stream(stream)))


def fp8lin_fwd_mx(xq, sf_x, wq, sf_w, y, stream=None) -> None:
    """Y = X . W^T on the row copies of X [M x K] and W [N x K] (fp8lin_cast_mx)."""
    M, K = xq.shape
    N = wq.shape[0]
    _mx_gemm("fp8lin_fwd_mx", xq, sf_x, wq, sf_w, y, M, N, K, sf_atom_bytes(M, K), sf_atom_bytes(N, K), (M, N),
             stream)


def fp8lin_dgrad_mx(dyq, sf_dy, wq, sf_w, dx, stream=None) -> None:
    """dX = dY . W on the row copy of dY [M x N] and the column copy of W [N x K]."""
    M, N = dyq.shape
    K = wq.shape[1]
    _mx_gemm("fp8lin_dgrad_mx", dyq, sf_dy, wq, sf_w, dx, M, N, K, sf_atom_bytes(M, N), sf_atom_bytes(K, N),
             (M, K), stream)


def fp8lin_wgrad_mx(dyq, sf_dy, xq, sf_x, dw, stream=None) -> None:
    """dW = dY^T . X on the column copies of dY [M x N] and X [M x K]."""
    M, N = dyq.shape
    K = xq.shape[1]
    _mx_gemm("fp8lin_wgrad_mx", dyq, sf_dy, xq, sf_x, dw, M, N, K, sf_atom_bytes(N, M), sf_atom_bytes(K, M),
             (N, K), stream)


def fp8lin_fwd_rowwise(xq, inv_x_rows, wq, inv_w_rows, y, stream=None) -> None:
    """Y = bf16((Xq . Wq^T)[m, n] * inv_x_rows[m] * inv_w_rows[n])."""
    M, K = xq.shape
    _gemm_call("fp8lin_fwd_rowwise", xq, inv_x_rows, wq, inv_w_rows, y, M, wq.shape[0], K, stream)


def fp8lin_dgrad_rowwise(dyq, inv_dy_rows, wqT, inv_w_cols, dx, stream=None) -> None:
    """dX = bf16((dYq . WqT^T)[m, k] * inv_dy_rows[m] * inv_w_cols[k])."""
    M, N = dyq.shape
    _gemm_call("fp8lin_dgrad_rowwise", dyq, inv_dy_rows, wqT, inv_w_cols, dx, M, N, wqT.shape[0], stream)


def fp8lin_wgrad_rowwise(dyqT, inv_dy_cols, xqT, inv_x_cols, dw, stream=None) -> None:
    """dW = bf16((dYqT . XqT^T)[n, k] * inv_dy_cols[n] * inv_x_cols[k])."""
    N, M = dyqT.shape
    _gemm_call("fp8lin_wgrad_rowwise", dyqT, inv_dy_cols, xqT, inv_x_cols, dw, M, N, xqT.shape[0], stream)


def fp8lin_fwd(xq, inv_x, wq, inv_w, y, stream=None) -> None:
    """Y [M x N] = bf16((Xq . Wq^T) * inv_x * inv_w); Xq [M x K], Wq [N x K]."""
    M, K = xq.shape
    N = wq.shape[0]
    for t, n in ((xq, "xq"), (wq, "wq"), (inv_x, "inv_x"), (inv_w, "inv_w"), (y, "y")):
        _dev(t, n)
    if wq.shape[1] != K or tuple(y.shape) != (M, N) or y.dtype != torch.bfloat16:
        raise ValueError("shape/dtype mismatch: xq [M,K], wq [N,K], y bf16 [M,N]")
    _check("fp8lin_fwd", _lib.fp8lin_fwd(_ptr(xq), _ptr(inv_x), _ptr(wq), _ptr(inv_w), _ptr(y),
                                         M, N, K, _stream(stream)))


def fp8lin_dgrad(dyq, inv_dy, wqT, inv_w, dx, stream=None) -> None:
    """dX [M x K] = bf16((dYq . WqT^T) * inv_dy * inv_w); dYq [M x N], WqT [K x N]."""
    M, N = dyq.shape
    K = wqT.shape[0]
    for t, n in ((dyq, "dyq"), (wqT, "wqT"), (inv_dy, "inv_dy"), (inv_w, "inv_w"), (dx, "dx")):
        _dev(t, n)
    if wqT.shape[1] != N or tuple(dx.shape) != (M, K) or dx.dtype != torch.bfloat16:
        raise ValueError("shape/dtype mismatch: dyq [M,N], wqT [K,N], dx bf16 [M,K]")
    _check("fp8lin_dgrad", _lib.fp8lin_dgrad(_ptr(dyq), _ptr(inv_dy), _ptr(wqT), _ptr(inv_w),
                                             _ptr(dx), M, N, K, _stream(stream)))


def fp8lin_dgrad_mn(dyq, inv_dy, wq, inv_w, dx, stream=None) -> None:
    """dX [M x K] = bf16((dYq . Wq) * inv_dy * inv_w); dYq [M x N], Wq [N x K] as cast (no transposed copy)."""
    M, N = dyq.shape
    K = wq.shape[1]
    for t, n in ((dyq, "dyq"), (wq, "wq"), (inv_dy, "inv_dy"), (inv_w, "inv_w"), (dx, "dx")):
        _dev(t, n)
    if wq.shape[0] != N or tuple(dx.shape) != (M, K) or dx.dtype != torch.bfloat16:
        raise ValueError("shape/dtype mismatch: dyq [M,N], wq [N,K], dx bf16 [M,K]")
    _check("fp8lin_dgrad_mn", _lib.fp8lin_dgrad_mn(_ptr(dyq), _ptr(inv_dy), _ptr(wq), _ptr(inv_w),
                                                   _ptr(dx), M, N, K, _stream(stream)))


def fp8lin_wgrad_mn(dyq, inv_dy, xq, inv_x, dw, stream=None) -> None:
    """dW [N x K] = bf16((dYq^T . Xq) * inv_dy * inv_x); dYq [M x N], Xq [M x K] as cast (no transposed copy)."""
    M, N = dyq.shape
    K = xq.shape[1]
    for t, n in ((dyq, "dyq"), (xq, "xq"), (inv_dy, "inv_dy"), (inv_x, "inv_x"), (dw, "dw")):
        _dev(t, n)
    if xq.shape[0] != M or tuple(dw.shape) != (N, K) or dw.dtype != torch.bfloat16:
        raise ValueError("shape/dtype mismatch: dyq [M,N], xq [M,K], dw bf16 [N,K]")
    _check("fp8lin_wgrad_mn", _lib.fp8lin_wgrad_mn(_ptr(dyq), _ptr(inv_dy), _ptr(xq), _ptr(inv_x),
                                                   _ptr(dw), M, N, K, _stream(stream)))


def fp8lin_wgrad(dyqT, inv_dy, xqT, inv_x, dw, stream=None) -> None:
    """dW [N x K] = bf16((dYqT . XqT^T) * inv_dy * inv_x); dYqT [N x M], XqT [K x M]."""
    N, M = dyqT.shape
    K = xqT.shape[0]
    for t, n in ((dyqT, "dyqT"), (xqT, "xqT"), (inv_dy, "inv_dy"), (inv_x, "inv_x"), (dw, "dw")):
        _dev(t, n)
    if xqT.shape[1] != M or tuple(dw.shape) != (N, K) or dw.dtype != torch.bfloat16:
        raise ValueError("shape/dtype mismatch: dyqT [N,M], xqT [K,M], dw bf16 [N,K]")
    _check("fp8lin_wgrad", _lib.fp8lin_wgrad(_ptr(dyqT), _ptr(inv_dy), _ptr(xqT), _ptr(inv_x),
                                             _ptr(dw), M, N, K, _stream(stream)))


def fp8lin_device_error(stream=None) -> int:
    """Raw device error word since the last call (0 = none); synchronises."""
    word = ctypes.c_uint32(0)
    st = _lib.fp8lin_device_error(_stream(stream), ctypes.addressof(word))
    if st not in (0, 5):
        _check("fp8lin_device_error", st)
    return int(word.value)


def fp8lin_selftest_bounded_wait(limit_ns: int, stream=None) -> None:
    """Launch a wait that runs out after limit_ns (see include/fp8lin.h)."""
    _check("fp8lin_selftest_bounded_wait", _lib.fp8lin_selftest_bounded_wait(int(limit_ns), _stream(stream)))


# ----------------------------------------------------------- one linear

class Float8Tensor:
    """Per-tensor FP8 state of one bf16 matrix: the scale, its inverse and
    the FP8 copies (device buffers, caller-visible): q [rows x cols] and,
    with ``transpose`` (always for row-wise scaling), qT [cols x rows].

    scaling = "dynamic": amax of this tensor, then scale + cast (default);
              "delayed": scale from an amax history ring (``history_len``
                         slots), this tensor's amax recorded by the cast; the
                         first call seeds the ring with one amax pass;
              "static":  a fixed scale set with ``set_scale``;
              "rowwise": one scale per row of q and per row of qT (per
                         column of the source): per-block scaling with
                         blocks that do not cross the GEMM contraction;
              "block":   blocks of 128 along the contraction, one pass with
                         no amax call: ``blocks="rowcol"`` (activations,
                         gradients) gives q in 1 x 128 blocks (row_inv
                         [ceil(cols/128) x rows]) and qc in 128 x 1 blocks
                         (col_inv [ceil(rows/128) x cols]); ``blocks="tile"``
                         (weights) gives q in 128 x 128 blocks (tile_inv);
              "mx":      power-of-two scales in blocks of 32 along the
                         contraction, applied by the tensor cores, one pass
                         with no amax call: q in 1 x 32 blocks (scale atoms
                         sf_row) and qc in 32 x 1 blocks (sf_col); mx_rule
                         "floor" (the largest power of two not above
                         fmt_max / amax) or "ocp" (the OCP Microscaling rule)."""

    def __init__(self, rows: int, cols: int, fmt: int, device, fmt_max: float = FMT_MAX,
                 scaling: str = "dynamic", history_len: int = 16, transpose: bool = True, blocks: str = "rowcol",
                 mx_rule: str = "floor"):
        if scaling not in ("dynamic", "delayed", "static", "rowwise", "block", "mx"):
            raise ValueError(f"unknown scaling {scaling!r}")
        if scaling == "mx":
            if mx_rule not in ("floor", "ocp"):
                raise ValueError(f"unknown mx_rule {mx_rule!r}")
            self.rows, self.cols, self.fmt, self.fmt_max, self.scaling = rows, cols, fmt, fmt_max, scaling
            self.mx_rule = mx_rule
            self.q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
            self.qc = torch.empty((rows, cols), dtype=torch.uint8, device=device)
            self.qT = None
            self.sf_row = torch.empty(sf_atom_bytes(rows, cols), dtype=torch.uint8, device=device)
            self.sf_col = torch.empty(sf_atom_bytes(cols, rows), dtype=torch.uint8, device=device)
            return
        if scaling == "block":
            if blocks not in ("rowcol", "tile"):
                raise ValueError(f"unknown blocks {blocks!r}")
            self.rows, self.cols, self.fmt, self.fmt_max, self.scaling, self.blocks = (rows, cols, fmt, fmt_max,
                                                                                      scaling, blocks)
            nr, nc = (rows + 127) // 128, (cols + 127) // 128
            self.q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
            self.qT = None
            if blocks == "rowcol":
                self.row_inv = torch.zeros((nc, rows), dtype=torch.float32, device=device)   # block-major
                self.qc = torch.empty((rows, cols), dtype=torch.uint8, device=device)
                self.col_inv = torch.zeros((nr, cols), dtype=torch.float32, device=device)
            else:
                self.tile_inv = torch.zeros((nr, nc), dtype=torch.float32, device=device)
            return
        if scaling == "rowwise" and not transpose:
            raise ValueError("row-wise scaling needs the transposed copy (its scales run along columns)")
        self.rows, self.cols, self.fmt, self.fmt_max = rows, cols, fmt, fmt_max
        self.scaling = scaling
        scalars = torch.zeros(3, dtype=torch.float32, device=device)
        self.amax, self.scale, self.inv_scale = scalars[0:1], scalars[1:2], scalars[2:3]
        self.q = torch.empty((rows, cols), dtype=torch.uint8, device=device)
        self.qT = torch.empty((cols, rows), dtype=torch.uint8, device=device) if transpose else None
        if scaling == "rowwise":
            self.row_amax = torch.zeros(rows, dtype=torch.float32, device=device)
            self.col_amax = torch.zeros(cols, dtype=torch.float32, device=device)
            self.row_inv = torch.zeros(rows, dtype=torch.float32, device=device)
            self.col_inv = torch.zeros(cols, dtype=torch.float32, device=device)
        if scaling == "delayed":
            self.history = torch.zeros(history_len, dtype=torch.float32, device=device)
            self.slot = 0
            self.seeded = False

    def set_scale(self, value: float) -> "Float8Tensor":
        """The fixed scale of static scaling."""
        self.scale.fill_(float(value))
        return self

    def quantize(self, x: torch.Tensor, stream=None, alone: bool = False) -> "Float8Tensor":
        """Scale, cast and transpose x according to this tensor's scaling.
        alone: nothing runs beside this cast (dynamic scaling then takes the
        one-call fp8lin_quantize, tuned for running alone)."""
        if self.scaling == "mx":
            fp8lin_cast_mx(x, self.fmt, q_row=self.q, sf_row=self.sf_row, q_col=self.qc, sf_col=self.sf_col,
                           fmt_max=self.fmt_max, stream=stream, rule=self.mx_rule)
        elif self.scaling == "block":
            if self.blocks == "rowcol":
                fp8lin_cast_blockwise(x, self.fmt, q_row=self.q, inv_row=self.row_inv, q_col=self.qc,
                                      inv_col=self.col_inv, fmt_max=self.fmt_max, stream=stream)
            else:
                fp8lin_cast_blockwise(x, self.fmt, q_tile=self.q, inv_tile=self.tile_inv, fmt_max=self.fmt_max,
                                      stream=stream)
        elif self.scaling == "dynamic" and alone:
            fp8lin_quantize(x, self.fmt, self.amax, self.scale, self.inv_scale, self.q, self.qT, self.fmt_max, stream)
        elif self.scaling == "dynamic":
            fp8lin_amax(x, self.amax, stream)
            fp8lin_cast_transpose(x, self.fmt, self.amax, self.scale, self.inv_scale, self.q, self.qT,
                                  self.fmt_max, stream)
        elif self.scaling == "rowwise":
            fp8lin_amax_rowcol(x, self.row_amax, self.col_amax, stream)
            fp8lin_cast_transpose_rowwise(x, self.fmt, self.row_amax, self.col_amax, self.row_inv, self.col_inv,
                                          self.q, self.qT, self.fmt_max, stream)
        elif self.scaling == "static":
            fp8lin_cast_transpose_static(x, self.fmt, self.scale, self.inv_scale, self.q, self.qT,
                                         self.amax, stream)
        else:
            n = self.history.numel()
            if not self.seeded:
                fp8lin_amax(x, self.history[(self.slot - 1) % n:(self.slot - 1) % n + 1], stream)
                self.seeded = True
            fp8lin_cast_transpose_delayed(x, self.fmt, self.history, self.slot, self.scale, self.inv_scale,
                                          self.q, self.qT, self.fmt_max, stream)
            self.slot = (self.slot + 1) % n
        return self


def quantize_alone(pairs, stream=None) -> None:
    """Cast each (Float8Tensor, x) of `pairs` with nothing running beside the
    casts.  The dynamic casts without a transposed copy, grouped by format,
    share one fp8lin_quantize_batch launch; every other cast runs on its own."""
    groups = {}
    for t8, x in pairs:
        if t8.scaling == "dynamic" and t8.qT is None:
            groups.setdefault((t8.fmt, t8.fmt_max), []).append((t8, x))
        else:
            t8.quantize(x, stream, alone=True)
    for (fmt, fmt_max), members in groups.items():
        for i in range(0, len(members), MAX_QUANTIZE_BATCH):
            chunk = members[i:i + MAX_QUANTIZE_BATCH]
            fp8lin_quantize_batch([(x, t8.amax, t8.scale, t8.inv_scale, t8.q) for t8, x in chunk], fmt, fmt_max,
                                  stream)


class Float8Linear:
    """The nine calls of one Float8 linear's forward and backward pass, on
    caller-owned bf16 X [M x K], W [N x K], dY [M x N].  Buffers for the FP8
    copies and the outputs are allocated once and reused every step; the FP8
    copies of X and W made in forward are what backward reads.

    transpose = False (default for per-tensor scaling): one FP8 copy per
    tensor, and the backward GEMMs read Wq, dYq and Xq MN-major
    (fp8lin_dgrad_mn / fp8lin_wgrad_mn).  transpose = True: the casts also
    write the transposed copies and the backward GEMMs read those (always so
    for row-wise scaling)."""

    def __init__(self, M: int, K: int, N: int, device="cuda", fmt_max: float = FMT_MAX,
                 scaling: str = "dynamic", history_len: int = 16, transpose: bool | None = None,
                 mx_rule: str = "floor"):
        self.M, self.K, self.N = M, K, N
        self.transpose = (scaling == "rowwise") if transpose is None else bool(transpose)
        if scaling in ("block", "mx") and self.transpose:
            raise ValueError("block scaling writes no transposed copies")
        args = (device, fmt_max, scaling, history_len, self.transpose)
        self.x8 = Float8Tensor(M, K, E4M3, *args, blocks="rowcol", mx_rule=mx_rule)
        self.w8 = Float8Tensor(N, K, E4M3, *args, blocks="tile", mx_rule=mx_rule)
        self.dy8 = Float8Tensor(M, N, E5M2, *args, blocks="rowcol", mx_rule=mx_rule)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=device)
        self.dw = torch.empty((N, K), dtype=torch.bfloat16, device=device)

    @property
    def flops(self) -> int:
        return 6 * self.M * self.N * self.K

    def forward(self, x: torch.Tensor, w: torch.Tensor, stream=None) -> torch.Tensor:
        # the step runs on one stream: nothing runs beside the casts, and
        # X's and W's share one launch where they can
        quantize_alone([(self.x8, x), (self.w8, w)], stream)
        if self.x8.scaling == "mx":
            fp8lin_fwd_mx(self.x8.q, self.x8.sf_row, self.w8.q, self.w8.sf_row, self.y, stream)
        elif self.x8.scaling == "block":
            fp8lin_fwd_block(self.x8.q, self.x8.row_inv, self.w8.q, self.w8.tile_inv, self.y, stream)
        elif self.x8.scaling == "rowwise":
            fp8lin_fwd_rowwise(self.x8.q, self.x8.row_inv, self.w8.q, self.w8.row_inv, self.y, stream)
        else:
            fp8lin_fwd(self.x8.q, self.x8.inv_scale, self.w8.q, self.w8.inv_scale, self.y, stream)
        return self.y

    def backward(self, dy: torch.Tensor, stream=None):
        self.dy8.quantize(dy, stream, alone=True)
        if self.dy8.scaling == "mx":
            fp8lin_dgrad_mx(self.dy8.q, self.dy8.sf_row, self.w8.qc, self.w8.sf_col, self.dx, stream)
            fp8lin_wgrad_mx(self.dy8.qc, self.dy8.sf_col, self.x8.qc, self.x8.sf_col, self.dw, stream)
        elif self.dy8.scaling == "block":
            fp8lin_dgrad_block(self.dy8.q, self.dy8.row_inv, self.w8.q, self.w8.tile_inv, self.dx, stream)
            fp8lin_wgrad_block(self.dy8.qc, self.dy8.col_inv, self.x8.qc, self.x8.col_inv, self.dw, stream)
        elif self.dy8.scaling == "rowwise":
            fp8lin_dgrad_rowwise(self.dy8.q, self.dy8.row_inv, self.w8.qT, self.w8.col_inv, self.dx, stream)
            fp8lin_wgrad_rowwise(self.dy8.qT, self.dy8.col_inv, self.x8.qT, self.x8.col_inv, self.dw, stream)
        elif self.transpose:
            fp8lin_dgrad(self.dy8.q, self.dy8.inv_scale, self.w8.qT, self.w8.inv_scale, self.dx, stream)
            fp8lin_wgrad(self.dy8.qT, self.dy8.inv_scale, self.x8.qT, self.x8.inv_scale, self.dw, stream)
        else:
            fp8lin_dgrad_mn(self.dy8.q, self.dy8.inv_scale, self.w8.q, self.w8.inv_scale, self.dx, stream)
            fp8lin_wgrad_mn(self.dy8.q, self.dy8.inv_scale, self.x8.q, self.x8.inv_scale, self.dw, stream)
        return self.dx, self.dw

    def step(self, x, w, dy, stream=None):
        self.forward(x, w, stream)
        self.backward(dy, stream)
        return self.y, self.dx, self.dw

    # kernels one dynamic step launches at most (amax x3, cast x3, three GEMMs;
    # fewer where casts take the one-launch path: X and W together, then dY)
    KERNELS_PER_STEP = 9


# the autograd / nn.Module front end (imports the names above)
from .nn import Float8LinearFunction, Float8LinearModule, swap_linear_layers  # noqa: E402

"""The C ABI on the host: the library loads without a GPU, exports every
entry point include/fp8lin.h declares, and rejects bad arguments before
touching CUDA (no GPU needed: argument checks run first)."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

HEADER = os.path.join(ROOT, "include", "fp8lin.h")


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    path = __graft_entry__._build_module().build()
    return ctypes.CDLL(path)


def declared_entry_points():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8lin_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_five_calls():
    names = declared_entry_points()
    for n in ("fp8lin_amax", "fp8lin_cast_transpose", "fp8lin_fwd", "fp8lin_dgrad", "fp8lin_wgrad"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_entry_points():
        assert hasattr(lib, name), f"{name} declared in fp8lin.h but not exported"


def test_binding_lists_every_declared_symbol(lib):
    import float8_linear_layers_gb300 as fl
    assert sorted(fl.ENTRY_POINTS) == declared_entry_points()


def declared_parameter_types():
    """name -> list of C parameter types, from the header's prototypes."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(fp8lin_[a-z_0-9]+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        types = []
        for p in params.split(","):
            p = " ".join(p.split())
            if p in ("", "void"):
                continue
            types.append(p.rsplit(" ", 1)[0] if "*" not in p else "pointer")
        out[name] = types
    return out


def test_binding_signatures_match_the_header(lib):
    """Every argument type the binding declares is the header's: an
    undeclared or narrowed pointer would reach the kernels truncated."""
    import float8_linear_layers_gb300 as fl
    ctype_of = {"pointer": ctypes.c_void_p, "cudaStream_t": ctypes.c_void_p, "int64_t": ctypes.c_int64,
                "uint64_t": ctypes.c_uint64, "float": ctypes.c_float, "fp8lin_fmt": ctypes.c_int,
                "fp8lin_status": ctypes.c_int, "int": ctypes.c_int}
    decl = declared_parameter_types()
    assert set(decl) == set(fl.ENTRY_POINTS)
    for name, types in decl.items():
        if name == "fp8lin_status_str":
            continue
        want = [ctype_of[t.replace("const ", "")] for t in types]
        assert fl.SIGNATURES[name] == want, f"{name}: binding {fl.SIGNATURES[name]} vs header {types}"


def test_status_strings(lib):
    lib.fp8lin_status_str.restype = ctypes.c_char_p
    for s in range(7):
        assert lib.fp8lin_status_str(s)
    assert b"unknown" in lib.fp8lin_status_str(99)


def _c(lib, name, *args):
    fn = getattr(lib, name)
    fn.restype = ctypes.c_int
    return fn(*args)


V = ctypes.c_void_p
I = ctypes.c_int64
F = ctypes.c_float


def test_argument_checks_without_gpu(lib):
    a16 = V(4096)      # 16-byte-aligned fake addresses: never dereferenced on these paths
    a4 = V(4100)
    # amax: null out / negative n / misaligned input
    assert _c(lib, "fp8lin_amax", a16, I(16), V(0), V(0)) == 1
    assert _c(lib, "fp8lin_amax", a16, I(-1), a16, V(0)) == 1
    assert _c(lib, "fp8lin_amax", V(4098), I(16), a16, V(0)) == 2
    assert _c(lib, "fp8lin_amax", a16, I(16), V(4098), V(0)) == 2
    # cast: bad format, bad fmt_max, shape not a multiple of 16, misaligned
    ct = lib.fp8lin_cast_transpose
    ct.restype = ctypes.c_int
    ct.argtypes = [V, I, I, ctypes.c_int, F, V, V, V, V, V, V]
    assert ct(a16, 32, 32, 2, 448.0, a16, a16, a16, a16, a16, None) == 1
    assert ct(a16, 32, 32, 0, 0.0, a16, a16, a16, a16, a16, None) == 1
    assert ct(a16, 32, 32, 0, float("nan"), a16, a16, a16, a16, a16, None) == 1
    assert ct(a16, 32, 24, 0, 448.0, a16, a16, a16, a16, a16, None) == 3
    assert ct(a16, 1 << 31, 32, 0, 448.0, a16, a16, a16, a16, a16, None) == 3
    assert ct(a16, 32, 32, 0, 448.0, a16, a16, a16, a4, a16, None) == 2
    assert ct(a16, 32, 32, 0, 448.0, None, a16, a16, a16, a16, None) == 1
    # GEMMs: null scales, misaligned operand, ragged dims
    for name in ("fp8lin_fwd", "fp8lin_dgrad", "fp8lin_wgrad"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [V, V, V, V, V, I, I, I, V]
        assert fn(a16, None, a16, a16, a16, 128, 128, 128, None) == 1
        assert fn(a16, a16, a16, a16, a16, -16, 128, 128, None) == 1
        assert fn(a4, a16, a16, a16, a16, 128, 128, 128, None) == 2
        assert fn(a16, a16, a16, a16, a16, 128, 120, 128, None) == 3
        assert fn(a16, a16, a16, a16, a16, 128, 128, 8, None) == 3


def test_argument_checks_of_mn_and_block_entry_points(lib):
    a16 = V(4096)      # 16-byte-aligned fake addresses: never dereferenced on these paths
    a4 = V(4100)
    # GEMMs on the row-major copies and the block-scaled GEMMs: same checks as fp8lin_fwd
    for name in ("fp8lin_dgrad_mn", "fp8lin_wgrad_mn", "fp8lin_fwd_block", "fp8lin_dgrad_block",
                 "fp8lin_wgrad_block"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [V, V, V, V, V, I, I, I, V]
        assert fn(a16, None, a16, a16, a16, 128, 128, 128, None) == 1, name
        assert fn(a16, a16, a16, a16, a16, 128, -16, 128, None) == 1, name
        assert fn(a16, a16, a4, a16, a16, 128, 128, 128, None) == 2, name
        assert fn(a16, a16, a16, a16, a4, 128, 128, 128, None) == 2, name
        assert fn(a16, a16, a16, a16, a16, 136, 128, 128, None) == 3, name
    # the block GEMMs read the row (and column) block scales four at a time
    for name in ("fp8lin_fwd_block", "fp8lin_dgrad_block", "fp8lin_wgrad_block"):
        assert getattr(lib, name)(a16, V(4100), a16, a16, a16, 128, 128, 128, None) == 2, name
    assert lib.fp8lin_fwd_block(a16, a16, a16, V(4100), a16, 128, 128, 128, None) != 2   # inv_w: 4 bytes
    fn = lib.fp8lin_wgrad_block
    assert fn(a16, a16, a16, V(4100), a16, 128, 128, 128, None) == 2
    # block cast: each copy with its scales, at least one copy, formats, alignment, shapes
    cb = lib.fp8lin_cast_blockwise
    cb.restype = ctypes.c_int
    cb.argtypes = [V, I, I, ctypes.c_int, F, V, V, V, V, V, V, V]
    assert cb(a16, 32, 32, 0, 448.0, a16, None, None, None, None, None, None) == 1   # q without scales
    assert cb(a16, 32, 32, 0, 448.0, None, a16, None, None, None, None, None) == 1   # scales without q
    assert cb(a16, 32, 32, 0, 448.0, None, None, None, None, None, None, None) == 1  # nothing asked for
    assert cb(a16, 32, 32, 3, 448.0, a16, a16, None, None, None, None, None) == 1    # format
    assert cb(a16, 32, 32, 0, -1.0, a16, a16, None, None, None, None, None) == 1     # fmt_max
    assert cb(a16, 32, 32, 0, 448.0, a4, a16, None, None, None, None, None) == 2     # misaligned copy
    assert cb(a16, 32, 32, 0, 448.0, a16, V(4098), None, None, None, None, None) == 2  # misaligned scales
    assert cb(a16, 32, 40, 0, 448.0, a16, a16, None, None, None, None, None) == 3    # ragged shape


def test_argument_checks_of_power_of_two_block_entry_points(lib):
    a16 = V(4096)      # 16-byte-aligned fake addresses: never dereferenced on these paths
    a8 = V(4104)
    for name in ("fp8lin_fwd_mx", "fp8lin_dgrad_mx", "fp8lin_wgrad_mx"):
        fn = getattr(lib, name)
        fn.restype = ctypes.c_int
        fn.argtypes = [V, V, V, V, V, I, I, I, V]
        assert fn(a16, None, a16, a16, a16, 128, 128, 128, None) == 1, name     # no scales for A
        assert fn(a16, a16, a16, None, a16, 128, 128, 128, None) == 1, name     # no scales for B
        assert fn(a16, a16, a16, a16, a16, 128, -16, 128, None) == 1, name
        assert fn(a16, a8, a16, a16, a16, 128, 128, 128, None) == 2, name       # scale atoms: 16 bytes
        assert fn(a16, a16, a16, a8, a16, 128, 128, 128, None) == 2, name
        assert fn(a16, a16, a8, a16, a16, 128, 128, 128, None) == 2, name
        assert fn(a16, a16, a16, a16, a16, 136, 128, 128, None) == 3, name
        assert fn(a16, a16, a16, a16, a16, 128, 128, 8, None) == 3, name
    cm = lib.fp8lin_cast_mx
    cm.restype = ctypes.c_int
    cm.argtypes = [V, I, I, ctypes.c_int, F, V, V, V, V, V]
    assert cm(a16, 32, 32, 0, 448.0, a16, None, None, None, None) == 1       # q without scales
    assert cm(a16, 32, 32, 0, 448.0, None, None, None, a16, None) == 1       # scales without q
    assert cm(a16, 32, 32, 0, 448.0, None, None, None, None, None) == 1      # nothing asked for
    assert cm(a16, 32, 32, 2, 448.0, a16, a16, None, None, None) == 1        # format
    assert cm(a16, 32, 32, 0, 0.0, a16, a16, None, None, None) == 1          # fmt_max
    assert cm(a16, 32, 32, 0, 1e-40, a16, a16, None, None, None) == 1        # subnormal fmt_max
    assert cm(a16, 32, 32, 0, float("inf"), a16, a16, None, None, None) == 1
    assert cm(a16, 32, 32, 0, 448.0, a16, a8, None, None, None) == 2         # misaligned atoms
    assert cm(V(4098), 32, 32, 0, 448.0, a16, a16, None, None, None) == 2    # misaligned input
    assert cm(a16, 32, 40, 0, 448.0, None, None, a16, a16, None) == 3        # ragged shape


def test_argument_checks_of_the_ocp_cast(lib):
    a16, a8 = V(4096), V(4104)
    cm = lib.fp8lin_cast_mx_ocp
    cm.restype = ctypes.c_int
    cm.argtypes = [V, I, I, ctypes.c_int, V, V, V, V, V]
    assert cm(a16, 32, 32, 0, a16, None, None, None, None) == 1          # q without scales
    assert cm(a16, 32, 32, 0, None, None, None, None, None) == 1         # nothing asked for
    assert cm(a16, 32, 32, 2, a16, a16, None, None, None) == 1           # format
    assert cm(a16, 32, 32, 0, a16, a8, None, None, None) == 2            # misaligned atoms
    assert cm(a16, 32, 40, 0, None, None, a16, a16, None) == 3           # ragged shape


def test_tile_count_limit_of_the_block_casts(lib):
    """The block casts index 128 x 128 tiles (and their ring's lookahead) with
    32-bit integers: a matrix of more than 2^31 - 2^20 - 1 tiles is refused
    as an unsupported shape before the device is touched, even though each
    dimension is within FP8LIN_MAX_DIM."""
    a16 = V(4096)
    big = 1 << 30                                    # 2^23 x 2^23 tiles
    cm = lib.fp8lin_cast_mx
    cm.restype = ctypes.c_int
    cm.argtypes = [V, I, I, ctypes.c_int, F, V, V, V, V, V]
    assert cm(a16, big, big, 0, 448.0, a16, a16, None, None, None) == 3
    co = lib.fp8lin_cast_mx_ocp
    co.restype = ctypes.c_int
    co.argtypes = [V, I, I, ctypes.c_int, V, V, V, V, V]
    assert co(a16, big, big, 0, None, None, a16, a16, None) == 3
    cb = lib.fp8lin_cast_blockwise
    cb.restype = ctypes.c_int
    cb.argtypes = [V, I, I, ctypes.c_int, F, V, V, V, V, V, V, V]
    assert cb(a16, big, big, 0, 448.0, a16, a16, None, None, None, None, None) == 3


def test_argument_checks_of_the_one_call_dynamic_cast(lib):
    """fp8lin_quantize checks every argument of its amax and its cast before
    launching either."""
    a16, a4 = V(4096), V(4100)
    fq = lib.fp8lin_quantize
    fq.restype = ctypes.c_int
    fq.argtypes = [V, I, I, ctypes.c_int, F, V, V, V, V, V, V]
    assert fq(a16, 32, 32, 0, 448.0, None, a16, a16, a16, None, None) == 1   # no amax slot
    assert fq(a16, 32, 32, 0, 448.0, a16, None, a16, a16, None, None) == 1   # no scale slot
    assert fq(a16, 32, 32, 0, 448.0, a16, a16, None, a16, None, None) == 1   # no inverse-scale slot
    assert fq(a16, 32, 32, 2, 448.0, a16, a16, a16, a16, None, None) == 1    # format
    assert fq(a16, 32, 32, 0, 0.0, a16, a16, a16, a16, None, None) == 1      # fmt_max
    assert fq(a16, -16, 32, 0, 448.0, a16, a16, a16, a16, None, None) == 1   # negative rows
    assert fq(a16, 32, 32, 0, 448.0, V(4098), a16, a16, a16, None, None) == 2  # misaligned amax
    assert fq(V(4098), 32, 32, 0, 448.0, a16, a16, a16, a16, None, None) == 2  # misaligned input
    assert fq(a16, 32, 32, 0, 448.0, a16, a16, a16, a4, None, None) == 2     # misaligned copy
    assert fq(a16, 32, 24, 0, 448.0, a16, a16, a16, a16, None, None) == 3    # ragged shape
    assert fq(a16, 1 << 31, 32, 0, 448.0, a16, a16, a16, a16, None, None) == 3


class QItem(ctypes.Structure):
    _fields_ = [("x", V), ("rows", ctypes.c_int64), ("cols", ctypes.c_int64), ("amax", V), ("scale", V),
                ("inv_scale", V), ("q", V)]


def test_argument_checks_of_the_batched_dynamic_cast(lib):
    """fp8lin_quantize_batch checks every item, and that no two slots of a
    call coincide, before launching anything."""
    fb = lib.fp8lin_quantize_batch
    fb.restype = ctypes.c_int
    fb.argtypes = [V, ctypes.c_int, ctypes.c_int, F, V]
    a16 = 4096

    def items(*specs):
        arr = (QItem * len(specs))()
        for k, sp in enumerate(specs):
            arr[k] = QItem(*sp)
        return arr

    def ok_item(base):  # x, 32 x 32, three slots, q
        return (a16, 32, 32, base, base + 4, base + 8, a16)

    two = items(ok_item(8192), ok_item(8448))
    assert fb(None, 1, 0, 448.0, None) == 1                        # no items
    assert fb(two, 0, 0, 448.0, None) == 1                         # empty batch
    five = items(*[ok_item(8192 + 256 * k) for k in range(5)])
    assert fb(five, 5, 0, 448.0, None) == 1                        # beyond the limit
    assert fb(two, 2, 2, 448.0, None) == 1                         # format
    assert fb(two, 2, 0, 0.0, None) == 1                           # fmt_max
    assert fb(items(ok_item(8192), (a16, 32, 32, 0, 8708, 8712, a16)), 2, 0, 448.0, None) == 1  # no amax slot
    assert fb(items(ok_item(8192), (a16, 32, 32, 8705, 8708, 8712, a16)), 2, 0, 448.0, None) == 2  # misaligned slot
    assert fb(items(ok_item(8192), (a16 + 4, 32, 32, 8704, 8708, 8712, a16)), 2, 0, 448.0, None) == 2  # input
    assert fb(items(ok_item(8192), (a16, 32, 24, 8704, 8708, 8712, a16)), 2, 0, 448.0, None) == 3  # ragged
    assert fb(items(ok_item(8192), (a16, 32, 32, 8704, 8708, 8712, 0)), 2, 0, 448.0, None) == 1   # no copy
    assert fb(items(ok_item(8192), ok_item(8192)), 2, 0, 448.0, None) == 1   # slots shared by two tensors
    assert fb(items(ok_item(8192), (a16, 32, 32, 8704, 8704, 8712, a16)), 2, 0, 448.0, None) == 1  # within one
    assert fb(items(ok_item(8192), (a16, 32, 32, 8704, 8708, 8200, a16)), 2, 0, 448.0, None) == 1  # across

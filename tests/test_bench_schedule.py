"""The benchmark's step schedules (pure host logic, no GPU): every cast is
issued before the first GEMM that reads it and never before its data
exists; the FFN step keeps its documented schedule."""
import bench


def _check(spec, overlap):
    main, side, needed, beside = bench.plan(spec, overlap)
    idx = {g: i for i, g in enumerate(spec.gemms)}
    placed = {}
    for i, keys in main.items():
        for k in keys:
            placed[k] = ("main", i)
    for i, keys in beside.items():
        for k in keys:
            assert needed[k] == i and k not in placed
            placed[k] = ("beside", i)
    for i, keys in side.items():
        for k in keys:
            placed[k] = ("side", i)
    assert set(placed) == set(bench.cast_inputs(spec))          # every cast exactly once
    for k, (where, i) in placed.items():
        a = spec.avail[k]
        exists = 0 if a is None else idx[a] + 1
        assert exists <= i <= needed[k], k                       # after its data, before its reader
        if where == "side":
            assert i < needed[k]                                 # something to hide under
    return main, side


def test_ffn_schedule():
    spec = bench.SPECS["ffn8b"]
    main, side = _check(spec, True)
    assert main[0] == ["xf"] and main[2] == ["h"]
    assert side[0] == ["w:w3", "w:w2"] and side[2] == ["dy:w2"] and side[4] == ["dy:w1", "dy:w3"]
    assert bench.spec_flops(spec) == 3 * 6 * 8192 * 4096 * 14336


def test_block_schedule():
    spec = bench.SPECS["block8b"]
    main, side = _check(spec, True)
    assert main[0] == ["xa"] and "xo" in main[1] and "xf" in main[2]
    assert "dy:o" in side[spec.gemms.index(("w3", "wgrad"))]
    assert "dy:qkv" in side[spec.gemms.index(("o", "wgrad"))]
    assert len(spec.gemms) == 15 and len(bench.cast_inputs(spec)) == 14


def test_serial_puts_everything_on_main():
    for spec in bench.SPECS.values():
        main, side = _check(spec, False)
        assert not any(side.values())


def test_attainable_bound():
    # cast traffic of one linear with both FP8 copies: 6 B per element of X, W
    # and dY (1,258 MB for the 8B FFN w1 shape); 5 B with one copy
    w13 = bench.SPECS["w13_8b"]
    per_linear = 8192 * 4096 + 14336 * 4096 + 8192 * 14336
    assert bench.cast_bytes(w13, "dynamic", transpose=True) == 6 * per_linear
    assert 1258e6 < 6 * per_linear < 1259e6
    assert bench.cast_bytes(w13, "dynamic") == 5 * per_linear
    # the FFN step casts X once for w1 and w3, and w2's input H (M x 14336) and dY2 (M x 4096)
    ffn = bench.SPECS["ffn8b"]
    elems = 8192 * 4096 + 2 * 14336 * 4096 + 2 * 8192 * 14336 + 8192 * 14336 + 4096 * 14336 + 8192 * 4096
    assert bench.cast_bytes(ffn, "delayed") == 3 * elems
    assert bench.cast_bytes(ffn, "delayed", transpose=True) == 4 * elems
    # row-wise scaling always writes both copies
    assert bench.cast_bytes(ffn, "rowwise") == bench.cast_bytes(ffn, "dynamic", transpose=True) == 6 * elems
    # with unlimited bandwidth the bound is the tensor peak; with casts it lies below
    assert abs(bench.attainable(w13, "dynamic", 3423.0, 1e30)["frac_of_peak"] - 1.0) < 1e-9
    a = bench.attainable(w13, "dynamic", 3423.0, 6775.9, transpose=True)
    gemm_ms = 6 * 8192 * 4096 * 14336 / 3423e12 * 1e3       # 0.843 ms
    cast_ms = 6 * per_linear / 6775.9e9 * 1e3                # 0.186 ms
    assert abs(a["frac_of_peak"] - gemm_ms / (gemm_ms + cast_ms)) < 1e-9
    assert 0.81 < a["frac_of_peak"] < 0.83
    assert bench.attainable(w13, "dynamic", 3423.0, 6775.9)["frac_of_peak"] > a["frac_of_peak"]
    # block scaling: one pass per tensor, two copies for activations and gradients, one for weights
    w_elems = 2 * 14336 * 4096 + 4096 * 14336
    assert bench.cast_bytes(ffn, "block") == 4 * (elems - w_elems) + 3 * w_elems
    # power-of-two blocks: every tensor, weights included, gets a 1 x 32 and a
    # 32 x 1 copy (2 B read, 2 x 1 B written; the scale bytes, 1/16 B, are
    # left out): 2,382,364,672 B for the FFN step, whose serialised bound at
    # 3423 TFLOP/s and 6775.9 GB/s is 3005 TFLOPS
    assert bench.cast_bytes(ffn, "mx") == 4 * elems == 2382364672
    m = bench.attainable(ffn, "mx", 3423.0, 6775.9)
    gemm_ms = 6 * (2 * 8192 * 4096 * 14336 + 8192 * 14336 * 4096) / 3423e12 * 1e3
    assert abs(m["frac_of_peak"] - gemm_ms / (gemm_ms + 4 * elems / 6775.9e9 * 1e3)) < 1e-9
    assert 3004.0 < m["serial_bound_tflops"] < 3006.0


def test_traffic_record_keys_on_the_per_tensor_kernel(tmp_path):
    """The committed DRAM-traffic record stays valid across edits to the
    block-scaled kernel and is voided by edits to the per-tensor kernel."""
    src = open(bench.GEMM_SRC).read()
    base = bench.gemm_kernel_sha256()
    block = src.index("// ------------------------------------------------- block-scaled kernel")
    edited_block = tmp_path / "block.cu"
    edited_block.write_text(src[:block + 80] + "// edit\n" + src[block + 80:])
    assert bench.gemm_kernel_sha256(str(edited_block)) == base
    kern = src.index("fp8_gemm_tn_kernel(")
    edited_kernel = tmp_path / "kernel.cu"
    edited_kernel.write_text(src[:kern] + "/* edit */ " + src[kern:])
    assert bench.gemm_kernel_sha256(str(edited_kernel)) != base


class _T8:
    """A cast target's host-side attributes (no device memory)."""

    def __init__(self, fmt, qT=None):
        self.fmt, self.fmt_max, self.qT = fmt, 448.0, qT


class _Fl:
    MAX_QUANTIZE_BATCH = 4


def _step(name, overlap, scaling, transpose=False):
    g = bench.StepGraph.__new__(bench.StepGraph)
    g.spec, g.overlap, g.scaling, g.fl = bench.SPECS[name], overlap, scaling, _Fl()
    g.t8 = {k: _T8(v[2], object() if transpose else None) for k, v in bench.cast_inputs(g.spec).items()}
    g._plan()
    return g


def test_gating_casts_share_launches_and_the_launch_count():
    """The casts issued right before a GEMM: with dynamic scaling and one FP8
    copy per tensor they share one fp8lin_quantize_batch launch; the bench's
    gpu_launches claim counts one kernel for that launch, two (amax + cast)
    for every dynamic or row-wise cast beside the GEMMs, one for any other
    recipe's cast, and one per GEMM."""
    g = _step("ffn8b", True, "dynamic")
    assert g._gate(0) == (["w:w1", "xf"], []) and g._gate(2) == (["h"], [])
    assert not any(g._gate(i)[0] or g._gate(i)[1] for i in (1, 3, 4, 5, 6, 7, 8))
    assert g._kernels_per_step() == 9 + 2 + 2 * 5
    # one stream: every cast gates its first GEMM; same-format casts share a launch
    g = _step("ffn8b", False, "dynamic")
    assert g._gate(2) == (["h", "w:w2"], [])
    assert g._kernels_per_step() == 9 + 6
    # both FP8 copies asked for: the gating casts go amax + cast, one tensor at a time
    g = _step("ffn8b", True, "dynamic", transpose=True)
    assert g._gate(0) == ([], ["w:w1", "xf"])
    assert g._kernels_per_step() == 9 + 2 * 3 + 2 * 5
    for scaling, per_cast in (("rowwise", 2), ("delayed", 1), ("block", 1), ("mx", 1)):
        g = _step("ffn8b", True, scaling)
        assert g._gate(0) == ([], ["xf"])                 # W1 runs beside X on the side stream
        assert g._kernels_per_step() == 9 + per_cast * 8
    g = _step("tiny", True, "dynamic")
    assert g._kernels_per_step() == 3 + 2              # X and W in one launch, then dY
    g = _step("block8b", True, "dynamic")
    assert g._kernels_per_step() == 15 + 4 + 2 * 9     # 15 GEMMs, four gates, nine casts beside the GEMMs

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

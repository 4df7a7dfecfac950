"""Parity of the schedule the benchmark times.

``bench.StepGraph`` issues a whole training step over several Float8 linears
on two CUDA streams: casts that gate the next GEMM on a high-priority main
stream, the others on a low-priority side stream under the GEMMs, joined by
events; X cast once for w1 and w3; the backward GEMMs reading the one
row-major FP8 copy of each tensor MN-major.  These tests run that object as
``bench.py`` runs it, at full size:

* the Llama-3.1-8B SwiGLU FFN (w1, w3 sharing X; w2) under dynamic, delayed,
  fp32-block and power-of-two-block scaling, and every linear of one
  Llama-3.1-8B block (QKV, O, w1, w3, w2) under dynamic scaling;
* two steps issued back to back on two different input sets (activations,
  weights and gradients all differ), so a buffer written by the second step
  while the first still reads it would show;
* after each step: every amax, scale, inverse scale, history entry, scale
  byte and FP8 byte of every cast input bit-exact against the oracle, and
  seeded sampled rows (first and last row included) of every Y, dX and dW
  within |y - ref| <= 2^-7 |ref| + 1e-3 rms(ref).

The state after the first step is copied on the main stream before the
second step is issued, so the copy is ordered exactly where the second
step's work starts.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads as wl
from gpu_helpers import assert_gemm_close, bf16_to_f64, to_dev_bf16

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
E4M3, E5M2 = oracle.E4M3, oracle.E5M2
SAMPLED_ROWS = 24
STATE = ("amax", "scale", "inv_scale", "history", "q", "qT", "qc", "row_inv", "col_inv", "tile_inv",
         "sf_row", "sf_col")


def _inputs(bench, spec, variant):
    """bf16 bits of every cast input; variant 0 is exactly bench.host_inputs(spec, 0)."""
    out = {}
    for key, (rows, cols, _, w, dist, seed, tid, outl) in bench.cast_inputs(spec).items():
        out[key] = wl.generate((rows, cols), *dist, seed=seed + 7919 * variant, tensor_id=tid, outlier_frac=outl)
    return out


def _rows(n, seed):
    rng = np.random.default_rng(seed)
    pick = rng.choice(n, size=min(n, SAMPLED_ROWS - 2), replace=False)
    return np.unique(np.concatenate([[0, n - 1], pick])).astype(np.int64)


def _snapshot(step):
    """Copies of every FP8 buffer, scale and output, made on the main stream."""
    snap = {"t8": {}, "out": {}}
    with torch.cuda.stream(step.main):
        for key, t8 in step.t8.items():
            snap["t8"][key] = {a: getattr(t8, a).clone() for a in STATE if getattr(t8, a, None) is not None}
        for name, outs in step.out.items():
            snap["out"][name] = {w: t.clone() for w, t in outs.items()}
    return snap


def _bits(t):
    return t.contiguous().cpu().numpy().view(np.uint32)


def _f32(v):
    return np.asarray(v, dtype=np.float32).view(np.uint32)


class _Oracle:
    """The oracle's view of one StepGraph: per cast input the recipe's FP8
    copies and scales, and (delayed scaling) the amax history the step
    carries from one call to the next."""

    def __init__(self, step, scaling):
        self.step, self.scaling = step, scaling
        self.hist, self.slot = {}, {}

    def quantize(self, key, bits):
        t8 = self.step.t8[key]
        fmt = t8.fmt
        if self.scaling == "dynamic":
            return oracle.quantize(bits, fmt)
        if self.scaling == "delayed":
            n = t8.history.numel()
            if key not in self.hist:                 # the first call seeds the slot before its own
                self.hist[key] = np.zeros(n, np.float32)
                self.slot[key] = 0
                self.hist[key][(0 - 1) % n] = oracle.amax(bits)
            r = oracle.quantize_delayed(bits, fmt, self.hist[key], self.slot[key])
            self.hist[key] = r["history"]
            self.slot[key] = (self.slot[key] + 1) % n
            return r
        if self.scaling == "block":
            if key.startswith("w:"):
                return {"tile": oracle.quantize_blocks(bits, fmt, 128, 128)}
            return {"row": oracle.quantize_blocks(bits, fmt, 1, 128), "col": oracle.quantize_blocks(bits, fmt, 128, 1)}
        assert self.scaling == "mx"
        rows, cols = bits.shape
        out = {}
        for k, along in (("row", "cols"), ("col", "rows")):
            d = oracle.quantize_mx(bits, fmt, along)
            P, K = (rows, cols) if along == "cols" else (cols, rows)
            d["atoms"] = oracle.pack_sf(oracle.sf_by_operand_row(d["sf"], along), P, K).reshape(-1)
            out[k] = d
        return out


def _check_casts(what, scaling, key, got, r):
    tag = f"{what} {key}"
    if scaling in ("dynamic", "delayed"):
        if scaling == "dynamic":
            assert _bits(got["amax"])[0] == _f32(r["amax"]), f"{tag} amax"
        else:
            assert np.array_equal(_bits(got["history"]), _f32(r["history"])), f"{tag} amax history"
        assert _bits(got["scale"])[0] == _f32(r["scale"]), f"{tag} scale"
        assert _bits(got["inv_scale"])[0] == _f32(r["inv_scale"]), f"{tag} inv_scale"
        assert np.array_equal(got["q"].cpu().numpy(), r["q"]), f"{tag} FP8 bytes"
    elif scaling == "block":
        if "tile" in r:
            assert np.array_equal(_bits(got["tile_inv"]), _f32(r["tile"]["inv_scale"])), f"{tag} tile scales"
            assert np.array_equal(got["q"].cpu().numpy(), r["tile"]["q"]), f"{tag} 128x128 FP8 bytes"
        else:
            assert np.array_equal(_bits(got["row_inv"].t()), _f32(r["row"]["inv_scale"])), f"{tag} 1x128 scales"
            assert np.array_equal(got["q"].cpu().numpy(), r["row"]["q"]), f"{tag} 1x128 FP8 bytes"
            assert np.array_equal(_bits(got["col_inv"]), _f32(r["col"]["inv_scale"])), f"{tag} 128x1 scales"
            assert np.array_equal(got["qc"].cpu().numpy(), r["col"]["q"]), f"{tag} 128x1 FP8 bytes"
    else:
        assert np.array_equal(got["sf_row"].cpu().numpy(), r["row"]["atoms"]), f"{tag} 1x32 scale atoms"
        assert np.array_equal(got["q"].cpu().numpy(), r["row"]["q"]), f"{tag} 1x32 FP8 bytes"
        assert np.array_equal(got["sf_col"].cpu().numpy(), r["col"]["atoms"]), f"{tag} 32x1 scale atoms"
        assert np.array_equal(got["qc"].cpu().numpy(), r["col"]["q"]), f"{tag} 32x1 FP8 bytes"


def _gemm_refs(scaling, rx, rw, rd, rm, rn):
    """Oracle rows of Y (rm), dX (rm) and dW (rn) of one linear."""
    if scaling in ("dynamic", "delayed"):
        return {"fwd": oracle.fwd_ref(rx["q"], rx["inv_scale"], rw["q"], rw["inv_scale"], rm),
                "dgrad": oracle.dgrad_ref(rd["q"], rd["inv_scale"], rw["qT"], rw["inv_scale"], rm),
                "wgrad": oracle.wgrad_ref(rd["qT"], rd["inv_scale"], rx["qT"], rx["inv_scale"], rn)}
    if scaling == "block":
        return {"fwd": oracle.fwd_block_ref(rx["row"]["q"], rx["row"]["inv_scale"], rw["tile"]["q"],
                                            rw["tile"]["inv_scale"], rm),
                "dgrad": oracle.dgrad_block_ref(rd["row"]["q"], rd["row"]["inv_scale"], rw["tile"]["q"],
                                                rw["tile"]["inv_scale"], rm),
                "wgrad": oracle.wgrad_block_ref(rd["col"]["q"], rd["col"]["inv_scale"], rx["col"]["q"],
                                                rx["col"]["inv_scale"], rn)}
    return {"fwd": oracle.fwd_mx_ref(rx["row"]["q"], rx["row"]["sf"], rw["row"]["q"], rw["row"]["sf"], rm),
            "dgrad": oracle.dgrad_mx_ref(rd["row"]["q"], rd["row"]["sf"], rw["col"]["q"], rw["col"]["sf"], rm),
            "wgrad": oracle.wgrad_mx_ref(rd["col"]["q"], rd["col"]["sf"], rx["col"]["q"], rx["col"]["sf"], rn)}


def _check_step(bench, what, step, scaling, orc, bits, snap):
    refs = {key: orc.quantize(key, bits[key]) for key in step.t8}
    for key in step.t8:
        _check_casts(what, scaling, key, snap["t8"][key], refs[key])
    for l in step.spec.linears:
        w = wl.WORKLOADS[l.workload]
        rm, rn = _rows(w.M, w.seed), _rows(w.N, w.seed + 1)
        ref = _gemm_refs(scaling, refs[l.x], refs["w:" + l.name], refs["dy:" + l.name], rm, rn)
        for which, rows in (("fwd", rm), ("dgrad", rm), ("wgrad", rn)):
            got = bf16_to_f64(snap["out"][l.name][which][torch.from_numpy(rows).cuda()])
            assert_gemm_close(got, ref[which], f"{what} {l.name}.{which}")


def _run_two_steps(fp8lin, workload, scaling):
    import bench
    spec = bench.SPECS[workload]
    dev = torch.device("cuda", 0)
    bits = [_inputs(bench, spec, v) for v in (0, 1)]
    dev_in = [{k: to_dev_bf16(b, dev) for k, b in bs.items()} for bs in bits]
    step = bench.StepGraph(fp8lin, spec, dev, dev_in[0], scaling=scaling)
    assert step.overlap and not step.transpose            # the default two-stream schedule, one copy per tensor
    torch.cuda.synchronize()
    step.run()                                            # step 1 on input set 0
    first = _snapshot(step)
    step.inp = dev_in[1]
    step.run()                                            # step 2 on input set 1, issued without a host sync
    second = _snapshot(step)
    torch.cuda.synchronize()
    assert fp8lin.fp8lin_device_error() == 0
    del dev_in
    orc = _Oracle(step, scaling)
    _check_step(bench, f"{workload}/{scaling} step 1", step, scaling, orc, bits[0], first)
    _check_step(bench, f"{workload}/{scaling} step 2", step, scaling, orc, bits[1], second)


@pytest.mark.parametrize("scaling", ["dynamic", "delayed", "block", "mx"])
def test_ffn8b_schedule_matches_oracle(fp8lin, scaling):
    _run_two_steps(fp8lin, "ffn8b", scaling)


def test_block8b_schedule_matches_oracle(fp8lin):
    _run_two_steps(fp8lin, "block8b", "dynamic")

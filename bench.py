"""Benchmark: Float8 linear fwd+bwd TFLOPS (amax and cast included).

Default workload: the Llama-3.1-8B SwiGLU FFN (``--workload ffn8b``).  One
step is the whole hot path for the FFN's three linears on one batch of 8192
tokens: for each of w1 and w3 (X [8192 x 4096], W [14336 x 4096],
dY [8192 x 14336]) and w2 (H [8192 x 14336], W [4096 x 14336],
dY [8192 x 4096]): the statistics and casts of X, W and dY (X once for w1
and w3) and the forward, input-gradient and weight-gradient FP8 GEMMs.
``--workload block8b`` adds the attention block's fused QKV [4096 -> 6144]
and output [4096 -> 4096] projections: every linear of one Llama-3.1-8B
transformer block.  Nothing is cached across steps (dynamic scaling
recomputes every statistic every step).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload ffn8b|block8b|...] [--scaling dynamic|delayed|rowwise|block|mx]

Prints one JSON line on rank 0.  N > 1 runs under torchrun: each rank runs
its own replica on its own batch (the path has no exchange step), timing is
bracketed by a barrier + synchronize and the max over ranks is reported.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from dataclasses import dataclass

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

METRIC = "FP8 linear fwd+bwd TFLOPS incl. amax/cast, % of GB300 dense FP8 peak"
FP8_PER_BF16 = 2.0            # nominal dense fp8 : bf16 tensor rate (4.5 : 2.25 PFLOP/s)
FALLBACK = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
E4M3, E5M2 = 0, 1
L2_FLUSH_BYTES = 512 << 20    # four times GB300's L2
BURST_REGION_MS = 2000.0      # timed regions shorter than this run at the burst clock


# ---------------------------------------------------------- step graphs

@dataclass(frozen=True)
class Linear:
    name: str
    workload: str          # key of workloads.WORKLOADS (shape, distributions, seed)
    x: str                 # key of the activation it reads (shared keys are cast once)
    w_id: int              # tensor ids of W and dY inside the workload's streams
    dy_id: int


@dataclass(frozen=True)
class Spec:
    """One training step over several Float8 linears.

    gemms: issue order on the main stream, as (linear, "fwd"|"dgrad"|"wgrad").
    avail: for every cast input, the GEMM after which its bf16 data exists
           (None = at the start of the step).  A cast that its first consumer
           needs right after the data appears runs on the main stream; any
           other runs on the side stream, released just before the GEMM that
           follows its producer, so it hides under GEMMs."""
    name: str
    description: str
    linears: tuple
    gemms: tuple
    avail: dict


_FFN_LINEARS = (Linear("w1", "llama3_8b_ffn_w13", "xf", wl.W, wl.DY),
                Linear("w3", "llama3_8b_ffn_w13", "xf", wl.W3, wl.DY3),
                Linear("w2", "llama3_8b_ffn_w2", "h", wl.W, wl.DY))
_FFN_GEMMS = (("w1", "fwd"), ("w3", "fwd"), ("w2", "fwd"), ("w2", "dgrad"), ("w2", "wgrad"),
              ("w1", "dgrad"), ("w1", "wgrad"), ("w3", "dgrad"), ("w3", "wgrad"))
_FFN_AVAIL = {
    "xf": None, "w:w1": None, "w:w3": None, "w:w2": None,
    "h": ("w3", "fwd"),          # H = silu(Y1) * Y3
    "dy:w2": ("w3", "fwd"),      # upstream gradient: cast under w2's forward (a deeper layer's wgrad in a full model)
    "dy:w1": ("w2", "dgrad"),    # dY1, dY3 derive from dH through the SwiGLU backward
    "dy:w3": ("w2", "dgrad"),
}

SPECS = {
    "ffn8b": Spec(
        "llama3.1-8b-swiglu-ffn",
        "Llama-3.1-8B SwiGLU FFN: w1, w3 (M8192 K4096 N14336, shared X) and w2 (M8192 K14336 N4096)",
        _FFN_LINEARS, _FFN_GEMMS, _FFN_AVAIL),
    "block8b": Spec(
        "llama3.1-8b-block-linears",
        "every linear of one Llama-3.1-8B block: fused QKV (M8192 K4096 N6144), O (M8192 K4096 N4096), "
        "w1, w3 (M8192 K4096 N14336, shared X) and w2 (M8192 K14336 N4096)",
        (Linear("qkv", "llama3_8b_qkv", "xa", wl.W, wl.DY), Linear("o", "llama3_8b_o", "xo", wl.W, wl.DY))
        + _FFN_LINEARS,
        (("qkv", "fwd"), ("o", "fwd")) + _FFN_GEMMS
        + (("o", "dgrad"), ("o", "wgrad"), ("qkv", "dgrad"), ("qkv", "wgrad")),
        {**_FFN_AVAIL, "xa": None, "w:qkv": None, "w:o": None,
         "xo": ("qkv", "fwd"),       # attention output
         "xf": ("o", "fwd"),         # FFN input: residual + norm after the attention block
         "dy:o": ("w3", "dgrad"),    # dX of w1 and w3 summed, through the residual
         "dy:qkv": ("o", "dgrad")}), # through the attention backward
}


def _single(key: str, wname: str, desc: str) -> Spec:
    """One linear's step: forward, then the gradient dY arrives (upstream)."""
    return Spec(key, desc, (Linear("l", wname, "x", wl.W, wl.DY),),
                (("l", "fwd"), ("l", "dgrad"), ("l", "wgrad")),
                {"x": None, "w:l": None, "dy:l": ("l", "fwd")})


SPECS.update({
    "tiny": _single("tiny", "tiny", "one linear M256 K512 N1024"),
    "qkv8b": _single("llama3.1-8b-qkv", "llama3_8b_qkv", "Llama-3.1-8B fused QKV, M8192 K4096 N6144"),
    "w13_8b": _single("llama3.1-8b-ffn-w1", "llama3_8b_ffn_w13", "Llama-3.1-8B FFN w1 (= w3), M8192 K4096 N14336"),
    "w2_8b": _single("llama3.1-8b-ffn-w2", "llama3_8b_ffn_w2", "Llama-3.1-8B FFN w2, M8192 K14336 N4096"),
    "w1_70b": _single("llama3.1-70b-ffn-w1", "llama3_70b_ffn_w1",
                      "Llama-3.1-70B FFN w1 with 0.1% x100 outliers in X, M16384 K8192 N28672"),
    "w1_405b": _single("llama3.1-405b-ffn-w1", "llama3_405b_ffn_w1",
                       "Llama-3.1-405B FFN w1 (Laplace dY), M8192 K16384 N53248"),
})


def spec_flops(spec: Spec) -> int:
    return sum(wl.WORKLOADS[l.workload].flops for l in spec.linears)


def cast_elem_bytes(scaling: str, transpose: bool, weight: bool = False) -> int:
    """HBM bytes per cast element in one step: the cast reads x (2 B) and
    writes one FP8 copy, or two with the transposed copy (always for
    row-wise scaling; for block scaling, activations and gradients get a
    row-block and a column-block copy, weights one 128 x 128-block copy);
    dynamic and row-wise scaling read x once more for the amax pass, delayed,
    static and block scaling do not.  Power-of-two block scaling ("mx")
    writes a row-block and a column-block copy of every tensor (plus one
    scale byte per 32 elements per copy, left out here)."""
    if scaling == "block":
        return 2 + (1 if weight else 2)
    if scaling == "mx":
        return 2 + 2
    two_copies = transpose or scaling == "rowwise"
    return 2 + 1 + (1 if two_copies else 0) + (2 if scaling in ("dynamic", "rowwise") else 0)


def cast_bytes(spec: Spec, scaling: str, transpose: bool = False) -> int:
    return sum(r * c * cast_elem_bytes(scaling, transpose, key.startswith("w:"))
               for key, (r, c, *_) in cast_inputs(spec).items())


def attainable(spec: Spec, scaling: str, peak_tflops: float, hbm_gbs: float, transpose: bool = False) -> dict:
    """Bound if every GEMM ran at the tensor peak and every amax / cast alone
    at the copy bandwidth, one after another: flop / (flop / P + cast bytes / BW).
    Running the casts beside the GEMMs can beat it."""
    flop, b = spec_flops(spec), cast_bytes(spec, scaling, transpose)
    t = flop / (peak_tflops * 1e12) + b / (hbm_gbs * 1e9)
    return {"serial_bound_tflops": flop / t / 1e12, "frac_of_peak": flop / t / 1e12 / peak_tflops,
            "cast_bytes_per_step": b,
            "note": "6MNK / (6MNK/P + cast bytes/BW): GEMMs at the peak and every amax/cast alone at the copy "
                    "bandwidth, serialised; overlapping casts with GEMMs can exceed it"}


def cast_inputs(spec: Spec):
    """Every bf16 tensor the step casts: key -> (rows, cols, fmt, workload, dist, seed, tensor id, outliers)."""
    out = {}
    for l in spec.linears:
        w = wl.WORKLOADS[l.workload]
        out.setdefault(l.x, (w.M, w.K, E4M3, w, w.x, w.seed, wl.X, w.x_outlier_frac))
        out["w:" + l.name] = (w.N, w.K, E4M3, w, w.w, w.seed, l.w_id, 0.0)
        out["dy:" + l.name] = (w.M, w.N, E5M2, w, w.dy, w.seed, l.dy_id, 0.0)
    return out


def host_inputs(spec: Spec, rank: int):
    """bf16 bit patterns of every cast input; activations and gradients per rank."""
    out = {}
    for key, (rows, cols, _, w, dist, seed, tid, outl) in cast_inputs(spec).items():
        per_rank = not key.startswith("w:")
        out[key] = wl.generate((rows, cols), *dist, seed=seed + (1000 * rank if per_rank else 0),
                               tensor_id=tid, outlier_frac=outl)
    return out


# ------------------------------------------------------------------ peaks

GEMM_SRC = os.path.join(ROOT, "float8_linear_layers_gb300", "csrc", "gemm.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "fp8_gemm_tn_kernel__ffn8b_step_traffic.json")


# The parts of the GEMM source the per-tensor kernel's traffic depends on:
# the device code up to the block-scaled kernel (helpers, tile map, kernel)
# and the host code from the raster to the per-tensor launch.
GEMM_REGIONS = (("namespace {", "// ------------------------------------------------- block-scaled kernel"),
                ("// Raster: keep", "std::atomic<bool> g_blk_attr_set"))


def gemm_kernel_sha256(path: str = GEMM_SRC) -> str:
    """SHA-256 over the per-tensor GEMM's device and host code (GEMM_REGIONS)."""
    import hashlib
    with open(path) as f:
        text = f.read()
    h = hashlib.sha256()
    for start, end in GEMM_REGIONS:
        i = text.index(start)
        h.update(text[i:text.index(end, i)].encode())
    return h.hexdigest()


def gemm_traffic(workload: str, scaling: str):
    """Mean DRAM bytes per GEMM launch of one step of `workload`, from the
    committed ncu capture of the per-tensor-scale GEMM; None when that
    kernel's source changed since the counters were taken, no capture covers
    this workload, or the step runs the row-wise- or block-scaled GEMM
    instead."""
    try:
        with open(TRAFFIC_FILE) as f:
            t = json.load(f)
        sha = gemm_kernel_sha256()
    except (OSError, ValueError):
        return None
    if t.get("gemm_kernel_sha256") != sha or t.get("workload") != workload or scaling in ("rowwise", "block", "mx"):
        return None
    return int(t["mean_dram_bytes_per_launch"])


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK), "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().strip().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        load = [s for s in sm if smax and s > 0.5 * max(smax)] or sm
        return {"sm_mhz": statistics.median(load) if load else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------- oracle (CPU)

def sha256_of(bits: np.ndarray) -> str:
    import hashlib
    return hashlib.sha256(np.ascontiguousarray(bits).view(np.uint8)).hexdigest()


class OracleSample:
    """The CPU oracle on a bounded sample of one step: the per-tensor scaling
    (amax, scale, cast, transpose) of the first `frac` of every cast input's
    rows and every GEMM on the first `frac` of its output rows (the whole
    tensors' FP8 copies, which the GEMMs read, prepared once, untimed).
    Work scales linearly with rows, so the sample does `frac` of the step's
    work.  The inputs are generated here, independently of the GPU leg, and
    fingerprinted (SHA-256 of the bf16 bytes) so the two legs can be shown
    to have seen the same bits."""

    def __init__(self, spec: Spec, frac: float):
        import oracle
        self.o, self.spec, self.frac = oracle, spec, frac
        self.inputs, self.sha256 = {}, {}
        for key, (rows, cols, fmt, w, dist, seed, tid, outl) in cast_inputs(spec).items():
            bits = wl.generate((rows, cols), *dist, seed=seed, tensor_id=tid, outlier_frac=outl)
            self.sha256[key] = sha256_of(bits)
            self.inputs[key] = (bits, fmt, oracle.quantize(bits, fmt))
        self.rows = {}
        for l in spec.linears:
            w = wl.WORKLOADS[l.workload]
            self.rows[l.name] = (np.arange(max(1, int(round(w.M * frac)))), np.arange(max(1, int(round(w.N * frac)))))
        self.last = {}

    def flops(self) -> int:
        """Multiply-adds x 2 of the sample's GEMM rows."""
        f = 0
        for l in self.spec.linears:
            w = wl.WORKLOADS[l.workload]
            rm, rn = self.rows[l.name]
            f += 2 * (2 * rm.size * w.N * w.K + rn.size * w.M * w.K)
        return f

    def run(self) -> float:
        o, f = self.o, self.frac
        t0 = time.perf_counter()
        for key, (bits, fmt, _) in self.inputs.items():
            rows = max(16, int(round(bits.shape[0] * f)))
            o.quantize(bits[:rows], fmt)
        last = {}
        for l in self.spec.linears:
            qx, qw, qd = (self.inputs[k][2] for k in (l.x, "w:" + l.name, "dy:" + l.name))
            rm, rn = self.rows[l.name]
            last[l.name] = {"fwd": o.fwd_ref(qx["q"], qx["inv_scale"], qw["q"], qw["inv_scale"], rm),
                            "dgrad": o.dgrad_ref(qd["q"], qd["inv_scale"], qw["qT"], qw["inv_scale"], rm),
                            "wgrad": o.wgrad_ref(qd["qT"], qd["inv_scale"], qx["qT"], qx["inv_scale"], rn)}
        secs = time.perf_counter() - t0
        self.last = last
        return secs

    def check(self, gpu: dict) -> dict:
        """Compare one GPU step (``StepGraph.parity_state``) with the oracle:
        amax, scale and inverse scale bits and every FP8 byte of every cast
        input; the sample's rows of every Y, dX and dW within the GEMM
        tolerance |y - ref| <= 2^-7 |ref| + 1e-3 rms(ref)."""
        o = self.o
        bad = []
        for key, (bits, fmt, r) in self.inputs.items():
            g = gpu["casts"][key]
            for a in ("amax", "scale", "inv_scale"):
                if g[a] != int(np.float32(r[a]).view(np.uint32)):
                    bad.append(f"{key} {a}")
            if not np.array_equal(g["q"], r["q"]):
                bad.append(f"{key} FP8 bytes")
        worst = 0.0
        for l in self.spec.linears:
            for which, ref in self.last[l.name].items():
                got = gpu["outputs"][l.name][which][:ref.shape[0]]
                ok, ratio = o.within_tolerance(got, ref, float(np.sqrt(np.mean(ref ** 2))))
                worst = max(worst, ratio)
                if not ok:
                    bad.append(f"{l.name}.{which}")
        return {"ok": not bad, "failures": bad, "worst_err_over_bound": worst,
                "checked": "amax, scale, inverse scale and every FP8 byte of every cast input bit-exact; the "
                           f"first {self.frac:.5g} of the rows of every Y, dX and dW within the GEMM tolerance"}

    def time_for(self, seconds: float, at_least: int = 1):
        """Run the sample until `seconds` have passed (at least `at_least` runs); the run times."""
        times = []
        while len(times) < at_least or sum(times) < seconds:
            times.append(self.run())
        return times

    def describe(self) -> str:
        return (f"one step of {self.spec.description}, sampled at {self.frac:.5g} of its rows: "
                f"amax/scale/cast/transpose of that share of every cast input (shared X once) and that share "
                f"of the output rows of every fwd/dgrad/wgrad GEMM ({self.flops() / 1e9:.4g} GFLOP)")


# ------------------------------------------------------------ reference

def run_reference(args, rank: int) -> None:
    """The oracle as the reference arm: each step is one run of the bounded
    sample of the workload (OracleSample); value = the sample's flops / its
    time, so ms_per_step x steps is the wall time spent."""
    if rank != 0:
        return
    import oracle
    spec = SPECS[args.workload]
    frac = args.cpu_frac
    s = OracleSample(spec, frac)
    for _ in range(args.warmup):
        s.run()
    times = [s.run() for _ in range(args.steps)]
    step_s = sum(times) / len(times)
    value = s.flops() / step_s / 1e12
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
        "extrapolated_ms_per_step": step_s / frac * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": {"workload": spec.name, "scaling": "dynamic"},
        "cpu_baseline": {"value": value, "unit": "TFLOPS", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": s.describe()},
        "e2e": {"value": value, "unit": "TFLOPS", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "inputs_sha256": s.sha256,
        "gpu_launches": 0,
        "note": "each step is one run of the sample; extrapolated_ms_per_step = ms_per_step / share",
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------- ours

def plan(spec: Spec, overlap: bool = True):
    """Where each cast runs.  Returns (main_casts, side_casts, needed_by):
    main_casts[i] are issued on the main stream right before GEMM i;
    side_casts[i] are released on the side stream just before GEMM i
    launches; needed_by[key] is the first GEMM that reads the cast."""
    lin = {l.name: l for l in spec.linears}
    idx = {g: i for i, g in enumerate(spec.gemms)}
    first_use = {}
    for i, (name, which) in enumerate(spec.gemms):
        l = lin[name]
        uses = {"fwd": (l.x, "w:" + name), "dgrad": ("dy:" + name, "w:" + name),
                "wgrad": ("dy:" + name, l.x)}[which]
        for k in uses:
            first_use.setdefault(k, i)
    main_casts = {i: [] for i in range(len(spec.gemms))}
    side_casts = {i: [] for i in range(len(spec.gemms))}
    beside = {i: [] for i in range(len(spec.gemms))}
    for key in cast_inputs(spec):
        a = spec.avail[key]
        release = 0 if a is None else idx[a] + 1
        n = first_use[key]
        if release > n:
            raise ValueError(f"{key} is read by GEMM {n} before it exists")
        if not overlap or release == n:
            main_casts[n].append(key)
        else:
            side_casts[release].append(key)
    if overlap:
        # several casts gating the same GEMM with nothing to hide under: the
        # first stays on the main stream, the others run beside it
        for i in main_casts:
            main_casts[i], beside[i] = main_casts[i][:1], main_casts[i][1:]
    for i in side_casts:
        side_casts[i].sort(key=lambda k: first_use[k])
    return main_casts, side_casts, first_use, beside


class StepGraph:
    """A Spec issued through the public entry points on two CUDA streams.

    With overlap, casts that have a GEMM to hide under run on a low-priority
    side stream; the GEMMs, and casts that gate the next GEMM, run on a
    high-priority main stream.  Side-stream work waits for a marker recorded
    on the main stream just before the GEMM it should run under is launched,
    so that GEMM's persistent CTAs are resident first and the HBM-bound
    kernels fill the SM resources it leaves free -- the overlap window the
    pages describe for FP8 scaling work.  Each step starts after the previous
    one has finished (FP8 buffers and outputs are reused)."""

    def __init__(self, fl, spec: Spec, dev, dev_in, overlap=True, scaling="dynamic", streams=None,
                 transpose=False, mx_rule="floor"):
        import torch
        self.fl, self.t, self.spec = fl, torch, spec
        self.overlap, self.scaling, self.mx_rule = overlap, scaling, mx_rule
        # one FP8 copy per tensor (backward GEMMs read it MN-major) unless the
        # transposed copies are asked for; row-wise scaling always needs them,
        # block scaling never writes them
        self.transpose = (transpose or scaling == "rowwise") and scaling not in ("block", "mx")
        self.inp = dev_in
        self.lin = {l.name: l for l in spec.linears}
        self.t8 = {}
        for key, (rows, cols, fmt, *_) in cast_inputs(spec).items():
            if scaling == "mx":      # every tensor: a 1 x 32 and a 32 x 1 block copy
                self.t8[key] = fl.Float8Tensor(rows, cols, fmt, dev, scaling=scaling, transpose=False,
                                               mx_rule=mx_rule)
            elif scaling == "block":   # weights in 128 x 128 blocks, activations and gradients in row / column blocks
                self.t8[key] = fl.Float8Tensor(rows, cols, fmt, dev, scaling=scaling, transpose=False,
                                               blocks="tile" if key.startswith("w:") else "rowcol")
            else:
                self.t8[key] = fl.Float8Tensor(rows, cols, fmt, dev, scaling=scaling, transpose=self.transpose)
        bf = torch.bfloat16
        self.out = {}
        for l in spec.linears:
            w = wl.WORKLOADS[l.workload]
            self.out[l.name] = {"fwd": torch.empty((w.M, w.N), dtype=bf, device=dev),
                                "dgrad": torch.empty((w.M, w.K), dtype=bf, device=dev),
                                "wgrad": torch.empty((w.N, w.K), dtype=bf, device=dev)}
        if streams is not None:
            self.main, self.side = streams
        elif overlap:
            self.main = torch.cuda.Stream(device=dev, priority=-1)
            self.side = torch.cuda.Stream(device=dev, priority=0)
        else:
            # one stream; not the legacy default stream, so the step can be captured in a CUDA graph
            self.main = self.side = torch.cuda.Stream(device=dev)
        self._plan()
        self.kernels_per_step = self._kernels_per_step()

    def _plan(self):
        self.main_casts, self.side_casts, self.needed_by, self.beside = plan(self.spec, self.overlap)

    def _gate(self, i):
        """The casts issued on the main stream right before GEMM i, split
        into the dynamic casts without a transposed copy, which share
        fp8lin_quantize_batch launches (one per format, at most four tensors
        each), and the others."""
        keys = (self.beside[i] if self.scaling == "dynamic" else []) + self.main_casts[i]
        batch = [k for k in keys if self.scaling == "dynamic" and self.t8[k].qT is None]
        return batch, [k for k in keys if k not in batch]

    def _kernels_per_step(self) -> int:
        """Kernels one step launches: the GEMMs; one per batched launch of
        gating casts; amax + cast for any other dynamic or row-wise cast; one
        for each block, power-of-two block, delayed and static cast."""
        per_cast = 2 if self.scaling in ("dynamic", "rowwise") else 1
        n = len(self.spec.gemms) + per_cast * sum(len(v) for v in self.side_casts.values())
        if self.scaling != "dynamic":
            n += per_cast * sum(len(v) for v in self.beside.values())
        for i in range(len(self.spec.gemms)):
            batch, rest = self._gate(i)
            fmts = {}
            for k in batch:
                fmts[(self.t8[k].fmt, self.t8[k].fmt_max)] = fmts.get((self.t8[k].fmt, self.t8[k].fmt_max), 0) + 1
            n += sum(-(-c // self.fl.MAX_QUANTIZE_BATCH) for c in fmts.values()) + per_cast * len(rest)
        return n

    def _cast_alone(self, rec, keys_batch, keys_rest, stream):
        for key in keys_rest:
            self._cast(rec, key, stream, alone=True)
        if keys_batch:
            # amax read, cast read and the FP8 copy: 5 B per element
            work = sum(5 * self.inp[k].numel() for k in keys_batch)
            self._mark(stream, rec, "quantize", "+".join(keys_batch), work, lambda: self.fl.quantize_alone(
                [(self.t8[k], self.inp[k]) for k in keys_batch], stream))

    def describe(self):
        how = {"rowwise": "row-wise (per-block) scaling",
               "block": "block scaling (1 x 128 / 128 x 128 blocks, fp32 scales, partial sums promoted per block)",
               "mx": "power-of-two block scaling (1 x 32 / 32 x 1 blocks, scales applied by the tensor cores)"}.get(
            self.scaling, f"{self.scaling} per-tensor scaling")
        if not self.overlap:
            return how + "; serial: one stream, shared X cast once"
        return how + ("; two streams: casts that the data dependencies leave hidable run on a low-priority side "
                      "stream under the GEMMs of a high-priority main stream; casts that gate the next GEMM run on "
                      "the main stream; shared X cast once")

    def outputs(self):
        return [self.out[l.name][w] for l in self.spec.linears for w in ("fwd", "dgrad", "wgrad")]

    def parity_state(self, frac: float) -> dict:
        """Host copies of what the last step left on the device, for the
        oracle comparison (per-tensor scaling): the amax, scale and inverse
        scale bits and the FP8 copy of every cast input, and the first
        `frac` of the rows of every Y, dX and dW (as float64)."""
        t = self.t
        casts = {}
        for key, t8 in self.t8.items():
            bits = lambda v: int(v.cpu().view(t.int32).item()) & 0xFFFFFFFF
            casts[key] = {"amax": bits(t8.amax), "scale": bits(t8.scale), "inv_scale": bits(t8.inv_scale),
                          "q": t8.q.cpu().numpy()}
        outputs = {}
        for l in self.spec.linears:
            w = wl.WORKLOADS[l.workload]
            nm, nn = max(1, int(round(w.M * frac))), max(1, int(round(w.N * frac)))
            o = self.out[l.name]
            outputs[l.name] = {"fwd": o["fwd"][:nm].float().cpu().numpy().astype(np.float64),
                               "dgrad": o["dgrad"][:nm].float().cpu().numpy().astype(np.float64),
                               "wgrad": o["wgrad"][:nn].float().cpu().numpy().astype(np.float64)}
        return {"casts": casts, "outputs": outputs}

    # -- issue -------------------------------------------------------------
    def _ev(self):
        return self.t.cuda.Event(enable_timing=True)

    def _mark(self, stream, rec, kind, label, work, fn):
        if rec is None or (kind != "gemm" and getattr(rec, "gemm_only", False)):
            fn()
            return
        e0, e1 = self._ev(), self._ev()
        e0.record(stream)
        fn()
        e1.record(stream)
        rec.append((kind, label, e0, e1, work))

    def _cast(self, rec, key, stream, alone=False):
        """Cast one input.  alone: no GEMM runs beside it (a cast that gates
        the next GEMM, or one running next to such a cast): dynamic scaling
        then takes the one-call fp8lin_quantize."""
        fl, x, t8 = self.fl, self.inp[key], self.t8[key]
        n = x.numel()
        two_copies = t8.qT is not None or getattr(t8, "blocks", None) == "rowcol" or t8.scaling == "mx"
        cast_bytes = (4 if two_copies else 3) * n   # read bf16, write one or two FP8 copies
        if t8.scaling == "dynamic" and alone:
            self._mark(stream, rec, "quantize", key, 2 * n + cast_bytes, lambda: fl.fp8lin_quantize(
                x, t8.fmt, t8.amax, t8.scale, t8.inv_scale, t8.q, t8.qT, t8.fmt_max, stream))
        elif t8.scaling in ("block", "mx"):
            self._mark(stream, rec, "cast", key, cast_bytes, lambda: t8.quantize(x, stream))
        elif t8.scaling == "rowwise":
            self._mark(stream, rec, "amax", key, 2 * n,
                       lambda: fl.fp8lin_amax_rowcol(x, t8.row_amax, t8.col_amax, stream))
            self._mark(stream, rec, "cast", key, cast_bytes, lambda: fl.fp8lin_cast_transpose_rowwise(
                x, t8.fmt, t8.row_amax, t8.col_amax, t8.row_inv, t8.col_inv, t8.q, t8.qT, t8.fmt_max, stream))
        elif t8.scaling == "dynamic":
            self._mark(stream, rec, "amax", key, 2 * n, lambda: fl.fp8lin_amax(x, t8.amax, stream))
            self._mark(stream, rec, "cast", key, cast_bytes, lambda: fl.fp8lin_cast_transpose(
                x, t8.fmt, t8.amax, t8.scale, t8.inv_scale, t8.q, t8.qT, t8.fmt_max, stream))
        else:
            self._mark(stream, rec, "cast", key, cast_bytes, lambda: t8.quantize(x, stream))

    def _gemm(self, rec, name, which):
        fl, m = self.fl, self.main
        l = self.lin[name]
        w = wl.WORKLOADS[l.workload]
        x8, w8, d8 = self.t8[l.x], self.t8["w:" + name], self.t8["dy:" + name]
        out = self.out[name][which]
        if self.scaling == "mx":
            fn = {"fwd": lambda: fl.fp8lin_fwd_mx(x8.q, x8.sf_row, w8.q, w8.sf_row, out, m),
                  "dgrad": lambda: fl.fp8lin_dgrad_mx(d8.q, d8.sf_row, w8.qc, w8.sf_col, out, m),
                  "wgrad": lambda: fl.fp8lin_wgrad_mx(d8.qc, d8.sf_col, x8.qc, x8.sf_col, out, m)}[which]
        elif self.scaling == "block":
            fn = {"fwd": lambda: fl.fp8lin_fwd_block(x8.q, x8.row_inv, w8.q, w8.tile_inv, out, m),
                  "dgrad": lambda: fl.fp8lin_dgrad_block(d8.q, d8.row_inv, w8.q, w8.tile_inv, out, m),
                  "wgrad": lambda: fl.fp8lin_wgrad_block(d8.qc, d8.col_inv, x8.qc, x8.col_inv, out, m)}[which]
        elif self.scaling == "rowwise":
            fn = {"fwd": lambda: fl.fp8lin_fwd_rowwise(x8.q, x8.row_inv, w8.q, w8.row_inv, out, m),
                  "dgrad": lambda: fl.fp8lin_dgrad_rowwise(d8.q, d8.row_inv, w8.qT, w8.col_inv, out, m),
                  "wgrad": lambda: fl.fp8lin_wgrad_rowwise(d8.qT, d8.col_inv, x8.qT, x8.col_inv, out, m)}[which]
        elif self.transpose:
            fn = {"fwd": lambda: fl.fp8lin_fwd(x8.q, x8.inv_scale, w8.q, w8.inv_scale, out, m),
                  "dgrad": lambda: fl.fp8lin_dgrad(d8.q, d8.inv_scale, w8.qT, w8.inv_scale, out, m),
                  "wgrad": lambda: fl.fp8lin_wgrad(d8.qT, d8.inv_scale, x8.qT, x8.inv_scale, out, m)}[which]
        else:
            fn = {"fwd": lambda: fl.fp8lin_fwd(x8.q, x8.inv_scale, w8.q, w8.inv_scale, out, m),
                  "dgrad": lambda: fl.fp8lin_dgrad_mn(d8.q, d8.inv_scale, w8.q, w8.inv_scale, out, m),
                  "wgrad": lambda: fl.fp8lin_wgrad_mn(d8.q, d8.inv_scale, x8.q, x8.inv_scale, out, m)}[which]
        self._mark(m, rec, "gemm", f"{name}.{which}", 2 * w.M * w.N * w.K, fn)

    def run(self, rec=None):
        m, s = self.main, self.side
        ready = {}
        for i, (name, which) in enumerate(self.spec.gemms):
            if self.beside[i] and self.scaling != "dynamic":
                marker = self.t.cuda.Event()
                marker.record(m)                      # the casts gating GEMM i start together
                s.wait_event(marker)
                for key in self.beside[i]:
                    self._cast(rec, key, s, alone=True)
                    e = self.t.cuda.Event()
                    e.record(s)
                    ready[key] = e
            # the one-launch dynamic cast occupies every SM: the casts gating
            # this GEMM run on the main stream, in one launch where they can
            self._cast_alone(rec, *self._gate(i), m)
            if self.side_casts[i]:
                marker = self.t.cuda.Event()
                marker.record(m)                      # this GEMM is about to launch
                s.wait_event(marker)
                for key in self.side_casts[i]:
                    self._cast(rec, key, s)
                    e = self.t.cuda.Event()
                    e.record(s)
                    ready[key] = e
            for key, e in list(ready.items()):
                if self.needed_by[key] == i:
                    m.wait_event(e)
                    del ready[key]
            self._gemm(rec, name, which)


def run_e2e(args, fl, spec, dev, host, step, world, dist, barrier):
    """The same step measured end to end from pinned host memory: every step
    uploads every bf16 input and reads back every output (Y, dX, dW of each
    linear).  Inputs and outputs are double buffered so that step i+1's
    upload and step i's readback run on their own copy streams while step i
    computes."""
    import torch
    pinned = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).pin_memory() for k, v in host.items()}
    h2d_bytes = sum(t.numel() * 2 for t in pinned.values())
    sets = []
    for k in range(2):
        din = {key: torch.empty(t.shape, dtype=torch.bfloat16, device=dev) for key, t in pinned.items()}
        g = step if k == 0 else StepGraph(fl, spec, dev, din, overlap=step.overlap, scaling=step.scaling,
                                          streams=(step.main, step.side), transpose=step.transpose,
                                          mx_rule=step.mx_rule)
        g.inp = din
        outs = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in g.outputs()]
        sets.append((g, din, outs))
    d2h_bytes = sum(t.numel() * t.element_size() for t in sets[0][2])
    copy_in = torch.cuda.Stream(device=dev)
    copy_out = torch.cuda.Stream(device=dev)
    main = step.main

    def run(n, timed):
        ev = lambda: torch.cuda.Event(enable_timing=timed)
        ev_in, ev_done, ev_out = [None, None], [None, None], [None, None]
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

        def upload(k):
            with torch.cuda.stream(copy_in):
                for key, t in pinned.items():
                    sets[k][1][key].copy_(t, non_blocking=True)
            e = ev()
            e.record(copy_in)
            ev_in[k] = e

        t0.record(copy_in)
        upload(0)
        for i in range(n):
            k, j = i % 2, (i + 1) % 2
            if i + 1 < n:
                if ev_done[j] is not None:
                    copy_in.wait_event(ev_done[j])       # step i-1 is done reading set j
                upload(j)
            main.wait_event(ev_in[k])
            if ev_out[k] is not None:
                main.wait_event(ev_out[k])               # step i-2's outputs have left set k
            g, _, outs = sets[k]
            g.run()
            e = ev()
            e.record(main)
            ev_done[k] = e
            copy_out.wait_event(e)
            with torch.cuda.stream(copy_out):
                for o, d in zip(outs, g.outputs()):
                    o.copy_(d, non_blocking=True)
            e = ev()
            e.record(copy_out)
            ev_out[k] = e
        t1.record(copy_out)
        return t0, t1

    run(2, False)
    barrier()
    t0, t1 = run(args.e2e_steps, True)
    barrier()
    e_ms = max_over_ranks(t0.elapsed_time(t1) / args.e2e_steps, dist, dev)
    return {"value": world * spec_flops(spec) / (e_ms * 1e-3) / 1e12, "unit": "TFLOPS",
            "h2d_bytes_per_step": int(h2d_bytes), "d2h_bytes_per_step": int(d2h_bytes), "ms_per_step": e_ms,
            "steps": args.e2e_steps,
            "pipeline": "double-buffered: upload of step i+1 and readback of step i overlap step i's compute; "
                        "the average includes the first upload and the last readback"}


def max_over_ranks(value: float, dist, device=None) -> float:
    """The largest of every rank's value (the job's time is its slowest rank's)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def run_ours(args, rank: int, world: int, local_rank: int) -> None:
    import torch
    import float8_linear_layers_gb300 as fl

    spec = SPECS[args.workload]
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    host = host_inputs(spec, rank)
    host_sha = {k: sha256_of(v) for k, v in host.items()} if rank == 0 else None
    dev_in = {k: torch.from_numpy(v.view(np.int16)).view(torch.bfloat16).to(dev) for k, v in host.items()}
    step = StepGraph(fl, spec, dev, dev_in, overlap=not args.serial, scaling=args.scaling,
                     transpose=args.transpose, mx_rule=args.mx_rule)
    stream = step.main
    torch.cuda.set_stream(stream)

    def barrier():
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        step.run()
    barrier()

    # ---- timed region (device-resident inputs): every step runs after an L2
    # flush (a buffer four times the L2 rewritten on the main stream, outside
    # the step's events, so no operand is L2-resident when the step starts);
    # each step is timed by its own pair of events on the main stream, which
    # every side-stream cast joins.
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sampler = ClockSampler(dev.index if dev.index is not None else 0)
    sampler.start()
    time.sleep(0.3)
    class _GemmEvents(list):
        gemm_only = True          # the timed region brackets only the GEMMs (the roofline's launches)

    events = _GemmEvents()
    new_ev = lambda: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
    ev_step = [new_ev() for _ in range(args.steps)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier()
    t_start.record(stream)
    for i in range(args.steps):
        flush.fill_(i & 0x7F)
        ev_step[i][0].record(stream)
        step.run(events)
        ev_step[i][1].record(stream)
    t_end.record(stream)
    barrier()
    # the same number of steps back to back, no flush (run after the flushed
    # ones, so later in the GPU's clock and power history)
    u0, u1 = new_ev()
    u0.record(stream)
    for _ in range(args.steps):
        step.run()
    u1.record(stream)
    barrier()
    clocks = sampler.stop()
    flushed_ms = max_over_ranks(sum(a.elapsed_time(b) for a, b in ev_step), dist, dev)
    region_ms = max_over_ranks(t_start.elapsed_time(t_end), dist, dev)
    unflushed_ms = max_over_ranks(u0.elapsed_time(u1), dist, dev)
    assert fl.fp8lin_device_error() == 0, "a GEMM kernel reported a timed-out wait"
    # per-kernel breakdown of amax / cast from separate, fully instrumented steps
    detail = []
    for _ in range(3):
        step.run(detail)
    barrier()

    # per-kernel times from the events (each pair brackets one launch on its stream)
    kern = {"gemm": [0.0, 0], "amax": [0.0, 0], "cast": [0.0, 0], "quantize": [0.0, 0]}
    per_layer = {}
    w1_fwd_ms, w1_fwd_n = 0.0, 0
    # the roofline's launch: w1's forward GEMM where the step has one, else the linear's forward
    roof_name = "w1" if "w1" in {l.name for l in spec.linears} else spec.linears[0].name
    roof_label = roof_name + ".fwd"
    for kind, label, e0, e1, work in list(events) + [d for d in detail if d[0] != "gemm"]:
        ms = e0.elapsed_time(e1) / (3 if kind != "gemm" else 1) * (args.steps if kind != "gemm" else 1)
        kern[kind][0] += ms
        kern[kind][1] += work / 3 * args.steps if kind != "gemm" else work
        if kind == "gemm":
            pl = per_layer.setdefault(label.split(".")[0], [0.0, 0])
            pl[0] += ms
            pl[1] += work
            if label == roof_label:
                w1_fwd_ms += ms
                w1_fwd_n += 1
    gemm_evs = [(label, e0, e1) for kind, label, e0, e1, _ in events if kind == "gemm"]
    per_step = len(gemm_evs) // args.steps
    gaps = {}
    for k in range(args.steps):
        seq = gemm_evs[k * per_step:(k + 1) * per_step]
        prev = ev_step[k][0]
        for label, e0, e1 in seq:
            gaps[label] = gaps.get(label, 0.0) + prev.elapsed_time(e0) / args.steps
            prev = e1
    gemm_ms, gemm_flops = kern["gemm"]
    amax_ms, amax_bytes = kern["amax"]
    cast_ms, cast_bytes = kern["cast"]
    rw = wl.WORKLOADS[next(l.workload for l in spec.linears if l.name == roof_name)]
    w1_fwd_flops = 2 * rw.M * rw.N * rw.K

    peaks, peak_src = load_peaks()
    fp8_peak_sustained = peaks["bf16_tflops_sustained"] * FP8_PER_BF16
    fp8_peak_burst = peaks["bf16_tflops"] * FP8_PER_BF16
    # the burst peak for a timed region of under two seconds at full clock,
    # the sustained one (taken seconds into a loop under the power cap) else
    burst = region_ms < BURST_REGION_MS
    fp8_peak = fp8_peak_burst if burst else fp8_peak_sustained
    peak_kind = "burst" if burst else "sustained"
    ms_per_step = flushed_ms / args.steps
    value = world * spec_flops(spec) / (ms_per_step * 1e-3) / 1e12
    gemm_tflops = gemm_flops / (gemm_ms * 1e-3) / 1e12
    w1_fwd_tflops = w1_fwd_flops / (w1_fwd_ms / w1_fwd_n * 1e-3) / 1e12

    # ---- sustained: steps back to back for about --sustain-seconds, the last
    # --steps of them timed; under this load the GPU reaches its power cap
    # within tens of milliseconds and settles at a lower SM clock, the state a
    # training loop runs in.  Compared with the sustained peak.
    sustained = None
    if args.sustain_seconds > 0:
        n_lead = max(0, int(args.sustain_seconds / (ms_per_step * 1e-3)) - args.steps)
        sampler2 = ClockSampler(dev.index if dev.index is not None else 0)
        sampler2.start()
        time.sleep(0.3)
        barrier()
        for _ in range(n_lead):
            step.run()
        s0, s1 = new_ev()
        s0.record(stream)
        for _ in range(args.steps):
            step.run()
        s1.record(stream)
        barrier()
        clocks2 = sampler2.stop()
        s_ms = max_over_ranks(s0.elapsed_time(s1) / args.steps, dist, dev)
        s_value = world * spec_flops(spec) / (s_ms * 1e-3) / 1e12
        sustained = {"ms_per_step": s_ms, "value": s_value, "unit": "TFLOPS", "steps": args.steps,
                     "steps_before": n_lead, "pct_of_fp8_peak_sustained": 100.0 * s_value / world / fp8_peak_sustained,
                     "clocks": clocks2,
                     "note": "the last steps of about --sustain-seconds of back-to-back steps (no flush), against "
                             "the sustained peak (cuBLAS bf16 x 2 taken seconds into a loop under the power cap)"}

    graph = None
    if args.graph:
        # the same step captured once in a CUDA graph and replayed: no host
        # launch cost per kernel (what launch-bound small shapes need)
        cg = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cg, stream=stream):
            step.run()
        for _ in range(args.warmup):
            cg.replay()
        barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            cg.replay()
        g1.record(stream)
        barrier()
        g_ms = max_over_ranks(g0.elapsed_time(g1) / args.steps, dist, dev)
        graph = {"ms_per_step": g_ms, "value": world * spec_flops(spec) / (g_ms * 1e-3) / 1e12, "unit": "TFLOPS",
                 "note": "same step replayed from a captured CUDA graph"}

    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(args, fl, spec, dev, host, step, world, dist, barrier)

    cpu, parity = None, None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle on a bounded sample of the same step, timed on the host
        # cores; the sample's results are then compared with one GPU step
        import oracle
        gpu_state = step.parity_state(args.cpu_frac) if args.scaling == "dynamic" else None
        s = OracleSample(spec, args.cpu_frac)
        times = s.time_for(args.cpu_seconds)
        secs = sum(times) / len(times)
        cpu = {"value": s.flops() / secs / 1e12, "unit": "TFLOPS", "cores": oracle.num_threads(),
               "kind": "oracle", "sample": s.describe(), "sample_seconds": secs, "runs": len(times),
               "extrapolated_step_seconds": secs / args.cpu_frac}
        if gpu_state is not None:
            parity = s.check(gpu_state)
            parity["inputs_sha256_match"] = s.sha256 == host_sha
            parity["ok"] = parity["ok"] and parity["inputs_sha256_match"]

    if dist is not None:
        dist.barrier()
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOPS", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp8 (e4m3/e5m2 operands, fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": spec.name, "scaling": args.scaling + ("-ocp" if args.scaling == "mx" and
                                                                       args.mx_rule == "ocp" else ""),
                   "linears": spec.description,
                   "fp8_copies": ("row-major and transposed; backward GEMMs read the transposed copies"
                                  if step.transpose else
                                  "two row-major copies per tensor (blocks along each GEMM's contraction); "
                                  "GEMMs read them K- or MN-major" if args.scaling in ("block", "mx") else
                                  "one row-major copy per tensor; backward GEMMs read it MN-major"),
                   "l2": f"flushed: a {L2_FLUSH_BYTES >> 20} MiB buffer is rewritten on the main stream before "
                         "every timed step, outside the step's events (the step's own operands, several GB, "
                         "exceed the 129 MB L2 as well); the unflushed back-to-back time is reported beside",
                   "parallelism": f"replicas x{world}"},
        "unflushed": {"ms_per_step": unflushed_ms / args.steps,
                      "value": world * spec_flops(spec) / (unflushed_ms / args.steps * 1e-3) / 1e12,
                      "unit": "TFLOPS", "steps": args.steps,
                      "note": "the same number of steps back to back with no flush, right after the flushed "
                              "ones (later in the clock and power history: see sustained)"},
        "sustained": sustained,
        "pct_of_fp8_peak": 100.0 * value / world / fp8_peak,
        "pct_of_fp8_peak_sustained": 100.0 * value / world / fp8_peak_sustained,
        "attainable": attainable(spec, args.scaling, fp8_peak, peaks["hbm_gbs"], step.transpose),
        "fp8_peak_tflops": {"used": peak_kind, "sustained": fp8_peak_sustained, "burst": fp8_peak_burst,
                            "timed_region_ms": region_ms,
                            "source": f"{peak_src} bf16 x {FP8_PER_BF16:g} (nominal fp8:bf16); burst for a timed "
                                      f"region under {BURST_REGION_MS / 1e3:g} s, sustained otherwise"},
        "roofline": {"bound": "tensor", "achieved": gemm_tflops, "peak": fp8_peak,
                     "unit": "TFLOP/s", "frac": gemm_tflops / fp8_peak,
                     "frac_of_sustained": gemm_tflops / fp8_peak_sustained,
                     "traffic": gemm_traffic(args.workload, args.scaling),
                     "kernel": {"block": "fp8_gemm_block_kernel", "mx": "fp8_gemm_mx_kernel"}.get(
                                   args.scaling, "fp8_gemm_tn_kernel") +
                               ", every launch of the timed region: mean 2*M*N*K flop per "
                               "launch / mean event-timed launch duration (launches run beside the side-stream "
                               "casts); traffic = mean DRAM bytes per GEMM launch of one step (ncu)",
                     "peak_source": f"{peak_src} {peak_kind} bf16 x {FP8_PER_BF16:g} (nominal fp8:bf16)",
                     "launches_timed": len(gemm_evs),
                     f"{roof_label}_tflops": w1_fwd_tflops},
        "kernels": {
            "gemm": {"ms_per_step": gemm_ms / args.steps, "tflops": gemm_tflops},
            "amax": {"ms_per_step": amax_ms / args.steps,
                     "note": "amax and cast times from 3 extra fully instrumented steps; may overlap GEMMs",
                     "gbs": amax_bytes / (amax_ms * 1e-3) / 1e9 if amax_ms else None},
            "cast_transpose": {"ms_per_step": cast_ms / args.steps,
                               "gbs": cast_bytes / (cast_ms * 1e-3) / 1e9 if cast_ms else None},
            "quantize": {"ms_per_step": kern["quantize"][0] / args.steps,
                         "gbs": kern["quantize"][1] / (kern["quantize"][0] * 1e-3) / 1e9 if kern["quantize"][0]
                         else None,
                         "note": "amax + cast of the casts nothing runs beside (fp8lin_quantize), one span each"},
            "hbm_peak_gbs": peaks["hbm_gbs"],
        },
        "per_linear_gemm_tflops": {k: v[1] / (v[0] * 1e-3) / 1e12 for k, v in per_layer.items()},
        "schedule": step.describe(),
        "main_stream_idle_before_gemm_ms": {k: round(v, 4) for k, v in gaps.items()},
        "clocks": clocks,
        "graph": graph,
        "e2e": e2e,
        "gpu_launches": step.kernels_per_step * args.steps,
        "cpu_baseline": cpu,
        "parity": None if parity is None else parity["ok"],
        "parity_detail": parity if parity is not None else
        "not checked: the oracle leg runs on rank 0 of a one-GPU run with dynamic scaling",
        "inputs_sha256": host_sha,
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


# ------------------------------------------------------- profiling cases

def run_profile_case(args) -> None:
    """One kernel of the w1 linear (M 8192, K 4096, N 14336), launched
    warmup + steps times on a small device footprint, for ncu captures."""
    import torch
    import float8_linear_layers_gb300 as fl

    w = wl.WORKLOADS["llama3_8b_ffn_w13"]
    dev = torch.device("cuda", 0)
    up = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(dev)
    case = args.profile_case
    need_x = case in ("gemm_fwd", "gemm_wgrad", "gemm_wgrad_mn")
    need_w = case in ("gemm_fwd", "gemm_dgrad", "gemm_dgrad_mn")
    need_dy = case in ("gemm_dgrad", "gemm_wgrad", "gemm_dgrad_mn", "gemm_wgrad_mn", "amax", "cast", "cast_q", "quantize",
                       "amax_rowcol", "cast_rowwise", "gemm_fwd_block", "gemm_dgrad_block", "gemm_wgrad_block",
                       "cast_block", "gemm_fwd_mx", "gemm_dgrad_mx", "gemm_wgrad_mx", "cast_mx")  # dY: 235 MB > L2
    x8 = w8 = d8 = None
    if need_x:
        x = up(w.make_x())
        x8 = fl.Float8Tensor(w.M, w.K, fl.E4M3, dev).quantize(x)
    if need_w:
        x_w = up(w.make_w())
        w8 = fl.Float8Tensor(w.N, w.K, fl.E4M3, dev).quantize(x_w)
        del x_w
    if need_dy:
        dy = up(w.make_dy())
        d8 = fl.Float8Tensor(w.M, w.N, fl.E5M2, dev).quantize(dy)
    if case == "gemm_fwd":
        out = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
        launch = lambda: fl.fp8lin_fwd(x8.q, x8.inv_scale, w8.q, w8.inv_scale, out)
        work, unit = 2 * w.M * w.N * w.K, "flop"
    elif case == "gemm_dgrad":
        out = torch.empty((w.M, w.K), dtype=torch.bfloat16, device=dev)
        launch = lambda: fl.fp8lin_dgrad(d8.q, d8.inv_scale, w8.qT, w8.inv_scale, out)
        work, unit = 2 * w.M * w.N * w.K, "flop"
    elif case == "gemm_wgrad":
        out = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev)
        launch = lambda: fl.fp8lin_wgrad(d8.qT, d8.inv_scale, x8.qT, x8.inv_scale, out)
        work, unit = 2 * w.M * w.N * w.K, "flop"
    elif case in ("gemm_fwd_block", "gemm_dgrad_block", "gemm_wgrad_block", "cast_block"):
        xb = fl.Float8Tensor(w.M, w.K, fl.E4M3, dev, scaling="block", blocks="rowcol")
        wb = fl.Float8Tensor(w.N, w.K, fl.E4M3, dev, scaling="block", blocks="tile")
        db = fl.Float8Tensor(w.M, w.N, fl.E5M2, dev, scaling="block", blocks="rowcol")
        if case != "cast_block":
            xb.quantize(up(w.make_x()))
            wb.quantize(up(w.make_w()))
        db.quantize(dy)
        torch.cuda.synchronize()
        if case == "gemm_fwd_block":
            out = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
            launch = lambda: fl.fp8lin_fwd_block(xb.q, xb.row_inv, wb.q, wb.tile_inv, out)
        elif case == "gemm_dgrad_block":
            out = torch.empty((w.M, w.K), dtype=torch.bfloat16, device=dev)
            launch = lambda: fl.fp8lin_dgrad_block(db.q, db.row_inv, wb.q, wb.tile_inv, out)
        elif case == "gemm_wgrad_block":
            out = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev)
            launch = lambda: fl.fp8lin_wgrad_block(db.qc, db.col_inv, xb.qc, xb.col_inv, out)
        if case == "cast_block":
            launch = lambda: db.quantize(dy)
            work, unit = 4 * w.M * w.N, "byte"
        else:
            work, unit = 2 * w.M * w.N * w.K, "flop"
    elif case in ("gemm_fwd_mx", "gemm_dgrad_mx", "gemm_wgrad_mx", "cast_mx"):
        xm = fl.Float8Tensor(w.M, w.K, fl.E4M3, dev, scaling="mx")
        wm = fl.Float8Tensor(w.N, w.K, fl.E4M3, dev, scaling="mx")
        dm = fl.Float8Tensor(w.M, w.N, fl.E5M2, dev, scaling="mx")
        if case != "cast_mx":
            xm.quantize(up(w.make_x()))
            wm.quantize(up(w.make_w()))
        dm.quantize(dy)
        torch.cuda.synchronize()
        if case == "gemm_fwd_mx":
            out = torch.empty((w.M, w.N), dtype=torch.bfloat16, device=dev)
            launch = lambda: fl.fp8lin_fwd_mx(xm.q, xm.sf_row, wm.q, wm.sf_row, out)
        elif case == "gemm_dgrad_mx":
            out = torch.empty((w.M, w.K), dtype=torch.bfloat16, device=dev)
            launch = lambda: fl.fp8lin_dgrad_mx(dm.q, dm.sf_row, wm.qc, wm.sf_col, out)
        elif case == "gemm_wgrad_mx":
            out = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev)
            launch = lambda: fl.fp8lin_wgrad_mx(dm.qc, dm.sf_col, xm.qc, xm.sf_col, out)
        if case == "cast_mx":
            launch = lambda: dm.quantize(dy)
            work, unit = 4 * w.M * w.N, "byte"
        else:
            work, unit = 2 * w.M * w.N * w.K, "flop"
    elif case == "gemm_dgrad_mn":
        out = torch.empty((w.M, w.K), dtype=torch.bfloat16, device=dev)
        launch = lambda: fl.fp8lin_dgrad_mn(d8.q, d8.inv_scale, w8.q, w8.inv_scale, out)
        work, unit = 2 * w.M * w.N * w.K, "flop"
    elif case == "gemm_wgrad_mn":
        out = torch.empty((w.N, w.K), dtype=torch.bfloat16, device=dev)
        launch = lambda: fl.fp8lin_wgrad_mn(d8.q, d8.inv_scale, x8.q, x8.inv_scale, out)
        work, unit = 2 * w.M * w.N * w.K, "flop"
    elif case == "cast_q":
        launch = lambda: fl.fp8lin_cast_transpose(dy, fl.E5M2, d8.amax, d8.scale, d8.inv_scale, d8.q, None)
        work, unit = 3 * w.M * w.N, "byte"
    elif case == "amax":
        launch = lambda: fl.fp8lin_amax(dy, d8.amax)
        work, unit = 2 * w.M * w.N, "byte"
    elif case == "quantize":
        # the one-launch dynamic cast: amax, scale and q (2 B read + 1 B written per element, algorithmic)
        launch = lambda: fl.fp8lin_quantize(dy, fl.E5M2, d8.amax, d8.scale, d8.inv_scale, d8.q, None)
        work, unit = 3 * w.M * w.N, "byte"
    elif case == "amax_rowcol":
        ra = torch.zeros(w.M, device=dev)
        ca = torch.zeros(w.N, device=dev)
        launch = lambda: fl.fp8lin_amax_rowcol(dy, ra, ca)
        work, unit = 2 * w.M * w.N, "byte"
    elif case == "cast_rowwise":
        ra, ca = torch.zeros(w.M, device=dev), torch.zeros(w.N, device=dev)
        ri, ci = torch.zeros(w.M, device=dev), torch.zeros(w.N, device=dev)
        fl.fp8lin_amax_rowcol(dy, ra, ca)
        launch = lambda: fl.fp8lin_cast_transpose_rowwise(dy, fl.E5M2, ra, ca, ri, ci, d8.q, d8.qT)
        work, unit = 4 * w.M * w.N, "byte"
    else:
        launch = lambda: fl.fp8lin_cast_transpose(dy, fl.E5M2, d8.amax, d8.scale, d8.inv_scale, d8.q, d8.qT)
        work, unit = 4 * w.M * w.N, "byte"
    for _ in range(args.warmup):
        launch()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    ev[0].record()
    for _ in range(args.steps):
        launch()
    ev[1].record()
    torch.cuda.synchronize()
    ms = ev[0].elapsed_time(ev[1]) / args.steps
    rate = work / (ms * 1e-3) / (1e12 if unit == "flop" else 1e9)
    print(json.dumps({"profile_case": case, "ms_per_launch": ms,
                      ("tflops" if unit == "flop" else "gbs"): rate}), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(SPECS), default="ffn8b")
    ap.add_argument("--scaling", choices=["dynamic", "delayed", "rowwise", "block", "mx"], default="dynamic",
                    help="scaling recipe (the headline metric is dynamic per-tensor)")
    ap.add_argument("--mx-rule", choices=["floor", "ocp"], default="floor",
                    help="power-of-two scale rule of --scaling mx: the largest power of two not above "
                         "fmt_max / amax, or the OCP Microscaling rule")
    ap.add_argument("--serial", action="store_true", help="issue the whole step on one stream")
    ap.add_argument("--transpose", action="store_true",
                    help="casts also write the transposed FP8 copies and the backward GEMMs read those "
                         "(default: one copy per tensor, read MN-major by the backward GEMMs)")
    ap.add_argument("--graph", action="store_true", help="also time the step replayed from a CUDA graph")
    ap.add_argument("--sustain-seconds", type=float, default=1.5,
                    help="length of the back-to-back run whose last --steps steps give the sustained number "
                         "(0: skip)")
    ap.add_argument("--e2e-steps", type=int, default=32,
                    help="steps of the end-to-end run; the average includes one pipeline fill and drain")
    ap.add_argument("--cpu-frac", type=float, default=1.0 / 64,
                    help="share of the step's rows the CPU oracle runs on (cpu_baseline and --impl reference)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="cpu_baseline: repeat the oracle sample until this much CPU time has been timed")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--profile-case", choices=["gemm_fwd", "gemm_dgrad", "gemm_wgrad", "gemm_dgrad_mn",
                                               "gemm_wgrad_mn", "gemm_fwd_block", "gemm_dgrad_block",
                                               "gemm_wgrad_block", "amax", "cast", "cast_q", "cast_block",
                                               "amax_rowcol", "cast_rowwise", "gemm_fwd_mx", "gemm_dgrad_mx",
                                               "gemm_wgrad_mx", "cast_mx", "quantize"],
                    help="run one kernel of the w1 linear alone (for ncu captures)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # timing rule: at least three warm-up steps
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args, rank)
    else:
        run_ours(args, rank, world, local_rank)


if __name__ == "__main__":
    main()

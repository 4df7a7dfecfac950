"""The benchmark's JSON contract.

CPU: the reference arm (the CPU oracle on a bounded sample of the FFN step)
prints one JSON line with the fields the driver reads.
GPU: our arm prints one JSON line with metric, value, roofline, clocks,
e2e, cpu_baseline and gpu_launches."""
import json
import os
import subprocess
import sys

import pytest

from conftest import ROOT

BASE_KEYS = {"metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
             "scaling", "vs_baseline", "dtype", "data", "config", "e2e", "gpu_launches", "cpu_baseline"}


def _run(args, timeout):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT,
                         capture_output=True, text=True, timeout=timeout)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_json_line():
    import time
    t0 = time.perf_counter()
    d = _run(["--impl", "reference", "--steps", "2", "--warmup", "3", "--cpu-frac", "0.001"], 900)
    wall = time.perf_counter() - t0
    assert BASE_KEYS <= set(d) and d["impl"] == "reference"
    # each step is one run of the sample: the steps' time fits in the run
    assert d["steps"] * d["ms_per_step"] * 1e-3 < wall
    assert abs(d["extrapolated_ms_per_step"] - d["ms_per_step"] / 0.001) < 1e-6 * d["extrapolated_ms_per_step"]
    assert len(d["inputs_sha256"]) == 8 and all(len(h) == 64 for h in d["inputs_sha256"].values())
    assert d["unit"] == "TFLOPS" and d["higher_is_better"] is True and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["warmup"] >= 3 and d["config"]["workload"]


@pytest.mark.gpu
def test_our_arm_json_line(fp8lin):
    d = _run(["--steps", "3", "--warmup", "3", "--e2e-steps", "2", "--cpu-frac", "0.002", "--cpu-seconds", "0"], 900)
    assert BASE_KEYS <= set(d) and "impl" not in d
    assert d["n_gpus"] == 1 and d["steps"] == 3 and d["value"] > 0
    r = d["roofline"]
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and 0 < r["frac"] < 2
    assert abs(r["frac"] - r["achieved"] / r["peak"]) < 1e-9
    # the FFN step: 9 GEMMs, 2 one-launch casts (X and W1 together before
    # w1's forward, H before w2's) and 5 amax + cast pairs under the GEMMs
    assert d["gpu_launches"] == (9 + 2 + 2 * 5) * 3
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] > 0
    assert "sm_mhz" in d["clocks"] and "reasons" in d["clocks"]
    # the oracle leg's check of one GPU step, on inputs with the same fingerprints
    assert d["parity"] is True and d["parity_detail"]["inputs_sha256_match"] is True
    assert d["unflushed"]["value"] > 0 and "flushed" in d["config"]["l2"]
    assert d["fp8_peak_tflops"]["used"] == "burst" and r["peak"] == d["fp8_peak_tflops"]["burst"]
    # the steady state under the power cap, against the sustained peak
    su = d["sustained"]
    assert su["value"] > 0 and su["steps"] == 3 and "sm_mhz" in su["clocks"]
    assert abs(su["pct_of_fp8_peak_sustained"] - 100 * su["value"] / d["fp8_peak_tflops"]["sustained"]) < 1e-6

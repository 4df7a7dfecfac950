"""Build libfp8lin.so in-tree with nvcc for sm_103a.

Each translation unit under csrc/ compiles in parallel to an object file; the
objects link into one shared library with the CUDA runtime linked statically,
so the library needs only the NVIDIA driver at run time.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libfp8lin.so")
# A second library for the tests only: the GEMM built with a fault injector
# (its producers can withhold one slab's copies) and a 20 ms wait limit, so
# a test can drive the kernel's abort path.  The product library never has it.
FAULT_LIB = os.path.join(OUT, "libfp8lin_faultinj.so")
FAULT_FLAGS = ["-DFP8LIN_FAULT_INJECTION", "-DFP8LIN_WAIT_LIMIT_NS=20000000ull"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "-I" + INCLUDE, "-I" + CSRC]
# extra nvcc flags (e.g. -DFP8LIN_GEMM_STAGES=5 to size the GEMM's shared-memory ring)
EXTRA = os.environ.get("FP8LIN_NVCC_FLAGS", "").split()


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libfp8lin")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def up_to_date() -> bool:
    if EXTRA or not all(os.path.exists(p) for p in (LIB, FAULT_LIB)):
        return False
    t = min(os.path.getmtime(LIB), os.path.getmtime(FAULT_LIB))
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile and link libfp8lin.so; returns its path."""
    if not force and up_to_date():
        return LIB
    os.makedirs(os.path.join(OUT, "obj"), exist_ok=True)
    cc = nvcc()
    procs = []
    jobs = [(src, os.path.join(OUT, "obj", os.path.basename(src)[:-3] + ".o"), []) for src in _sources()]
    objs = [obj for _, obj, _ in jobs]
    fault_obj = os.path.join(OUT, "obj", "gemm_faultinj.o")
    jobs.append((os.path.join(CSRC, "gemm.cu"), fault_obj, FAULT_FLAGS))
    for src, obj, flags in jobs:
        cmd = [cc, *ARCH, *NVCC_FLAGS, *EXTRA, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd))
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((src, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(f"--- {s}\n{o}" for s, o in failed))
    fault_objs = [fault_obj] + [os.path.join(OUT, "obj", n) for n in ("api.o", "quantize.o")]
    for lib, lib_objs in ((LIB, objs), (FAULT_LIB, fault_objs)):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *lib_objs], check=True)
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose=True))

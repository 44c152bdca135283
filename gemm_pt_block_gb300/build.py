"""Builds libmxfp4.so in place with nvcc for sm_103a (GB300).

Each translation unit is compiled in parallel, then linked into one shared
library with a static CUDA runtime. The quantizer unit is compiled with
``--fmad=false`` (its arithmetic must not be contracted; it also uses explicit
round-to-nearest intrinsics) and nothing is built with flush-to-zero.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmxfp4.so")
# The bounds-checking build (every kernel store checked against its output's
# extent; for tests): its own objects and library.
BUILD_BC = os.path.join(HERE, "_build_bc")
LIB_BC = os.path.join(HERE, "libmxfp4_bc.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-ftz=false", "-prec-div=true",
          "-prec-sqrt=true", f"-I{os.path.join(ROOT, 'include')}", f"-I{CSRC}"]
UNITS = {
    "api.cu": [],
    "quant.cu": ["--fmad=false"],
    "gemm.cu": ["--fmad=false"],
}
HEADERS = ["internal.h", "mx_device.cuh", "ptx.cuh", "quant_device.cuh", "tma_host.h"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_v: bool = False,
          bounds_check: bool = False) -> str:
    build_dir, lib_out = (BUILD_BC, LIB_BC) if bounds_check else (BUILD, LIB)
    flags = ["-DMXFP4_BOUNDS_CHECK"] if bounds_check else []
    os.makedirs(build_dir, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(ROOT, "include", "mxfp4.h")]
    objs, jobs = [], []
    for unit, extra in UNITS.items():
        src = os.path.join(CSRC, unit)
        obj = os.path.join(build_dir, unit.replace(".cu", ".o"))
        objs.append(obj)
        if force or ptxas_v or _stale(obj, [src, __file__] + hdrs):
            cmd = [nvcc(), *ARCH, *COMMON, *flags, *extra, "-c", src, "-o", obj]
            if ptxas_v:
                cmd.insert(1, "-Xptxas=-v")
            jobs.append(cmd)

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(max_workers=len(UNITS)) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_v or r.returncode:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode:
                raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")
    if force or jobs or _stale(lib_out, objs):
        tmp = lib_out + f".{os.getpid()}.tmp"
        cmd = [nvcc(), *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("nvcc link failed")
        os.replace(tmp, lib_out)
    return lib_out


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True, ptxas_v="--ptxas-v" in sys.argv)

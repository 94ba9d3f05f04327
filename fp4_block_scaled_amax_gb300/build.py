"""Build libfp4.so in-tree with nvcc for sm_103a (no cmake, one -gencode).

    python -m fp4_block_scaled_amax_gb300.build

Translation units compile in parallel; the shared object lands next to this
file, where the binding loads it.  Rebuilds only when a source is newer.

It also builds `tc_ceiling`, a standalone program (not part of the library)
that measures the tensor cores' FLOP per clock per SM for the bf16 and FP4
MMA forms; the benchmark reports the FP4 GEMM against it.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libfp4.so")
CEILING = os.path.join(HERE, "tc_ceiling")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
          "--expt-relaxed-constexpr"]
# the quantizer's float32 steps must stay single correctly rounded operations
PER_FILE = {"quantize.cu": ["-fmad=false"], "rht.cu": ["-fmad=false"]}
SOURCES = ["abi.cu", "quantize.cu", "rht.cu", "gemv.cu", "gemv_umma.cu", "gemm_sm103.cu"]
CEILING_SOURCE = "tc_ceiling.cu"


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _deps() -> list:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "fp4.h"))
    return files


def _stale(target: str, deps: list) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build_ceiling(force: bool = False) -> str:
    """The tensor-core ceiling program (one translation unit)."""
    src = os.path.join(CSRC, CEILING_SOURCE)
    deps = [src, os.path.join(CSRC, "async_sm103.cuh")]
    if not force and not _stale(CEILING, deps):
        return CEILING
    tmp = CEILING + ".tmp"
    r = subprocess.run([_nvcc(), *ARCH, "-O3", "-std=c++17", "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr",
                        src, "-o", tmp], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {CEILING_SOURCE}:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, CEILING)
    return CEILING


def build(verbose: bool = False, force: bool = False) -> str:
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    with cf.ThreadPoolExecutor(max_workers=1) as side:
        ceiling = side.submit(build_ceiling, force)
        lib = _build_lib(nvcc, verbose, force)
        ceiling.result()
    return lib


def _build_lib(nvcc: str, verbose: bool, force: bool) -> str:
    deps = [d for d in _deps() if not d.endswith(CEILING_SOURCE)]
    if not force and not _stale(LIB, deps):
        return LIB

    def compile_one(src: str) -> str:
        obj = os.path.join(BUILD, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *COMMON, *PER_FILE.get(src, []), "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB + ".tmp"
    r = subprocess.run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))

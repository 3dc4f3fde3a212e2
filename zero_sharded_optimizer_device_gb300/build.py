"""Build libzero.so in-tree with nvcc for sm_103a (GB300).

Translation units compile in parallel to objects under ``_build/`` and link
into ``zero_sharded_optimizer_device_gb300/libzero.so`` against the shared CUDA
runtime (the same libcudart PyTorch loads).
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libzero.so")
# Same sources with -DZERO_CHECKED: every kernel access tested against its
# buffer's extent and recorded when outside (zero_bounds_report in zero.h).
LIB_CHECKED = os.path.join(HERE, "libzero_checked.so")

SOURCES = ["zero_plan.cpp", "zero_api.cpp", "zero_sched.cpp", "zero_rs.cu", "zero_kernels.cu",
           "zero_noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-I", INCLUDE, "-I", CSRC,
          "-Xcompiler", "-fPIC,-ffp-contract=off,-O2"]


def nvcc() -> str:
    env = os.environ.get("NVCC")
    if env:
        return env
    cand = "/usr/local/cuda/bin/nvcc"
    return cand if os.path.exists(cand) else "nvcc"


def _compile(src: str, extra: list[str], outdir: str = BUILD) -> str:
    obj = os.path.join(outdir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *COMMON, *ARCH, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if src.endswith(".cpp"):
        cmd[cmd.index("-c"):cmd.index("-c")] = ["-x", "cu"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip() and "-Xptxas" in " ".join(extra):
        sys.stderr.write(r.stderr)
    return obj


def build(verbose: bool = False, ptxas_info: bool = False, checked: bool = False) -> str:
    """Compile and link libzero.so, or with ``checked`` libzero_checked.so."""
    outdir = os.path.join(BUILD, "checked") if checked else BUILD
    lib = LIB_CHECKED if checked else LIB
    os.makedirs(outdir, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    if checked:
        extra.append("-DZERO_CHECKED")
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, outdir), SOURCES))
    cmd = [nvcc(), "-shared", "-cudart", "shared", *ARCH, "-o", lib, *objs,
           "-Xlinker", "-rpath,/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose:
        print(f"built {lib}")
    return lib


if __name__ == "__main__":
    build(verbose=True, ptxas_info="-v" in sys.argv, checked="--checked" in sys.argv)

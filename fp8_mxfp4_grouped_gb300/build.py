"""Build libhg.so in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` is compiled in parallel, then linked
into ``fp8_mxfp4_grouped_gb300/libhg.so`` (static CUDA runtime, no libcuda
link: the TMA encoder is fetched through the runtime's driver entry point).

    python -m fp8_mxfp4_grouped_gb300.build [--verbose-ptxas]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD_DIR = os.path.join(os.path.dirname(HERE), "_build")
LIB_PATH = os.path.join(HERE, "libhg.so")
SOURCES = ["api.cu", "plan.cu", "gemm.cu", "moe_io.cu", "plan_noalloc.cu", "gemm_host.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    proc = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if proc.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + proc.stdout)
    return proc.stdout


def build(verbose_ptxas: bool = False, extra_flags=None) -> str:
    """Compile and link; returns the path of the shared library."""
    nvcc = _nvcc()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = list(extra_flags or [])
    if verbose_ptxas:
        extra += ["-Xptxas", "-v"]
    jobs = []
    for src in SOURCES:
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        jobs.append((obj, [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]))
    logs = []
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        for out in ex.map(lambda j: _run(j[1]), jobs):
            logs.append(out)
    tmp = LIB_PATH + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[j[0] for j in jobs]])
    os.replace(tmp, LIB_PATH)
    if verbose_ptxas:
        sys.stdout.write("".join(logs))
    return LIB_PATH


if __name__ == "__main__":
    build(verbose_ptxas="--verbose-ptxas" in sys.argv)
    print(LIB_PATH)

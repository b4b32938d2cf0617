"""Compile the CUDA library (libmoe_gb300.so) in-tree for sm_103a with nvcc.

Each translation unit is compiled in parallel, then linked with the static CUDA runtime so
the library loads on machines without a GPU (the driver is opened only when a call runs).
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
LIB = os.path.join(BUILD, "libmoe_gb300.so")
SOURCES = ["api.cu", "router.cu", "route_small.cu", "dispatch.cu", "experts.cu", "gemm.cu", "stream.cu", "decode.cu",
           "noalloc.cu", "stats.cu", "host_experts.cu", "host_io.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_gb300.so")


def _deps_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(HERE, "..", "include", "moe.h"))
    paths.append(os.path.abspath(__file__))
    return max(os.path.getmtime(p) for p in paths)


LIB_TIMELINE = os.path.join(BUILD, "libmoe_gb300_timeline.so")


def build(force: bool = False, verbose: bool = False, timeline: bool = False) -> str:
    """Build the library if any source is newer than it; return its path. timeline=True builds
    the variant whose one-token kernel records its in-kernel timeline (MOE_TIMELINE), for
    `python -m sparse_moe_ffn_router_gb300.timeline`."""
    os.makedirs(BUILD, exist_ok=True)
    lib = LIB_TIMELINE if timeline else LIB
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _deps_mtime():
        return lib
    nvcc = _nvcc()
    extra = ["-DMOE_TIMELINE"] if timeline else []
    suffix = "_tl.o" if timeline else ".o"

    def compile_one(src: str):
        obj = os.path.join(BUILD, src.replace(".cu", suffix))
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    with open(os.path.join(BUILD, "ptxas_timeline.log" if timeline else "ptxas.log"), "w") as f:
        for (_, log), src in zip(results, SOURCES):
            f.write(f"==== {src}\n{log}\n")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(f"built {lib}", file=sys.stderr)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

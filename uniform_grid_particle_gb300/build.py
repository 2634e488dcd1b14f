"""Build libugrid.so in-tree for sm_103a with nvcc (no cmake, no torch extension).

Each .cu file is compiled on its own (in parallel) and the objects are linked
into ``uniform_grid_particle_gb300/libugrid.so`` against the shared CUDA
runtime, so the library and PyTorch share one runtime in a process.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build")
LIBRARY = os.path.join(PKG, "libugrid.so")

SOURCES = ["abi.cu", "build_fused.cu", "build_bucketed.cu", "build_small.cu", "build_cluster.cu", "build_sparse.cu", "count.cu", "scan.cu", "scatter.cu", "reorder.cu", "segsort.cu",
           "scan_noalloc.cu", "diagnostics.cu", "reorder_many.cu",
           "density.cu"]
HEADERS = [os.path.join(CSRC, "ugrid_internal.cuh"), os.path.join(CSRC, "segsort_device.cuh"),
           os.path.join(CSRC, "fused_common.cuh"),
           os.path.join(INCLUDE, "ugrid.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    found = shutil.which("nvcc")
    if found:
        return found
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    return os.path.join(home, "bin", "nvcc")


def cuda_lib_dir() -> str:
    return os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc()))), "lib64")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, extra: list[str], verbose: bool) -> str:
    obj = os.path.join(OBJDIR, os.path.splitext(os.path.basename(src))[0] + ".o")
    cmd = [nvcc(), *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stderr}")
    if verbose and res.stderr:
        print(res.stderr, end="")
    return obj


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None) -> str:
    """Compile every .cu of the package and link libugrid.so; returns its path."""
    sources = [os.path.join(CSRC, s) for s in SOURCES]
    if not force and not extra_flags and not _stale(LIBRARY, sources + HEADERS + [__file__]):
        return LIBRARY
    os.makedirs(OBJDIR, exist_ok=True)
    extra = list(extra_flags or [])
    with cf.ThreadPoolExecutor(max_workers=len(sources)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose), sources))
    tmp = LIBRARY + ".tmp"
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath=" + cuda_lib_dir()]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    import sys

    print(build(force=True, verbose=True, extra_flags=sys.argv[1:]))

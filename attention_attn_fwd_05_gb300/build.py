"""Build the CUDA library in-tree: ``_build/libattn_gb300.so`` for sm_103a.

Each translation unit is compiled by its own nvcc process (in parallel), then
linked into one shared library against the shared CUDA runtime, so the
library and PyTorch use the same runtime instance.  Nothing is installed into
site-packages.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libattn_gb300.so")
# The bounds-checking debug build: the same sources compiled with
# -DATTN_DEBUG_BOUNDS into a library of its own, so it can never be loaded in
# place of the normal one by accident.
BUILD_BOUNDS = os.path.join(PKG, "_build_bounds")
LIB_BOUNDS = os.path.join(BUILD_BOUNDS, "libattn_gb300_bounds.so")
SOURCES = ["attn_api.cu", "attn_fwd_tc.cu", "attn_fwd_f32.cu", "row_softmax.cu",
           "attn_noalloc.cu", "add_rmsnorm.cu", "attn_bwd.cu", "attn_bwd_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-cudart", "shared",
              "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else (shutil.which("nvcc") or "nvcc")


def _inputs_mtime() -> float:
    paths = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    paths.append(os.path.join(os.path.dirname(PKG), "include", "attn_fwd.h"))
    return max(os.path.getmtime(p) for p in paths)


def build(force: bool = False, verbose: bool = False, bounds_checks: bool = False) -> str:
    """Compile and link the library if any source is newer than it; return its
    path.  ``bounds_checks`` builds the debug variant instead (every global
    index and TMA coordinate of the forward kernels checked before use, a
    failure recorded in the device status word)."""
    build_dir, lib = (BUILD_BOUNDS, LIB_BOUNDS) if bounds_checks else (BUILD, LIB)
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _inputs_mtime():
        return lib
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    extra = ["-DATTN_DEBUG_BOUNDS"] if bounds_checks else []

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    cuda_lib = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "lib64")
    tmp = lib + f".{os.getpid()}.tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs,
           f"-Xlinker=-rpath,{cuda_lib}"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force=True, verbose=True))

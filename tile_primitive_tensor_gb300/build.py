"""Build libtpgemm.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel to an object file under
``_build/`` and linked into ``_lib/libtpgemm.so`` (CUDA runtime linked
statically; the driver's tensor-map encoder is fetched at run time, so no
libcuda link is needed and the library loads on machines without a GPU).
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libtpgemm.so")
# The debug build (-DTPGEMM_DEBUG): device-side bounds checks that report
# TPGEMM_ERR_BOUNDS and skip the access. Built on request only.
BUILD_DIR_DEBUG = os.path.join(HERE, "_build_debug")
LIB_PATH_DEBUG = os.path.join(LIB_DIR, "libtpgemm_debug.so")
SOURCES = ["tpgemm_api.cu", "tc_gemm.cu", "mma_sync_gemm.cu", "tmem_copy.cu", "vec_copy.cu",
           "mx_scales.cu"]
HEADERS = ["ptx.cuh", "tpgemm_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False,
          debug: bool = False) -> str:
    """Compile and link the library (or, with debug, libtpgemm_debug.so) if any
    source changed; return its path."""
    nvcc = _nvcc()
    build_dir = BUILD_DIR_DEBUG if debug else BUILD_DIR
    lib_path = LIB_PATH_DEBUG if debug else LIB_PATH
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    headers = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "tpgemm.h")]
    flags = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                    "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr"]
    if debug:
        flags += ["-DTPGEMM_DEBUG"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]

    def compile_one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        if force or ptxas_verbose or _stale(o, [s] + headers):
            cmd = [nvcc] + flags + ["-c", s, "-o", o]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose or ptxas_verbose:
                sys.stderr.write(r.stdout + r.stderr)
        return o

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    if force or _stale(lib_path, objs):
        tmp = lib_path + f".tmp{os.getpid()}"
        cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                ptxas_verbose="--ptxas-verbose" in sys.argv, debug="--debug" in sys.argv))

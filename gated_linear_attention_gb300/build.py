"""Build step of the CUDA library: nvcc, sm_103a only, objects compiled in parallel.

``python -m gated_linear_attention_gb300.build`` (or ``build()``) writes
``gated_linear_attention_gb300/_build/libsala_gla.so``; ``build(debug=True)`` writes the debug
build ``_build_debug/libsala_gla_debug.so`` (compiled with ``SALA_GLA_DEBUG``: device code checks
the indices it derives from the inputs and records SALA_ERR_DEBUG_CHECK instead of making a
bad access), which the binding loads when the environment sets ``SALA_GLA_DEBUG=1``. The CUDA runtime is linked
statically, so the library loads on a machine without a GPU (its entry points then return
SALA_ERR_CUDA); the driver's tensor-map encoder is fetched at run time through the runtime's
driver entry-point query, so libcuda is not a link dependency either.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libsala_gla.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(BUILD_DEBUG, "libsala_gla_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) +
            glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h")))


def up_to_date(debug: bool = False) -> bool:
    lib = LIB_DEBUG if debug else LIB
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(), debug: bool = False) -> str:
    """Compile every ``csrc/*.cu`` for sm_103a and link ``libsala_gla.so`` (or, with
    ``debug``, ``libsala_gla_debug.so`` with the device-side index checks)."""
    lib, bdir = (LIB_DEBUG, BUILD_DEBUG) if debug else (LIB, BUILD)
    if debug:
        extra_flags = ("-DSALA_GLA_DEBUG", *extra_flags)
    if not force and up_to_date(debug):
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    srcs = _sources()

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as pool:
        objs = list(pool.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs, "-lpthread", "-ldl",
           "-lrt"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, extra_flags=[
        "-Xptxas", "-v"] if "--ptxas-v" in sys.argv else [], debug="--debug" in sys.argv))

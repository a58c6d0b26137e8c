"""Build the CUDA library ``libsage_gb300.so`` in-tree for sm_103a.

Each ``csrc/*.cu`` is compiled on its own (in parallel) with
``nvcc -gencode arch=compute_103a,code=sm_103a -O3 -lineinfo`` and the objects
are linked into ``_build/libsage_gb300.so``.  ``-Xptxas -v`` output (registers,
spills, shared memory) is kept in ``_build/ptxas.log``.

``build(debug_bounds=True)`` compiles the same sources with
``-DSAGE_DEBUG_BOUNDS`` into ``_build/debug/libsage_gb300_debug.so``: every
global access whose index a kernel computes is checked against its tensor's
extent, skipped when outside, and the first such site is recorded for
``sage_debug_bounds`` (the stand-in for a memory sanitizer).
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libsage_gb300.so")
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "libsage_gb300_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libsage_gb300.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile every kernel file for sm_103a and link the shared library
    (the bounds-checking debug library with ``debug_bounds=True``)."""
    out_dir, lib = (DEBUG_BUILD, DEBUG_LIB) if debug_bounds else (BUILD, LIB)
    if not force and not stale(lib):
        return lib
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                    "-Xptxas", "-v", "--expt-relaxed-constexpr"]
    if debug_bounds:
        flags.append("-DSAGE_DEBUG_BOUNDS")

    def compile_one(src):
        obj = os.path.join(out_dir, os.path.basename(src) + ".o")
        cmd = [nvcc] + flags + ["-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(compile_one, srcs))
    with open(os.path.join(out_dir, "ptxas.log"), "w") as f:
        for (obj, log), src in zip(results, srcs):
            f.write(f"==== {os.path.basename(src)}\n{log}\n")
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + [o for o, _ in results]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    if verbose:
        print(open(os.path.join(out_dir, "ptxas.log")).read())
    return lib


if __name__ == "__main__":
    build(force=True, verbose=True)

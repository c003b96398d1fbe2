"""In-tree build of libuniprefill.so (sm_103a) with nvcc; no cmake, translation units in parallel."""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIB = os.path.join(PKG, "libuniprefill.so")
# the bounds-checked build (-DUP_DEBUG_BOUNDS): every kernel range-checks its global indices and reports
# a violation in the status word; a development aid, not loaded by the package
DEBUG_LIB = os.path.join(PKG, "libuniprefill_debug.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["up_score.cu", "up_select.cu", "up_compact.cu", "up_meta.cu"]


def nvcc():
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libuniprefill")
    return exe


def _stale(out, deps):
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose=False, force=False, ptxas_verbose=False, debug_bounds=False):
    """Compile every translation unit for sm_103a and link the shared library; returns its path.
    debug_bounds=True builds the bounds-checked variant (libuniprefill_debug.so) instead."""
    deps_common = [os.path.join(CSRC, "up_internal.cuh"),
                   os.path.join(os.path.dirname(PKG), "include", "uniprefill.h"), __file__]
    objdir = os.path.join(PKG, "_build", "debug" if debug_bounds else "")
    os.makedirs(objdir, exist_ok=True)
    lib = DEBUG_LIB if debug_bounds else LIB
    flags = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr"]
    if debug_bounds:
        flags += ["-DUP_DEBUG_BOUNDS"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]

    def one(src):
        s = os.path.join(CSRC, src)
        o = os.path.join(objdir, src.replace(".cu", ".o"))
        if force or _stale(o, [s] + deps_common):
            cmd = [nvcc()] + flags + ["-c", s, "-o", o]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
            if verbose or ptxas_verbose:
                sys.stderr.write(r.stderr)
        return o

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(one, SOURCES))
    if force or _stale(lib, objs):
        tmp = lib + ".tmp"
        cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True, force="--force" in sys.argv, ptxas_verbose="-v" in sys.argv,
                debug_bounds="--debug-bounds" in sys.argv))

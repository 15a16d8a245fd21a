"""Builds libdiffattn.so in-tree with nvcc for sm_103a (no CMake).

Each .cu file under csrc/ compiles to an object in parallel; the objects link
into differential_attention_02_gb300/libdiffattn.so. Rebuilds only what is
older than its source or any header.

build(debug=True) makes libdiffattn_debug.so instead (objects in _build_debug/):
the same kernels compiled with DIFFATTN_DEBUG_CHECKS, whose device-side index
checks of TMA coordinates, paged block-table entries and split ranges record a
code in the error word (kind 2) instead of passing silently. Point the binding
at it with the DIFFATTN_LIBRARY environment variable.
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libdiffattn.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libdiffattn_debug.so")
SOURCES = ["api.cu", "fwd_simt_f32.cu", "decode_bf16.cu", "gemm_tcgen05.cu", "fwd_tcgen05.cu",
           "fwd_pair_tcgen05.cu", "layer_ops.cu", "bwd_simt.cu", "bwd_tcgen05.cu",
           "selftest.cu"]
HEADERS = [os.path.join(CSRC, "common.cuh"), os.path.join(CSRC, "kernels.h"),
           os.path.join(ROOT, "include", "diffattn.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(ptxas_verbose: bool, debug: bool = False):
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", CSRC,
                "-I", os.path.join(ROOT, "include")]
    if ptxas_verbose:
        f += ["-Xptxas", "-v"]
    if debug:
        f += ["-DDIFFATTN_DEBUG_CHECKS"]
    return f


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, debug: bool = False) -> str:
    """Compiles what is out of date and returns the path of the library
    (libdiffattn.so, or libdiffattn_debug.so with debug=True)."""
    bdir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug else (BUILD, LIB)
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + HEADERS):
            jobs.append([cc] + _flags(ptxas_verbose, debug) + ["-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        return cmd, r

    with ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        for cmd, r in ex.map(run, jobs):
            if verbose or ptxas_verbose or r.returncode:
                sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
            if r.returncode:
                raise RuntimeError(f"nvcc failed on {cmd[-3]}")
    if force or jobs or _stale(lib, objs):
        cmd = [cc] + ARCH + ["-shared", "-o", lib] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode:
            raise RuntimeError("link failed:\n" + r.stdout + r.stderr)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))

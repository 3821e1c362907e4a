"""Builds ``libconvfused.so`` in-tree with nvcc for sm_103a (tcgen05 needs the
architecture-specific ``compute_103a`` target).  Translation units compile in parallel;
the tcgen05 kernel is compiled once per tile width.

``build(debug_bounds=True)`` builds ``libconvfused_bounds.so`` instead (its own object folder):
the same sources with ``-DCONVF_DEBUG_BOUNDS``, whose kernels check every hand-computed global
index against the tensor their parameters describe and report a violation through the status
word (CONVF_ERR_BOUNDS) instead of making the access.  It is a testing aid: the environment
variable ``CONVF_DEBUG_BOUNDS=1`` makes the binding load it."""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIB_DIR, "libconvfused.so")
BUILD_DIR_BOUNDS = os.path.join(PKG, "_build", "bounds")
LIB_BOUNDS = os.path.join(LIB_DIR, "libconvfused_bounds.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-I", os.path.join(ROOT, "include"), "-I", CSRC]

UNITS = [("api.cu", []), ("k_depthwise.cu", []), ("k_int8.cu", []), ("k_watchdog.cu", []), ("k_pad.cu", []),
         ("tc_window.cu", []), ("tc_halo.cu", []), ("k_mbblock.cu", []), ("chain.cu", []),
         ("tc_chain.cu", [])] + [
    ("tc_conv_inst.cu", [f"-DCONVF_BN={bn}"]) for bn in (32, 64, 128, 256)]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    hdr = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [
        os.path.join(ROOT, "include", "conv_fused.h"), os.path.abspath(__file__)]
    return hdr


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(s) > t for s in _sources())


def build(force: bool = False, verbose: bool = False, extra_flags=None, debug_bounds: bool = False) -> str:
    """Compile (if needed) and return the path of the shared library (the bounds-checking one
    with ``debug_bounds``)."""
    lib = LIB_BOUNDS if debug_bounds else LIB
    build_dir = BUILD_DIR_BOUNDS if debug_bounds else BUILD_DIR
    if not force and not _stale(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    extra = list(extra_flags or []) + (["-DCONVF_DEBUG_BOUNDS"] if debug_bounds else [])

    def compile_unit(unit):
        src, defs = unit
        tag = src.replace(".cu", "") + "".join(d.split("=")[-1] for d in defs)
        obj = os.path.join(build_dir, tag + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, *defs, "-c", os.path.join(CSRC, src), "-o", obj]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} {defs}:\n{res.stderr}")
        if verbose and res.stderr.strip():
            print(res.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_unit, UNITS))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs, "-lcuda"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        # the driver library is resolved at run time through the runtime's entry-point query;
        # link without it if the stub is not on the linker path
        cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError("link failed:\n" + res.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None))

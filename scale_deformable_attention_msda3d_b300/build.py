"""Builds libmsda.so in-tree with nvcc for sm_103a (B300).

    python -m scale_deformable_attention_msda3d_b300.build [--force] [--debug-bounds]

Objects go to ``_build/`` next to this file; the shared library is written next to this
file as ``libmsda.so``.  Sources are compiled in parallel, then linked with the static
CUDA runtime so that loading the library needs no GPU.  ``--debug-bounds`` (or
build(debug=True)) compiles the same sources with MSDA_DEBUG_BOUNDS into ``_build_debug/``
and ``libmsda_debug.so``: every corner row index is checked before its access and the
first offender recorded (include/msda.h, bounds-checking build).
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from typing import List

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmsda.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libmsda_debug.so")
PROBES_SRC = os.path.join(CSRC, "probes", "msda_probes.cu")
LIB_PROBES = os.path.join(PKG, "libmsda_probes.so")
HEADERS = [os.path.join(ROOT, "include", "msda.h")]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "--expt-relaxed-constexpr", "-I" + os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: cannot build libmsda")


def sources() -> List[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                  if f.endswith((".cu", ".cpp")))


def _inputs() -> List[str]:
    return sources() + HEADERS + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                                  if f.endswith((".cuh", ".h"))] + [os.path.abspath(__file__)]


def is_stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags: List[str] = (),
          debug: bool = False) -> str:
    """Build libmsda.so (debug=True: libmsda_debug.so with the bounds checks)."""
    lib_out = LIB_DEBUG if debug else LIB
    build_dir = BUILD_DEBUG if debug else BUILD
    if debug:
        extra_flags = [*extra_flags, "-DMSDA_DEBUG_BOUNDS"]
    if not force and not is_stale(lib_out):
        return lib_out
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()

    def compile_one(src: str) -> str:
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib_out + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, lib_out)
    return lib_out


def build_probes(force: bool = False) -> str:
    """Build libmsda_probes.so, the on-chip rate microbenchmarks that bench.py --probe runs
    (not part of libmsda)."""
    if (not force and os.path.exists(LIB_PROBES)
            and os.path.getmtime(LIB_PROBES) >= os.path.getmtime(PROBES_SRC)):
        return LIB_PROBES
    tmp = LIB_PROBES + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
           "-cudart", "static", "-o", tmp, PROBES_SRC]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on msda_probes.cu:\n{r.stdout}{r.stderr}")
    os.replace(tmp, LIB_PROBES)
    return LIB_PROBES


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true")
    ap.add_argument("--ptxas-info", action="store_true",
                    help="print registers / spills / shared memory per kernel")
    ap.add_argument("--debug-bounds", action="store_true",
                    help="build libmsda_debug.so (corner row indices checked before access)")
    a = ap.parse_args(argv)
    extra = ["-Xptxas", "-v"] if a.ptxas_info else []
    print(build(force=a.force or a.ptxas_info, verbose=a.verbose or a.ptxas_info,
                extra_flags=extra, debug=a.debug_bounds))
    return 0


if __name__ == "__main__":
    sys.exit(main())

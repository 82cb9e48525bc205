"""Builds libvce.so in-tree with nvcc for sm_103a (GB300).

    python -m vocabulary_cross_entropy_gb300.build [-v] [-f] [--bounds-check]

Each translation unit is compiled in parallel to an object file under
``_build/`` next to this file, then linked into ``libvce.so`` beside the
package's Python sources.  The CUDA runtime is linked statically; the driver
entry point for tensor-map encoding is resolved at run time through the
runtime, so no libcuda link is needed at build time.

``build_bounds_check()`` (``--bounds-check``) makes the debugging variant
``libvce_bounds.so`` with -DVCE_BOUNDS_CHECK: every kernel checks the
addresses it computes and reports VCE_DEVSTATUS_BOUNDS instead of making an
access that fails a check.  A process selects it by setting VCE_LIBRARY to
its path before the package loads the library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libvce.so")
BOUNDS_BUILD = os.path.join(HERE, "_build_bounds")
BOUNDS_LIB = os.path.join(HERE, "libvce_bounds.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
         "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)) + [os.path.join(INCLUDE, "vce.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(verbose: bool = False, force: bool = False, extra_flags=(), lib: str = LIB,
          build_dir: str = BUILD) -> str:
    if not force and up_to_date(lib):
        return lib
    nvcc = _nvcc()
    os.makedirs(build_dir, exist_ok=True)
    srcs = sources()

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, flush=True)
        return obj

    with ThreadPoolExecutor(max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


def build_bounds_check(verbose: bool = False, force: bool = False) -> str:
    """The debugging variant with every kernel's address checks compiled in."""
    return build(verbose, force, ("-DVCE_BOUNDS_CHECK",), BOUNDS_LIB, BOUNDS_BUILD)


if __name__ == "__main__":
    v = "-v" in sys.argv
    if "--bounds-check" in sys.argv:
        print(build_bounds_check(verbose=v, force="-f" in sys.argv))
    else:
        print(build(verbose=v, force="-f" in sys.argv))

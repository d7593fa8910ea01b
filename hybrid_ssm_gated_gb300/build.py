"""Build the CUDA library (libgdn.so) for sm_103a with nvcc.

Each translation unit under csrc/ compiles in parallel; the objects are
linked into hybrid_ssm_gated_gb300/lib/libgdn.so against the shared CUDA
runtime. Rebuilds only when a source or header is newer than the library.
build(debug=True) builds the bounds-checking variant (GDN_DEBUG_BOUNDS: every
global copy and store checked against its array) into lib/debug/libgdn.so.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
LIBDIR = os.path.join(HERE, "lib")
LIB = os.path.join(LIBDIR, "libgdn.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "--expt-relaxed-constexpr",
                     "-I", INCLUDE]


def nvcc() -> str:
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libgdn.so")
    return path


def sources() -> list[str]:
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps() -> list[str]:
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        [os.path.join(INCLUDE, "gdn.h"), __file__]


def _paths(debug: bool) -> tuple[str, str]:
    """(library, object directory) of the normal or the bounds-checking build."""
    d = os.path.join(LIBDIR, "debug") if debug else LIBDIR
    return os.path.join(d, "libgdn.so"), os.path.join(d, "obj")


def _compile(src: str, extra: list[str], objdir: str) -> str:
    obj = os.path.join(objdir, os.path.basename(src) + ".o")
    os.makedirs(os.path.dirname(obj), exist_ok=True)
    if os.path.exists(obj) and os.path.getmtime(obj) >= max(os.path.getmtime(d) for d in _deps()):
        return obj
    cmd = [nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if r.stderr.strip():
        sys.stderr.write(r.stderr)
    os.replace(obj + ".tmp", obj)
    return obj


def build(force: bool = False, verbose_ptxas: bool = False, debug: bool = False) -> str:
    """Compile and link libgdn.so (debug: the bounds-checking build); returns its path."""
    lib, objdir = _paths(debug)
    os.makedirs(objdir, exist_ok=True)
    newest = max(os.path.getmtime(d) for d in _deps())
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= newest:
        return lib
    if force:
        shutil.rmtree(objdir, ignore_errors=True)
        os.makedirs(objdir, exist_ok=True)
    extra = (["-Xptxas", "-v"] if verbose_ptxas else []) + (["-DGDN_DEBUG_BOUNDS"] if debug else [])
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, objdir), sources()))
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "shared", "-o", lib + ".tmp"] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose_ptxas="-v" in sys.argv))

"""Build libgcl.so in-tree with nvcc for sm_103a (no cmake, no torch extension machinery).

Each .cu file is compiled in parallel to an object, then linked into a shared
library next to this file.  A file is recompiled when it or any header is newer
than its object.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(PKG, "_build", platform.machine())   # objects are per host arch
LIB = os.path.join(PKG, "libgcl.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hs), default=0.0)


def _compile(src: str, extra: list[str], verbose: bool, objdir: str = OBJDIR) -> str:
    obj = os.path.join(objdir, os.path.basename(src) + ".o")
    if (os.path.exists(obj) and os.path.getmtime(obj) >= os.path.getmtime(src)
            and os.path.getmtime(obj) >= _headers_mtime()):
        return obj
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return obj


DEBUG_LIB = os.path.join(PKG, "libgcl_debug.so")
DEBUG_FLAGS = ["-DGCL_DEBUG_BOUNDS"]


def build(verbose: bool = False, extra: list[str] | None = None, jobs: int | None = None,
          debug: bool = False) -> str:
    """Compile every csrc/*.cu and link libgcl.so; returns the library path.  debug=True builds
    libgcl_debug.so instead, with every checked index tested against its buffer
    (GCL_DEBUG_BOUNDS: an index outside records GCL_DEV_OUT_OF_BOUNDS and the access is
    skipped), in objects of its own."""
    objdir = OBJDIR + ("-debug" if debug else "")
    lib = DEBUG_LIB if debug else LIB
    os.makedirs(objdir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    extra = list(extra or []) + (DEBUG_FLAGS if debug else [])
    with cf.ThreadPoolExecutor(max_workers=jobs or min(8, len(srcs))) as ex:
        objs = list(ex.map(lambda s: _compile(s, extra, verbose, objdir), srcs))
    if (not os.path.exists(lib)
            or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs)):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(verbose=True))

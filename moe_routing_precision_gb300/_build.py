"""Build the in-tree CUDA library ``libmoe_route.so`` for sm_103a.

Each ``csrc/*.cu`` file is compiled by nvcc in parallel, then linked into one
shared library beside this file (shared CUDA runtime, so the process shares
the runtime PyTorch already loaded).  No torch extension machinery is used:
the library exposes a plain C ABI (``include/moe_route.h``).

The debug-bounds library ``libmoe_route_debug.so`` is the same sources with
``MOE_DEBUG_BOUNDS`` defined (the kernels' internal index and alignment
checks compiled in).  ``build()`` makes it instead of the normal library when
asked to, or when the environment variable ``MOE_DEBUG_BOUNDS`` is ``1``;
the binding then loads it (see ``lib_path``).
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_NAME = "libmoe_route.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
BUILD_DIR = os.path.join(PKG, "_build")
DEBUG_LIB_PATH = os.path.join(PKG, "libmoe_route_debug.so")
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", f"-I{INCLUDE}", f"-I{CSRC}"]


def nvcc_path() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmoe_route.so")
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def debug_bounds_requested() -> bool:
    """True when the environment asks for the debug-bounds library."""
    return os.environ.get("MOE_DEBUG_BOUNDS", "0") == "1"


def lib_path(debug_bounds: bool | None = None) -> str:
    """The library the binding loads: the debug-bounds one if requested."""
    if debug_bounds is None:
        debug_bounds = debug_bounds_requested()
    return DEBUG_LIB_PATH if debug_bounds else LIB_PATH


def is_stale(debug_bounds: bool = False) -> bool:
    path = lib_path(debug_bounds)
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(p) > t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags: list[str] | None = None,
          debug_bounds: bool | None = None) -> str:
    """Compile and link the library if any source is newer; return its path.
    debug_bounds: build libmoe_route_debug.so (None: as MOE_DEBUG_BOUNDS says)."""
    if debug_bounds is None:
        debug_bounds = debug_bounds_requested()
    out_path = lib_path(debug_bounds)
    if not force and not is_stale(debug_bounds):
        return out_path
    nvcc = nvcc_path()
    build_dir = DEBUG_BUILD_DIR if debug_bounds else BUILD_DIR
    os.makedirs(build_dir, exist_ok=True)
    flags = NVCC_FLAGS + (["-DMOE_DEBUG_BOUNDS=1"] if debug_bounds else []) + (extra_flags or [])

    def compile_one(src):
        obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout, r.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, _sources()))
    tmp = out_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, out_path)
    return out_path


if __name__ == "__main__":  # pragma: no cover
    import sys
    print(build(force="--force" in sys.argv, verbose=True))

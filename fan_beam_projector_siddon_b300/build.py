"""Build ``libctproj.so`` in-tree with nvcc for sm_103a (no JIT cache, no torch extension)."""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libctproj.so")
# Bounds-checking build (-DCT_DEBUG_BOUNDS): every data-dependent index is checked on the device
# and counted instead of used when out of range; for tests, not for timing.
LIB_BOUNDS = os.path.join(PKG, "libctproj_bounds.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
    "-Xptxas", "-v",
]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _stale(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(p) > t for p in deps)


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    lib = LIB_BOUNDS if debug_bounds else LIB
    if not force and not _stale(lib):
        return lib
    nvcc = os.environ.get("NVCC", "nvcc")
    tmp = lib + f".tmp{os.getpid()}"
    extra = ["-DCT_DEBUG_BOUNDS"] if debug_bounds else []
    cmd = [nvcc, *NVCC_FLAGS, *extra, "-shared", "-I", INCLUDE, "-I", CSRC, "-o", tmp, *sources()]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        sys.stderr.write(res.stdout + res.stderr)
        raise RuntimeError(f"nvcc failed building {os.path.basename(lib)}")
    if verbose:
        sys.stderr.write(res.stderr)
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)

"""Build libmoe_fp8.so in-tree with nvcc for sm_103a (GB300).

Each translation unit compiles in parallel to an object under ``_build/``;
the objects link into ``fp8_block_scale_gb300/libmoe_fp8.so``.  Nothing is
installed into site-packages.  ``build(debug_bounds=True)`` compiles the same
sources with ``-DMOE_DEBUG_BOUNDS`` (every data-derived global index and
tensor-copy coordinate checked, failures counted in a device-side record, no
trap) into ``_build_debug/`` and ``libmoe_fp8_debug.so``.
"""

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_fp8.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libmoe_fp8_debug.so")
SOURCES = ["api.cu", "plan.cu", "prep.cu", "forward.cu", "vector.cu", "noalloc.cu", "router.cu", "w4a8.cu", "w4a8_tc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "-I", os.path.join(ROOT, "include")]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose=False, force=False, debug_bounds=False):
    """Compile the CUDA library; returns the path of the shared object.

    debug_bounds: build the bounds-checking variant instead (its own objects
    and shared object, so both variants can exist side by side)."""
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug_bounds else (BUILD, LIB)
    defines = ["-DMOE_DEBUG_BOUNDS"] if debug_bounds else []
    os.makedirs(build_dir, exist_ok=True)
    nvcc = _nvcc()
    headers = [os.path.join(CSRC, h) for h in os.listdir(CSRC) if h.endswith((".cuh", ".h"))]
    inc = os.path.join(ROOT, "include")
    headers += [os.path.join(inc, h) for h in os.listdir(inc) if h.endswith(".h")]
    objs = []
    jobs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(build_dir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + headers):
            jobs.append([nvcc, *ARCH, *FLAGS, *defines, "-c", s, "-o", o])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode != 0:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed: {' '.join(cmd)}")

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        run([nvcc, *ARCH, "-shared", "-o", lib, *objs])
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, debug_bounds="--debug-bounds" in sys.argv))

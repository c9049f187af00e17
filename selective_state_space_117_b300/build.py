"""Build the CUDA library libssscan.so in-tree with nvcc for sm_103a.

Every translation unit under csrc/ is compiled in parallel into _build/ and
linked into selective_state_space_117_b300/libssscan.so (CUDA runtime linked
statically, so the library loads without any library path set).  With
--debug-bounds the same sources are compiled with SS_DEBUG_BOUNDS into
_build_debug/ and linked into libssscan_debug.so (device-side index checks
recorded in the status word; see include/ss_scan.h).

    python -m selective_state_space_117_b300.build [--force] [--debug-bounds] [-v]
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
BUILD_DEBUG = os.path.join(HERE, "_build_debug")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libssscan.so")
LIB_DEBUG = os.path.join(HERE, "libssscan_debug.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, verbose, build_dir, extra):
    obj = os.path.join(build_dir, src[:-3] + ".o")
    cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def build(force: bool = False, verbose: bool = False, debug_bounds: bool = False) -> str:
    """Compile and link the library (libssscan.so, or libssscan_debug.so with debug_bounds)."""
    build_dir, lib, extra = (BUILD_DEBUG, LIB_DEBUG, ["-DSS_DEBUG_BOUNDS"]) if debug_bounds else (BUILD, LIB, [])
    os.makedirs(build_dir, exist_ok=True)
    hdrs = headers()
    srcs = sources()
    todo = [s for s in srcs if force or _stale(os.path.join(build_dir, s[:-3] + ".o"), [os.path.join(CSRC, s), *hdrs])]
    if todo:
        with cf.ThreadPoolExecutor(max_workers=max(1, min(len(todo), os.cpu_count() or 1))) as ex:
            for obj, log in ex.map(lambda s: _compile(s, verbose, build_dir, extra), todo):
                if verbose and log:
                    sys.stderr.write(log)
    objs = [os.path.join(build_dir, s[:-3] + ".o") for s in srcs]
    if force or todo or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.check_call([NVCC, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return lib


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true", help="print ptxas resource usage")
    ap.add_argument("--debug-bounds", action="store_true", help="build libssscan_debug.so (SS_DEBUG_BOUNDS)")
    args = ap.parse_args()
    print(build(force=args.force, verbose=args.verbose, debug_bounds=args.debug_bounds))


if __name__ == "__main__":
    main()

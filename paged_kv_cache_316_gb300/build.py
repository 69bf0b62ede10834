"""Build libpagedkv.so in-tree with nvcc for sm_103a.

    python -m paged_kv_cache_316_gb300.build [--force] [--ptxas-verbose] [--debug-bounds | --all]

Each translation unit under csrc/ is compiled in parallel to an object in
_build/, then linked into paged_kv_cache_316_gb300/libpagedkv.so with the
CUDA runtime linked statically (the library needs no libcudart at load time
and no libcuda at link time).  The debug variant, libpagedkv_debug.so
(objects in _build/debug/), is the same source compiled with
-DPKV_DEBUG_BOUNDS=1: every offset the kernels derive is range-checked
before use (the PKV_DEV_ERR_BOUNDS bit of the error word).
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpagedkv.so")
LIB_DEBUG = os.path.join(HERE, "libpagedkv_debug.so")
INCLUDE = os.path.join(ROOT, "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found")
    return exe


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _variant(debug_bounds: bool):
    """(object folder, library path, extra nvcc flags) of one build."""
    if debug_bounds:
        return os.path.join(BUILD, "debug"), LIB_DEBUG, ["-DPKV_DEBUG_BOUNDS=1"]
    return BUILD, LIB, []


def _start(debug_bounds: bool, force: bool, ptxas_verbose: bool):
    """Start the nvcc jobs of one variant; returns (objects, library, jobs)."""
    obj_dir, lib, extra = _variant(debug_bounds)
    os.makedirs(obj_dir, exist_ok=True)
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "pagedkv.h"))
    objs, procs = [], []
    for src in sources():
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        if force or ptxas_verbose or _stale(obj, [src] + headers):
            cmd = [nvcc()] + ARCH + NVCC_FLAGS + extra + ["-c", src, "-o", obj]
            if ptxas_verbose:
                cmd += ["-Xptxas", "-v"]
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT, text=True)))
    return objs, lib, procs


def _finish(objs, lib, procs, force: bool, ptxas_verbose: bool, quiet: bool) -> str:
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if pr.returncode != 0:
            failed.append((src, out))
        elif out and (ptxas_verbose or not quiet):
            sys.stdout.write(out)
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    if force or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        subprocess.run([nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs,
                       check=True)
        os.replace(tmp, lib)
    return lib


def build(force: bool = False, ptxas_verbose: bool = False, quiet: bool = True,
          debug_bounds: bool = False) -> str:
    """Build one variant: libpagedkv.so, or with debug_bounds the range-checking
    libpagedkv_debug.so (-DPKV_DEBUG_BOUNDS=1); returns its path."""
    objs, lib, procs = _start(debug_bounds, force, ptxas_verbose)
    return _finish(objs, lib, procs, force, ptxas_verbose, quiet)


def build_all(force: bool = False, quiet: bool = True):
    """Build both variants, all translation units compiled in parallel;
    returns (release library, debug library)."""
    jobs = [_start(d, force, False) for d in (False, True)]
    return tuple(_finish(*j, force, False, quiet) for j in jobs)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    ap.add_argument("--debug-bounds", action="store_true", help="build libpagedkv_debug.so only")
    ap.add_argument("--all", action="store_true", help="build both libraries")
    a = ap.parse_args()
    if a.all:
        print("\n".join(build_all(force=a.force, quiet=False)))
    else:
        print(build(force=a.force, ptxas_verbose=a.ptxas_verbose, quiet=False,
                    debug_bounds=a.debug_bounds))


if __name__ == "__main__":
    main()

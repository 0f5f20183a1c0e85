"""Builds libmtsgemm.so from csrc/*.cu with nvcc for sm_103a.

Each translation unit compiles in its own nvcc process (in parallel), then
one nvcc call links the shared library.  Objects and the library go to
``tiled_fp32_gemm_gb300/_build/``; a source newer than its object (or any
header newer than it) triggers a rebuild.

``checked=True`` builds the same sources with ``-DMT_BOUNDS_CHECK=1`` into
``_build/checked/libmtsgemm_checked.so``: the FFMA path's kernels (the FFMA
GEMM, its operand copies and K-slice reduce, the one-warp kernel) test every
global and shared access against its buffer, skip any that falls outside and
count it (``mt_bounds_status``).  For tests; slower than the normal build.

    python -m tiled_fp32_gemm_gb300.build [--force] [--verbose] [--checked]
"""
from __future__ import annotations

import argparse
import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libmtsgemm.so")
CHECKED_BUILD = os.path.join(BUILD, "checked")
CHECKED_LIB = os.path.join(CHECKED_BUILD, "libmtsgemm_checked.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden",
                     "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    exe = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(exe):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build")
    return exe


def _headers():
    return glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src: str, obj: str, verbose: bool, defines=()) -> str:
    cmd = [nvcc(), *NVCC_FLAGS, *defines, "-c", src, "-o", obj]
    if verbose:
        cmd += ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stderr}")
    return r.stderr if verbose else ""


def _variant(checked: bool):
    """(object dir, library, extra nvcc flags) of the normal or checked build."""
    if checked:
        return CHECKED_BUILD, CHECKED_LIB, ["-DMT_BOUNDS_CHECK=1"]
    return BUILD, LIB, []


def build_many(variants, force: bool = False, verbose: bool = False):
    """Compile the stale objects of every requested variant (False: normal,
    True: checked) in one pool of nvcc processes, then link each library.
    Returns the library paths in the order asked."""
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    headers = _headers()
    jobs, plans = [], []
    for checked in variants:
        out_dir, lib, defines = _variant(checked)
        os.makedirs(out_dir, exist_ok=True)
        objects = []
        for src in sources:
            obj = os.path.join(out_dir, os.path.basename(src)[:-3] + ".o")
            objects.append(obj)
            if force or _stale(obj, [src, *headers]):
                jobs.append((src, obj, defines))
        plans.append((lib, objects))
    if jobs:
        # The longest translation units first, so they overlap the rest.
        jobs.sort(key=lambda j: -os.path.getsize(j[0]))
        with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            logs = list(ex.map(lambda j: _compile(j[0], j[1], verbose, j[2]), jobs))
        if verbose:
            for (src, obj, _), log in zip(jobs, logs):
                print(f"== {os.path.relpath(obj, BUILD)}\n{log}", file=sys.stderr)
    for lib, objects in plans:
        if force or jobs or _stale(lib, objects):
            tmp = lib + f".tmp{os.getpid()}"
            cmd = [nvcc(), *ARCH, "-shared", "-o", tmp, *objects, "-cudart", "static"]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed:\n{r.stderr}")
            os.replace(tmp, lib)
    return [lib for lib, _ in plans]


def build(force: bool = False, verbose: bool = False, checked: bool = False) -> str:
    """Compile and link the library if anything changed; returns its path.
    checked=True: the bounds-checked build instead (see the module doc)."""
    return build_many([checked], force=force, verbose=verbose)[0]


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose", action="store_true", help="print -Xptxas -v")
    ap.add_argument("--checked", action="store_true", help="the bounds-checked build")
    ap.add_argument("--all", action="store_true", help="the normal and the checked build")
    a = ap.parse_args()
    if a.all:
        print("\n".join(build_many([False, True], force=a.force, verbose=a.verbose)))
    else:
        print(build(force=a.force, verbose=a.verbose, checked=a.checked))

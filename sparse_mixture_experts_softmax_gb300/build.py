"""Build step of the CUDA library ``libmoe_gb300.so`` (sm_103a only).

Each ``csrc/*.cu`` file is compiled by nvcc in parallel and the objects are
linked into one shared library next to this file.  Rebuilds only what changed.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe_gb300.so")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the MoE CUDA library cannot be built")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return hs


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


LIB_DEBUG = os.path.join(PKG, "libmoe_gb300_debug.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")


def _variant(debug: bool):
    """(object directory, library path, extra nvcc flags) of the release or
    the MOE_DEBUG build (device-side index checks; see csrc/common.cuh)."""
    if debug:
        return BUILD_DEBUG, LIB_DEBUG, ["-DMOE_DEBUG"]
    return BUILD, LIB, []


def _run(cmd, verbose):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr)
    return cmd


def build_library(verbose: bool = False, extra_flags=None, debug: bool = False,
                  also_debug: bool = False) -> str:
    """Compile and link the library (or, with debug=True, its MOE_DEBUG
    variant); also_debug builds both, their files compiled in one pool.
    Returns the path of the (first) library."""
    nvcc = _nvcc()
    headers = _headers()
    variants = [debug] + ([not debug] if also_debug else [])
    compile_jobs, links = [], []
    for dbg in variants:
        bdir, lib, vflags = _variant(dbg)
        os.makedirs(bdir, exist_ok=True)
        flags = NVCC_FLAGS + vflags + list(extra_flags or [])
        objs = []
        for src in _sources():
            obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            if _stale(obj, [src] + headers):
                compile_jobs.append([nvcc] + ARCH + flags + ["-I", INCLUDE, "-c", src, "-o", obj])
        links.append((lib, objs))
    if compile_jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(compile_jobs), os.cpu_count() or 4)) as ex:
            list(ex.map(lambda c: _run(c, verbose), compile_jobs))
    for lib, objs in links:
        if _stale(lib, objs):
            _run([nvcc] + ARCH + ["-shared", "-o", lib] + objs, verbose)
    return links[0][0]


if __name__ == "__main__":
    print(build_library(verbose=True))

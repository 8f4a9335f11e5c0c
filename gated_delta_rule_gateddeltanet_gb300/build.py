"""Builds libgdn.so in-tree with nvcc for sm_103a (GB300).

Each translation unit under ``csrc/`` is compiled in parallel to an object in
``_build/`` and the objects are linked into ``libgdn.so`` next to this file.
Rebuilds happen only when a source or header is newer than the library.
``ptxas`` resource usage (registers, spills, shared memory) is kept in
``_build/ptxas.log``.

``build(debug=True)`` makes ``libgdn_debug.so`` beside it: the translation
units that hold precondition checks (``DEBUG_SOURCES``) compiled again with
``GDN_DEBUG_CHECKS`` into ``_build_debug/``, linked with the release objects
of every other unit (whose code the macro does not change).
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgdn.so")
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libgdn_debug.so")
DEBUG_SOURCES = ("gdn_api.cu", "gdn_debug.cu")  # the units whose code GDN_DEBUG_CHECKS changes

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _inputs():
    return _sources() + sorted(glob.glob(os.path.join(CSRC, "*.cuh"))) + \
        sorted(glob.glob(os.path.join(INCLUDE, "*.h"))) + [os.path.abspath(__file__)]


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src, build_dir=BUILD, extra=()):
    obj = os.path.join(build_dir, os.path.basename(src)[:-3] + ".o")
    cmd = [_nvcc(), *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    return obj, r.stderr


def _link(objs, lib):
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [_nvcc(), *ARCH, "-shared", "-o", tmp, *objs, "-lcudart_static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)


def _build_debug(force: bool) -> str:
    build(force=force)  # the release objects of the other units
    if not force and not needs_build(LIB_DEBUG):
        return LIB_DEBUG
    os.makedirs(BUILD_DEBUG, exist_ok=True)
    srcs = _sources()
    dbg = [s for s in srcs if os.path.basename(s) in DEBUG_SOURCES]
    with ThreadPoolExecutor(max_workers=len(dbg)) as ex:
        dobjs = [o for o, _ in ex.map(lambda s: _compile(s, BUILD_DEBUG, ["-DGDN_DEBUG_CHECKS"]), dbg)]
    objs = [os.path.join(BUILD, os.path.basename(s)[:-3] + ".o") for s in srcs if s not in dbg]
    _link(objs + dobjs, LIB_DEBUG)
    return LIB_DEBUG


def build(force: bool = False, verbose: bool = False, debug: bool = False) -> str:
    """Compile every kernel for sm_103a and link libgdn.so (with ``debug``:
    libgdn_debug.so, see above); returns the library's path."""
    if debug:
        return _build_debug(force)
    if not force and not needs_build():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    with ThreadPoolExecutor(max_workers=min(8, len(srcs))) as ex:
        results = list(ex.map(_compile, srcs))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for (obj, log), src in zip(results, srcs):
            f.write(f"==== {os.path.basename(src)}\n{log}\n")
    _link([o for o, _ in results], LIB)
    if verbose:
        print(open(os.path.join(BUILD, "ptxas.log")).read())
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv))

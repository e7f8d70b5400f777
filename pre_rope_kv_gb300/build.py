"""Compile the CUDA library (sm_103a) into pre_rope_kv_gb300/_build/libkvi.so.

Each translation unit is compiled in parallel with nvcc for
``arch=compute_103a,code=sm_103a`` only, then linked into one shared library
with the CUDA runtime linked statically.  Nothing is installed: the library
stays in the source tree, next to the binding that loads it.

``build(debug=True)`` compiles the same sources with ``-DKVI_DEBUG_CHECKS``
into ``_build/libkvi_debug.so``: the checks and the failure hook that
``include/kvi_debug.h`` describes.  Only the tests use it.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libkvi.so")
DEBUG_LIB_PATH = os.path.join(OUT_DIR, "libkvi_debug.so")
SOURCES = ["kvi_host.cu", "kvi_retrieve.cu", "kvi_inject.cu", "kvi_noalloc.cu", "kvi_shared.cu",
           "kvi_store_io.cu", "kvi_graph.cu", "kvi_selftest.cu"]
HEADERS = [os.path.join(CSRC, "kvi_internal.cuh"), os.path.join(CSRC, "kvi_dot2.cuh"),
           os.path.join(CSRC, "kvi_sync.cuh"),
           os.path.join(INCLUDE, "kvi.h"), os.path.join(INCLUDE, "kvi_debug.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvi")


def _stale(path: str) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    deps = [os.path.join(CSRC, s) for s in SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False) -> str:
    """Build libkvi.so (or, with debug, libkvi_debug.so) if it is missing or
    older than its sources."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    if not force and not _stale(lib_path):
        return lib_path
    os.makedirs(OUT_DIR, exist_ok=True)
    nvcc = _nvcc()
    common = ["-std=c++17", "-O3", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]
    if debug:
        common += ["-DKVI_DEBUG_CHECKS"]
    if ptxas_info:
        common += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(OUT_DIR, src.replace(".cu", f"{'.dbg' if debug else ''}.{os.getpid()}.o"))
        objs.append(obj)
        cmd = [nvcc, *common, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
    failed = []
    for src, pr in procs:
        out, _ = pr.communicate()
        if out and (verbose or ptxas_info or pr.returncode):
            print(out, file=sys.stderr)
        if pr.returncode:
            failed.append(src)
    if failed:
        for o in objs:
            if os.path.exists(o):
                os.remove(o)
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, "-shared", *ARCH, "-o", tmp, *objs, "-Xcompiler", "-fPIC"]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.check_call(cmd)
    os.replace(tmp, lib_path)
    for o in objs:
        os.remove(o)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))

"""Build libpagedkv.so in-tree (nvcc for sm_103a, g++ for the host bookkeeping).

Objects go to ``_build/`` next to this file; the library to
``libpagedkv.so`` next to this file. Translation units compile in parallel
and only when a source or header is newer than the library.
``build_traced()`` builds the tracing variant of the prefill kernel
(``-DKVP_PREFILL_TRACE``) as ``libpagedkv_trace.so`` from objects in
``_build/trace/``; it is a measuring tool, never the product.
"""

from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpagedkv.so")
TRACE_LIB = os.path.join(HERE, "libpagedkv_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedkv")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu"))) + sorted(glob.glob(os.path.join(CSRC, "*.cpp")))


def _deps():
    return _sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h")) + [__file__]


def needs_build(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(p) > t for p in _deps())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("build step failed:\n" + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, lib: str = LIB, objdir: str = BUILD,
          defines: tuple = ()) -> str:
    """Compile every translation unit and link ``lib`` (libpagedkv.so by
    default); returns its path."""
    if not force and not needs_build(lib):
        return lib
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    jobs = []
    for src in _sources():
        obj = os.path.join(objdir, os.path.basename(src) + ".o")
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                   *[f"-D{d}" for d in defines], "-Xptxas", "-v", "-c", src, "-o", obj]
        else:
            cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-Wall", "-I", INCLUDE, "-c", src, "-o", obj]
        jobs.append((cmd, obj))
    with ThreadPoolExecutor(max_workers=min(8, len(jobs))) as ex:
        logs = list(ex.map(lambda j: _run(j[0]), jobs))
    if verbose:
        for log in logs:
            sys.stdout.write(log)
    tmp = lib + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *[o for _, o in jobs], "-o", tmp])
    os.replace(tmp, lib)
    return lib


def build_traced(force: bool = False) -> str:
    """The tracing variant of the library (the prefill kernel's stamps on)."""
    return build(force=force, lib=TRACE_LIB, objdir=os.path.join(BUILD, "trace"), defines=("KVP_PREFILL_TRACE",))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

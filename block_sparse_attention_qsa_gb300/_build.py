"""Builds libqsa.so in-tree for sm_103a with nvcc (no cmake, no torch build).

Each .cu under csrc/ compiles to an object in parallel; the objects link into
``block_sparse_attention_qsa_gb300/libqsa.so`` with the CUDA runtime linked
statically, so the library only needs the NVIDIA driver at run time.

``build(trace=True)`` makes the tracing build instead, ``libqsa_trace.so``
(the same sources with ``-DQSA_TRACE``: the step's kernels record per-CTA
phase stamps, read back with ``qsa_trace_read``); ``timeline.py`` uses it.
"""

from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libqsa.so")
BUILD_TRACE = os.path.join(PKG, "_build_trace")
LIB_TRACE = os.path.join(PKG, "libqsa_trace.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the QSA library needs the CUDA toolkit to build")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _newest_input() -> float:
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    files += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build(force: bool = False, verbose: bool = False, extra_flags=(), trace: bool = False) -> str:
    """Compile and link libqsa.so (or, with ``trace``, libqsa_trace.so);
    returns its path. Skips work when the library is newer than every source
    unless ``force``."""
    lib, bdir = (LIB_TRACE, BUILD_TRACE) if trace else (LIB, BUILD)
    if trace:
        extra_flags = (*extra_flags, "-DQSA_TRACE")
    if not force and os.path.exists(lib) and os.path.getmtime(lib) >= _newest_input():
        return lib
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    objs = []
    cmds = []
    for src in sources():
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmds.append([cc, *ARCH, *FLAGS, *extra_flags, "-c", src, "-o", obj])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), flush=True)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        return r.stderr

    with concurrent.futures.ThreadPoolExecutor(max_workers=min(8, len(cmds))) as ex:
        logs = list(ex.map(run, cmds))
    if verbose:
        for lg in logs:
            if lg.strip():
                print(lg)
    tmp = lib + ".tmp"
    run([cc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    v = "-v" in sys.argv
    extra = ["-Xptxas", "-v"] if "--ptxas" in sys.argv else []
    print(build(force=True, verbose=v or bool(extra), extra_flags=extra))

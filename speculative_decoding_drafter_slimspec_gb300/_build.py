"""Builds libslimspec.so in-tree for sm_103a with nvcc.

Each .cu file under csrc/ is compiled to an object in parallel, then the
objects are linked into a shared library with the CUDA runtime linked
statically (so loading the library needs no libcudart on the loader path).
The library lands next to this file; build products are git-ignored.

Beside it, libsstimeline.so (csrc/timeline.cpp, host C++ against CUPTI) is
the benchmark's kernel timeline; it is built when the toolkit has CUPTI and
skipped otherwise (the library itself never uses it).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libslimspec.so")
TIMELINE_LIB = os.path.join(HERE, "libsstimeline.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA 13 toolkit is required to build libslimspec")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _newest_input() -> float:
    files = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                         if f.endswith((".cuh", ".h"))]
    files.append(os.path.join(os.path.dirname(HERE), "include", "slimspec.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def build_timeline(force: bool = False):
    """Compiles libsstimeline.so (if out of date); returns its path, or None
    when the toolkit has no CUPTI or no host compiler."""
    src = os.path.join(CSRC, "timeline.cpp")
    if not force and os.path.exists(TIMELINE_LIB) and \
            os.path.getmtime(TIMELINE_LIB) >= os.path.getmtime(src):
        return TIMELINE_LIB
    cuda = os.path.dirname(os.path.dirname(os.path.realpath(_nvcc())))
    inc, lib = os.path.join(cuda, "include"), os.path.join(cuda, "lib64")
    cxx = shutil.which("g++") or shutil.which("c++")
    if cxx is None or not os.path.exists(os.path.join(inc, "cupti.h")):
        return None
    tmp = TIMELINE_LIB + ".tmp"
    r = subprocess.run([cxx, "-O2", "-shared", "-fPIC", "-std=c++17", f"-I{inc}", src, "-o", tmp,
                        f"-L{lib}", "-lcupti", f"-Wl,-rpath,{lib}"], capture_output=True,
                       text=True)
    if r.returncode != 0:
        sys.stderr.write(f"libsstimeline.so not built (no kernel timeline):\n{r.stderr[-2000:]}")
        return None
    os.replace(tmp, TIMELINE_LIB)
    return TIMELINE_LIB


def build(force: bool = False, verbose: bool = False) -> str:
    """Compiles (if out of date) and returns the path of libslimspec.so."""
    build_timeline(force)
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= _newest_input():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)
    extra = ["-Xptxas", "-v"] if verbose else []

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stderr}")
        if verbose and r.stderr:
            sys.stderr.write(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", *objs, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

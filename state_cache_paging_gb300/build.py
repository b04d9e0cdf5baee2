"""Builds liblmc.so in-tree for sm_103a (nvcc + g++, no cmake).

Usage: ``python state_cache_paging_gb300/build.py [--force] [-v]`` (run by
path: importing the package itself requires the built library). The translation units
compile in parallel; the CUDA runtime is linked statically, so the library
loads without torch and shares the primary context with whatever else runs
in the process.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
import tempfile

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "liblmc.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")
HOST_UNITS = ("layout", "checks")  # host C++ translation units in csrc/
CXX = os.environ.get("CXX", "g++")


def _sources():
    out = []
    for name in sorted(os.listdir(CSRC)):
        if name.endswith((".cu", ".cpp", ".h", ".map")):
            out.append(os.path.join(CSRC, name))
    out.append(os.path.join(INCLUDE, "lmc.h"))
    return out


def _stale(target: str) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in _sources())


def build_library(force: bool = False, extra_nvcc=(), out_path: str | None = None, verbose: bool = False) -> str:
    """Compiles and links liblmc.so; returns its path. `extra_nvcc` adds flags
    (e.g. -D tuning constants) to the CUDA translation unit."""
    out = out_path or LIB_PATH
    if not force and not extra_nvcc and out_path is None and not _stale(out):
        return out
    os.makedirs(BUILD_DIR, exist_ok=True)
    work = tempfile.mkdtemp(dir=BUILD_DIR)  # private per build (builds may run concurrently)
    cu_obj = os.path.join(work, "paging.o")
    cpp_objs = [os.path.join(work, name + ".o") for name in HOST_UNITS]
    ptxas_log = os.path.join(BUILD_DIR, "ptxas.log")
    cmds = [
        [NVCC, "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xptxas", "-v", "-Xcompiler", "-fPIC,-fvisibility=hidden",
         "-I", INCLUDE, "-I", CSRC, *extra_nvcc, "-c", os.path.join(CSRC, "paging.cu"), "-o", cu_obj],
        *[[CXX, "-O2", "-std=c++17", "-fPIC", "-fvisibility=hidden", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE,
           "-I", CSRC, "-c", os.path.join(CSRC, name + ".cpp"), "-o", obj]
          for name, obj in zip(HOST_UNITS, cpp_objs)],
    ]
    procs = [subprocess.Popen(c, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True) for c in cmds]
    logs = [p.communicate()[0] for p in procs]
    for c, p, log in zip(cmds, procs, logs):
        if p.returncode != 0:
            raise RuntimeError(f"compile failed: {' '.join(c)}\n{log}")
    with open(ptxas_log, "w") as f:
        f.write(logs[0])
    if verbose:
        print(logs[0])
    tmp = os.path.join(work, "liblmc.so")
    link = [NVCC, "-shared", *ARCH, "-Xlinker", "--version-script=" + os.path.join(CSRC, "liblmc.map"),
            "-o", tmp, cu_obj, *cpp_objs]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed: {' '.join(link)}\n{r.stdout}{r.stderr}")
    os.replace(tmp, out)
    shutil.rmtree(work, ignore_errors=True)
    return out


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))

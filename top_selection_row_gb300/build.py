"""Build the selection library in-tree: ``libqrita.so`` next to this file.

One nvcc invocation for sm_103a (GB300) compiles the kernel and the C ABI.
The result is git-ignored; ``__graft_entry__.build()`` runs this on every
machine that needs the library (nothing compiled elsewhere is reused).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB_PATH = os.path.join(PKG_DIR, "libqrita.so")

SOURCES = ["qrita_kernel.cu", "qrita_outputs.cu", "qrita_api.cpp"]
HEADERS = ["qrita_device.cuh", "qrita_internal.h"]

GENCODE = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libqrita.so")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "qrita.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile libqrita.so for sm_103a; returns its path."""
    if not force and up_to_date():
        return LIB_PATH
    import tempfile

    base = [nvcc_path(), *GENCODE, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]
    if extra_flags:
        base[1:1] = list(extra_flags)
    tmp = LIB_PATH + ".tmp"
    with tempfile.TemporaryDirectory(prefix="qrita_build_") as td:
        # every translation unit compiles at once, then one link
        objs, procs = [], []
        for src in SOURCES:
            obj = os.path.join(td, os.path.splitext(src)[0] + ".o")
            cmd = [*base, "-c", os.path.join(CSRC, src), "-o", obj]
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((cmd, subprocess.Popen(cmd)))
            objs.append(obj)
        for cmd, pr in procs:
            if pr.wait() != 0:
                raise subprocess.CalledProcessError(pr.returncode, cmd)
        link = [nvcc_path(), *GENCODE, "-shared", "-o", tmp, *objs]
        if verbose:
            print(" ".join(link), file=sys.stderr)
        subprocess.run(link, check=True)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose=True))

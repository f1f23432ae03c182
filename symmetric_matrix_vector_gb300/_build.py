"""Build the xsymv CUDA library (libxsymv.so) in-tree with nvcc for sm_103a.

Each translation unit is compiled in parallel, then linked into one shared
library that exports only the C-ABI declared in include/xsymv.h.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBDIR = os.path.join(PKG, "_lib")
LIBNAME = "libxsymv.so"
LIBPATH = os.path.join(LIBDIR, LIBNAME)

UNITS = ["xsymv_api", "xsymv_probe", "xsymv_s", "xsymv_d", "xsymv_c", "xsymv_z", "xsymv_w",
         "xsymv_gemv"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden",
                     "-I", INCLUDE]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the xsymv CUDA library cannot be built")


def _inputs():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh", ".h"))]
    files.append(os.path.join(INCLUDE, "xsymv.h"))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIBPATH):
        return False
    t = os.path.getmtime(LIBPATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile and link libxsymv.so; returns its path."""
    if not force and up_to_date():
        return LIBPATH
    exe = nvcc()
    objdir = os.path.join(LIBDIR, "obj")
    os.makedirs(objdir, exist_ok=True)
    procs = []
    for u in UNITS:
        src = os.path.join(CSRC, u + ".cu")
        obj = os.path.join(objdir, u + ".o")
        cmd = [exe, *NVCC_FLAGS, *extra_flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((u, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                          text=True)))
    failed = []
    for u, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((u, out))
        elif verbose and out:
            print(out, file=sys.stderr)
    if failed:
        msg = "\n".join("%s:\n%s" % (u, o) for u, o in failed)
        raise RuntimeError("nvcc failed:\n" + msg)
    tmp = LIBPATH + ".tmp%d" % os.getpid()
    objs = [os.path.join(objdir, u + ".o") for u in UNITS]
    subprocess.run([exe, *ARCH, "-shared", "-o", tmp, *objs], check=True)
    os.replace(tmp, LIBPATH)
    return LIBPATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""Build liblayerattn.so in-tree for sm_103a (GB300) with nvcc.

Each translation unit compiles in parallel to an object; one link makes the
shared library with the CUDA runtime linked statically, so the library loads
on a machine with no GPU driver (the test suite checks its exports there).
The same sources compiled with -DLA_CHECKED=1 give liblayerattn_checked.so,
the build with bounds checks on every global store of the kernels.
Rebuilds only when a source or header is newer than the library.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "liblayerattn.so")
LIB_CHECKED = os.path.join(BUILD, "liblayerattn_checked.so")
SOURCES = ["la_api.cu", "la_attn.cu", "la_proj.cu", "la_misc.cu"]
HEADERS = ["la_device.cuh", "la_internal.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("CUDA_HOME", ""), "/usr/local/cuda"):
        p = os.path.join(cand, "bin", "nvcc") if cand else ""
        if p and os.path.exists(p):
            return p
    return "nvcc"


def _inputs():
    files = [os.path.join(CSRC, f) for f in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "layerattn.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    for lib in (LIB, LIB_CHECKED):
        if not os.path.exists(lib):
            return False
        t = os.path.getmtime(lib)
        if any(os.path.getmtime(f) > t for f in _inputs()):
            return False
    return True


def _compile(src: str, checked: bool, verbose: bool) -> str:
    out_dir = os.path.join(BUILD, "checked") if checked else BUILD
    obj = os.path.join(out_dir, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), "-c", os.path.join(CSRC, src), "-o", obj, "-O3", "-std=c++17", *ARCH, "-lineinfo",
           "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC, "-Xptxas", "-v"]
    if checked:
        cmd.append("-DLA_CHECKED=1")
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = os.path.join(out_dir, os.path.splitext(src)[0] + ".log")
    with open(log, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed for {src} (log: {log})")
    if verbose:
        sys.stderr.write(r.stderr)
    return obj


def _link(objs, lib: str) -> None:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc(), "-shared", *ARCH, "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc link failed")
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False) -> str:
    """Build liblayerattn.so and liblayerattn_checked.so; returns the former's path."""
    os.makedirs(os.path.join(BUILD, "checked"), exist_ok=True)
    if not force and up_to_date():
        return LIB
    jobs = [(s, c) for c in (False, True) for s in SOURCES]
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        objs = list(ex.map(lambda j: _compile(j[0], j[1], verbose), jobs))
    _link(objs[:len(SOURCES)], LIB)
    _link(objs[len(SOURCES):], LIB_CHECKED)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

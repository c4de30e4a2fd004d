"""Compile the CUDA sources into ``libengram.so`` inside the package (sm_103a only).

Each translation unit is compiled in parallel with nvcc, then linked into one
shared library. No fast-math: the dequant relies on IEEE fp32 multiplies
without flush-to-zero.
"""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(os.path.dirname(PKG), "include")
LIB = os.path.join(PKG, "libengram.so")
BUILD_DIR = os.path.join(PKG, "_build")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE]


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _stale(out: str, deps) -> bool:
    if not os.path.exists(out):
        return True
    t = os.path.getmtime(out)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, extra_flags=None, lib_path: str = LIB) -> str:
    """Build `lib_path` (default: the package's libengram.so) when it is older than its sources.
    A library built with extra flags (e.g. the checked build, -DENGRAM_CHECKED=1) goes to its own
    path and object directory."""
    nvcc = os.environ.get("NVCC", "nvcc")
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(INCLUDE, "engram.h"))
    srcs = sources()
    if not force and not _stale(lib_path, srcs + headers + [__file__]):
        return lib_path
    build_dir = BUILD_DIR if lib_path == LIB else BUILD_DIR + "_" + os.path.splitext(os.path.basename(lib_path))[0]
    os.makedirs(build_dir, exist_ok=True)
    flags = NVCC_FLAGS + list(extra_flags or [])
    procs, objs = [], []
    for src in srcs:
        obj = os.path.join(build_dir, os.path.basename(src) + ".o")
        objs.append(obj)
        cmd = [nvcc, *ARCH, *flags, "-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for cmd, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stderr.write(out.decode(errors="replace"))
        if p.returncode != 0:
            failed.append(" ".join(cmd))
    if failed:
        raise RuntimeError("nvcc failed:\n" + "\n".join(failed))
    tmp = lib_path + ".tmp"
    subprocess.check_call([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))

"""Build libamk.so in-tree with nvcc for sm_103a.

The translation units compiled in parallel, then linked with the static
CUDA runtime.  No cmake, no torch extension machinery: the library is a
plain C-ABI shared object loaded through ctypes.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libamk.so")

SOURCES = ["decode_kernel.cu", "amk_api.cpp", "schedule.cpp", "static_scratch.cu", "prefill.cu", "hbm_probe.cu"]
HEADERS = ["device_model.hpp", "schedule.hpp", "prefill.hpp", "ptx.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")
FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE]


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "amk.h"))
    files.append(os.path.abspath(__file__))
    return files


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("command failed: " + " ".join(cmd) + "\n" + r.stdout + r.stderr)
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, extra_flags=None) -> str:
    """Compile and link libamk.so; returns its path.  extra_flags (e.g.
    -DAMK_STAGE_BYTES=16384 to build 16 KB tiles) force a rebuild."""
    if not force and not extra_flags and not stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    flags = FLAGS + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(BUILD, src + ".o")
        cmd = [NVCC] + ARCH + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        out = _run(cmd)
        return obj, cmd, out

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    objs = [r[0] for r in results]
    tmp = LIB + ".tmp"
    link = [NVCC] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
    _run(link)
    os.replace(tmp, LIB)
    if verbose:
        for _, cmd, out in results:
            print(" ".join(cmd), file=sys.stderr)
            if out.strip():
                print(out, file=sys.stderr)
        print(" ".join(link), file=sys.stderr)
    return LIB


if __name__ == "__main__":
    extra = sys.argv[1:]
    print(build(force=True, verbose=True, extra_flags=extra))

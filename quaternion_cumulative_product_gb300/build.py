"""Builds ``libquatscan.so`` (the CUDA library behind ``include/quat_cumprod.h``).

One translation unit, compiled for sm_103a only, with the static CUDA runtime,
in place next to this file.  Used by ``__graft_entry__.build()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SOURCES = [os.path.join(HERE, "csrc", "quat_scan.cu")]
HEADERS = [os.path.join(HERE, "csrc", f) for f in
           ("quat_device.cuh", "quat_common.cuh", "quat_tiles.cuh", "quat_chain.cuh", "quat_walk.cuh",
            "quat_segwalk.cuh", "quat_segwalk_ws.cuh", "quat_segwalk_bwd.cuh", "quat_segwalk_tab.cuh",
            "quat_short.cuh")]
DEPS = SOURCES + HEADERS + [os.path.join(ROOT, "include", "quat_cumprod.h")]
LIB = os.path.join(HERE, "libquatscan.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_path() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found (CUDA toolkit required to build libquatscan.so)")


def command(out: str = LIB, extra=()) -> list:
    return [nvcc_path(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
            "-shared", "-I", os.path.join(ROOT, "include"), *extra, *SOURCES, "-o", out]


def is_stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not is_stale():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    extra = ("-Xptxas", "-v") if verbose else ()
    proc = subprocess.run(command(tmp, extra), capture_output=True, text=True)
    if proc.returncode != 0:
        sys.stderr.write(proc.stdout + proc.stderr)
        raise RuntimeError("nvcc failed to build libquatscan.so")
    if verbose:
        sys.stderr.write(proc.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)

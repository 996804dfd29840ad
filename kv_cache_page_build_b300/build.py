"""Build libkvr.so in-tree with nvcc for sm_103a.

    python -m kv_cache_page_build_b300.build [--force]

The library is one translation unit (csrc/kvr.cu includes the kernel
headers), linked against the static CUDA runtime so that it only needs the
driver at run time.  ptxas resource usage (registers, spills, shared memory)
is written to ``build.log`` next to the library.
"""
from __future__ import annotations

import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(PKG, "libkvr.so")
LOG = os.path.join(PKG, "build.log")
ARCH = "-gencode=arch=compute_103a,code=sm_103a"


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh"))
                  + [os.path.join(INCLUDE, "kvr.h")])


def up_to_date() -> bool:
    if not os.path.exists(LIB):
        return False
    t = os.path.getmtime(LIB)
    return all(os.path.getmtime(s) <= t for s in _sources())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and up_to_date():
        return LIB
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc(), ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xptxas", "-v",
           "-Xcompiler", "-fPIC,-O2", "-shared", "-cudart", "static",
           f"-I{INCLUDE}", f"-I{CSRC}", os.path.join(CSRC, "kvr.cu"), "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    with open(LOG, "w") as f:
        f.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError(f"nvcc failed ({r.returncode}); see {LOG}")
    if verbose:
        sys.stdout.write(r.stderr)
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)

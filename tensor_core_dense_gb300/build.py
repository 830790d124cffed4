"""Compiles the CUDA library (csrc/*.cu) into _lib/libtcgemm.so for sm_103a
(one nvcc per translation unit, in parallel, then one link).

nvcc cross-compiles without a GPU.  The library links the CUDA runtime
statically and reaches the driver's tensor-map encoder through
cudaGetDriverEntryPointByVersion, so it needs no libcuda at link time.
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(LIB_DIR, "libtcgemm.so")
SOURCES = [os.path.join(CSRC, "tcgemm.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cuh")] + [
    os.path.join(ROOT, "include", "tcgemm.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "--expt-relaxed-constexpr",
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False, extra=None) -> str:
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(LIB_DIR, exist_ok=True)
    tag = f"{os.getpid()}.tmp"
    objs = [os.path.join(LIB_DIR, os.path.basename(src)[:-3] + f".{tag}.o") for src in SOURCES]
    cmds = [[nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-I", CSRC,
             *(extra or []), "-c", src, "-o", obj] for src, obj in zip(SOURCES, objs)]
    for c in cmds:
        if verbose:
            print(" ".join(c), file=sys.stderr)
    # one nvcc per translation unit, in parallel, then one link
    with ThreadPoolExecutor(len(cmds)) as ex:
        for f in [ex.submit(subprocess.check_call, c) for c in cmds]:
            f.result()
    tmp = f"{LIB_PATH}.{tag}"
    subprocess.check_call([nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared",
                           *objs, "-o", tmp])
    for o in objs:
        os.remove(o)
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None)

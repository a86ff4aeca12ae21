"""Build libmqconv.so (all CUDA kernels + the C ABI) in-tree for sm_103a.

Each translation unit compiles to its own object in parallel (the kernels do
not call device code across units), then one link step makes the library.
"""
from __future__ import annotations

import concurrent.futures
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
OBJ = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmqconv.so")
SOURCES = ["api.cu", "quantize.cu", "conv.cu", "conv_halo.cu", "conv_halo_fwd_a.cu", "conv_halo_fwd_b.cu", "conv_halo_dgrad_a.cu",
           "conv_halo_dgrad_b.cu"]
HEADERS = ["common.cuh", "conv_halo.cuh", "kernels.h", os.path.join("..", "..", "include", "mqconv.h")]

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC",
    "-Xptxas", "-warn-spills",
]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def _obj(src: str) -> str:
    return os.path.join(OBJ, os.path.splitext(src)[0] + ".o")


def _newest_header() -> float:
    deps = [os.path.join(CSRC, h) for h in HEADERS]
    return max((os.path.getmtime(d) for d in deps if os.path.exists(d)), default=0.0)


def _obj_stale(src: str) -> bool:
    o = _obj(src)
    if not os.path.exists(o):
        return True
    t = os.path.getmtime(o)
    return os.path.getmtime(os.path.join(CSRC, src)) > t or _newest_header() > t


def stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    return any(os.path.getmtime(d) > t for d in deps if os.path.exists(d))


def _compile(src: str, verbose: bool) -> None:
    o = _obj(src)
    cmd = [_nvcc(), *NVCC_FLAGS, "-c", "-o", o + ".tmp", os.path.join(CSRC, src)]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(o + ".tmp", o)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not stale():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    todo = [s for s in SOURCES if force or _obj_stale(s)]
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(SOURCES), os.cpu_count() or 4)) as ex:
        for f in [ex.submit(_compile, s, verbose) for s in todo]:
            f.result()
    cmd = [_nvcc(), "-gencode", "arch=compute_103a,code=sm_103a", "-shared", "-Xcompiler", "-fPIC",
           "-o", LIB + ".tmp", *[_obj(s) for s in SOURCES]]
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True)
    print(LIB)

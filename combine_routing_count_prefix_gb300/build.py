"""Build libllmoe.so (the CUDA library behind include/llmoe.h) for sm_103a.

One translation unit, one -gencode; nvcc cross-compiles without a GPU.  The
library links the CUDA runtime statically and exports only the llmoe_* C ABI.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
SRC = os.path.join(PKG, "csrc", "llmoe.cu")
HDR = os.path.join(ROOT, "include", "llmoe.h")
OUT_DIR = os.path.join(PKG, "_build")
SO = os.path.join(OUT_DIR, "libllmoe.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-Xcompiler", "-fPIC,-fvisibility=hidden", "-shared",
]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand) and shutil.which(cand) is None:
        raise RuntimeError("nvcc not found: the CUDA library cannot be built")
    return cand


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if not force and os.path.exists(SO) and os.path.getmtime(SO) >= newest:
        return SO
    tmp = f"{SO}.{os.getpid()}.tmp"
    cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-o", tmp, SRC]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, SO)
    return SO


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

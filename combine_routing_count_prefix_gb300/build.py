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
# the phase-trace build (-DLLMOE_PHASE_TRACE=1): the same library with per-CTA
# timer stamps in the dispatch and combine kernels, for phase_budget.py only
TRACE_SO = os.path.join(OUT_DIR, "libllmoe_trace.so")

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


def build(force: bool = False, verbose: bool = False, trace: bool = False) -> str:
    """Compile the library (or, with trace=True, its phase-trace build) unless
    it is newer than its sources; returns the path of the shared object."""
    out = TRACE_SO if trace else SO
    os.makedirs(OUT_DIR, exist_ok=True)
    newest = max(os.path.getmtime(SRC), os.path.getmtime(HDR))
    if not force and os.path.exists(out) and os.path.getmtime(out) >= newest:
        return out
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = [nvcc(), *NVCC_FLAGS, "-I", os.path.join(ROOT, "include"), "-o", tmp, SRC]
    if trace:
        cmd.insert(1, "-DLLMOE_PHASE_TRACE=1")
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

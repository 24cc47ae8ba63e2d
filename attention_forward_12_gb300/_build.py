"""In-tree build of the CUDA library ``libattn.so`` (nvcc, sm_103a only)."""
from __future__ import annotations

import os
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SOURCES = [os.path.join(CSRC, "attn_fwd.cu")]
DEPS = SOURCES + [os.path.join(CSRC, "sm103_primitives.cuh"), os.path.join(ROOT, "include", "attn.h")]
LIB_PATH = os.path.join(PKG, "libattn.so")

NVCC_FLAGS = [
    "-gencode", "arch=compute_103a,code=sm_103a",
    "-O3", "-lineinfo", "-std=c++17",
    "-shared", "-Xcompiler", "-fPIC",
    "-I", os.path.join(ROOT, "include"),
]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile ``libattn.so`` next to this file if it is missing or stale."""
    stale = (not os.path.exists(LIB_PATH)) or any(
        os.path.getmtime(LIB_PATH) < os.path.getmtime(d) for d in DEPS)
    if force or stale:
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        cmd = [nvcc(), *NVCC_FLAGS, *SOURCES, "-o", tmp]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        subprocess.run(cmd, check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH

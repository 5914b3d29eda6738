"""Build the in-tree CUDA library ``libneox_attn.so`` for sm_103a with nvcc.

``python -m causal_rope_self_neox_b300.build`` (or ``build()``) compiles
``csrc/neox_attn.cu`` into ``causal_rope_self_neox_b300/libneox_attn.so``.  The
library links the CUDA runtime statically and reaches the driver's tensor-map
encoder through the runtime's entry-point query, so it needs no -lcuda.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
LIB = os.path.join(PKG, "libneox_attn.so")
SRC = os.path.join(PKG, "csrc", "neox_attn.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc_command(out: str = LIB, extra=()) -> list:
    return ["nvcc", *ARCH, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
            "-I", os.path.join(ROOT, "include"), "-I", os.path.join(PKG, "csrc"), *extra, SRC, "-o", out]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = glob.glob(os.path.join(PKG, "csrc", "*")) + glob.glob(os.path.join(ROOT, "include", "*.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if force or _stale():
        tmp = LIB + f".tmp{os.getpid()}"
        cmd = nvcc_command(tmp, ["-Xptxas", "-v"] if verbose else [])
        subprocess.check_call(cmd)
        os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

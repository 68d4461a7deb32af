"""Build libflint_moe.so in-tree for sm_103a (nvcc cross-compiles; no GPU needed)."""
from __future__ import annotations

import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCES = [os.path.join(HERE, "csrc", "flint_moe.cu")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def build(verbose: bool = False) -> str:
    out = os.path.join(HERE, "libflint_moe.so")
    cmd = ["nvcc", "-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-shared",
           "-o", out, *SOURCES]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd))
    subprocess.check_call(cmd)
    return out


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))

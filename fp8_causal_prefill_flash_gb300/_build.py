"""Build libfp8attn.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SO = os.path.join(PKG, "libfp8attn.so")
SOURCES = [os.path.join(CSRC, "api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("attn_fwd.cuh", "ptx.cuh", "quant.cuh")] + [
    os.path.join(ROOT, "include", "fp8attn.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
              "-Xcompiler", "-fPIC", "-shared"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date() -> bool:
    if not os.path.exists(SO):
        return False
    t = os.path.getmtime(SO)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile the CUDA library (skipped when it is newer than its sources)."""
    if not force and up_to_date():
        return SO
    tmp = SO + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *SOURCES, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, SO)
    return SO


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

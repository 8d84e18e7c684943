"""Build libfp8attn.so in-tree with nvcc for sm_103a (GB300)."""
from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
SO = os.path.join(PKG, "libfp8attn.so")
# debug build with the clock64 role timeline (attn_debug_timeline)
SO_TIMELINE = os.path.join(PKG, "libfp8attn_timeline.so")
SOURCES = [os.path.join(CSRC, "api.cu")]
DEPS = SOURCES + [os.path.join(CSRC, f) for f in ("attn_fwd.cuh", "ptx.cuh", "quant.cuh",
                                                   "split_plan.h")] + [
    os.path.join(ROOT, "include", "fp8attn.h")]

NVCC_FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
              "-Xcompiler", "-fPIC", "-shared"]


def nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def up_to_date(so: str = SO) -> bool:
    if not os.path.exists(so):
        return False
    t = os.path.getmtime(so)
    return all(os.path.getmtime(d) <= t for d in DEPS)


def build(force: bool = False, verbose: bool = False, timeline: bool = False) -> str:
    """Compile the CUDA library (skipped when it is newer than its sources).
    ``timeline`` builds the separate debug library with the role timeline."""
    so = SO_TIMELINE if timeline else SO
    if not force and up_to_date(so):
        return so
    tmp = so + f".tmp{os.getpid()}"
    cmd = [nvcc(), *NVCC_FLAGS, *(["-DFA8_TIMELINE"] if timeline else []), *SOURCES, "-o", tmp]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
        print(" ".join(cmd), file=sys.stderr)
    subprocess.run(cmd, check=True)
    os.replace(tmp, so)
    return so


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))

"""The C ABI used from plain C (tests/c_abi_check.c): it must compile and link
against include/fp8attn.h, libfp8attn.so and the CUDA runtime on any machine
(CPU test), and run on a GPU with exact results (GPU test)."""
import os
import subprocess

import pytest

import fp8_causal_prefill_flash_gb300 as fa

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _build(tmp_path):
    fa.build()
    lib_dir = os.path.dirname(fa.LIBRARY_PATH)
    exe = os.path.join(str(tmp_path), "c_abi_check")
    cmd = ["gcc", "-O2", "-std=c11", "-Wall", "-Werror", os.path.join(HERE, "c_abi_check.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           "-L", lib_dir, "-lfp8attn", "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
           "-Wl,-rpath," + lib_dir, "-Wl,-rpath," + os.path.join(CUDA, "lib64"), "-o", exe]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_compiles_and_links(tmp_path):
    assert os.access(_build(tmp_path), os.X_OK)


@pytest.mark.gpu
def test_c_program_runs(tmp_path):
    exe = _build(tmp_path)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "C ABI check ok" in r.stdout

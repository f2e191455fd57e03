"""CPU check of the vectorised kernels' mask decode and lane gather: builds
tests/decode_host_check.cu for the host with nvcc (the product's
Pattern<N, M>::decode and ::dot compiled for the CPU) and runs it over every
valid chunk mask of 2:4, 1:4, 2:8, 4:8 and the dense patterns, and a sample
of 1:8; and the tensor-core product's 2:4 group expansion table.  No GPU is
used."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "decode_host_check.cu")
CSRC = os.path.join(ROOT, "sparse_spmv_memory_02_b300", "csrc")
INCLUDE = os.path.join(ROOT, "include")


def _nvcc():
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    return None


def test_mask_decode_and_gather_on_the_host(tmp_path):
    nvcc = _nvcc()
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path / "decode_host_check")
    build = subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
                            "-DNM_USE_MIXED_FMA=1", "-I", INCLUDE, "-I", CSRC, SRC, "-o", exe],
                           capture_output=True, text=True, timeout=600)
    assert build.returncode == 0, build.stdout + build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert run.returncode == 0 and run.stdout.strip().endswith("OK"), run.stdout + run.stderr
    # every pattern reported, none with failures
    for pat in ("2:4", "1:4", "2:8", "4:8", "1:8", "4:4", "8:8", "2:4x", "2:4s"):
        line = [l for l in run.stdout.splitlines() if l.startswith(pat + " ")]
        assert line and line[0].endswith(" 0 failures"), run.stdout

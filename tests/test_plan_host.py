"""CPU check of the streaming kernels' launch planning: builds
tests/plan_host_check.cu with the library's planner (csrc/nm_bulk_plan.cu)
for the host and runs it under the default tuning and the forced tunings the
GPU tests use.  Every plan must fit shared memory, cover K and the rows
exactly, keep regions 16-byte aligned and bound the partial sums; the
tensor-core product's K-split plans must respect the SM count, the resident
clusters and the tile sizes.  No GPU is used."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "plan_host_check.cu")
CSRC = os.path.join(ROOT, "sparse_spmv_memory_02_b300", "csrc")
INCLUDE = os.path.join(ROOT, "include")

TUNINGS = ["", "rows_xtile=1024", "rows_task=512", "rows_R=4,rows_warps=3", "rows_ring=4096",
           "ctas=2", "rows_warps=1,rows_xtile=2048,rows_task=512", "rows_R=1",
           "rows_xtile=4096,rows_task=1000,rows_pre=1", "sp_split=0", "sp_k=2", "sp_k=8,sp_units=40"]


@pytest.fixture(scope="module")
def checker(tmp_path_factory):
    nvcc = next((c for c in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc")
                 if c and os.path.exists(c)), None)
    if nvcc is None:
        pytest.skip("nvcc not available")
    exe = str(tmp_path_factory.mktemp("plan") / "plan_host_check")
    build = subprocess.run([nvcc, "-std=c++17", "-O2", "-gencode", "arch=compute_103a,code=sm_103a",
                            "-DNM_USE_MIXED_FMA=1", "-I", INCLUDE, "-I", CSRC, SRC,
                            os.path.join(CSRC, "nm_bulk_plan.cu"), "-o", exe],
                           capture_output=True, text=True, timeout=600)
    assert build.returncode == 0, build.stdout + build.stderr
    return exe


@pytest.mark.parametrize("tune", TUNINGS)
def test_launch_plans_hold_their_invariants(checker, tune):
    env = dict(os.environ, NM_BULK_TUNE=tune)
    run = subprocess.run([checker], capture_output=True, text=True, timeout=300, env=env)
    assert run.returncode == 0 and run.stdout.strip().endswith("OK"), run.stdout[-3000:]
    assert " 0 failures" in run.stdout

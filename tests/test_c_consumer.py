"""The headers are usable from C: tests/c_consumer.c includes include/nm.h
and include/nm_probe.h, compiles with gcc as C99 (-Wall -Werror), links
against libnm.so and calls the entry points that need no GPU."""
import os
import shutil
import subprocess

import pytest

from sparse_spmv_memory_02_b300 import build as nmbuild
from sparse_spmv_memory_02_b300 import nm

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_builds_links_and_runs(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    nmbuild.build()
    exe = str(tmp_path / "c_consumer")
    libdir = os.path.dirname(nm.LIB_PATH)
    build = subprocess.run(
        ["gcc", "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
         "-I", os.path.join(ROOT, "include"), os.path.join(ROOT, "tests", "c_consumer.c"),
         "-L", libdir, "-l:libnm.so", "-Wl,-rpath," + libdir, "-o", exe],
        capture_output=True, text=True, timeout=300)
    assert build.returncode == 0, build.stdout + build.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0 and run.stdout.strip().endswith("OK"), run.stdout + run.stderr

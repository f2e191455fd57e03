"""The device-side failure path, exercised on the GPU without a fault: with
NM_BULK_TUNE=wait_fault_test=1 the streaming SpMV kernel issues no copies, so
nothing ever completes its slot barriers and no copy is in flight; every
wait gives up after 2 ms, sets NM_DEVERR_PIPE_TIMEOUT in the device error
word and the kernel returns.  The host reads the word, clears it, and the
CUDA context is still usable.  The tuning is read once per process, so the
check runs in a child process."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys
sys.path.insert(0, %r)
import torch
import nm_synth
from sparse_spmv_memory_02_b300 import nm
W = nm_synth.weights(300, 1024, 0, "cuda")
A = nm.nm_pack(W, nm_synth.topn_mask(W, 2, 4), 2, 4)
x = nm_synth.activations(1024, 1, 1, True, "cuda")[0]
assert nm.nm_device_errors() == 0
nm.nm_spmv(A, x)                     # every slot wait runs out after 2 ms
flags = nm.nm_device_errors()        # synchronises and clears
assert flags & nm.NM_DEVERR_PIPE_TIMEOUT, flags
assert nm.nm_device_errors() == 0
assert (torch.ones(1000, device="cuda") * 2).sum().item() == 2000.0
print("TIMEOUT REPORTED", flags)
""" % ROOT


def test_slot_wait_timeout_is_reported_and_the_context_survives():
    env = dict(os.environ, NM_BULK_TUNE="wait_fault_test=1")
    r = subprocess.run([sys.executable, "-c", CHILD], env=env, capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0 and "TIMEOUT REPORTED" in r.stdout, r.stdout + r.stderr

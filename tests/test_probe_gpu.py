"""The read-only HBM stream (include/nm_probe.h) reads every byte it is
given: its XOR of all 32-bit words equals the XOR computed on the host, for
sizes that fill several grid sweeps and leave a ragged last sweep."""
import numpy as np
import pytest
import torch

from sparse_spmv_memory_02_b300 import nm

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 48, 4096, 1 << 20, (1 << 24) + 16 * 12345])
def test_probe_reads_every_word(nbytes):
    g = torch.Generator(device="cuda").manual_seed(nbytes)
    buf = torch.randint(-2 ** 31, 2 ** 31 - 1, (nbytes // 4,), generator=g, dtype=torch.int64,
                        device="cuda").to(torch.int32)
    sink = nm.nm_probe_read_stream(buf)
    torch.cuda.synchronize()
    want = np.bitwise_xor.reduce(buf.cpu().numpy().view(np.uint32))
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(want)


def test_probe_empty_and_offset():
    buf = torch.zeros(64, dtype=torch.int32, device="cuda")
    buf[4:8] = torch.tensor([1, 2, 4, 8], dtype=torch.int32)
    sink = torch.full((1,), 77, dtype=torch.int32, device="cuda")
    nm.nm_probe_read_stream(buf[:0], sink)  # nothing read, sink untouched
    torch.cuda.synchronize()
    assert int(sink.item()) == 77
    nm.nm_probe_read_stream(buf[4:], sink)  # 16-byte aligned view
    torch.cuda.synchronize()
    assert int(sink.item()) == 15

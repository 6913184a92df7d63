"""The read-only streaming self-test reads every word of its buffer once:
its XOR fold equals the XOR of the buffer's 32-bit words computed on the
host; misaligned buffers and sizes are refused without a launch."""

import numpy as np
import pytest
import torch

import paged_kv_cache_145_gb300 as pkv

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("nbytes", [16, 4096 + 48, 3 << 20, (1 << 24) + 16 * 7])
def test_fold_covers_every_word(nbytes):
    g = torch.Generator().manual_seed(nbytes % 9973)
    host = torch.randint(0, 256, (nbytes,), dtype=torch.uint8, generator=g)
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    pkv.paged_selftest_read_stream(host.cuda(), sink)
    want = np.bitwise_xor.reduce(host.numpy().view(np.uint32))
    assert int(sink.cpu().numpy().view(np.uint32)[0]) == int(want)


def test_refusals():
    buf = torch.zeros(64, dtype=torch.uint8, device="cuda")
    sink = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(RuntimeError):
        pkv.paged_selftest_read_stream(buf[1:17], sink)   # not 16-byte aligned
    with pytest.raises(RuntimeError):
        pkv.paged_selftest_read_stream(buf[:24], sink)    # not a multiple of 16 bytes
    pkv.paged_selftest_read_stream(buf[:0], sink)         # nothing to read
    assert int(sink.item()) == 0

"""Failure detection on the GPU without a fault: a bounded wait that runs
out reports PKV_DEV_TIMEOUT through the device error word, and the context
stays usable for the next call."""

import time

import numpy as np
import pytest
import torch

import paged_kv_cache_145_gb300 as pkv

pytestmark = pytest.mark.gpu


def test_wait_timeout_is_reported_and_context_survives():
    assert pkv.paged_get_device_error() == 0
    t0 = time.perf_counter()
    pkv.paged_selftest_wait_timeout(20_000_000)  # 20 ms
    assert pkv.paged_get_device_error() == pkv.PKV_DEV_TIMEOUT
    assert time.perf_counter() - t0 >= 0.02
    # The error word was read and cleared; later work runs normally.
    assert pkv.paged_get_device_error() == 0
    k = torch.randn(4, 2, 16, 64).cuda()
    v = torch.randn(4, 2, 16, 64).cuda()
    cache = pkv.PagedKVCache(k, v)
    q = torch.randn(1, 2, 64).cuda()
    out = pkv.paged_attention_decode(cache, q, torch.tensor([[2, 0]], dtype=torch.int32).cuda(),
                                     torch.tensor([20], dtype=torch.int32).cuda(), 0.125)
    assert pkv.paged_get_device_error() == 0
    assert np.all(np.isfinite(out.cpu().numpy()))


def test_wait_timeout_limit_is_checked():
    with pytest.raises(RuntimeError):
        pkv.paged_selftest_wait_timeout(0)
    with pytest.raises(RuntimeError):
        pkv.paged_selftest_wait_timeout(2_000_000_000)

"""Decode attention with the library's fixed scratch (no caller workspace).

paged_attention_decode_static_ws serves callers that cannot allocate device
memory themselves -- for example a plug-in inside a host program that owns
and reserves GPU memory up front, or a latency-critical path where a
cudaMalloc could synchronise the device.  This file checks, through the C
ABI, that two calls in a row give results identical to the allocating
entry point's (both run the same kernels on the same inputs, so every
element must be equal), that sampled rows match the float64 oracle, that a
call changes neither the device's free memory nor torch's allocation count,
that nothing from the first call leaks into the second, and that requests
larger than the fixed scratch are refused.  It is collected last so a
failure here cannot hide other tests.
"""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_145_gb300 as pkv
from oracle import attention as A
from paged_kv_cache_145_gb300 import _lib, synth
from tests.workload import TOL, gpu_out_f64

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def make_case(seed, num_seqs, heads, kv_heads, lo, hi, dtype=torch.bfloat16, b=16, d=128):
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(lo, hi + 1, (num_seqs,), generator=g, dtype=torch.int32)
    nblk = [-(-int(x) // b) for x in lens]
    n = sum(nblk) + 5
    perm = torch.randperm(n, generator=g)
    width = max(nblk)
    tables = torch.full((num_seqs, width), -1, dtype=torch.int32)
    pos = 0
    for i, k in enumerate(nblk):
        tables[i, :k] = perm[pos:pos + k]
        pos += k
    k_cache = torch.randn(n, kv_heads, b, d, generator=g).to(dtype).cuda()
    v_cache = torch.randn(n, kv_heads, b, d, generator=g).to(dtype).cuda()
    q = torch.randn(num_seqs, heads, d, generator=g).to(dtype).cuda()
    return pkv.PagedKVCache(k_cache, v_cache), q, tables.cuda(), lens.cuda(), int(lens.max())


def call_static(cache, q, tables, lens, scale, out, max_len, part):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return _lib.lib().paged_attention_decode_static_ws(
        cache.ref, _p(q), _p(tables), tables.shape[1], _p(lens), q.shape[0], q.shape[1],
        max_len, float(scale), _p(out), part, stream)


def test_two_calls_match_the_allocating_entry_point():
    cases = [dict(seed=1, num_seqs=24, heads=32, kv_heads=8, lo=200, hi=3000),
             dict(seed=2, num_seqs=40, heads=16, kv_heads=16, lo=1, hi=2100)]
    for i, spec in enumerate(cases):  # two calls in a row, different shapes: stale scratch must not matter
        cache, q, tables, lens, max_len = make_case(**spec)
        scale = 1.0 / np.sqrt(q.shape[-1])
        need = pkv.paged_attention_workspace_bytes(cache, q.shape[0], q.shape[1], max_len, 512)
        assert 0 < need <= _lib.PKV_STATIC_WS_BYTES  # split-K is exercised
        ref = pkv.paged_attention_decode(cache, q, tables, lens, scale, max_seq_len=max_len,
                                         partition_size=512)
        out = torch.full_like(q, float("nan"))
        torch.cuda.synchronize()
        free_before, allocated_before = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated()
        assert call_static(cache, q, tables, lens, scale, out, max_len, 512) == 0
        torch.cuda.synchronize()
        # The call allocates nothing: torch's allocation count is the same
        # after it as before, and so is the device's free memory once the
        # array is resident (under lazy module loading the first call on a
        # device is when the driver commits the fixed array itself).
        assert torch.cuda.memory_allocated() == allocated_before
        if i > 0:
            assert torch.cuda.mem_get_info()[0] == free_before
        assert pkv.paged_get_device_error() == 0
        assert torch.equal(out, ref)
        # Sampled rows against the float64 oracle (first, middle, last).
        got = gpu_out_f64(out)
        rows = sorted({0, q.shape[0] // 2, q.shape[0] - 1})
        want, bad = A.attention(synth.storage_numpy(q.cpu(), "bf16"),
                                synth.storage_numpy(cache.k_cache.cpu(), "bf16"),
                                synth.storage_numpy(cache.v_cache.cpu(), "bf16"),
                                [list(r) for r in tables.cpu().numpy()], lens.cpu().tolist(),
                                scale, 16, "bf16", seqs=rows)
        assert bad == []
        assert np.all(np.isfinite(got))
        assert max(float(np.max(np.abs(got[s] - want[s]))) for s in rows) <= TOL["bf16"]


def test_oversized_request_is_refused():
    cache, q, tables, lens, _ = make_case(seed=3, num_seqs=4, heads=8, kv_heads=8, lo=10, hi=20)
    out = torch.empty_like(q)
    # 4096 sequences x 32 heads x 64 partitions of scratch is far above the
    # fixed array; the pointers are never dereferenced because the call
    # refuses before enqueuing anything.
    big = _lib.lib().paged_attention_decode_static_ws(
        cache.ref, _p(q), _p(tables), 2048, _p(lens), 4096, 32, 32768, 0.1, _p(out), 512,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert big == _lib.PKV_ERR_WORKSPACE
    assert pkv.paged_get_device_error() == 0

"""GPU block swap between the device pool and pinned host memory, against
the oracle: bit-exact both ways, out-of-range pairs, unpinned memory, and a
preempt-by-swap round trip through decode attention."""

import ctypes

import numpy as np
import pytest
import torch

import paged_kv_cache_145_gb300 as pkv
from oracle import attention as A
from paged_kv_cache_145_gb300 import _lib, synth

pytestmark = pytest.mark.gpu


def host(t, dt):
    return synth.storage_numpy(t, dt)


def pools(dt, n, hk, b, d, seed, device="cpu"):
    g = torch.Generator().manual_seed(seed)
    t = synth.TORCH_DTYPE[dt]
    return (torch.randn(n, hk, b, d, generator=g).to(t).to(device),
            torch.randn(n, hk, b, d, generator=g).to(t).to(device))


@pytest.mark.parametrize("dt,hk,b,d", [("bf16", 8, 16, 128), ("f16", 40, 16, 128), ("f32", 4, 32, 64)])
def test_swap_out_and_in_bit_exact(dt, hk, b, d):
    dk, dv = pools(dt, 40, hk, b, d, 1)
    hk_, hv_ = pools(dt, 25, hk, b, d, 2)
    hk_, hv_ = hk_.pin_memory(), hv_.pin_memory()
    cache = pkv.PagedKVCache(dk.cuda(), dv.cuda())
    perm = np.random.default_rng(3).permutation(40)
    out_pairs = [(int(perm[i]), int(i)) for i in range(20)]
    pkv.paged_block_swap(cache, hk_, hv_, torch.tensor(out_pairs).cuda(), pkv.PKV_SWAP_OUT)
    assert pkv.paged_get_device_error() == 0
    ek, ev, ehk, ehv, bad = A.swap_blocks(host(dk, dt), host(dv, dt), host(pools(dt, 25, hk, b, d, 2)[0], dt),
                                          host(pools(dt, 25, hk, b, d, 2)[1], dt), out_pairs, "out")
    assert bad == []
    assert np.array_equal(host(hk_, dt), ehk) and np.array_equal(host(hv_, dt), ehv)
    assert np.array_equal(host(cache.k_cache, dt), ek)
    in_pairs = [(int(i), int(perm[39 - i])) for i in range(12)]
    pkv.paged_block_swap(cache, hk_, hv_, torch.tensor(in_pairs).cuda(), pkv.PKV_SWAP_IN)
    assert pkv.paged_get_device_error() == 0
    ek2, ev2, _, _, bad = A.swap_blocks(ek, ev, ehk, ehv, in_pairs, "in")
    assert bad == []
    assert np.array_equal(host(cache.k_cache, dt), ek2) and np.array_equal(host(cache.v_cache, dt), ev2)


def test_swap_bad_pairs_flagged():
    dk, dv = pools("bf16", 10, 2, 16, 64, 4)
    hk_, hv_ = pools("bf16", 3, 2, 16, 64, 5)
    hk_, hv_ = hk_.pin_memory(), hv_.pin_memory()
    before_h = host(hk_, "bf16").copy()
    cache = pkv.PagedKVCache(dk.cuda(), dv.cuda())
    pairs = [(1, 0), (10, 1), (2, 3), (-1, 2)]
    pkv.paged_block_swap(cache, hk_, hv_, torch.tensor(pairs).cuda(), pkv.PKV_SWAP_OUT)
    assert pkv.paged_get_device_error() == pkv.PKV_DEV_PAIR_RANGE
    _, _, ehk, _, bad = A.swap_blocks(host(dk, "bf16"), host(dv, "bf16"), before_h,
                                      host(pools("bf16", 3, 2, 16, 64, 5)[1], "bf16"), pairs, "out")
    assert bad == [1, 2, 3]
    assert np.array_equal(host(hk_, "bf16"), ehk)


def test_unpinned_host_memory_is_refused():
    dk, dv = pools("f16", 4, 1, 16, 64, 6)
    cache = pkv.PagedKVCache(dk.cuda(), dv.cuda())
    hk_ = torch.zeros(2, 1, 16, 64, dtype=torch.float16)  # pageable
    pairs = torch.tensor([[0, 1]]).cuda()
    rc = _lib.lib().paged_block_swap(cache.ref, ctypes.c_void_p(hk_.data_ptr()),
                                     ctypes.c_void_p(hk_.data_ptr()), 2,
                                     ctypes.c_void_p(pairs.data_ptr()), 1, 0,
                                     ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -3
    with pytest.raises(ValueError):
        pkv.paged_block_swap(cache, hk_, hk_, pairs, pkv.PKV_SWAP_OUT)


def test_preempt_by_swap_round_trip_through_decode():
    # A batch decodes; sequence 1 is preempted: its blocks go to host memory,
    # the device blocks are reused (overwritten), later the data comes back
    # into other free blocks and its table is remapped.  The decode output
    # after restoring must equal the output before preemption, bit for bit.
    b, hk, d, G = 16, 8, 128, 4
    lens = [300, 517, 64]
    nblk = [-(-L // b) for L in lens]
    n = sum(nblk) + nblk[1] + 4
    dk, dv = pools("bf16", n, hk, b, d, 7)
    cache = pkv.PagedKVCache(dk.cuda(), dv.cuda())
    tables = np.full((3, max(nblk)), -1, dtype=np.int32)
    pos = 0
    for i, k in enumerate(nblk):
        tables[i, :k] = np.arange(pos, pos + k)
        pos += k
    spare = list(range(pos, n))
    q = torch.randn(3, hk * G, d, generator=torch.Generator().manual_seed(8)).bfloat16().cuda()
    lens_t = torch.tensor(lens, dtype=torch.int32).cuda()
    out1 = pkv.paged_attention_decode(cache, q, torch.from_numpy(tables).cuda(), lens_t, 0.088)
    hk_ = torch.empty(nblk[1], hk, b, d, dtype=torch.bfloat16).pin_memory()
    hv_ = torch.empty_like(hk_).pin_memory()
    victim = tables[1, :nblk[1]].copy()
    pkv.paged_block_swap(cache, hk_, hv_, torch.tensor([[int(x), i] for i, x in enumerate(victim)]).cuda(),
                         pkv.PKV_SWAP_OUT)
    cache.k_cache[torch.from_numpy(victim).long().cuda()] = 0   # blocks reused by someone else
    cache.v_cache[torch.from_numpy(victim).long().cuda()] = 0
    fresh = spare[:nblk[1]]
    pkv.paged_block_swap(cache, hk_, hv_, torch.tensor([[i, f] for i, f in enumerate(fresh)]).cuda(),
                         pkv.PKV_SWAP_IN)
    tables[1, :nblk[1]] = fresh
    out2 = pkv.paged_attention_decode(cache, q, torch.from_numpy(tables).cuda(), lens_t, 0.088)
    assert pkv.paged_get_device_error() == 0
    assert torch.equal(out1, out2)

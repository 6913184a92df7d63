"""GPU KV write and block copy against the oracle: bit-exact over every byte
of both pools, plus padding, out-of-range and no-op cases."""

import numpy as np
import pytest
import torch

import paged_kv_cache_145_gb300 as pkv
from oracle import attention as A
from paged_kv_cache_145_gb300 import synth

pytestmark = pytest.mark.gpu


def pools(dtype, n, hk, b, d, seed):
    g = torch.Generator().manual_seed(seed)
    t = synth.TORCH_DTYPE[dtype]
    return (torch.randn(n, hk, b, d, generator=g).to(t), torch.randn(n, hk, b, d, generator=g).to(t))


def host(t, dtype):
    return synth.storage_numpy(t, dtype)


@pytest.mark.parametrize("dtype,hk,b,d", [("f32", 4, 16, 64), ("f16", 40, 16, 128),
                                          ("bf16", 8, 16, 128), ("bf16", 8, 32, 128),
                                          ("f16", 2, 8, 64), ("f32", 3, 5, 4)])
def test_write_bit_exact(dtype, hk, b, d):
    n = 23
    kp, vp = pools(dtype, n, hk, b, d, 1)
    g = torch.Generator().manual_seed(2)
    slots = torch.randperm(n * b, generator=g)[:37].to(torch.int64)
    slots[5] = -1                      # padding token
    slots[9] = -3
    kn = torch.randn(37, hk, d, generator=g).to(kp.dtype)
    vn = torch.randn(37, hk, d, generator=g).to(kp.dtype)
    cache = pkv.PagedKVCache(kp.cuda(), vp.cuda())
    pkv.paged_kv_write(cache, kn.cuda(), vn.cuda(), slots.cuda())
    assert pkv.paged_get_device_error() == 0
    ek, ev, bad = A.write_tokens(host(kp, dtype), host(vp, dtype), host(kn, dtype), host(vn, dtype),
                                 slots.tolist(), b)
    assert bad == []
    assert np.array_equal(host(cache.k_cache, dtype), ek)
    assert np.array_equal(host(cache.v_cache, dtype), ev)


def test_write_out_of_range_slot_is_flagged_and_skipped():
    kp, vp = pools("f16", 6, 2, 16, 64, 3)
    slots = torch.tensor([3, 6 * 16, 40, 10 ** 9], dtype=torch.int64)
    kn, vn = torch.randn(4, 2, 64).half(), torch.randn(4, 2, 64).half()
    cache = pkv.PagedKVCache(kp.cuda(), vp.cuda())
    pkv.paged_kv_write(cache, kn.cuda(), vn.cuda(), slots.cuda())
    assert pkv.paged_get_device_error() == pkv.PKV_DEV_SLOT_RANGE
    assert pkv.paged_get_device_error() == 0  # reading clears the word
    ek, ev, bad = A.write_tokens(host(kp, "f16"), host(vp, "f16"), host(kn, "f16"), host(vn, "f16"),
                                 slots.tolist(), 16)
    assert bad == [1, 3]
    assert np.array_equal(host(cache.k_cache, "f16"), ek)
    assert np.array_equal(host(cache.v_cache, "f16"), ev)


def test_prefill_sized_write_fills_whole_sequences():
    # Every position of two sequences written in one call, through their tables.
    b, hk, d = 16, 8, 128
    kp, vp = pools("bf16", 40, hk, b, d, 4)
    tables = [[31, 2, 17, 9, 0], [5, 38, 21]]
    lens = [70, 41]
    slots = [tables[s][t // b] * b + t % b for s in range(2) for t in range(lens[s])]
    n = len(slots)
    g = torch.Generator().manual_seed(5)
    kn = torch.randn(n, hk, d, generator=g).bfloat16()
    vn = torch.randn(n, hk, d, generator=g).bfloat16()
    cache = pkv.PagedKVCache(kp.cuda(), vp.cuda())
    pkv.paged_kv_write(cache, kn.cuda(), vn.cuda(), torch.tensor(slots).cuda())
    assert pkv.paged_get_device_error() == 0
    ek, ev, _ = A.write_tokens(host(kp, "bf16"), host(vp, "bf16"), host(kn, "bf16"),
                               host(vn, "bf16"), slots, b)
    assert np.array_equal(host(cache.k_cache, "bf16"), ek)
    assert np.array_equal(host(cache.v_cache, "bf16"), ev)


def test_empty_write_is_a_no_op():
    kp, vp = pools("f32", 3, 1, 16, 64, 6)
    cache = pkv.PagedKVCache(kp.cuda(), vp.cuda())
    e = torch.empty(0, 1, 64, device="cuda")
    pkv.paged_kv_write(cache, e, e, torch.empty(0, dtype=torch.int64, device="cuda"))
    assert torch.equal(cache.k_cache.cpu(), kp)


@pytest.mark.parametrize("dtype,hk,b,d", [("bf16", 8, 16, 128), ("f16", 40, 16, 128),
                                          ("f32", 4, 32, 64), ("bf16", 1, 8, 64)])
def test_copy_bit_exact(dtype, hk, b, d):
    n = 50
    kp, vp = pools(dtype, n, hk, b, d, 7)
    perm = np.random.default_rng(8).permutation(n)
    pairs = [(int(perm[i]), int(perm[25 + i])) for i in range(20)]
    cache = pkv.PagedKVCache(kp.cuda(), vp.cuda())
    pkv.paged_block_copy(cache, torch.tensor(pairs, dtype=torch.int64).cuda())
    assert pkv.paged_get_device_error() == 0
    ek, ev, bad = A.copy_blocks(host(kp, dtype), host(vp, dtype), pairs)
    assert bad == []
    assert np.array_equal(host(cache.k_cache, dtype), ek)
    assert np.array_equal(host(cache.v_cache, dtype), ev)


def test_copy_bad_pairs_flagged_and_self_copy_no_op():
    kp, vp = pools("bf16", 10, 8, 16, 128, 9)
    pairs = [(1, 2), (3, 10), (-1, 4), (5, 5), (6, 7)]
    cache = pkv.PagedKVCache(kp.cuda(), vp.cuda())
    pkv.paged_block_copy(cache, torch.tensor(pairs, dtype=torch.int64).cuda())
    assert pkv.paged_get_device_error() == pkv.PKV_DEV_PAIR_RANGE
    ek, ev, bad = A.copy_blocks(host(kp, "bf16"), host(vp, "bf16"), pairs)
    assert bad == [1, 2]
    assert np.array_equal(host(cache.k_cache, "bf16"), ek)
    assert np.array_equal(host(cache.v_cache, "bf16"), ev)


def test_cow_demo_on_device():
    # The pages' copy-on-write demo with real K/V rows: a pool of 6 blocks of
    # width 4; A holds positions 1..5, C forks A and appends a sixth.  After
    # the copy and the write, A's rows are unchanged and C's read A's prefix
    # followed by the new row; the first block stays shared.
    hk, b, d = 2, 4, 64
    bm = pkv.BlockManager(6, b)
    bm.admit(0, 5)
    bm.fork(0, 1)
    kp, vp = pools("f16", 6, hk, b, d, 10)
    cache = pkv.PagedKVCache(kp.cuda(), vp.cuda())
    tab_before, _ = bm.tables([0], 2)
    slots, pairs = bm.append([1])
    assert len(pairs) == 1 and pairs[0][0] == tab_before[0][1]
    kn, vn = torch.randn(1, hk, d).half(), torch.randn(1, hk, d).half()
    pkv.paged_block_copy(cache, torch.from_numpy(pairs).cuda())
    pkv.paged_kv_write(cache, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    assert pkv.paged_get_device_error() == 0
    tabs, lens = bm.tables([0, 1], 2)
    assert list(lens) == [5, 6] and tabs[0][0] == tabs[1][0] and tabs[0][1] != tabs[1][1]
    k = cache.k_cache.cpu()

    def rows(s, n):
        return torch.stack([k[int(tabs[s][t // b]), :, t % b] for t in range(n)])

    orig = torch.stack([kp[int(tab_before[0][t // b]), :, t % b] for t in range(5)])
    assert torch.equal(rows(0, 5), orig)
    assert torch.equal(rows(1, 5), orig) and torch.equal(rows(1, 6)[5], kn[0])

"""The native host block manager against the oracle's block pool (no GPU).

Both are driven with the same free-list order and the same operations; their
tables, slots, copy-on-write pairs, reference counts and free counts must be
identical, entry for entry."""

import random

import numpy as np
import pytest

from oracle import blocks as B
from oracle import paging as P
from paged_kv_cache_145_gb300 import BlockManager
from paged_kv_cache_145_gb300 import synth


def same_state(bm, pool, names):
    for n in names:
        width = max(1, bm.num_seq_blocks(n))
        tab, lens = bm.tables([n], width)
        assert list(tab[0]) == pool.table(n)
        assert int(lens[0]) == pool.length(n) == bm.seq_len(n)
    assert bm.num_free() == pool.num_free()
    counts = pool.refcounts()
    for blk in range(pool.num_blocks):
        assert bm.refcount(blk) == counts[blk]
    assert bm.check()


def test_random_operations_match_oracle():
    rng = random.Random(5)
    n, b = 48, 4
    order = rng.sample(range(n), n)
    bm = BlockManager(n, b, order)
    pool = B.BlockPool(n, b, free_order=order)
    live = []
    for step in range(600):
        op = rng.random()
        if op < 0.2 or not live:
            ln = rng.randint(1, 14)
            try:
                pool.admit(step, list(range(ln)))
            except MemoryError:
                with pytest.raises(MemoryError):
                    bm.admit(step, ln)
                continue
            bm.admit(step, ln)
            live.append(step)
        elif op < 0.35:
            src = rng.choice(live)
            pool.fork(src, step)
            bm.fork(src, step)
            live.append(step)
        elif op < 0.85:
            batch = [rng.choice(live) for _ in range(rng.randint(1, 4))]
            snap = (pool.num_free(), {x: pool.table(x) for x in live})
            try:
                expect = []
                for x in batch:
                    r = pool.append(x, 0)
                    expect.append(r)
            except MemoryError:
                # The native step is all-or-nothing; rebuild the oracle to
                # the pre-step state by replaying is not possible, so only
                # check that the native side refuses and stays unchanged.
                with pytest.raises(MemoryError):
                    bm.append(batch)
                pool = None
                break
            slots, pairs = bm.append(batch)
            assert list(slots) == [r.slot for r in expect]
            assert [tuple(p) for p in pairs] == [r.copy for r in expect if r.copy]
        else:
            x = live.pop(rng.randrange(len(live)))
            pool.release(x)
            bm.release(x)
        same_state(bm, pool, live)


def test_worked_example_tables():
    # b = 16: 50 tokens take 4 blocks; the 51st position is at offset 2 of the
    # 4th entry; 65 tokens take 5 blocks.
    order = [7, 3, 12, 5] + [i for i in range(16) if i not in (7, 3, 12, 5)]
    bm = BlockManager(16, 16, order)
    bm.admit(1, 50)
    tab, lens = bm.tables([1], 4)
    slots, pairs = bm.append([1])
    assert list(tab[0]) == [7, 3, 12, 5] and lens[0] == 50
    assert slots[0] == 5 * 16 + 2 and len(pairs) == 0
    bm.admit(2, 65)
    assert bm.num_seq_blocks(2) == 5 == P.blocks_needed(65, 16)


def test_fork_workload_copies():
    b, prompt, forks = 16, 1031, 8
    n = synth.pool_with_slack(P.blocks_needed(prompt, b) + forks, 0.1)
    order = synth.free_order(3, n)
    bm = BlockManager(n, b, order)
    pool = B.BlockPool(n, b, free_order=order, auto_verify=False)
    bm.admit(0, prompt)
    pool.admit(0, list(range(prompt)))
    for f in range(1, forks):
        bm.fork(0, f)
        pool.fork(0, f)
    slots, pairs = bm.append(list(range(forks)))
    expect = [pool.append(f, 0) for f in range(forks)]
    assert list(slots) == [r.slot for r in expect]
    assert [tuple(p) for p in pairs] == [r.copy for r in expect if r.copy]
    assert len(pairs) == forks - 1
    pool.verify()
    same_state(bm, pool, list(range(forks)))


def test_append_is_all_or_nothing():
    bm = BlockManager(2, 4)
    bm.admit(0, 4)            # full block
    bm.admit(1, 2)
    bm.fork(1, 2)             # shared partial block, no free block left
    before = (bm.tables([0, 1, 2], 2), bm.num_free())
    with pytest.raises(MemoryError):
        bm.append([1, 0])     # needs two fresh blocks, none free
    after = (bm.tables([0, 1, 2], 2), bm.num_free())
    assert all(np.array_equal(a, c) for a, c in zip(before[0], after[0])) and before[1] == after[1]
    assert bm.check()


def test_bad_arguments():
    with pytest.raises(ValueError):
        BlockManager(4, 16, [0, 1, 1, 2])
    bm = BlockManager(4, 16)
    with pytest.raises(RuntimeError):
        bm.admit(0, 0)
    bm.admit(0, 5)
    with pytest.raises(RuntimeError):
        bm.admit(0, 5)
    with pytest.raises(RuntimeError):
        bm.fork(9, 1)
    with pytest.raises(RuntimeError):
        bm.release(9)
    with pytest.raises(RuntimeError):
        bm.tables([0], 0)


def test_oversized_requests_change_nothing():
    # Requests whose rounded-up block count or position range would overflow
    # 64 bits are refused, and the manager is left as it was.
    bm = BlockManager(8, 16)
    bm.admit(0, 20)
    free = bm.num_free()
    for n in (2**62, 2**63 - 1):
        with pytest.raises(MemoryError):
            bm.admit(1, n)
    assert bm.num_free() == free and bm.seq_len(1) == -1 and bm.check()
    assert bm._lib.pkv_bm_slots(bm._h, 0, 1, 2**63 - 1, None) == -3   # start + count overflows
    assert list(bm.slots(0, 0, 20)) == [bm.tables([0], 2)[0][0][t // 16] * 16 + t % 16
                                        for t in range(20)]


def test_slots_query_matches_oracle_translation():
    rng = random.Random(9)
    order = rng.sample(range(64), 64)
    bm = BlockManager(64, 8, order)
    pool = B.BlockPool(64, 8, free_order=order)
    for s, n in enumerate([13, 1, 40, 8]):
        bm.admit(s, n)
        pool.admit(s, list(range(n)))
        table = pool.table(s)
        expect = [P.translate(t, 8, table)[3] for t in range(n)]
        assert list(bm.slots(s, 0, n)) == expect
        assert list(bm.slots(s, n // 2, n - n // 2)) == expect[n // 2:]
    with pytest.raises(RuntimeError):
        bm.slots(0, 10, 4)   # past the sequence end

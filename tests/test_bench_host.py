"""Host-side logic of bench.py (no GPU): byte accounting pinned to the pages'
per-token KV figure, and the rank-combining rule run on 2 gloo ranks."""

import os
import socket

import numpy as np
import torch.multiprocessing as tmp

import bench
from oracle import paging as P


def test_decode_bytes_per_position_match_kv_sizing():
    # OPT-13B: about 800 KB of KV per token over 40 layers ("vLLM and
    # PagedAttention: Virtual Memory for LLM Serving", sizing paragraph), so
    # one layer's keys + values are 1/40 of the oracle's per-token figure.
    w = bench.Workload("opt13b")
    _, kv = w.decode_bytes(512)
    per_pos = kv / int(w.seq_lens.sum())
    assert per_pos == P.kv_bytes_per_token(40, 5120, 2) / 40 == 20480
    g = bench.Workload("gqa")
    _, kv = g.decode_bytes(512)
    assert kv / int(g.seq_lens.sum()) == 2 * 8 * 128 * 2


def test_workload_plans_one_new_position_per_sequence():
    w = bench.Workload("opt13b")
    assert len(w.slots) == w.S == 64 and len(w.pairs) == 0
    assert np.all(w.seq_lens == bench.synth.lengths("opt13b") + 1)
    f = bench.Workload("fork")
    assert len(f.pairs) == 16 * 7


def test_unique_bytes_count_shared_pages_once():
    # Parallel sampling: each group's 64 full prompt blocks are shared by its
    # 8 forks; copy-on-write gave 7 forks a private copy of the partial last
    # block and the 8th kept the original, each now holding 8 positions.
    f = bench.Workload("fork")
    per_pos = 2 * 8 * 128 * 2
    assert f.unique_kv_bytes() == 16 * (64 * 16 + 8 * 8) * per_pos
    _, logical = f.decode_bytes(512)
    assert logical == 16 * 8 * 1032 * per_pos
    # No sharing: unique equals logical.
    w = bench.Workload("opt13b")
    assert w.unique_kv_bytes() == w.decode_bytes(512)[1]


def test_reference_arm_steps_are_bounded_and_counted():
    # K + W steps of the oracle in one process; the head count per step is
    # chosen so the whole run stays near its time target.
    b, secs, steps, h, hk = bench._reference_steps("tiny", 6, 2, 4242, distinct=2, target_s=60.0)
    assert steps == 6 and 1 <= h <= hk == 4 and secs > 0
    lens = bench._lengths("tiny")
    per = [2 * (int(lens[i]) + 1) * h * 64 * 4 for i in range(2)]
    assert b == 3 * per[0] + 3 * per[1]
    _, _, _, h_small, _ = bench._reference_steps("tiny", 20, 0, 4242, distinct=1, target_s=1e-6)
    assert h_small == 1


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, results):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    b, s = bench.combine_ranks(1000 * (rank + 1), 0.5 + rank)
    results[rank] = (b, s)
    dist.barrier()
    dist.destroy_process_group()


def test_combine_ranks_two_gloo_ranks():
    port = _free_port()
    mgr = tmp.Manager()
    results = mgr.dict()
    tmp.spawn(_rank, args=(2, port, results), nprocs=2, join=True)
    assert results[0] == results[1] == (3000.0, 1.5)


def test_slot_utilization_matches_oracle_closed_form():
    # The bench's utilization (positions over allocated slots, from the native
    # block manager) equals the oracle's sum(T) / sum(b * ceil(T / b)).
    for b in (8, 16, 32, 64):
        for table in ("shuffled", "identity"):
            w = bench.Workload("opt13b", block_size=b, table=table)
            lens = [int(x) for x in w.seq_lens]
            assert abs(w.utilization - float(P.paged_utilization(lens, b))) < 1e-12


def test_cpu_baseline_samples_count_their_work():
    # Prefill: one (sequence, KV head) pair of the chunked workload covers
    # 512 queries x 4 query heads, query i seeing 4096 + i + 1 positions;
    # QK^T and PV are 2 * 128 FLOPs each per visible position.
    f, secs, pairs, q = bench._oracle_prefill_sample("chunked", 1e-9, 4242, False)
    assert pairs == 1 and q == 512 and secs > 0
    assert f == 4 * 128 * 4 * (512 * 4097 + 511 * 512 // 2)
    # Data movers: bytes counted as the GPU line counts them.
    blk = 40 * 16 * 128 * 2
    b, secs, units = bench._oracle_op_sample("opt13b", "copy", 1e-9, 4242)
    assert units == 256 and b == 2 * 2 * 256 * blk + 16 * 256
    b, secs, units = bench._oracle_op_sample("opt13b", "swap", 1e-9, 4242)
    assert units == 256 and b == 2 * (2 * 256 * blk + 16 * 256)
    b, secs, units = bench._oracle_op_sample("gqa", "write", 1e-9, 4242)
    n = int(bench._lengths("gqa")[0])
    assert units == n and b == 2 * 2 * n * 8 * 128 * 2 + 8 * n

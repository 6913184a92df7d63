"""GPU parity: the CUDA path against the float64 oracle, on every workload.

Each test plans a decode step with both allocators (which must agree entry
for entry), runs copy-on-write, KV write and decode attention on the GPU,
and compares: pools bit-exact over every byte, attention within the stated
tolerance.  Full-size workloads compare the whole pool and a seeded sample
of attention rows.
"""

import numpy as np
import pytest
import torch

import paged_kv_cache_145_gb300 as pkv
from paged_kv_cache_145_gb300 import synth
from tests.workload import (TOL, Sequences, StepData, gpu_out_f64, max_err, run_gpu,
                            run_oracle)

pytestmark = pytest.mark.gpu


def sample_rows(n, k, seed):
    if n <= k:
        return list(range(n))
    rows = np.random.default_rng(seed).choice(n, size=k, replace=False)
    return sorted(int(x) for x in rows)


def check_step(seqs, data, sample=None, partition_size=0):
    seqs.check_plans_agree()
    cache, out, err = run_gpu(seqs, data, partition_size=partition_size)
    assert err == 0
    kp, vp, ref = run_oracle(seqs, data, sample=sample)
    dt = data.dtype
    assert np.array_equal(synth.storage_numpy(cache.k_cache, dt), kp)
    assert np.array_equal(synth.storage_numpy(cache.v_cache, dt), vp)
    rows = range(len(seqs.ids)) if sample is None else sample
    got = gpu_out_f64(out)
    assert np.all(np.isfinite(got))
    e = max_err(got, ref, rows)
    assert e <= TOL[dt], "max abs error %.3g > %.3g" % (e, TOL[dt])
    return got, ref, e


def test_tiny_step():
    seqs = Sequences("tiny")
    check_step(seqs, StepData(seqs))


def test_tiny_step_worked_example_table():
    # The first sequence (50 cached tokens) gets the table 7 3 12 5; its new
    # token, zero-based position 50, lands at offset 2 of physical block 5.
    seqs = Sequences("tiny", pinned_prefix=[7, 3, 12, 5])
    assert list(seqs.tables[0][:4]) == [7, 3, 12, 5]
    assert seqs.slots[0] == 5 * 16 + 2
    # 65 cached tokens need a fifth block; the new position 65 is offset 1
    # of that fifth block.
    assert seqs.bm.num_seq_blocks(2) == 5
    assert seqs.slots[2] == int(seqs.tables[2][4]) * 16 + 1
    check_step(seqs, StepData(seqs))


@pytest.mark.parametrize("part", [16, 32, 48])
def test_tiny_step_split(part):
    seqs = Sequences("tiny")
    check_step(seqs, StepData(seqs), partition_size=part)


def test_opt13b_full_size():
    seqs = Sequences("opt13b")
    data = StepData(seqs, pool_device="cuda")
    check_step(seqs, data, sample=sample_rows(len(seqs.ids), 6, 11))


def test_gqa_full_size():
    seqs = Sequences("gqa")
    data = StepData(seqs, pool_device="cuda")
    check_step(seqs, data, sample=sample_rows(len(seqs.ids), 12, 12))


def test_fork_full_size():
    seqs = Sequences("fork")
    assert len(seqs.pairs) == seqs.groups * (seqs.forks - 1)
    prompt_blocks = seqs.prompt // seqs.b
    for g in range(seqs.groups):
        shared = seqs.tables[g * seqs.forks][:prompt_blocks]
        for f in range(seqs.forks):
            row = seqs.tables[g * seqs.forks + f]
            assert np.array_equal(row[:prompt_blocks], shared)
            assert seqs.bm.refcount(int(row[prompt_blocks])) == 1
        assert all(seqs.bm.refcount(int(x)) == seqs.forks for x in shared)
    data = StepData(seqs, pool_device="cuda")
    check_step(seqs, data, sample=sample_rows(len(seqs.ids), 12, 13))


@pytest.mark.parametrize("block_size", [16, 32])
def test_long_context_split_k(block_size):
    seqs = Sequences("long", block_size=block_size)
    data = StepData(seqs, pool_device="cuda")
    part = synth.CONFIGS["long"]["partition_size"]
    # All 8 sequences: the only full-size case with 33-65 partition merges.
    check_step(seqs, data, sample=list(range(len(seqs.ids))), partition_size=part)

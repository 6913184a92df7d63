"""Builds one decode step of a named workload on both sides, independently.

Product side: the native BlockManager decides tables, slots and copy pairs;
the CUDA kernels copy, write and attend.  Oracle side: the oracle's
BlockPool decides the same things from the same free-list order; the
oracle's float64 functions copy, write and attend.  Only the seeded inputs
from ``synth`` are shared.
"""

import math

import numpy as np
import torch

import paged_kv_cache_145_gb300 as pkv
from oracle import attention as A
from oracle import blocks as B
from oracle import paging as P
from paged_kv_cache_145_gb300 import synth

# Attention tolerances (max abs error vs the float64 oracle): fp16 2e-3 and
# bf16 8e-3 are the stated bars at fp32 accumulation; fp32 1e-5 is derived
# (fp32 rounding of ~D-term dot products and a ~T-term weighted mean).
TOL = {"f32": 1e-5, "f16": 2e-3, "bf16": 8e-3}


def edge_tol(dtype, ref):
    """Tolerance for edge cases whose outputs are not small (|out| >~ 1).

    The output is rounded once to its dtype, so the bar is the stated
    tolerance or one unit in the last place at the reference's magnitude,
    whichever is larger.
    """
    mant = {"f32": 23, "f16": 10, "bf16": 7}[dtype]
    mag = np.maximum(np.abs(ref), 2.0 ** -14)
    ulp = 2.0 ** (np.floor(np.log2(mag)) - mant)
    return np.maximum(TOL[dtype], ulp)


class Sequences:
    """Sequence ids and the host-side plan of one step (both allocators)."""

    def __init__(self, name, batch=None, free_order_seed=None, block_size=None, lengths=None,
                 pinned_prefix=None):
        cfg = synth.CONFIGS[name]
        self.name = name
        self.cfg = cfg
        self.b = block_size or cfg["block_size"]
        b = self.b
        if name == "fork":
            groups, forks, prompt = cfg["groups"], cfg["forks"], cfg["prompt"]
            self.groups, self.forks, self.prompt = groups, forks, prompt
            self.ids = [g * forks + f for g in range(groups) for f in range(forks)]
            need = groups * (P.blocks_needed(prompt, b) + forks - 1)
            self.num_blocks = synth.pool_with_slack(need, cfg["slack"])
        else:
            self.lengths = (np.asarray(lengths, dtype=np.int64) if lengths is not None
                            else synth.lengths(name, batch))
            self.ids = list(range(len(self.lengths)))
            need = sum(P.blocks_needed(int(t) + 1, b) for t in self.lengths)
            self.num_blocks = cfg.get("pool_blocks") or synth.pool_with_slack(need, cfg["slack"])
        seed = synth.seed_of(name, 2) if free_order_seed is None else free_order_seed
        order = list(synth.free_order(seed, self.num_blocks))
        if pinned_prefix:
            order = list(pinned_prefix) + [x for x in order if x not in pinned_prefix]
        self.order = order

        # product side
        bm = pkv.BlockManager(self.num_blocks, b, order)
        if name == "fork":
            for g in range(self.groups):
                root = g * self.forks
                bm.admit(root, self.prompt)
                for f in range(1, self.forks):
                    bm.fork(root, root + f)
        else:
            for i, t in enumerate(self.lengths):
                bm.admit(i, int(t))
        self.slots, self.pairs = bm.append(self.ids)
        self.max_blocks = max(bm.num_seq_blocks(i) for i in self.ids)
        self.tables, self.seq_lens = bm.tables(self.ids, self.max_blocks)
        self.bm = bm

        # oracle side
        pool = B.BlockPool(self.num_blocks, b, free_order=order, auto_verify=False)
        if name == "fork":
            for g in range(self.groups):
                root = g * self.forks
                pool.admit(root, list(range(self.prompt)))
                for f in range(1, self.forks):
                    pool.fork(root, root + f)
        else:
            for i, t in enumerate(self.lengths):
                pool.admit(i, list(range(int(t))))
        res = [pool.append(i, -1) for i in self.ids]
        pool.verify()
        self.o_slots = [r.slot for r in res]
        self.o_pairs = [r.copy for r in res if r.copy]
        self.o_tables = [pool.table(i) for i in self.ids]
        self.o_lens = [pool.length(i) for i in self.ids]
        self.pool = pool

    def check_plans_agree(self):
        assert list(self.slots) == self.o_slots
        assert [tuple(p) for p in self.pairs] == self.o_pairs
        for row, t in zip(self.tables, self.o_tables):
            assert list(row[: len(t)]) == t and all(x == -1 for x in row[len(t):])
        assert list(self.seq_lens) == self.o_lens
        counts = self.pool.refcounts()
        for blk in range(self.num_blocks):
            assert self.bm.refcount(blk) == counts[blk]
        assert self.bm.check()


class StepData:
    """Seeded tensors of one step (pool, new keys/values, queries)."""

    def __init__(self, seqs, pool_device="cpu", heads=None, kv_heads=None, head_dim=None,
                 dtype=None, seed_base=0):
        cfg = seqs.cfg
        self.H = heads or cfg["heads"]
        self.Hk = kv_heads or cfg["kv_heads"]
        self.D = head_dim or cfg["head_dim"]
        self.dtype = dtype or cfg["dtype"]
        n, S = seqs.num_blocks, len(seqs.ids)
        sd = lambda k: synth.seed_of(seqs.name, k) + seed_base  # noqa: E731
        shape = (n, self.Hk, seqs.b, self.D)
        self.k_pool = synth.normal(sd(3), shape, self.dtype, device=pool_device)
        self.v_pool = synth.normal(sd(4), shape, self.dtype, device=pool_device)
        self.k_new = synth.normal(sd(5), (S, self.Hk, self.D), self.dtype)
        self.v_new = synth.normal(sd(6), (S, self.Hk, self.D), self.dtype)
        self.q = synth.normal(sd(7), (S, self.H, self.D), self.dtype)
        self.scale = 1.0 / math.sqrt(self.D)


def run_gpu(seqs, data, partition_size=0, max_seq_len=None):
    """Copy-on-write, KV write and decode on the GPU; returns (cache, out, err)."""
    dev = torch.device("cuda")
    cache = pkv.PagedKVCache(data.k_pool.to(dev).clone(), data.v_pool.to(dev).clone())
    pairs = torch.from_numpy(np.asarray(seqs.pairs, dtype=np.int64).reshape(-1, 2)).to(dev)
    slots = torch.from_numpy(np.asarray(seqs.slots, dtype=np.int64)).to(dev)
    tables = torch.from_numpy(seqs.tables).to(dev)
    lens = torch.from_numpy(seqs.seq_lens).to(dev)
    pkv.paged_block_copy(cache, pairs)
    pkv.paged_kv_write(cache, data.k_new.to(dev), data.v_new.to(dev), slots)
    bound = int(seqs.seq_lens.max()) if max_seq_len is None else max_seq_len
    out = pkv.paged_attention_decode(cache, data.q.to(dev), tables, lens, data.scale,
                                     max_seq_len=bound, partition_size=partition_size)
    err = pkv.paged_get_device_error()
    return cache, out, err


def run_oracle(seqs, data, sample=None):
    """The oracle's copy, write and attention; returns (k_pool, v_pool, out)."""
    dt = data.dtype
    kp = synth.storage_numpy(data.k_pool, dt)
    vp = synth.storage_numpy(data.v_pool, dt)
    kp, vp, bad = A.copy_blocks(kp, vp, seqs.o_pairs)
    assert bad == []
    kp, vp, bad = A.write_tokens(kp, vp, synth.storage_numpy(data.k_new, dt),
                                 synth.storage_numpy(data.v_new, dt), seqs.o_slots, seqs.b)
    assert bad == []
    out, bad = A.attention(synth.storage_numpy(data.q, dt), kp, vp, seqs.o_tables, seqs.o_lens,
                           data.scale, seqs.b, dt, seqs=sample)
    assert bad == []
    return kp, vp, out


def gpu_out_f64(out):
    return out.detach().float().cpu().numpy().astype(np.float64)


def max_err(gpu, ref, rows):
    return max(float(np.max(np.abs(gpu[s] - ref[s]))) for s in rows)

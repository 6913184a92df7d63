"""Shared-prefix decode (paged_attention_decode_shared) on the GPU against
the oracle: groups of sequences whose tables share their first blocks
(forks of one prompt) give the attention of every sequence over its own
table; the parallel-sampling workload at full size with all 128 sequences;
identical forks stay bit-identical; relabelling the pool is bit-exact; a
member that breaks its group's contract is flagged and zeroed; sequences
outside every group and pools without group support decode in full; the
partition pass's tail grid (tail_parts) gives the full grid's bits (one
slice: merged in place, against the oracle) and flags the sequences it does
not cover."""

import numpy as np
import pytest
import torch

import paged_kv_cache_145_gb300 as pkv
from oracle import attention as A
from paged_kv_cache_145_gb300 import _lib, synth
from tests.workload import Sequences, StepData, TOL, edge_tol, gpu_out_f64, run_oracle

pytestmark = pytest.mark.gpu
TORCH = synth.TORCH_DTYPE


class GroupCase:
    """Groups of sequences sharing ceil(prefix / b) table entries (the
    group's first blocks), each member with private blocks after them."""

    def __init__(self, dtype, Hk, G, D, b, groups, seed=0, spare=4):
        # groups: list of (size, prefix, [member lengths])
        rng = np.random.default_rng(seed)
        self.dtype, self.Hk, self.G, self.D, self.b = dtype, Hk, G, D, b
        self.lens, starts, prefixes = [], [0], []
        need = 0
        for size, prefix, lens in groups:
            assert len(lens) == size and all(L >= prefix for L in lens)
            shared = -(-prefix // b)
            need += shared + sum(-(-L // b) - shared for L in lens)
            self.lens += list(lens)
            starts.append(starts[-1] + size)
            prefixes.append(prefix)
        self.N = need + spare
        perm = list(rng.permutation(self.N))
        width = max(-(-L // b) for L in self.lens) + 1
        self.tables = np.full((len(self.lens), width), -1, dtype=np.int32)
        s = 0
        for size, prefix, lens in groups:
            shared_blocks = [perm.pop() for _ in range(-(-prefix // b))]
            for L in lens:
                own = [perm.pop() for _ in range(-(-L // b) - len(shared_blocks))]
                self.tables[s, :len(shared_blocks) + len(own)] = shared_blocks + own
                s += 1
        self.starts = np.asarray(starts, dtype=np.int32)
        self.prefixes = np.asarray(prefixes, dtype=np.int32)
        self.max_group = max(g[0] for g in groups)
        g = torch.Generator().manual_seed(seed)
        shape = (self.N, Hk, b, D)
        self.k = torch.randn(*shape, generator=g).to(TORCH[dtype])
        self.v = torch.randn(*shape, generator=g).to(TORCH[dtype])
        self.q = torch.randn(len(self.lens), Hk * G, D, generator=g).to(TORCH[dtype])
        self.scale = 1.0 / np.sqrt(D)

    def run(self, part=0, plain=False, tables=None, k=None, v=None, q=None, tail_parts=0):
        cache = pkv.PagedKVCache((self.k if k is None else k).cuda(),
                                 (self.v if v is None else v).cuda())
        tab = torch.from_numpy(self.tables if tables is None else tables).cuda()
        ln = torch.tensor(self.lens, dtype=torch.int32).cuda()
        qq = (self.q if q is None else q).cuda()
        if plain:
            out = pkv.paged_attention_decode(cache, qq, tab, ln, self.scale, partition_size=part)
        else:
            out = pkv.paged_attention_decode_shared(
                cache, qq, tab, ln, self.scale, torch.from_numpy(self.starts).cuda(),
                torch.from_numpy(self.prefixes).cuda(), self.max_group, partition_size=part,
                tail_parts=tail_parts)
        return out, pkv.paged_get_device_error()

    def oracle(self):
        dt = self.dtype
        out, bad = A.attention(synth.storage_numpy(self.q, dt), synth.storage_numpy(self.k, dt),
                               synth.storage_numpy(self.v, dt), [list(r) for r in self.tables],
                               self.lens, self.scale, self.b, dt)
        assert bad == []
        return out


GRID = [("bf16", 2, 4, 128, 16), ("f16", 2, 4, 128, 16), ("bf16", 1, 8, 128, 8), ("f16", 2, 1, 128, 32),
        ("bf16", 2, 2, 64, 16), ("f16", 1, 8, 64, 64)]


@pytest.mark.parametrize("dt,Hk,G,D,b", GRID)
@pytest.mark.parametrize("part", [64, 0])
def test_groups_match_oracle(dt, Hk, G, D, b, part):
    if part and part % b:
        part = b * 4
    groups = [(3, 200, [205, 260, 200]), (1, 50, [77]), (8, 130, [131 + 7 * i for i in range(8)]),
              (2, 0, [40, 5]), (5, 64, [64, 65, 100, 300, 64])]
    c = GroupCase(dt, Hk, G, D, b, groups, seed=hash((dt, Hk, G, D, b, part)) % 997)
    out, err = c.run(part=part)
    assert err == 0
    got, ref = gpu_out_f64(out), c.oracle()
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= edge_tol(dt, ref))
    plain, err = c.run(part=part, plain=True)
    assert err == 0
    assert np.all(np.abs(got - gpu_out_f64(plain)) <= edge_tol(dt, ref))
    # Tail grids: as many slices as the longest tail needs (one: the tails
    # are computed and merged in one pass), and one more.
    ps = part if part else pkv.paged_attention_partition_size(
        pkv.PagedKVCache(c.k[:1].cuda(), c.v[:1].cuda()), len(c.lens), Hk * G, c.tables.shape[1] * b)
    own = {}
    for gi in range(len(c.starts) - 1):
        for s_ in range(c.starts[gi], c.starts[gi + 1]):
            own[s_] = c.prefixes[gi] // ps
    need = max(-(-L // ps) - own.get(i, 0) for i, L in enumerate(c.lens))
    for tp in (max(need, 1), need + 1):
        out, err = c.run(part=part, tail_parts=tp)
        assert err == 0, (tp, need)
        assert np.all(np.abs(gpu_out_f64(out) - ref) <= edge_tol(dt, ref)), tp


def test_group_larger_than_one_row_block():
    # 12 members x 8 query heads = 96 stacked rows: three row blocks.
    groups = [(12, 256, [256 + 3 * i for i in range(12)]), (1, 0, [33])]
    c = GroupCase("bf16", 1, 8, 128, 16, groups, seed=5)
    ref = c.oracle()
    for tp in (0, 1):  # every tail (<= 33 positions) within one 64-position partition
        out, err = c.run(part=64, tail_parts=tp)
        assert err == 0
        got = gpu_out_f64(out)
        assert np.all(np.abs(got - ref) <= edge_tol("bf16", ref))


def test_parallel_sampling_workload_full_size_all_sequences():
    # The parallel-sampling workload: 16 groups x 8 forks of a 1031-token
    # prompt (64 shared full blocks; each fork's last block copied on
    # write), GQA 32/8, bf16, block 16; every one of the 128 sequences
    # against the oracle, after the step's copy-on-write and KV write.
    seqs = Sequences("fork")
    data = StepData(seqs, pool_device="cuda")
    seqs.check_plans_agree()
    dev = torch.device("cuda")
    cache = pkv.PagedKVCache(data.k_pool.to(dev).clone(), data.v_pool.to(dev).clone())
    pkv.paged_block_copy(cache, torch.from_numpy(np.asarray(seqs.pairs, dtype=np.int64).reshape(-1, 2)).to(dev))
    pkv.paged_kv_write(cache, data.k_new.to(dev), data.v_new.to(dev),
                       torch.from_numpy(np.asarray(seqs.slots, dtype=np.int64)).to(dev))
    starts = torch.arange(0, len(seqs.ids) + 1, seqs.forks, dtype=torch.int32, device=dev)
    prefix = (seqs.prompt // seqs.b) * seqs.b
    prefixes = torch.full((seqs.groups,), prefix, dtype=torch.int32, device=dev)
    tables = torch.from_numpy(seqs.tables).to(dev)
    lens = torch.from_numpy(seqs.seq_lens).to(dev)
    part = synth.CONFIGS["fork"].get("partition_size", 0)
    out = pkv.paged_attention_decode_shared(cache, data.q.to(dev), tables, lens, data.scale, starts,
                                            prefixes, seqs.forks, partition_size=part)
    assert pkv.paged_get_device_error() == 0
    _, _, ref = run_oracle(seqs, data)
    got = gpu_out_f64(out)
    assert np.all(np.isfinite(got))
    assert float(np.max(np.abs(got - ref))) <= TOL["bf16"]
    # Every fork's tail (the prompt's last 7 tokens and the new one) lies in
    # one partition: a one-slice tail grid, merged in place, on all 128.
    out1 = pkv.paged_attention_decode_shared(cache, data.q.to(dev), tables, lens, data.scale, starts,
                                             prefixes, seqs.forks, partition_size=part, tail_parts=1)
    assert pkv.paged_get_device_error() == 0
    assert float(np.max(np.abs(gpu_out_f64(out1) - ref))) <= TOL["bf16"]


def test_identical_forks_are_bit_identical():
    # Eight forks with the same table, length and query: every output row
    # of the group is the same bits.
    groups = [(8, 320, [333] * 8)]
    c = GroupCase("bf16", 2, 4, 128, 16, groups, seed=9)
    c.tables[1:] = c.tables[0]
    c.q[1:] = c.q[0]
    for tp in (0, 1):
        out, err = c.run(part=64, tail_parts=tp)
        assert err == 0
        o = out.cpu()
        for i in range(1, 8):
            assert torch.equal(o[i], o[0])


@pytest.mark.parametrize("groups,tps", [
    ([(4, 160, [170, 200, 161, 300]), (2, 32, [40, 90])], (0, 3)),
    ([(4, 128, [130, 150, 170, 191]), (2, 64, [70, 100])], (0, 1, 2)),
])
def test_relabelling_blocks_is_bit_exact(groups, tps):
    c = GroupCase("f16", 2, 4, 128, 16, groups, seed=11)
    perm = np.random.default_rng(3).permutation(c.N)
    inv = np.argsort(perm)
    k2, v2 = torch.empty_like(c.k), torch.empty_like(c.v)
    k2[torch.from_numpy(perm)] = c.k
    v2[torch.from_numpy(perm)] = c.v
    tables = np.where(c.tables >= 0, perm[np.maximum(c.tables, 0)], -1).astype(np.int32)
    assert np.array_equal(inv[perm], np.arange(c.N))
    for tp in tps:
        out0, err = c.run(part=64, tail_parts=tp)
        assert err == 0
        out1, err = c.run(part=64, tables=tables, k=k2, v=v2, tail_parts=tp)
        assert err == 0
        assert torch.equal(out0.cpu(), out1.cpu())


def test_broken_member_is_flagged_and_zeroed():
    # Member 2 of the first group names another block inside the shared
    # prefix: its row is zero and PKV_DEV_SHARING is set; every other
    # sequence is still right.
    groups = [(4, 128, [130, 140, 150, 160]), (2, 64, [70, 80])]
    c = GroupCase("bf16", 2, 4, 128, 16, groups, seed=13, spare=6)
    tables = c.tables.copy()
    used = set(int(x) for x in tables.ravel() if x >= 0)
    spare_block = next(i for i in range(c.N) if i not in used)
    tables[2, 1] = spare_block
    out, err = c.run(part=64, tables=tables)
    assert err & _lib.PKV_DEV_SHARING
    got = gpu_out_f64(out)
    assert np.all(got[2] == 0.0)
    c.tables = tables
    ref = c.oracle()
    rows = [0, 1, 3, 4, 5]
    assert np.all(np.abs(got[rows] - ref[rows]) <= edge_tol("bf16", ref[rows]))


def test_sequences_outside_groups_and_empty_groups():
    # Groups [0, 3), [3, 3) (empty) and [3, 5); sequences 5 and 6 belong to
    # no group and are decoded in full.
    groups = [(3, 96, [100, 120, 96]), (2, 48, [60, 50]), (2, 0, [30, 200])]
    c = GroupCase("bf16", 2, 4, 128, 16, groups, seed=17)
    c.starts = np.asarray([0, 3, 3, 5], dtype=np.int32)
    c.prefixes = np.asarray([96, 999, 48], dtype=np.int32)
    out, err = c.run(part=32)
    assert err == 0
    got, ref = gpu_out_f64(out), c.oracle()
    assert np.all(np.abs(got - ref) <= edge_tol("bf16", ref))


def test_fp8_pool_decodes_in_full():
    # Groups apply to 16-bit pools; an FP8 pool gives the plain decode.
    n, hk, b, d = 40, 2, 16, 128
    g = torch.Generator().manual_seed(21)
    kc = synth.random_codes(21, (n, hk, b, d)).cuda()
    vc = synth.random_codes(22, (n, hk, b, d)).cuda()
    sc = torch.full((hk,), 1.0 / 64, device="cuda")
    cache = pkv.PagedKVCache(kc, vc, sc, sc.clone(), torch.bfloat16)
    tables = torch.tensor([[0, 1, 2, 3, 4], [0, 1, 2, 5, 6]], dtype=torch.int32).cuda()
    lens = torch.tensor([70, 75], dtype=torch.int32).cuda()
    q = torch.randn(2, hk * 4, d, generator=g).bfloat16().cuda()
    starts = torch.tensor([0, 2], dtype=torch.int32).cuda()
    prefix = torch.tensor([48], dtype=torch.int32).cuda()
    a = pkv.paged_attention_decode_shared(cache, q, tables, lens, 0.088, starts, prefix, 2)
    bb = pkv.paged_attention_decode(cache, q, tables, lens, 0.088)
    assert pkv.paged_get_device_error() == 0
    assert torch.equal(a, bb)


@pytest.mark.parametrize("dt", ["bf16", "f16"])
def test_tail_grid(dt):
    # Tails: group 0 (prefix 128 = two 64-position partitions) ends in
    # partition 2, group 1 (prefix 192) in partition 3, group 2 (prefix 64)
    # in partition 1: one slice covers every sequence.  Member 0 of group 3
    # has no tail (length = prefix = 128: the CTA merges the two shared
    # partitions alone), group 4's member is one shared partition (written
    # by the shared-prefix kernel).  Two or more slices give the full
    # grid's bits; one slice merges in place.
    groups = [(3, 128, [140, 150, 191]), (4, 192, [200, 230, 250, 255]), (1, 64, [100]),
              (2, 128, [128, 129]), (1, 64, [64])]
    c = GroupCase(dt, 2, 4, 128, 16, groups, seed=23)
    full, err = c.run(part=64)
    assert err == 0
    got, ref = gpu_out_f64(full), c.oracle()
    assert np.all(np.abs(got - ref) <= edge_tol(dt, ref))
    for tp in (2, 9):
        out, err = c.run(part=64, tail_parts=tp)
        assert err == 0
        assert torch.equal(out.cpu(), full.cpu())
    out, err = c.run(part=64, tail_parts=1)
    assert err == 0
    assert np.all(np.abs(gpu_out_f64(out) - ref) <= edge_tol(dt, ref))


def test_tail_grid_flags_uncovered_sequences():
    # With 64-position partitions: members of length 200 and 250 (prefix
    # 128) need partitions 2 and 3; sequence 6 (outside every group, length
    # 150) needs partitions 0-2.  A one-slice tail grid zeroes and flags
    # exactly those; three slices cover everyone.
    groups = [(3, 128, [140, 200, 250]), (2, 64, [70, 80]), (2, 0, [30, 150])]
    c = GroupCase("bf16", 2, 4, 128, 16, groups, seed=29)
    c.starts = np.asarray([0, 3, 5], dtype=np.int32)
    c.prefixes = np.asarray([128, 64], dtype=np.int32)
    ref = c.oracle()
    out, err = c.run(part=64, tail_parts=1)
    assert err & _lib.PKV_DEV_SHARING
    got = gpu_out_f64(out)
    uncovered, covered = [1, 2, 6], [0, 3, 4, 5]
    assert np.all(got[uncovered] == 0.0)
    assert np.all(np.abs(got[covered] - ref[covered]) <= edge_tol("bf16", ref[covered]))
    out, err = c.run(part=64, tail_parts=3)
    assert err == 0
    assert np.all(np.abs(gpu_out_f64(out) - ref) <= edge_tol("bf16", ref))
    # Two slices (merge launch): the same rows zeroed, as member 1 and 2
    # need two tail partitions and sequence 6 three.
    out, err = c.run(part=64, tail_parts=2)
    assert err & _lib.PKV_DEV_SHARING
    got = gpu_out_f64(out)
    assert np.all(got[[6]] == 0.0)
    ok = [0, 1, 2, 3, 4, 5]
    assert np.all(np.abs(got[ok] - ref[ok]) <= edge_tol("bf16", ref[ok]))

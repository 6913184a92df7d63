"""GPU decode attention against the oracle over the supported geometry grid,
plus edge cases and invariants, with hand-built tables (no allocator)."""

import numpy as np
import pytest
import torch

import paged_kv_cache_145_gb300 as pkv
from oracle import attention as A
from paged_kv_cache_145_gb300 import synth
from tests.workload import TOL, edge_tol, gpu_out_f64

pytestmark = pytest.mark.gpu

TORCH = synth.TORCH_DTYPE


class Case:
    """Random pool, scattered tables and queries for given lengths."""

    def __init__(self, dtype, H, Hk, D, b, lens, seed=0, spare=3, width_extra=1):
        rng = np.random.default_rng(seed)
        self.dtype, self.H, self.Hk, self.D, self.b = dtype, H, Hk, D, b
        self.lens = [int(x) for x in lens]
        nblk = [-(-max(L, 1) // b) for L in self.lens]
        self.N = sum(nblk) + spare
        perm = rng.permutation(self.N)
        self.width = max(nblk) + width_extra
        self.tables = np.full((len(self.lens), self.width), -1, dtype=np.int32)
        pos = 0
        for i, k in enumerate(nblk):
            self.tables[i, :k] = perm[pos:pos + k]
            pos += k
        g = torch.Generator().manual_seed(seed)
        shape = (self.N, Hk, b, D)
        self.k = torch.randn(*shape, generator=g).to(TORCH[dtype])
        self.v = torch.randn(*shape, generator=g).to(TORCH[dtype])
        self.q = torch.randn(len(self.lens), H, D, generator=g).to(TORCH[dtype])
        self.scale = 1.0 / np.sqrt(D)

    def cache(self):
        return pkv.PagedKVCache(self.k.cuda().clone(), self.v.cuda().clone())

    def gpu(self, part=0, max_len=0, cache=None, q=None, tables=None, lens=None, workspace=None):
        cache = cache or self.cache()
        tab = torch.from_numpy(self.tables if tables is None else tables).cuda()
        ln = torch.tensor(self.lens if lens is None else lens, dtype=torch.int32).cuda()
        q = (self.q if q is None else q).cuda()
        out = pkv.paged_attention_decode(cache, q, tab, ln, self.scale, max_seq_len=max_len,
                                         partition_size=part, workspace=workspace)
        return out, pkv.paged_get_device_error()

    def oracle(self, tables=None, lens=None, max_len=None):
        dt = self.dtype
        return A.attention(synth.storage_numpy(self.q, dt), synth.storage_numpy(self.k, dt),
                           synth.storage_numpy(self.v, dt),
                           [list(r) for r in (self.tables if tables is None else tables)],
                           self.lens if lens is None else lens, self.scale, self.b, dt,
                           max_len=max_len)


GRID = [(dt, D, b, G, part)
        for dt in ("f32", "f16", "bf16")
        for D in (64, 128)
        for b in (8, 16, 32)
        for G in (1, 4)
        for part in (0, 2)]
GRID += [("f16", 128, 16, 2, 0), ("f16", 128, 16, 8, 0), ("bf16", 128, 16, 8, 2),
         ("bf16", 64, 8, 2, 2), ("f32", 128, 32, 8, 0)]
GRID += [(dt, 128, 64, G, part) for dt in ("f16", "bf16") for G in (1, 4) for part in (0, 2)]
GRID += [("f32", 64, 64, 2, 2)]


@pytest.fixture(params=["auto", "simt"])
def kernel(request, monkeypatch):
    """Runs a test with the automatic kernel choice (tensor cores for grouped
    fp16/bf16 heads) and again with the CUDA-core kernel forced."""
    if request.param == "simt":
        monkeypatch.setenv("PKV_DECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("PKV_DECODE_KERNEL", raising=False)
    return request.param


@pytest.mark.parametrize("dt,D,b,G,part", GRID)
def test_geometry_grid(dt, D, b, G, part, kernel):
    # part = 2 means two blocks per partition: many partitions, ragged tails.
    lens = [1, b - 1, b, b + 1, 97, 300, 2 * b * 3 + 5]
    c = Case(dt, 2 * G, 2, D, b, lens, seed=hash((dt, D, b, G, part)) % 1000)
    out, err = c.gpu(part=part * b)
    assert err == 0
    ref, bad = c.oracle()
    assert bad == []
    got = gpu_out_f64(out)
    tol = edge_tol(dt, ref)
    assert np.all(np.abs(got - ref) <= tol)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_length_one_is_the_value_row(dt):
    c = Case(dt, 4, 4, 128, 16, [1, 1, 1], seed=3)
    out, err = c.gpu()
    assert err == 0
    got = gpu_out_f64(out)
    for s in range(3):
        blk = int(c.tables[s, 0])
        v0 = c.v[blk, :, 0, :].to(torch.float64).numpy()
        assert np.array_equal(got[s], v0)  # weight 1 exactly, value round-trips


@pytest.mark.parametrize("part", [0, 32])
def test_equal_keys_give_mean_of_values(part):
    c = Case("f32", 4, 2, 64, 16, [77, 130], seed=4)
    c.k[:] = c.k[0, 0, 0]
    out, err = c.gpu(part=part)
    got = gpu_out_f64(out)
    for s, L in enumerate(c.lens):
        for h in range(4):
            rows = [c.v[c.tables[s, t // 16], h // 2, t % 16].double().numpy() for t in range(L)]
            assert np.max(np.abs(got[s, h] - np.mean(rows, axis=0))) < 1e-5


@pytest.mark.parametrize("part", [0, 64])
def test_partition_boundaries(part, kernel):
    lens = [63, 64, 65, 127, 128, 129, 511, 512, 513, 1023, 1024, 1025]
    c = Case("bf16", 8, 2, 128, 16, lens, seed=5)
    out, err = c.gpu(part=part)
    assert err == 0
    ref, _ = c.oracle()
    assert np.max(np.abs(gpu_out_f64(out) - ref)) <= TOL["bf16"]


@pytest.mark.parametrize("dt,G,b", [("f16", 1, 8), ("bf16", 4, 16), ("f32", 2, 32)])
def test_largest_partition(dt, G, b, kernel):
    # Partitions of 8192 positions, the largest accepted: one CTA stages
    # 8192 / b table entries and streams the whole partition; lengths just
    # below, at and past it give one full partition, a full one merged with
    # a one-position one, and a ragged second partition.
    lens = [1, 8191, 8192, 8193, 9000]
    c = Case(dt, 2 * G, 2, 128, b, lens, seed=11 + G)
    out, err = c.gpu(part=8192)
    assert err == 0
    ref, bad = c.oracle()
    assert bad == []
    assert np.all(np.abs(gpu_out_f64(out) - ref) <= edge_tol(dt, ref))


def test_largest_batch(kernel):
    # 65535 sequences, the most the launch grid indexes: the first, the last
    # and a seeded spread of sequences against the oracle.
    S = 65535
    rng = np.random.default_rng(17)
    c = Case("bf16", 2, 1, 64, 16, rng.integers(1, 49, S), seed=17, spare=1, width_extra=0)
    out, err = c.gpu()
    assert err == 0
    seqs = sorted({0, 1, S - 2, S - 1, *rng.choice(S, 200, replace=False).tolist()})
    ref, bad = A.attention(synth.storage_numpy(c.q, "bf16"), synth.storage_numpy(c.k, "bf16"),
                           synth.storage_numpy(c.v, "bf16"), c.tables, c.lens, c.scale, 16,
                           "bf16", seqs=seqs)
    assert bad == []
    got = gpu_out_f64(out)[seqs]
    assert np.all(np.abs(got - ref[seqs]) <= edge_tol("bf16", ref[seqs]))


def test_invalid_lengths_zero_rows():
    c = Case("f16", 4, 4, 128, 16, [40, 40, 40, 40], seed=6)
    lens = [40, 0, 40, c.width * 16 + 1]
    out, err = c.gpu(lens=lens, max_len=c.width * 16)
    assert err == pkv.PKV_DEV_SEQ_LEN
    got = gpu_out_f64(out)
    assert np.all(got[1] == 0) and np.all(got[3] == 0)
    ref, bad = c.oracle(lens=lens, max_len=c.width * 16)
    assert sorted(bad) == [1, 3]
    assert np.max(np.abs(got[[0, 2]] - ref[[0, 2]])) <= TOL["f16"]
    # A length above the caller's bound (but inside the table) is invalid too.
    out, err = c.gpu(lens=[40, 40, 40, 40], max_len=39)
    assert err == pkv.PKV_DEV_SEQ_LEN and np.all(gpu_out_f64(out) == 0)


@pytest.mark.parametrize("part", [0, 32])
def test_bad_table_entry_zero_row(part, kernel):
    c = Case("bf16", 8, 2, 128, 16, [100, 100, 100], seed=7)
    tables = c.tables.copy()
    tables[1, 3] = c.N + 7
    tables[2, 0] = -5
    out, err = c.gpu(part=part, tables=tables)
    assert err == pkv.PKV_DEV_TABLE_RANGE
    got = gpu_out_f64(out)
    assert np.all(got[1] == 0) and np.all(got[2] == 0)
    ref, bad = c.oracle(tables=tables)
    assert sorted(bad) == [1, 2]
    assert np.max(np.abs(got[0] - ref[0])) <= TOL["bf16"]


def test_unused_table_entries_are_not_read():
    c = Case("f16", 4, 4, 64, 16, [20, 33], seed=8, width_extra=3)
    tables = c.tables.copy()
    tables[0, 2:] = 10 ** 6          # beyond the sequence: never dereferenced
    out, err = c.gpu(tables=tables)
    assert err == 0
    ref, _ = c.oracle()
    assert np.max(np.abs(gpu_out_f64(out) - ref)) <= TOL["f16"]


@pytest.mark.parametrize("part", [0, 48])
def test_relabelling_blocks_is_bit_exact(part, kernel):
    c = Case("bf16", 16, 4, 128, 16, [200, 17, 700, 1], seed=9)
    out1, _ = c.gpu(part=part)
    perm = torch.from_numpy(np.random.default_rng(1).permutation(c.N))
    k2 = torch.empty_like(c.k)
    v2 = torch.empty_like(c.v)
    k2[perm] = c.k
    v2[perm] = c.v
    tables = c.tables.copy()
    used = tables >= 0
    tables[used] = perm.numpy()[tables[used]]
    cache = pkv.PagedKVCache(k2.cuda(), v2.cuda())
    out2, err = c.gpu(part=part, cache=cache, tables=tables)
    assert err == 0
    assert torch.equal(out1, out2)


def test_shared_prefix_forks_identical(kernel):
    c = Case("bf16", 32, 8, 128, 16, [1031] * 4, seed=10)
    tables = np.repeat(c.tables[:1], 4, axis=0)
    q = c.q.clone()
    q[:] = q[0]
    out, err = c.gpu(tables=tables, q=q)
    assert err == 0
    for s in range(1, 4):
        assert torch.equal(out[s], out[0])


def test_workspace_partials_match_oracle():
    c = Case("f32", 8, 2, 128, 16, [300, 1000, 64], seed=11)
    part = 128
    max_len = max(c.lens)
    cache = c.cache()
    nbytes = pkv.paged_attention_workspace_bytes(cache, 3, 8, max_len, part)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out, err = c.gpu(part=part, max_len=max_len, cache=cache, workspace=ws)
    assert err == 0
    P = -(-max_len // part)
    ml = ws[: 3 * 8 * P * 8].view(torch.float32).view(3, 8, P, 2).cpu().numpy().astype(np.float64)
    o_off = ((3 * 8 * P * 8 + 255) // 256) * 256
    o = ws[o_off:o_off + 3 * 8 * P * 128 * 4].view(torch.float32).view(3, 8, P, 128).cpu().numpy()
    dt = "f32"
    stats = A.partition_stats(synth.storage_numpy(c.q, dt), synth.storage_numpy(c.k, dt),
                              synth.storage_numpy(c.v, dt), [list(r) for r in c.tables], c.lens,
                              c.scale, 16, dt, part)
    for s, L in enumerate(c.lens):
        n = -(-L // part)
        if n == 1:
            continue  # written straight to the output
        for h in range(8):
            m, l, oo = stats[(s, h)]
            # The kernel keeps maxima in base-2 units: m2 = m * log2(e).
            assert np.max(np.abs(ml[s, h, :n, 0] * np.log(2.0) - m)) < 1e-5
            # Sums are relative to each maximum, so they agree directly.
            assert np.max(np.abs(ml[s, h, :n, 1] / l - 1.0)) < 1e-5
            assert np.max(np.abs(o[s, h, :n] - oo)) < 1e-5


def test_empty_batch_is_a_no_op():
    c = Case("f16", 4, 4, 64, 16, [5], seed=12)
    cache = c.cache()
    q = torch.empty(0, 4, 64, dtype=torch.float16, device="cuda")
    out = pkv.paged_attention_decode(cache, q, torch.empty(0, 1, dtype=torch.int32, device="cuda"),
                                     torch.empty(0, dtype=torch.int32, device="cuda"), 0.1)
    assert out.shape == (0, 4, 64) and pkv.paged_get_device_error() == 0


@pytest.mark.parametrize("dt,G,b", [("bf16", 4, 16), ("f16", 8, 16), ("f16", 1, 16), ("f32", 4, 16),
                                    ("bf16", 4, 8), ("f16", 2, 32), ("bf16", 8, 64)])
def test_stale_nan_slots_never_reach_the_output(dt, G, b, kernel):
    # Slots past each sequence's end inside its last block hold NaN; the
    # kernels must neither use them nor let 0 * NaN into the sums.
    lens = [1, 5, 8, 9, 16, 17, 31, 250]
    c = Case(dt, 2 * G, 2, 128, b, lens, seed=13)
    for s_, L in enumerate(lens):
        last = int(c.tables[s_, (L - 1) // b])
        c.k[last, :, (L - 1) % b + 1:] = float("nan")
        c.v[last, :, (L - 1) % b + 1:] = float("nan")
    out, err = c.gpu(part=max(32, 2 * b))  # several partitions, each a multiple of b
    assert err == 0
    got = gpu_out_f64(out)
    ref, _ = c.oracle()
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= edge_tol(dt, ref))

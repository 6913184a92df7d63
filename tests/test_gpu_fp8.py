"""FP8 E4M3 KV cache on the GPU against the oracle: the quantizing write is
bit-exact (codes equal e4m3(x / scale) with saturation), decode over FP8
pools matches attention over the dequantized values, and the byte movers
(copy, swap) work on FP8 pools unchanged."""

import numpy as np
import pytest
import torch

import paged_kv_cache_145_gb300 as pkv
from oracle import attention as A
from paged_kv_cache_145_gb300 import synth
from tests.workload import TOL, edge_tol, gpu_out_f64

pytestmark = pytest.mark.gpu
IO = {"f16": torch.float16, "bf16": torch.bfloat16}


def fp8_cache(n, hk, b, d, io, seed, k_scale=None, v_scale=None):
    kc = synth.random_codes(seed, (n, hk, b, d)).cuda()
    vc = synth.random_codes(seed + 1, (n, hk, b, d)).cuda()
    g = torch.Generator().manual_seed(seed + 2)
    ks = torch.rand(hk, generator=g) * 0.02 + 0.002 if k_scale is None else k_scale
    vs = torch.rand(hk, generator=g) * 0.02 + 0.002 if v_scale is None else v_scale
    return pkv.PagedKVCache(kc, vc, ks.float().cuda(), vs.float().cuda(), IO[io])


@pytest.mark.parametrize("io,hk,d", [("f16", 8, 128), ("bf16", 40, 128), ("bf16", 2, 64)])
def test_quantizing_write_bit_exact(io, hk, d):
    n, b = 30, 16
    cache = fp8_cache(n, hk, b, d, io, 1)
    kp = synth.storage_numpy(cache.k_cache, "e4m3").copy()
    vp = synth.storage_numpy(cache.v_cache, "e4m3").copy()
    g = torch.Generator().manual_seed(3)
    slots = torch.randperm(n * b, generator=g)[:50].to(torch.int64)
    slots[7] = -1
    kn = (torch.randn(50, hk, d, generator=g) * 3).to(IO[io])
    vn = (torch.randn(50, hk, d, generator=g) * 3).to(IO[io])
    kn[0, 0, :4] = torch.tensor([60.0, -60.0, 1e-5, 0.0])   # saturating / tiny values
    pkv.paged_kv_write(cache, kn.cuda(), vn.cuda(), slots.cuda())
    assert pkv.paged_get_device_error() == 0
    ek, ev, bad = A.write_tokens_fp8(kp, vp, synth.storage_numpy(kn, io), synth.storage_numpy(vn, io),
                                     slots.tolist(), b, cache.k_scale.cpu().numpy(),
                                     cache.v_scale.cpu().numpy(), io)
    assert bad == []
    assert np.array_equal(synth.storage_numpy(cache.k_cache, "e4m3"), ek)
    assert np.array_equal(synth.storage_numpy(cache.v_cache, "e4m3"), ev)


def decode_case(io, G, b, d, lens, part, seed, hk=2, q_mult=None, k_scale=None, v_scale=None):
    nblk = [-(-L // b) for L in lens]
    n = sum(nblk) + 3
    cache = fp8_cache(n, hk, b, d, io, seed, k_scale=k_scale, v_scale=v_scale)
    perm = np.random.default_rng(seed).permutation(n)
    tables = np.full((len(lens), max(nblk)), -1, dtype=np.int32)
    pos = 0
    for i, k in enumerate(nblk):
        tables[i, :k] = perm[pos:pos + k]
        pos += k
    q = torch.randn(len(lens), hk * G, d, generator=torch.Generator().manual_seed(seed + 9))
    if q_mult is not None:
        q = q * torch.as_tensor(q_mult, dtype=torch.float32).view(-1, 1, 1)
    q = q.to(IO[io])
    out = pkv.paged_attention_decode(cache, q.cuda(), torch.from_numpy(tables).cuda(),
                                     torch.tensor(lens, dtype=torch.int32).cuda(), 1 / np.sqrt(d),
                                     partition_size=part)
    assert pkv.paged_get_device_error() == 0
    ref, bad = A.attention(synth.storage_numpy(q, io), synth.storage_numpy(cache.k_cache, "e4m3"),
                           synth.storage_numpy(cache.v_cache, "e4m3"), [list(r) for r in tables], lens,
                           1 / np.sqrt(d), b, "e4m3", q_dtype=io, k_scale=cache.k_scale.cpu().numpy(),
                           v_scale=cache.v_scale.cpu().numpy())
    assert bad == []
    return gpu_out_f64(out), ref


@pytest.fixture(params=["auto", "simt"])
def kernel(request, monkeypatch):
    """Tensor-core FP8 kernel (default) and the CUDA-core one."""
    if request.param == "simt":
        monkeypatch.setenv("PKV_DECODE_KERNEL", "simt")
    else:
        monkeypatch.delenv("PKV_DECODE_KERNEL", raising=False)
    return request.param


@pytest.mark.parametrize("io,G,b,d,part", [
    ("f16", 1, 16, 128, 0), ("bf16", 1, 16, 128, 32), ("bf16", 4, 16, 128, 0), ("f16", 4, 32, 128, 64),
    ("bf16", 8, 8, 128, 16), ("f16", 2, 64, 64, 128), ("bf16", 4, 16, 64, 0), ("f16", 1, 8, 64, 16)])
def test_fp8_decode_matches_oracle(io, G, b, d, part, kernel):
    lens = [1, b - 1, b, b + 1, 97, 300, 777]
    got, ref = decode_case(io, G, b, d, lens, part, seed=hash((io, G, b, d, part)) % 1000)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= edge_tol(io, ref))


@pytest.mark.parametrize("io,vs,d", [("f16", 3e-3, 128), ("f16", 0.05, 128), ("bf16", 0.012, 128),
                                     ("bf16", 0.05, 128), ("f16", 0.05, 64)])
def test_fp8_decode_value_scales_either_side_of_the_split(io, vs, d, kernel):
    # Values up to 448 * v_scale (22 at 0.05): P enters P.V as one fp16 part
    # while 2^-11 * 448 * |v_scale| stays within half the output's bar, else
    # as two parts.  Both forms against the oracle at the stated bars.
    for seed in range(3):
        got, ref = decode_case(io, 4, 16, d, [5, 97, 300, 777, 2000], 0, seed=seed,
                               v_scale=torch.full((2,), vs))
        assert np.all(np.isfinite(got))
        assert np.all(np.abs(got - ref) <= edge_tol(io, ref))


@pytest.mark.parametrize("io,G,b,d", [("bf16", 4, 16, 128), ("f16", 2, 8, 64)])
def test_fp8_largest_partition(io, G, b, d, kernel):
    # 8192-position partitions (the largest accepted) over FP8 pools: lengths
    # below, at and past one partition.
    lens = [1, 8191, 8192, 8193, 9000]
    got, ref = decode_case(io, G, b, d, lens, 8192, seed=31 + G)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= edge_tol(io, ref))


def test_fp8_step_through_block_manager(kernel):
    # Decode step on an FP8 pool: the block manager plans the step, the new
    # token is quantized into its slot, then attention reads it back.
    b, hk, G, d, io = 16, 8, 4, 128, "bf16"
    lens = [300, 17, 1024, 5]
    n = sum(-(-(L + 1) // b) for L in lens) + 4
    order = synth.free_order(21, n)
    bm = pkv.BlockManager(n, b, order)
    for i, L in enumerate(lens):
        bm.admit(i, L)
    slots, pairs = bm.append(range(4))
    tables, seq_lens = bm.tables(range(4), max(bm.num_seq_blocks(i) for i in range(4)))
    cache = fp8_cache(n, hk, b, d, io, 22)
    kp = synth.storage_numpy(cache.k_cache, "e4m3").copy()
    vp = synth.storage_numpy(cache.v_cache, "e4m3").copy()
    g = torch.Generator().manual_seed(23)
    kn = torch.randn(4, hk, d, generator=g).bfloat16()
    vn = torch.randn(4, hk, d, generator=g).bfloat16()
    q = torch.randn(4, hk * G, d, generator=g).bfloat16()
    pkv.paged_kv_write(cache, kn.cuda(), vn.cuda(), torch.from_numpy(slots).cuda())
    out = pkv.paged_attention_decode(cache, q.cuda(), torch.from_numpy(tables).cuda(),
                                     torch.from_numpy(seq_lens).cuda(), 0.0884)
    assert pkv.paged_get_device_error() == 0
    ks, vs = cache.k_scale.cpu().numpy(), cache.v_scale.cpu().numpy()
    ek, ev, _ = A.write_tokens_fp8(kp, vp, synth.storage_numpy(kn, io), synth.storage_numpy(vn, io),
                                   list(slots), b, ks, vs, io)
    assert np.array_equal(synth.storage_numpy(cache.k_cache, "e4m3"), ek)
    ref, _ = A.attention(synth.storage_numpy(q, io), ek, ev, [list(r) for r in tables], list(seq_lens),
                         0.0884, b, "e4m3", q_dtype=io, k_scale=ks, v_scale=vs)
    # Uniformly random codes make value rows up to ~9, so outputs are not
    # small: the bar is the tolerance or one output ulp, whichever is larger.
    got = gpu_out_f64(out)
    assert np.all(np.abs(got - ref) <= edge_tol(io, ref))


def test_fp8_copy_and_swap_are_byte_moves():
    cache = fp8_cache(12, 8, 16, 128, "f16", 31)
    kp = synth.storage_numpy(cache.k_cache, "e4m3").copy()
    vp = synth.storage_numpy(cache.v_cache, "e4m3").copy()
    pairs = [(1, 7), (3, 9)]
    pkv.paged_block_copy(cache, torch.tensor(pairs).cuda())
    ek, ev, _ = A.copy_blocks(kp, vp, pairs)
    assert np.array_equal(synth.storage_numpy(cache.k_cache, "e4m3"), ek)
    hk_ = torch.zeros(4, 8, 16, 128, dtype=torch.uint8).view(torch.float8_e4m3fn).pin_memory()
    hv_ = torch.zeros_like(hk_).pin_memory()
    pkv.paged_block_swap(cache, hk_, hv_, torch.tensor([[7, 0], [2, 3]]).cuda(), pkv.PKV_SWAP_OUT)
    assert pkv.paged_get_device_error() == 0
    assert np.array_equal(synth.storage_numpy(hk_, "e4m3")[0], ek[7])
    assert np.array_equal(synth.storage_numpy(hv_, "e4m3")[3], ev[2])


def fp8_prefill_case(io, G, b, prefix, chunk, seed, hk=2, k_scale=None, q_mult=None, nan_tail=False,
                     seqs=None, v_scale=None):
    lens = [p_ + c for p_, c in zip(prefix, chunk)]
    nblk = [-(-L // b) for L in lens]
    n = sum(nblk) + 3
    cache = fp8_cache(n, hk, b, 128, io, seed, k_scale=k_scale, v_scale=v_scale)
    perm = np.random.default_rng(seed).permutation(n)
    tables = np.full((len(lens), max(nblk) + 1), -1, dtype=np.int32)
    pos = 0
    for i, k in enumerate(nblk):
        tables[i, :k] = perm[pos:pos + k]
        pos += k
    if nan_tail:  # NaN codes in the slots past each sequence's end
        codes = cache.k_cache.view(torch.uint8), cache.v_cache.view(torch.uint8)
        for i, L in enumerate(lens):
            last = int(tables[i, (L - 1) // b])
            for c in codes:
                c[last, :, (L - 1) % b + 1:] = 0x7F
    starts = np.concatenate([[0], np.cumsum(chunk)]).astype(np.int32)
    q = torch.randn(int(starts[-1]), hk * G, 128, generator=torch.Generator().manual_seed(seed + 5))
    if q_mult is not None:
        q = q * q_mult
    q = q.to(IO[io])
    scale = 1 / np.sqrt(128)
    out = pkv.paged_attention_prefill(cache, q.cuda(), torch.from_numpy(starts).cuda(),
                                      torch.from_numpy(tables).cuda(),
                                      torch.tensor(lens, dtype=torch.int32).cuda(), scale, max(chunk))
    assert pkv.paged_get_device_error() == 0
    ref = A.prefill_attention(synth.storage_numpy(q, io), synth.storage_numpy(cache.k_cache, "e4m3"),
                              synth.storage_numpy(cache.v_cache, "e4m3"), [list(r) for r in tables],
                              lens, starts, scale, b, "e4m3", seqs=seqs, q_dtype=io,
                              k_scale=cache.k_scale.cpu().numpy(), v_scale=cache.v_scale.cpu().numpy())
    return gpu_out_f64(out), ref


@pytest.mark.parametrize("io,G,b", [("f16", 4, 16), ("bf16", 4, 16), ("bf16", 1, 8), ("f16", 8, 64),
                                    ("bf16", 2, 32)])
def test_fp8_prefill_matches_oracle(io, G, b):
    got, ref = fp8_prefill_case(io, G, b, [0, 5, 100, 17], [37, 64, 3, 130], seed=31 + G + b)
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= edge_tol(io, ref))


@pytest.mark.parametrize("io,vs", [("f16", 3e-3), ("f16", 0.03), ("bf16", 0.012), ("bf16", 0.05)])
def test_fp8_prefill_value_scales_either_side_of_the_split(io, vs):
    # P enters P.V as one fp16 part while 2^-11 * 448 * |v_scale| stays
    # within half the output's bar, else as two parts: both forms against
    # the oracle at the stated bars, values reaching 448 * v_scale.
    got, ref = fp8_prefill_case(io, 4, 16, [0, 40, 300], [90, 17, 64], seed=71,
                                v_scale=torch.full((2,), vs))
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= edge_tol(io, ref))


def test_fp8_prefill_chunked_workload_full_size_sampled():
    # The benchmark's FP8 chunked-prefill workload at full size (8 x (4096
    # cached + 512 queries), GQA 32/8, bf16 I/O, block 16), in its launch
    # configuration; two whole sequences against the oracle.
    cfg = synth.CONFIGS["chunked"]
    S, G = cfg["batch"], cfg["heads"] // cfg["kv_heads"]
    chunk = [cfg["chunk"]] * S
    got, ref = fp8_prefill_case("bf16", G, cfg["block_size"], [cfg["prefix"]] * S, chunk,
                                      seed=47, hk=cfg["kv_heads"], seqs=[0, S - 1])
    assert np.all(np.isfinite(got))
    rows = np.concatenate([np.arange(0, chunk[0]), np.arange(sum(chunk) - chunk[-1], sum(chunk))])
    assert np.all(np.abs(got[rows] - ref[rows]) <= edge_tol("bf16", ref[rows]))


def test_fp8_prefill_bf16_queries_beyond_fp16_range():
    got, ref = fp8_prefill_case("bf16", 4, 16, [20, 0], [50, 70], seed=43, q_mult=1e5,
                                      k_scale=torch.full((2,), 3e-7))
    assert np.all(np.isfinite(got))
    assert np.all(np.abs(got - ref) <= edge_tol("bf16", ref))


def test_fp8_prefill_stale_nan_codes():
    got, ref = fp8_prefill_case("f16", 4, 16, [3, 0, 40], [5, 17, 9], seed=47, nan_tail=True)
    assert np.all(np.isfinite(got)) and np.all(np.abs(got - ref) <= edge_tol("f16", ref))


def test_fp8_prefill_refusals(monkeypatch):
    # head_dim 64 and the mma.sync prefill kernel do not take FP8 pools.
    cache = fp8_cache(4, 2, 16, 64, "f16", 41)
    q = torch.zeros(3, 2, 64, dtype=torch.float16).cuda()
    args = (torch.tensor([0, 3], dtype=torch.int32).cuda(), torch.zeros(1, 1, dtype=torch.int32).cuda(),
            torch.tensor([3], dtype=torch.int32).cuda(), 0.1, 3)
    with pytest.raises(RuntimeError):
        pkv.paged_attention_prefill(cache, q, *args)
    monkeypatch.setenv("PKV_PREFILL_KERNEL", "mma")
    cache = fp8_cache(4, 2, 16, 128, "f16", 41)
    with pytest.raises(RuntimeError):
        pkv.paged_attention_prefill(cache, torch.zeros(3, 2, 128, dtype=torch.float16).cuda(), *args)


def test_fp8_default_partition_follows_grid_size():
    """FP8 pools default to the longest of 2048 / 1536 / 1024 / 512 positions
    that still launches 8 thread blocks per SM; 16-bit pools keep 512."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    cache = fp8_cache(4, 8, 16, 128, "bf16", 5)

    def expect(S, L):
        for part in (2048, 1536, 1024):
            if S * 8 * -(-L // part) >= 8 * sms:
                return part
        return 512

    for S, L in [(256, 2001), (64, 2001), (8, 32768), (1, 100), (4096, 3000)]:
        assert pkv.paged_attention_partition_size(cache, S, 32, L) == expect(S, L)
    native = pkv.PagedKVCache(torch.zeros(4, 8, 16, 128, dtype=torch.bfloat16, device="cuda"),
                              torch.zeros(4, 8, 16, 128, dtype=torch.bfloat16, device="cuda"))
    assert pkv.paged_attention_partition_size(native, 256, 32, 2001) == 512


def test_fp8_bf16_queries_beyond_fp16_range(kernel):
    """bf16 queries up to ~5e5 (past fp16's 65504) with a small key scale:
    the scores stay O(1) and the output must still match the oracle, so the
    fp16 products may not overflow.  Sequence 0 keeps N(0, 1) queries."""
    lens = [70, 300, 33]
    ks = torch.full((2,), 3e-7)
    got, ref = decode_case("bf16", 4, 16, 128, lens, 64, 41, q_mult=[1.0, 1e5, 2.5e4],
                           k_scale=ks)
    assert np.isfinite(got).all()
    assert np.all(np.abs(got - ref) <= edge_tol("bf16", ref))


@pytest.mark.parametrize("b", [8, 16, 32])
def test_fp8_stale_nan_codes_never_reach_the_output(b, kernel):
    # Unused slots of each sequence's last block hold the NaN code 0x7F.
    lens = [1, 5, 8, 9, 16, 17, 250]
    nblk = [-(-L // b) for L in lens]
    n = sum(nblk) + 2
    cache = fp8_cache(n, 2, b, 128, "bf16", 51)
    tables = np.full((len(lens), max(nblk)), -1, dtype=np.int32)
    pos = 0
    for i, k in enumerate(nblk):
        tables[i, :k] = np.arange(pos, pos + k)
        pos += k
    kraw = cache.k_cache.view(torch.uint8)
    vraw = cache.v_cache.view(torch.uint8)
    for i, L in enumerate(lens):
        last = int(tables[i, (L - 1) // b])
        kraw[last, :, (L - 1) % b + 1:] = 0x7F
        vraw[last, :, (L - 1) % b + 1:] = 0x7F
    q = torch.randn(len(lens), 8, 128, generator=torch.Generator().manual_seed(52)).bfloat16()
    out = pkv.paged_attention_decode(cache, q.cuda(), torch.from_numpy(tables).cuda(),
                                     torch.tensor(lens, dtype=torch.int32).cuda(), 0.0884,
                                     partition_size=2 * b)
    assert pkv.paged_get_device_error() == 0
    got = gpu_out_f64(out)
    ref, _ = A.attention(synth.storage_numpy(q, "bf16"), synth.storage_numpy(cache.k_cache, "e4m3"),
                         synth.storage_numpy(cache.v_cache, "e4m3"), [list(r) for r in tables], lens,
                         0.0884, b, "e4m3", q_dtype="bf16", k_scale=cache.k_scale.cpu().numpy(),
                         v_scale=cache.v_scale.cpu().numpy())
    assert np.all(np.isfinite(got)) and np.all(np.abs(got - ref) <= edge_tol("bf16", ref))

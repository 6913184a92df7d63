"""Checks that pin the CPU oracle to facts other than itself.

Each ``check_*`` takes the oracle function(s) it pins as arguments, so the
same check runs against the real oracle (``test_oracle.py``) and against
copies with planted mistakes (``test_oracle_mutations.py``), which must fail.

What pins what:
* the pages' worked numbers (fixtures in ``tests/golden/``);
* closed forms computed a different way (residue counting, exact fractions);
* brute force over an enumerated slot list instead of div/mod;
* an independent library routine (``torch.softmax`` in float64, torch's
  bfloat16 conversion);
* mathematical invariants (relabelling physical blocks, shared prefixes,
  merging split partitions).
"""

import math
import random
from fractions import Fraction

import numpy as np
import torch

from tests.golden import ints, load


# ---------------------------------------------------------------------------
# helpers independent of the oracle
# ---------------------------------------------------------------------------
def enumerate_slots(table, b):
    """(block, offset) of every slot a table covers, in logical order.

    Built by walking the table block by block, without any division, so it
    is a second derivation of the address mapping.
    """
    out = []
    for blk in table:
        for off in range(b):
            out.append((blk, off))
    return out


def contiguous_rows(pool, table, length, b, head):
    return np.stack([pool[blk, head, off] for blk, off in enumerate_slots(table, b)[:length]])


def approx_equal(value, printed):
    """True when ``value`` rounds to ``printed`` at the precision printed."""
    text = str(printed)
    digits = len(text.split(".")[1]) if "." in text else 0
    return round(float(value), digits) == float(text)


# ---------------------------------------------------------------------------
# address arithmetic
# ---------------------------------------------------------------------------
def check_address_example(translate, blocks_needed, tail_waste):
    g = load("address_example.txt")
    b = int(g["block_size"])
    n = int(g["request_tokens"])
    assert blocks_needed(n, b) == int(g["request_blocks"])
    assert tail_waste(n, b) == int(g["request_unused_slots"])
    table = ints(g["example_table"])
    # The position being written lies in the block after the 50 stored tokens'
    # last full slot; the table has room for it (4 blocks = 64 slots).
    lb, off, pb, slot = translate(int(g["position"]), b, table)
    assert off == int(g["position_offset"])
    assert pb == int(g["position_physical_block"])
    assert slot == pb * b + off
    assert blocks_needed(65, b) == int(g["token_65_blocks"])
    assert blocks_needed(64, b) == int(g["token_65_blocks"]) - 1
    short = int(g["short_request_tokens"])
    assert blocks_needed(short, b) * b == int(g["short_request_slots"])
    assert tail_waste(short, b) == int(g["short_request_unused"])


def check_translate_enumeration(translate, seed=0):
    rng = random.Random(seed)
    for b in (1, 4, 8, 16, 32):
        for _ in range(20):
            nblk = rng.randint(1, 9)
            table = rng.sample(range(1000), nblk)
            slots = enumerate_slots(table, b)
            for t in range(len(slots)):
                lb, off, pb, slot = translate(t, b, table)
                assert (pb, off) == slots[t]
                assert table[lb] == pb
                assert slot == slots[t][0] * b + slots[t][1]


# ---------------------------------------------------------------------------
# fragmentation and sizing
# ---------------------------------------------------------------------------
def check_utilization(paged_utilization, reserved_utilization, mean_tail_waste, allocated_slots):
    g = load("utilization.txt")
    lo, hi, b = int(g["len_lo"]), int(g["len_hi"]), int(g["block_size"])
    lengths = list(range(lo, hi + 1))
    assert Fraction(sum(lengths), len(lengths)) == int(g["mean_length"])
    assert reserved_utilization(lengths, 2000) * 100 == int(g["reserve_2000_percent"])
    waste = mean_tail_waste(lengths, b)
    assert approx_equal(waste, g["mean_tail_waste_about"])
    assert approx_equal(paged_utilization(lengths, b) * 100, g["paged_utilization_percent_about"])
    assert approx_equal(reserved_utilization(lengths, 4096) * 100, g["reserve_4096_percent_about"])
    # Closed form by residue counting: a length with residue r = T mod b
    # wastes (b - r) mod b slots; count how many lengths fall in each class.
    counts = [0] * b
    for r in range(b):
        first = lo + ((r - lo) % b)
        counts[r] = 0 if first > hi else (hi - first) // b + 1
    total_waste = sum(c * ((b - r) % b) for r, c in enumerate(counts))
    assert waste == Fraction(total_waste, len(lengths))
    assert allocated_slots(lengths, b) == sum(lengths) + total_waste
    assert paged_utilization(lengths, b) == Fraction(sum(lengths), sum(lengths) + total_waste)
    # Bound printed next to the formula: total waste below b per request.
    assert allocated_slots(lengths, b) - sum(lengths) < b * len(lengths)


def check_kv_bytes(kv_bytes_per_token):
    g = load("opt13b_kv.txt")
    per_tok = kv_bytes_per_token(int(g["num_layers"]), int(g["hidden_size"]), int(g["elem_bytes"]))
    # "about 800 KB": binary kilobytes, and exactly so for this shape.
    assert approx_equal(per_tok / 1024, g["kv_kb_per_token_about"])
    seq = per_tok * int(g["sequence_tokens"])
    assert approx_equal(seq / 2 ** 30, g["sequence_gb_about"])


# ---------------------------------------------------------------------------
# block pool
# ---------------------------------------------------------------------------
def check_cow_demo(BlockPool):
    g = load("cow_demo.txt")
    pool = BlockPool(int(g["pool_blocks"]), int(g["block_width"]))
    pool.admit("A", ints(g["parent_tokens"]))
    pool.fork("A", "C")
    assert pool.table("A") == pool.table("C")
    res = pool.append("C", int(g["child_token"]))
    assert res.copy is not None and res.copy[0] == pool.table("A")[-1]
    assert pool.read("A") == ints(g["parent_after"])
    assert pool.read("C") == ints(g["child_after"])
    assert pool.table("A")[0] == pool.table("C")[0]
    assert pool.table("A")[-1] != pool.table("C")[-1]
    pool.release("A")
    assert pool.read("C") == ints(g["child_after"])
    pool.release("C")
    assert pool.num_free() == int(g["pool_blocks"])

    small = BlockPool(int(g["small_pool_blocks"]), int(g["block_width"]))
    small.admit("A", ints(g["small_parent_tokens"]))
    small.fork("A", "B")
    before = (small.read("A"), small.read("B"), small.refcounts(), list(small.slots))
    failed = False
    try:
        small.append("B", int(g["small_child_token"]))
    except MemoryError:
        failed = True
    assert failed
    assert before == (small.read("A"), small.read("B"), small.refcounts(), list(small.slots))
    # Negative control: B's next token written straight into the shared tail
    # (no copy) lands in the block A reads through, which then holds 1, 2, 99,
    # and the recomputed invariants flag the block as shared with two fills.
    t, w = small.length("B"), small.width
    small.slots[small.table("B")[t // w] * w + t % w] = int(g["negative_control_token"])
    small.lengths["B"] = t + 1
    assert small.block_contents(small.table("A")[-1]) == ints(g["negative_control_parent_after"])
    try:
        small.verify()
        caught = False
    except AssertionError:
        caught = True
    assert caught


def check_fork_workload(BlockPool, b=16, prompt=1031, forks=8):
    """One prompt forked into ``forks`` sequences, each appending a token.

    Following the append rule, every fork but the last to append finds the
    shared partial block held by others and copies it; the last holder
    writes in place.
    """
    full = prompt // b
    pool = BlockPool(200, b)
    pool.admit(0, list(range(prompt)))
    for f in range(1, forks):
        pool.fork(0, f)
    pairs = []
    for f in range(forks):
        res = pool.append(f, 10_000 + f)
        if res.copy:
            pairs.append(res.copy)
    assert len(pairs) == forks - 1
    shared = pool.table(0)[:full]
    for f in range(forks):
        assert pool.table(f)[:full] == shared
        assert pool.read(f) == list(range(prompt)) + [10_000 + f]
        assert pool.refcounts()[pool.table(f)[-1]] == 1
    assert all(pool.refcounts()[blk] == forks for blk in shared)
    assert 200 - pool.num_free() == full + forks
    assert len({pool.table(f)[-1] for f in range(forks)}) == forks


def check_pool_vs_contiguous(BlockPool, allocated_slots, seed=1):
    """Random operations; every read equals a plain per-sequence list."""
    rng = random.Random(seed)
    b = 4
    pool = BlockPool(64, b, free_order=rng.sample(range(64), 64))
    plain = {}
    nxt = 0
    for step in range(400):
        op = rng.random()
        names = list(plain)
        try:
            if op < 0.25 or not names:
                n = rng.randint(1, 12)
                toks = list(range(nxt, nxt + n)); nxt += n
                pool.admit(step, toks)
                plain[step] = toks
            elif op < 0.45:
                src = rng.choice(names)
                pool.fork(src, step)
                plain[step] = list(plain[src])
            elif op < 0.85:
                name = rng.choice(names)
                pool.append(name, nxt)
                plain[name].append(nxt); nxt += 1
            else:
                name = rng.choice(names)
                pool.release(name)
                del plain[name]
        except MemoryError:
            pass
        for name, toks in plain.items():
            assert pool.read(name) == toks
        held = {blk for name in plain for blk in pool.table(name)}
        assert len(held) == 64 - pool.num_free()
    # Without sharing, slots held equal the closed form.
    solo = BlockPool(64, b)
    lens = [3, 4, 5, 9, 16, 1]
    for i, n in enumerate(lens):
        solo.admit(i, list(range(n)))
    assert (64 - solo.num_free()) * b == allocated_slots(lens, b)


# ---------------------------------------------------------------------------
# write and copy
# ---------------------------------------------------------------------------
def _flat_rows(pool):
    """View [N, Hk, b, D] as one row per slot: [N * b, Hk, D]."""
    n, hk, b, d = pool.shape
    return np.ascontiguousarray(np.moveaxis(pool, 1, 2)).reshape(n * b, hk, d)


def check_write(write_tokens, seed=2):
    rng = np.random.default_rng(seed)
    n, hk, b, d = 7, 3, 4, 8
    kp = rng.integers(0, 2 ** 16, size=(n, hk, b, d)).astype(np.uint16)
    vp = rng.integers(0, 2 ** 16, size=(n, hk, b, d)).astype(np.uint16)
    slots = [5, -1, 27, 0, 13, n * b + 3]
    kn = rng.integers(0, 2 ** 16, size=(len(slots), hk, d)).astype(np.uint16)
    vn = rng.integers(0, 2 ** 16, size=(len(slots), hk, d)).astype(np.uint16)
    k2, v2, bad = write_tokens(kp, vp, kn, vn, slots, b)
    assert bad == [5]
    fk, fv = _flat_rows(kp), _flat_rows(vp)
    for i, s in enumerate(slots):
        if 0 <= s < n * b:
            fk[s] = kn[i]
            fv[s] = vn[i]
    assert np.array_equal(_flat_rows(k2), fk) and np.array_equal(_flat_rows(v2), fv)
    assert k2.dtype == kp.dtype and not np.array_equal(k2, kp)


def check_copy(copy_blocks, seed=3):
    rng = np.random.default_rng(seed)
    kp = rng.standard_normal((6, 2, 4, 8)).astype(np.float32)
    vp = rng.standard_normal((6, 2, 4, 8)).astype(np.float32)
    k2, v2, bad = copy_blocks(kp, vp, [(1, 4), (2, 5), (0, 9)])
    assert bad == [2]
    for blk, src in enumerate([0, 1, 2, 3, 1, 2]):
        assert np.array_equal(k2[blk], kp[src]) and np.array_equal(v2[blk], vp[src])


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def tiny_case(seed=4, dtype=np.float32):
    """Tiny MHA case: 4 heads, D=8, b=4, scattered tables of lengths 9,3,13,1."""
    rng = np.random.default_rng(seed)
    n, hk, b, d = 12, 4, 4, 8
    perm = list(rng.permutation(n))
    lens = [9, 3, 13, 1]
    tables, pos = [], 0
    for L in lens:
        k = -(-L // b)
        tables.append([int(x) for x in perm[pos:pos + k]]); pos += k
    kp = rng.standard_normal((n, hk, b, d)).astype(dtype)
    vp = rng.standard_normal((n, hk, b, d)).astype(dtype)
    q = rng.standard_normal((len(lens), hk, d)).astype(dtype)
    return q, kp, vp, tables, lens, b


def check_bruteforce(attention):
    q, kp, vp, tables, lens, b = tiny_case()
    scale = 1 / math.sqrt(q.shape[-1])
    out, bad = attention(q, kp, vp, tables, lens, scale, b, "f32")
    assert bad == []
    for s, L in enumerate(lens):
        for h in range(q.shape[1]):
            keys = [[float(x) for x in row] for row in contiguous_rows(kp, tables[s], L, b, h)]
            vals = [[float(x) for x in row] for row in contiguous_rows(vp, tables[s], L, b, h)]
            ref = brute(list(map(float, q[s, h])), keys, vals, scale)
            assert np.max(np.abs(out[s, h] - np.array(ref))) < 1e-12


def brute(q_row, keys, vals, scale):
    z = [scale * math.fsum(a * c for a, c in zip(q_row, k)) for k in keys]
    top = max(z)
    w = [math.exp(x - top) for x in z]
    tot = math.fsum(w)
    return [math.fsum(w[t] * vals[t][i] for t in range(len(vals))) / tot for i in range(len(vals[0]))]


def check_contiguous_torch(attention, seed=5):
    """Identity table over a contiguous pool == torch softmax attention."""
    rng = np.random.default_rng(seed)
    b, hk, d, G = 4, 2, 16, 3
    L = 23
    nblk = -(-L // b)
    kp = rng.standard_normal((nblk, hk, b, d)).astype(np.float32)
    vp = rng.standard_normal((nblk, hk, b, d)).astype(np.float32)
    q = rng.standard_normal((1, hk * G, d)).astype(np.float32)
    out, _ = attention(q, kp, vp, [list(range(nblk))], [L], 0.3, b, "f32")
    kp, vp, q = kp.astype(np.float64), vp.astype(np.float64), q.astype(np.float64)
    kc = torch.from_numpy(kp).permute(1, 0, 2, 3).reshape(hk, nblk * b, d)[:, :L]
    vc = torch.from_numpy(vp).permute(1, 0, 2, 3).reshape(hk, nblk * b, d)[:, :L]
    qt = torch.from_numpy(q[0]).reshape(hk, G, d)
    w = torch.softmax(0.3 * qt @ kc.transpose(1, 2), dim=-1)
    ref = (w @ vc).reshape(hk * G, d).numpy()
    assert np.max(np.abs(out[0].astype(np.float64) - ref)) < 1e-12


def check_special_cases(attention, seed=6):
    rng = np.random.default_rng(seed)
    b, hk, d = 4, 1, 8
    kp = rng.standard_normal((5, hk, b, d)).astype(np.float32)
    vp = rng.standard_normal((5, hk, b, d)).astype(np.float32)
    q = rng.standard_normal((1, 1, d)).astype(np.float32)
    # Length 1: the output is the single value row.
    out, _ = attention(q, kp, vp, [[3]], [1], 0.7, b, "f32")
    assert np.array_equal(out[0, 0], vp[3, 0, 0].astype(np.float64))
    # All keys equal: uniform weights, the output is the mean of the values.
    kq = kp.copy()
    kq[:] = kp[0, 0, 0]
    out, _ = attention(q, kq, vp, [[2, 0, 4]], [10], 0.7, b, "f32")
    rows = np.concatenate([vp[2, 0], vp[0, 0], vp[4, 0, :2]]).astype(np.float64)
    assert np.max(np.abs(out[0, 0] - rows.mean(axis=0))) < 1e-12
    # Two keys: the weight of the first is a logistic of the score gap.
    kt = np.zeros((1, 1, b, d))
    vt = np.zeros((1, 1, b, d))
    kt[0, 0, 0, 0], kt[0, 0, 1, 1] = 1.0, 1.0
    vt[0, 0, 0, 2], vt[0, 0, 1, 3] = 1.0, 1.0
    qq = np.zeros((1, 1, d))
    qq[0, 0, 0], qq[0, 0, 1] = 2.0, -1.0
    scale = 0.5
    out, _ = attention(qq, kt, vt, [[0]], [2], scale, b, "f32")
    w0 = 1.0 / (1.0 + math.exp(-(scale * 2.0 - scale * -1.0)))
    assert abs(out[0, 0, 2] - w0) < 1e-15 and abs(out[0, 0, 3] - (1 - w0)) < 1e-15


def check_gqa_mapping(attention):
    """Query head h must read KV head h // (H / Hk)."""
    b, hk, G, d = 4, 3, 4, 4
    kp = np.zeros((2, hk, b, d))
    vp = np.zeros((2, hk, b, d))
    for k in range(hk):
        vp[:, k] = k + 1.0
    q = np.ones((1, hk * G, d))
    out, _ = attention(q, kp, vp, [[1, 0]], [7], 1.0, b, "f32")
    for h in range(hk * G):
        assert np.all(out[0, h] == h // G + 1.0)


def check_relabel_invariance(attention, seed=7):
    q, kp, vp, tables, lens, b = tiny_case(seed)
    out, _ = attention(q, kp, vp, tables, lens, 0.25, b, "f32")
    perm = np.random.default_rng(seed + 1).permutation(kp.shape[0])
    kq = np.empty_like(kp)
    vq = np.empty_like(vp)
    kq[perm] = kp
    vq[perm] = vp
    tq = [[int(perm[x]) for x in t] for t in tables]
    out2, _ = attention(q, kq, vq, tq, lens, 0.25, b, "f32")
    assert np.array_equal(out, out2)


def check_invalid_rows(attention):
    q, kp, vp, tables, lens, b = tiny_case()
    tables = [list(t) for t in tables]
    tables[1][0] = kp.shape[0] + 5
    lens = list(lens)
    lens[2] = 0
    out, bad = attention(q, kp, vp, tables, lens, 0.5, b, "f32")
    assert sorted(bad) == [1, 2]
    assert np.all(out[1] == 0) and np.all(out[2] == 0)
    assert np.all(np.isfinite(out[0])) and np.any(out[0] != 0)


def check_split_merge(attention, partition_stats, merge_partitions):
    q, kp, vp, tables, lens, b = tiny_case(8)
    out, _ = attention(q, kp, vp, tables, lens, 0.4, b, "f32")
    for ps in (4, 8):
        stats = partition_stats(q, kp, vp, tables, lens, 0.4, b, "f32", ps)
        for (s, h), (m, l, o) in stats.items():
            assert len(m) == -(-lens[s] // ps)
            assert np.max(np.abs(merge_partitions(m, l, o) - out[s, h])) < 1e-12
            # The first partition alone is plain attention over its positions.
            keys = contiguous_rows(kp, tables[s], min(ps, lens[s]), b, h).astype(np.float64)
            z = 0.4 * keys @ q[s, h].astype(np.float64)
            assert abs(m[0] - z.max()) < 1e-12
            assert abs(l[0] - np.exp(z - z.max()).sum()) < 1e-12


def check_bf16(to_f64, seed=9):
    bits = np.random.default_rng(seed).integers(0, 2 ** 16, size=4096).astype(np.uint16)
    bits = bits[((bits >> 7) & 0xFF) != 0xFF]  # drop inf/NaN patterns
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(to_f64(bits, "bf16"), ref)
    half = np.random.default_rng(seed).standard_normal(100).astype(np.float16)
    assert np.array_equal(to_f64(half, "f16"), half.astype(np.float64))


def check_swap(swap_blocks, copy_blocks, seed=10):
    """Swapping out then in restores blocks; it equals a copy within one
    pool made of the device pool followed by the host pool."""
    rng = np.random.default_rng(seed)
    dk = rng.integers(0, 2 ** 16, size=(6, 2, 4, 8)).astype(np.uint16)
    dv = rng.integers(0, 2 ** 16, size=(6, 2, 4, 8)).astype(np.uint16)
    hk = np.zeros((4, 2, 4, 8), dtype=np.uint16)
    hv = np.zeros((4, 2, 4, 8), dtype=np.uint16)
    out_pairs = [(5, 0), (2, 3), (1, 9)]
    dk1, dv1, hk1, hv1, bad = swap_blocks(dk, dv, hk, hv, out_pairs, "out")
    assert bad == [2]
    assert np.array_equal(dk1, dk) and np.array_equal(dv1, dv)
    both_k, both_v, _ = copy_blocks(np.concatenate([dk, hk]), np.concatenate([dv, hv]),
                                    [(s_, 6 + d_) for s_, d_ in out_pairs[:2]])
    assert np.array_equal(hk1, both_k[6:]) and np.array_equal(hv1, both_v[6:])
    # Reuse the device blocks, then bring the data back elsewhere.
    dk2 = dk1.copy()
    dk2[[5, 2]] = 0
    dk3, dv3, _, _, bad = swap_blocks(dk2, dv1, hk1, hv1, [(0, 4), (3, 0)], "in")
    assert bad == []
    assert np.array_equal(dk3[4], dk[5]) and np.array_equal(dk3[0], dk[2])
    assert np.array_equal(dv3[4], dv[5]) and np.array_equal(dv3[0], dv[2])


def check_prefill(prefill_attention, attention, seed=11):
    """Prefill pins: a one-query chunk is decode; with no cached prefix and an
    identity table it is torch's causal scaled-dot-product attention; the
    outputs of earlier queries do not depend on later keys."""
    rng = np.random.default_rng(seed)
    b, hk, G, d = 4, 2, 2, 8
    lens = [9, 6, 13]
    chunk = [3, 6, 1]                      # queries per sequence (6 = whole prompt)
    starts = np.concatenate([[0], np.cumsum(chunk)])
    nblk = [-(-L // b) for L in lens]
    perm = rng.permutation(sum(nblk) + 2)
    tables, pos = [], 0
    for k in nblk:
        tables.append([int(x) for x in perm[pos:pos + k]]); pos += k
    kp = rng.standard_normal((len(perm), hk, b, d)).astype(np.float32)
    vp = rng.standard_normal((len(perm), hk, b, d)).astype(np.float32)
    q = rng.standard_normal((int(starts[-1]), hk * G, d)).astype(np.float32)
    out = prefill_attention(q, kp, vp, tables, lens, starts, 0.35, b, "f32")
    # One-query chunk (sequence 2) and each query of a chunk = decode over its prefix.
    for s_ in range(3):
        for i in range(chunk[s_]):
            L = lens[s_] - chunk[s_] + i + 1
            ref, _ = attention(q[starts[s_] + i:starts[s_] + i + 1], kp, vp, [tables[s_]], [L],
                               0.35, b, "f32")
            assert np.max(np.abs(out[starts[s_] + i] - ref[0])) < 1e-12
    # Whole-prompt chunk (sequence 1, no prefix): torch causal attention.
    rows = lambda pool: np.stack([pool[tables[1][t // b], :, t % b] for t in range(6)])  # noqa: E731
    kc = torch.from_numpy(rows(kp).astype(np.float64)).permute(1, 0, 2)   # [Hk, 6, d]
    vc = torch.from_numpy(rows(vp).astype(np.float64)).permute(1, 0, 2)
    qc = torch.from_numpy(q[starts[1]:starts[2]].astype(np.float64)).permute(1, 0, 2)  # [H, 6, d]
    kc = kc.repeat_interleave(G, dim=0)
    vc = vc.repeat_interleave(G, dim=0)
    ref = torch.nn.functional.scaled_dot_product_attention(qc, kc, vc, is_causal=True, scale=0.35)
    assert np.max(np.abs(out[starts[1]:starts[2]] - ref.permute(1, 0, 2).numpy())) < 1e-12
    # Causality: changing the last position's key and value leaves every
    # query that cannot see it unchanged.
    k2, v2 = kp.copy(), vp.copy()
    last = lens[0] - 1
    k2[tables[0][last // b], :, last % b] += 5.0
    v2[tables[0][last // b], :, last % b] -= 3.0
    out2 = prefill_attention(q, k2, v2, tables, lens, starts, 0.35, b, "f32", seqs=[0])
    assert np.array_equal(out2[starts[0]:starts[0] + 2], out[starts[0]:starts[0] + 2])
    assert not np.allclose(out2[starts[0] + 2], out[starts[0] + 2])


def check_e4m3(e4m3_encode, e4m3_decode, seed=12):
    """E4M3 codes: torch's float8_e4m3fn cast (round to nearest even) on
    in-range values, the format's landmark codes, saturation, and the
    half-step error bound."""
    rng = np.random.default_rng(seed)
    x = np.concatenate([rng.standard_normal(4000) * 40, rng.uniform(-464, 464, 4000),
                        [0.0, 1.0, 448.0, -448.0, 2.0 ** -9, 1.0625, 1.1875, 464.0, 0.5, 240.0]])
    x = x.astype(np.float32)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3_encode(x), ref)
    # landmarks from the format: 1.0, the largest finite, the smallest subnormal
    assert e4m3_encode(np.float32(1.0)) == 0x38 and e4m3_decode(0x38) == 1.0
    assert e4m3_decode(0x7E) == 448.0 and e4m3_decode(0x01) == 2.0 ** -9
    assert np.isnan(e4m3_decode(0x7F)) and np.isnan(e4m3_decode(0xFF))
    # saturation instead of NaN beyond the largest finite
    assert e4m3_encode(np.float32(1e4)) == 0x7E and e4m3_encode(np.float32(-1e4)) == 0xFE
    # round trip within half a step (3 mantissa bits: relative 2^-4)
    y = np.abs(rng.uniform(2.0 ** -6, 448, 2000).astype(np.float32))
    assert np.all(np.abs(e4m3_decode(e4m3_encode(y)) - y) <= y * 2.0 ** -4)


def check_fp8_write_and_attention(write_tokens_fp8, dequantize_pool, attention, e4m3_encode):
    rng = np.random.default_rng(13)
    n, hk, b, d = 6, 2, 4, 8
    kp = rng.integers(0, 0x7E, size=(n, hk, b, d)).astype(np.uint8)
    vp = rng.integers(0, 0x7E, size=(n, hk, b, d)).astype(np.uint8)
    kn = rng.standard_normal((3, hk, d)).astype(np.float16)
    vn = rng.standard_normal((3, hk, d)).astype(np.float16)
    ks, vs = np.array([0.02, 0.5], np.float32), np.array([0.01, 0.25], np.float32)
    slots = [5, 17, 22]
    k2, v2, bad = write_tokens_fp8(kp, vp, kn, vn, slots, b, ks, vs, "f16")
    assert bad == []
    for i, sl in enumerate(slots):
        for h in range(hk):
            assert np.array_equal(k2[sl // b, h, sl % b],
                                  e4m3_encode(kn[i, h].astype(np.float32) / ks[h]))
    # Attention over an FP8 pool equals attention over its dequantized values.
    q = rng.standard_normal((2, hk * 2, d)).astype(np.float16)
    tables, lens = [[3, 1], [0, 5, 2]], [7, 10]
    out, _ = attention(q, k2, v2, tables, lens, 0.3, b, "e4m3", q_dtype="f16", k_scale=ks, v_scale=vs)
    ref, _ = attention(q.astype(np.float64), dequantize_pool(k2, ks), dequantize_pool(v2, vs), tables,
                       lens, 0.3, b, "f64")
    assert np.max(np.abs(out - ref)) < 1e-12


def check_fp8_prefill(prefill_attention, attention, dequantize_pool):
    """Causal prefill over an FP8 pool equals prefill over its dequantized
    float64 values, and one-query chunks equal FP8 decode attention."""
    rng = np.random.default_rng(17)
    n, hk, b, d, g = 8, 2, 4, 8, 2
    kp = rng.integers(0, 0x7E, size=(n, hk, b, d)).astype(np.uint8)
    vp = rng.integers(0, 0x7E, size=(n, hk, b, d)).astype(np.uint8)
    kp[kp % 3 == 0] |= 0x80  # some negative codes
    ks, vs = np.array([0.03, 0.2], np.float32), np.array([0.05, 0.01], np.float32)
    tables, lens = [[6, 1, 3], [0, 4, 2, 5]], [11, 14]
    starts = np.array([0, 4, 9])  # chunks of 4 and 5 new queries
    q = rng.standard_normal((9, hk * g, d)).astype(np.float16)
    out = prefill_attention(q, kp, vp, tables, lens, starts, 0.25, b, "e4m3", q_dtype="f16",
                            k_scale=ks, v_scale=vs)
    ref = prefill_attention(q.astype(np.float64), dequantize_pool(kp, ks), dequantize_pool(vp, vs),
                            tables, lens, starts, 0.25, b, "f64")
    assert np.max(np.abs(out - ref)) < 1e-12
    # The last query of each chunk sees the whole sequence: decode attention.
    last = [int(starts[1]) - 1, int(starts[2]) - 1]
    dec, _ = attention(q[last], kp, vp, tables, lens, 0.25, b, "e4m3", q_dtype="f16", k_scale=ks,
                       v_scale=vs)
    assert np.max(np.abs(out[last] - dec)) < 1e-12

"""KV write, block copy and paged single-query attention, in float64 (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

[vLLM-TGI] = "Inside vLLM and TGI: Paging, Versioned Schedulers and
Operations"; [VM-LLM] = "vLLM and PagedAttention: Virtual Memory for LLM
Serving" (transcript); [CB-PA] = "Continuous Batching & PagedAttention: vLLM
Memory Management Architecture".

Storage convention (a reading: [vLLM-TGI] "Block addresses and fragmentation
arithmetic" says the physical layout is backend-specific): the key pool and
the value pool are separate arrays of shape ``[num_blocks, kv_heads, b, D]``.
Row ``(blk, head, off)`` holds one token's key (or value) for one KV head.

Element types are named ``"f32"``, ``"f16"`` and ``"bf16"``.  NumPy has no
bfloat16, so bf16 arrays are carried as their raw ``uint16`` bit patterns; a
bf16 number is by definition the upper half of an IEEE binary32, which is how
:func:`to_f64` widens it.

Paging changes where keys and values are stored, not what attention
computes ([vLLM-TGI] opening section: kernels read a sequence through a
block table; [VM-LLM] paging paragraph: token order remains correct while
blocks come from anywhere in the pool).  The attention oracle is therefore
the textbook definition of one query attending over the gathered logical
sequence, evaluated in float64 on the stored (already rounded) inputs.
"""

import math

import numpy as np

DTYPES = ("f32", "f16", "bf16", "e4m3")


# ---------------------------------------------------------------------------
# FP8 E4M3 (OCP 8-bit floating point, "E4M3" variant): 1 sign bit, 4 exponent
# bits with bias 7, 3 mantissa bits; exponent 0 encodes subnormals
# (mantissa / 8 * 2^-6); the all-ones exponent with all-ones mantissa is NaN;
# there are no infinities, so the largest finite magnitude is 1.75 * 2^8 =
# 448.  Cache codes here are produced with round-to-nearest-even and
# saturation to +-448 ("satfinite").
# ---------------------------------------------------------------------------
def e4m3_decode(codes):
    """Codes (uint8) to float64 values; NaN for the two NaN codes."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    exp = (c >> 3) & 0xF
    man = (c & 7).astype(np.float64)
    val = np.where(exp == 0, man / 8.0 * 2.0 ** -6, (1.0 + man / 8.0) * 2.0 ** (exp - 7.0))
    val = np.where((exp == 15) & ((c & 7) == 7), np.nan, val)
    return sign * val


_E4M3_POS = e4m3_decode(np.arange(0x7F))  # codes 0x00..0x7E: 0 .. 448, increasing


def e4m3_encode(x):
    """float32 values to E4M3 codes: nearest value, ties to the even code
    (even mantissa), magnitudes beyond 448 saturate to 448, NaN to 0x7F."""
    x = np.asarray(x, dtype=np.float32).astype(np.float64)
    mag = np.abs(x)
    hi = np.clip(np.searchsorted(_E4M3_POS, mag, side="left"), 0, 0x7E)
    lo = np.clip(hi - 1, 0, 0x7E)
    d_hi = np.abs(_E4M3_POS[hi] - mag)
    d_lo = np.abs(mag - _E4M3_POS[lo])
    pick = np.where(d_lo < d_hi, lo, np.where(d_hi < d_lo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(mag >= 448.0, 0x7E, pick)
    code = (pick | np.where(np.signbit(x), 0x80, 0)).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def to_f64(x, dtype):
    """Widen stored elements to float64 exactly."""
    x = np.asarray(x)
    if dtype == "f64":
        return x.astype(np.float64)
    if dtype == "e4m3":
        return e4m3_decode(x)
    if dtype == "f32":
        return x.astype(np.float32, copy=False).astype(np.float64)
    if dtype == "f16":
        return x.astype(np.float16, copy=False).astype(np.float64)
    if dtype == "bf16":
        bits = x.astype(np.uint16, copy=False).astype(np.uint32) << np.uint32(16)
        return bits.view(np.float32).astype(np.float64)
    raise ValueError("unknown dtype %r" % (dtype,))


# ---------------------------------------------------------------------------
# KV write (reshape-and-cache)
# ---------------------------------------------------------------------------
def write_tokens(k_pool, v_pool, k_new, v_new, slot_mapping, b):
    """Store each new token's key and value rows at its slot.

    [VM-LLM] paging paragraph and [vLLM-TGI] "Exact CPU block manager and
    copy-on-write" (append): a token goes into its sequence's last block at
    the next free offset.  The slot is ``block * b + offset``, so the block
    is ``slot // b`` and the offset ``slot % b``.

    ``k_pool``/``v_pool``: ``[N, Hk, b, D]``; ``k_new``/``v_new``:
    ``[T, Hk, D]``; ``slot_mapping``: ``T`` integers.  Element values are
    copied as they are (any dtype, bit patterns included).  A negative slot
    marks a padding token and is skipped; a slot at or beyond ``N * b`` is
    skipped and reported.

    Returns ``(k_pool', v_pool', bad)`` where ``bad`` lists the token indices
    whose slot was out of range.  The input pools are not modified.
    """
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    n_blocks = k_out.shape[0]
    bad = []
    for i, slot in enumerate(slot_mapping):
        slot = int(slot)
        if slot < 0:
            continue
        blk, off = slot // b, slot % b
        if blk >= n_blocks:
            bad.append(i)
            continue
        for h in range(k_out.shape[1]):
            k_out[blk, h, off, :] = k_new[i, h, :]
            v_out[blk, h, off, :] = v_new[i, h, :]
    return k_out, v_out, bad


def write_tokens_fp8(k_pool, v_pool, k_new, v_new, slot_mapping, b, k_scale, v_scale, io_dtype):
    """KV write into an FP8 E4M3 pool with one scale per KV head.

    Like :func:`write_tokens`, but each new element x (stored in
    ``io_dtype``, widened exactly to float32) is stored as the code
    ``e4m3(x / scale[h])``, the division done in float32 (correctly
    rounded).  Reading the cache back gives ``value(code) * scale[h]``.
    """
    kq = np.empty(k_new.shape, dtype=np.uint8)
    vq = np.empty(v_new.shape, dtype=np.uint8)
    for h in range(k_new.shape[1]):
        kx = to_f64(k_new[:, h], io_dtype).astype(np.float32)
        vx = to_f64(v_new[:, h], io_dtype).astype(np.float32)
        kq[:, h] = e4m3_encode(kx / np.float32(k_scale[h]))
        vq[:, h] = e4m3_encode(vx / np.float32(v_scale[h]))
    return write_tokens(k_pool, v_pool, kq, vq, slot_mapping, b)


def dequantize_pool(codes, scales):
    """float64 values of an E4M3 pool ``[N, Hk, b, D]`` with per-head scales."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[None, :, None, None]


# ---------------------------------------------------------------------------
# Block copy (copy-on-write)
# ---------------------------------------------------------------------------
def copy_blocks(k_pool, v_pool, pairs):
    """Copy whole blocks: for each (src, dst), block dst := block src.

    [vLLM-TGI] "Exact CPU block manager and copy-on-write" (append to a
    shared partial block takes a fresh block and copies the old contents
    into it) and [VM-LLM] sharing paragraph (a private copy for the branch
    being modified).  Every KV head of the block is copied, for keys and
    values.  Pairs are applied in order.  A pair naming a block outside
    ``[0, N)`` is skipped and reported; returns ``(k', v', bad)``.
    """
    k_out = np.array(k_pool, copy=True)
    v_out = np.array(v_pool, copy=True)
    n_blocks = k_out.shape[0]
    bad = []
    for i, (src, dst) in enumerate(pairs):
        src, dst = int(src), int(dst)
        if not (0 <= src < n_blocks and 0 <= dst < n_blocks):
            bad.append(i)
            continue
        k_out[dst] = k_out[src]
        v_out[dst] = v_out[src]
    return k_out, v_out, bad


def swap_blocks(dev_k, dev_v, host_k, host_v, pairs, direction):
    """Move whole blocks between a device pool and a host pool.

    "vLLM and PagedAttention: Virtual Memory for LLM Serving" (preemption
    paragraph): KV data can be swapped into CPU memory and restored later.
    ``direction`` "out": host block dst := device block src; "in": device
    block dst := host block src.  Both pools are ``[blocks, Hk, b, D]``.
    Pairs naming a block outside its pool are skipped and reported.
    Returns ``(dev_k', dev_v', host_k', host_v', bad)``.
    """
    dk, dv = np.array(dev_k, copy=True), np.array(dev_v, copy=True)
    hk, hv = np.array(host_k, copy=True), np.array(host_v, copy=True)
    if direction == "out":
        src_k, src_v, dst_k, dst_v = dk, dv, hk, hv
    elif direction == "in":
        src_k, src_v, dst_k, dst_v = hk, hv, dk, dv
    else:
        raise ValueError("direction must be 'out' or 'in'")
    bad = []
    for i, (src, dst) in enumerate(pairs):
        src, dst = int(src), int(dst)
        if not (0 <= src < src_k.shape[0] and 0 <= dst < dst_k.shape[0]):
            bad.append(i)
            continue
        dst_k[dst] = src_k[src]
        dst_v[dst] = src_v[src]
    return dk, dv, hk, hv, bad


# ---------------------------------------------------------------------------
# Attention
# ---------------------------------------------------------------------------
def gather_rows(pool, table, length, b, kv_head):
    """Rows ``0..length-1`` of one KV head of a sequence, in logical order.

    Position t lives in physical block ``table[t // b]`` at offset ``t % b``
    ([vLLM-TGI] "Block addresses and fragmentation arithmetic").
    """
    return np.stack([pool[table[t // b], kv_head, t % b, :] for t in range(length)])


def _check_row(table, length, n_blocks, b, max_len):
    """True when a sequence's length and the table entries it uses are valid.

    [vLLM-TGI] "Exact CPU block manager and copy-on-write" asks that a
    kernel's table be validated (bounds, logical length) before use; an
    empty request is not admissible in the same section's model.
    """
    if length < 1 or length > max_len or length > len(table) * b:
        return False
    used = table[: -(-length // b)]
    return all(0 <= int(x) < n_blocks for x in used)


def attention(q, k_pool, v_pool, tables, seq_lens, scale, b, dtype, seqs=None, max_len=None,
              q_dtype=None, k_scale=None, v_scale=None):
    """Single-query attention of every sequence over its paged keys/values.

    For sequence s and query head h (KV head ``h // (H // Hk)``, query heads
    grouped contiguously), with ``L = seq_lens[s]`` and ``K_t``, ``V_t`` the
    rows gathered through the table:

        z_t = scale * (q[s, h] . K_t)          t = 0 .. L-1
        out[s, h] = sum_t exp(z_t - max z) V_t / sum_t exp(z_t - max z)

    ``q``: ``[S, H, D]``; pools ``[N, Hk, b, D]``; ``tables``: ``S`` lists
    (or a 2-D array) of physical block ids; all stored in ``dtype``.  For an
    FP8 (``"e4m3"``) pool, ``q`` is stored in ``q_dtype`` and key/value rows
    of KV head h are ``value(code) * k_scale[h]`` / ``* v_scale[h]``.  Rows
    whose length or table entries are invalid are set to zero and their
    sequence index is reported.  ``seqs`` restricts the work to a subset of
    sequences (other rows are NaN).  ``max_len`` is the caller's bound on
    lengths (default: the table width times b).

    Returns ``(out float64 [S, H, D], bad_sequences)``.
    """
    q = np.asarray(q)
    n_seq, n_heads, dim = q.shape
    n_blocks, kv_heads = k_pool.shape[0], k_pool.shape[1]
    if n_heads % kv_heads:
        raise ValueError("query heads must be a multiple of KV heads")
    group = n_heads // kv_heads
    out = np.full((n_seq, n_heads, dim), np.nan)
    bad = []
    for s in (range(n_seq) if seqs is None else seqs):
        table = [int(x) for x in tables[s]]
        length = int(seq_lens[s])
        bound = len(table) * b if max_len is None else max_len
        if not _check_row(table, length, n_blocks, b, bound):
            out[s] = 0.0
            bad.append(s)
            continue
        for kvh in range(kv_heads):
            keys = to_f64(gather_rows(k_pool, table, length, b, kvh), dtype)
            vals = to_f64(gather_rows(v_pool, table, length, b, kvh), dtype)
            if k_scale is not None:
                keys = keys * float(k_scale[kvh])
            if v_scale is not None:
                vals = vals * float(v_scale[kvh])
            for h in range(kvh * group, (kvh + 1) * group):
                z = scale * (keys @ to_f64(q[s, h], q_dtype or dtype))
                w = np.exp(z - z.max())
                out[s, h] = (w @ vals) / w.sum()
    return out, bad


def prefill_attention(q, k_pool, v_pool, tables, seq_lens, query_starts, scale, b, dtype,
                      seqs=None, q_dtype=None, k_scale=None, v_scale=None):
    """Causal attention of a chunk of new queries per sequence (prefill).

    "vLLM and PagedAttention: Virtual Memory for LLM Serving" (opening
    paragraph): during prefill all prompt tokens are known, so their queries
    are processed together; "Inside vLLM and TGI: Paging, Versioned
    Schedulers and Operations" (launch notes: chunked prefill) splits a long
    prompt into chunks.  Sequence s holds ``L = seq_lens[s]`` positions after
    its chunk of ``Q = query_starts[s + 1] - query_starts[s]`` queries was
    written; query i sits at position ``L - Q + i`` and attends, like a
    decode query, to positions ``0 .. L - Q + i`` of the sequence:

        out[query_starts[s] + i, h] = attention over the first L - Q + i + 1
                                      positions (see :func:`attention`)

    ``q``: ``[total queries, H, D]``; pools ``[N, Hk, b, D]``; returns
    ``out float64 [total queries, H, D]`` (rows of unlisted sequences NaN).
    For an FP8 (``"e4m3"``) pool, ``q`` is stored in ``q_dtype`` and the
    key/value rows of KV head kh are the codes' values times ``k_scale[kh]``
    / ``v_scale[kh]``, as in :func:`attention`.
    """
    q = np.asarray(q)
    _, n_heads, dim = q.shape
    kv_heads = k_pool.shape[1]
    group = n_heads // kv_heads
    out = np.full(q.shape, np.nan)
    n_seq = len(seq_lens)
    for s in (range(n_seq) if seqs is None else seqs):
        table = [int(x) for x in tables[s]]
        length = int(seq_lens[s])
        q0, q1 = int(query_starts[s]), int(query_starts[s + 1])
        first = length - (q1 - q0)
        for kvh in range(kv_heads):
            keys = to_f64(gather_rows(k_pool, table, length, b, kvh), dtype)
            vals = to_f64(gather_rows(v_pool, table, length, b, kvh), dtype)
            if k_scale is not None:
                keys = keys * float(k_scale[kvh])
            if v_scale is not None:
                vals = vals * float(v_scale[kvh])
            for h in range(kvh * group, (kvh + 1) * group):
                for i in range(q1 - q0):
                    visible = first + i + 1
                    z = scale * (keys[:visible] @ to_f64(q[q0 + i, h], q_dtype or dtype))
                    w = np.exp(z - z.max())
                    out[q0 + i, h] = (w @ vals[:visible]) / w.sum()
    return out


def partition_stats(q, k_pool, v_pool, tables, seq_lens, scale, b, dtype, partition_size, seqs=None):
    """Per-partition softmax statistics of a split-K decode.

    The keys of a sequence are cut into consecutive partitions of
    ``partition_size`` positions.  For partition p (positions
    ``p*P .. min(L, (p+1)*P) - 1``) and query head h:

        m_p = max_t z_t,  l_p = sum_t exp(z_t - m_p),
        o_p = sum_t exp(z_t - m_p) V_t / l_p

    with ``z_t`` as in :func:`attention` (natural-log domain).  Returns a
    dict ``{(s, h): (m[P], l[P], o[P, D])}`` for valid sequences.
    """
    q = np.asarray(q)
    n_seq, n_heads, _ = q.shape
    kv_heads = k_pool.shape[1]
    group = n_heads // kv_heads
    stats = {}
    for s in (range(n_seq) if seqs is None else seqs):
        table = [int(x) for x in tables[s]]
        length = int(seq_lens[s])
        n_part = -(-length // partition_size)
        for kvh in range(kv_heads):
            keys = to_f64(gather_rows(k_pool, table, length, b, kvh), dtype)
            vals = to_f64(gather_rows(v_pool, table, length, b, kvh), dtype)
            for h in range(kvh * group, (kvh + 1) * group):
                z = scale * (keys @ to_f64(q[s, h], dtype))
                m = np.empty(n_part)
                l = np.empty(n_part)
                o = np.empty((n_part, keys.shape[1]))
                for p in range(n_part):
                    lo, hi = p * partition_size, min(length, (p + 1) * partition_size)
                    m[p] = z[lo:hi].max()
                    w = np.exp(z[lo:hi] - m[p])
                    l[p] = w.sum()
                    o[p] = (w @ vals[lo:hi]) / l[p]
                stats[(s, h)] = (m, l, o)
    return stats


def merge_partitions(m, l, o):
    """Combine per-partition statistics into the full softmax output.

    With M = max_p m_p and weights c_p = exp(m_p - M) * l_p, the full
    result is sum_p c_p o_p / sum_p c_p: each partition's unnormalised sum
    is rescaled to the common maximum, which is exactly the softmax over the
    union of the partitions.
    """
    m = np.asarray(m, dtype=np.float64)
    big = m.max()
    c = np.exp(m - big) * np.asarray(l, dtype=np.float64)
    return (c @ np.asarray(o, dtype=np.float64)) / c.sum()


def attention_bruteforce(q_row, keys, vals, scale):
    """Pure-Python single-query attention using only the ``math`` module.

    Used to pin :func:`attention` on tiny inputs: ``q_row`` is a list of D
    floats, ``keys``/``vals`` lists of L lists of D floats.
    """
    z = [scale * math.fsum(a * c for a, c in zip(q_row, k)) for k in keys]
    top = max(z)
    w = [math.exp(x - top) for x in z]
    tot = math.fsum(w)
    dim = len(vals[0])
    return [math.fsum(w[t] * vals[t][d] for t in range(len(vals))) / tot for d in range(dim)]

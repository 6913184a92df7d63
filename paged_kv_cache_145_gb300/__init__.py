"""GB300-native paged KV cache: decode attention, KV write and block copy.

A thin binding over ``libpagedkv.so`` (C ABI: ``include/pagedkv.h``).  Each
function checks and marshals its tensors (device, dtype, contiguity) and
passes raw pointers and the CUDA stream to the library; every step of the
computation runs in the library's CUDA kernels.  PyTorch supplies device
memory and streams only.  There is no CPU fallback: if the library is not
built, the first call raises.

Cache layout: ``k_cache`` and ``v_cache`` are ``[num_blocks, kv_heads,
block_size, head_dim]`` tensors of one dtype (float32, float16 or bfloat16).
"""

import ctypes

import numpy as np
import torch

from . import _lib
from ._lib import (PKV_DEV_PAIR_RANGE, PKV_DEV_SEQ_LEN, PKV_DEV_SLOT_RANGE,  # noqa: F401
                   PKV_DEV_TABLE_RANGE, PKV_DEV_TIMEOUT, PKV_ERR_NOMEM, PKV_SWAP_IN,
                   PKV_SWAP_OUT)

_DTYPE_CODE = {torch.float32: _lib.PKV_F32, torch.float16: _lib.PKV_F16, torch.bfloat16: _lib.PKV_BF16,
               torch.float8_e4m3fn: _lib.PKV_FP8_E4M3}

__all__ = [
    "PagedKVCache", "BlockManager", "paged_kv_write", "paged_attention_decode",
    "paged_attention_prefill",
    "paged_attention_workspace_bytes", "paged_attention_partition_size",
    "paged_block_copy", "paged_block_swap", "paged_get_device_error",
    "paged_selftest_wait_timeout", "paged_selftest_read_stream", "paged_attention_decode_shared",
    "library_path",
]


def library_path():
    return _lib.LIB_PATH


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype=None, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must have dtype %s, got %s" % (name, dtype, t.dtype))
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the cache on %s" % (name, t.device, device))


class PagedKVCache:
    """The physical pool: two ``[N, Hk, b, D]`` tensors (keys, values).

    FP8 pools (``torch.float8_e4m3fn``) also take ``k_scale`` / ``v_scale``
    (float32 CUDA tensors ``[Hk]``: a key of head h is its code's value times
    ``k_scale[h]``) and ``io_dtype`` (float16 or bfloat16: the type of q, out
    and the new keys/values).  For other pools ``io_dtype`` is the pool's.
    """

    def __init__(self, k_cache, v_cache, k_scale=None, v_scale=None, io_dtype=None):
        _need(k_cache, "k_cache")
        _need(v_cache, "v_cache", k_cache.dtype, k_cache.device)
        if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
            raise ValueError("k_cache and v_cache must both be [N, Hk, b, D]")
        if k_cache.dtype not in _DTYPE_CODE:
            raise ValueError("cache dtype must be float32, float16, bfloat16 or float8_e4m3fn")
        self.k_cache, self.v_cache = k_cache, v_cache
        self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim = k_cache.shape
        self.dtype, self.device = k_cache.dtype, k_cache.device
        self.k_scale = self.v_scale = None
        if self.dtype == torch.float8_e4m3fn:
            if io_dtype not in (torch.float16, torch.bfloat16):
                raise ValueError("an FP8 pool needs io_dtype float16 or bfloat16")
            for t, name in ((k_scale, "k_scale"), (v_scale, "v_scale")):
                _need(t, name, torch.float32, self.device)
                if t.shape != (self.num_kv_heads,):
                    raise ValueError("%s must be [kv_heads]" % name)
            self.k_scale, self.v_scale = k_scale, v_scale
            self.io_dtype = io_dtype
        else:
            self.io_dtype = self.dtype
        self._c = _lib.pkv_cache(k_cache.data_ptr(), v_cache.data_ptr(), self.num_blocks,
                                 self.block_size, self.num_kv_heads, self.head_dim,
                                 _DTYPE_CODE[self.dtype],
                                 self.k_scale.data_ptr() if self.k_scale is not None else None,
                                 self.v_scale.data_ptr() if self.v_scale is not None else None,
                                 _DTYPE_CODE[self.io_dtype])

    @classmethod
    def empty(cls, num_blocks, block_size, num_kv_heads, head_dim, dtype, device="cuda"):
        shape = (num_blocks, num_kv_heads, block_size, head_dim)
        return cls(torch.empty(shape, dtype=dtype, device=device),
                   torch.empty(shape, dtype=dtype, device=device))

    @property
    def ref(self):
        return ctypes.byref(self._c)


def paged_kv_write(cache, k, v, slot_mapping, stream=None):
    """Store ``k``/``v`` ``[T, Hk, D]`` at ``slot_mapping`` (int64 ``[T]``)."""
    _need(k, "k", cache.io_dtype, cache.device)
    _need(v, "v", cache.io_dtype, cache.device)
    _need(slot_mapping, "slot_mapping", torch.int64, cache.device)
    n = slot_mapping.numel()
    if k.shape != (n, cache.num_kv_heads, cache.head_dim) or v.shape != k.shape:
        raise ValueError("k and v must be [num_tokens, kv_heads, head_dim]")
    _lib.check(_lib.lib().paged_kv_write(cache.ref, _ptr(k), _ptr(v), _ptr(slot_mapping), n,
                                         _stream(stream)), "paged_kv_write")


def paged_attention_partition_size(cache, num_seqs, num_heads, max_seq_len, partition_size=0):
    r = _lib.lib().paged_attention_partition_size(cache.ref, num_seqs, num_heads, max_seq_len,
                                                  partition_size)
    if r < 0:
        _lib.check(r, "paged_attention_partition_size")
    return r


def paged_attention_workspace_bytes(cache, num_seqs, num_heads, max_seq_len, partition_size=0):
    return int(_lib.lib().paged_attention_workspace_bytes(cache.ref, num_seqs, num_heads,
                                                          max_seq_len, partition_size))


def paged_attention_decode(cache, q, block_tables, seq_lens, scale, out=None, max_seq_len=0,
                           workspace=None, partition_size=0, stream=None):
    """Decode attention of ``q`` ``[S, H, D]`` through the block tables.

    ``block_tables``: int32 ``[S, max_blocks]``; ``seq_lens``: int32 ``[S]``;
    ``max_seq_len``: host bound on ``seq_lens`` (0 = table width x block
    size).  Allocates ``out`` and the split-K workspace when not given.
    Returns ``out``.
    """
    _need(q, "q", cache.io_dtype, cache.device)
    _need(block_tables, "block_tables", torch.int32, cache.device)
    _need(seq_lens, "seq_lens", torch.int32, cache.device)
    if q.dim() != 3 or q.shape[2] != cache.head_dim:
        raise ValueError("q must be [num_seqs, num_heads, head_dim]")
    num_seqs, num_heads = q.shape[0], q.shape[1]
    if block_tables.dim() != 2 or block_tables.shape[0] != num_seqs or seq_lens.shape != (num_seqs,):
        raise ValueError("block_tables must be [num_seqs, max_blocks] and seq_lens [num_seqs]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", cache.io_dtype, cache.device)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    bound = max_seq_len if max_seq_len else block_tables.shape[1] * cache.block_size
    need = paged_attention_workspace_bytes(cache, num_seqs, num_heads, bound, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=cache.device)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _lib.check(_lib.lib().paged_attention_decode(
        cache.ref, _ptr(q), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), num_seqs,
        num_heads, max_seq_len, float(scale), _ptr(out), ws_ptr, ws_len, partition_size,
        _stream(stream)), "paged_attention_decode")
    return out


def paged_attention_decode_shared(cache, q, block_tables, seq_lens, scale, group_starts,
                                  group_prefix, max_group_size, out=None, max_seq_len=0,
                                  workspace=None, partition_size=0, tail_parts=0, stream=None):
    """Decode attention like :func:`paged_attention_decode` for a batch whose
    groups of consecutive sequences share a table prefix.

    ``group_starts``: int32 ``[num_groups + 1]`` (group g is sequences
    ``group_starts[g] .. group_starts[g+1] - 1``); ``group_prefix``: int32
    ``[num_groups]`` positions shared by every member; ``max_group_size``:
    host bound on group sizes; ``tail_parts``: partitions per sequence that
    the partition pass covers after its group's shared ones (0: all of
    them).  Returns ``out``.
    """
    _need(q, "q", cache.io_dtype, cache.device)
    _need(block_tables, "block_tables", torch.int32, cache.device)
    _need(seq_lens, "seq_lens", torch.int32, cache.device)
    _need(group_starts, "group_starts", torch.int32, cache.device)
    _need(group_prefix, "group_prefix", torch.int32, cache.device)
    if q.dim() != 3 or q.shape[2] != cache.head_dim:
        raise ValueError("q must be [num_seqs, num_heads, head_dim]")
    num_seqs, num_heads = q.shape[0], q.shape[1]
    if block_tables.dim() != 2 or block_tables.shape[0] != num_seqs or seq_lens.shape != (num_seqs,):
        raise ValueError("block_tables must be [num_seqs, max_blocks] and seq_lens [num_seqs]")
    num_groups = group_prefix.numel()
    if group_starts.numel() != num_groups + 1:
        raise ValueError("group_starts must hold num_groups + 1 entries")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", cache.io_dtype, cache.device)
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    bound = max_seq_len if max_seq_len else block_tables.shape[1] * cache.block_size
    need = paged_attention_workspace_bytes(cache, num_seqs, num_heads, bound, partition_size)
    if need and workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=cache.device)
    ws_ptr = _ptr(workspace) if workspace is not None else ctypes.c_void_p(0)
    ws_len = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _lib.check(_lib.lib().paged_attention_decode_shared(
        cache.ref, _ptr(q), _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), num_seqs,
        num_heads, max_seq_len, float(scale), _ptr(out), _ptr(group_starts), _ptr(group_prefix),
        num_groups, int(max_group_size), int(tail_parts), ws_ptr, ws_len, partition_size,
        _stream(stream)),
        "paged_attention_decode_shared")
    return out


def paged_attention_prefill(cache, q, query_starts, block_tables, seq_lens, scale, max_queries,
                            out=None, stream=None):
    """Causal attention of each sequence's chunk of new queries.

    ``q``: ``[total_queries, H, D]``; ``query_starts``: int32 ``[S + 1]``;
    ``block_tables``: int32 ``[S, max_blocks]``; ``seq_lens``: int32 ``[S]``
    (positions including the chunk); ``max_queries``: host bound on any
    chunk's length.  Returns ``out``.
    """
    _need(q, "q", cache.io_dtype, cache.device)
    _need(query_starts, "query_starts", torch.int32, cache.device)
    _need(block_tables, "block_tables", torch.int32, cache.device)
    _need(seq_lens, "seq_lens", torch.int32, cache.device)
    if q.dim() != 3 or q.shape[2] != cache.head_dim:
        raise ValueError("q must be [total_queries, num_heads, head_dim]")
    num_seqs = seq_lens.shape[0]
    if query_starts.shape != (num_seqs + 1,) or block_tables.dim() != 2 or \
            block_tables.shape[0] != num_seqs:
        raise ValueError("query_starts must be [S + 1] and block_tables [S, max_blocks]")
    if out is None:
        out = torch.empty_like(q)
    _need(out, "out", cache.io_dtype, cache.device)
    _lib.check(_lib.lib().paged_attention_prefill(
        cache.ref, _ptr(q), q.shape[0], _ptr(query_starts), num_seqs, int(max_queries),
        _ptr(block_tables), block_tables.shape[1], _ptr(seq_lens), q.shape[1], float(scale),
        _ptr(out), _stream(stream)), "paged_attention_prefill")
    return out


def paged_block_copy(cache, pairs, stream=None):
    """Copy blocks ``pairs[i, 0] -> pairs[i, 1]`` (int64 ``[n, 2]``)."""
    _need(pairs, "pairs", torch.int64, cache.device)
    if pairs.numel() and (pairs.dim() != 2 or pairs.shape[1] != 2):
        raise ValueError("pairs must be [num_pairs, 2]")
    n = pairs.shape[0] if pairs.numel() else 0
    _lib.check(_lib.lib().paged_block_copy(cache.ref, _ptr(pairs), n, _stream(stream)),
               "paged_block_copy")


def paged_block_swap(cache, host_k, host_v, pairs, direction, stream=None):
    """Move blocks between the device pool and a pinned host pool.

    ``host_k``/``host_v``: pinned CPU tensors ``[M, Hk, b, D]`` of the cache
    dtype; ``pairs``: int64 ``[n, 2]`` on the device as (src, dst);
    ``direction``: ``PKV_SWAP_OUT`` (device -> host) or ``PKV_SWAP_IN``.
    """
    for t, name in ((host_k, "host_k"), (host_v, "host_v")):
        if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_pinned():
            raise ValueError("%s must be a pinned CPU tensor" % name)
        if not t.is_contiguous() or t.dtype != cache.dtype:
            raise ValueError("%s must be contiguous with the cache dtype" % name)
        if t.dim() != 4 or tuple(t.shape[1:]) != (cache.num_kv_heads, cache.block_size, cache.head_dim):
            raise ValueError("%s must be [M, kv_heads, block_size, head_dim]" % name)
    if host_k.shape != host_v.shape:
        raise ValueError("host_k and host_v must have one shape")
    _need(pairs, "pairs", torch.int64, cache.device)
    if pairs.numel() and (pairs.dim() != 2 or pairs.shape[1] != 2):
        raise ValueError("pairs must be [num_pairs, 2]")
    n = pairs.shape[0] if pairs.numel() else 0
    _lib.check(_lib.lib().paged_block_swap(cache.ref, _ptr(host_k), _ptr(host_v), host_k.shape[0],
                                           _ptr(pairs), n, int(direction), _stream(stream)),
               "paged_block_swap")


def paged_get_device_error(stream=None):
    """Synchronise the stream; return and clear the device error bits."""
    bits = ctypes.c_uint32(0)
    _lib.check(_lib.lib().paged_get_device_error(_stream(stream), ctypes.byref(bits)),
               "paged_get_device_error")
    return int(bits.value)


def paged_selftest_wait_timeout(limit_ns=10_000_000, stream=None):
    """Run the bounded-wait self-test: a wait that nothing completes gives up
    after ``limit_ns`` and sets PKV_DEV_TIMEOUT (read it with
    :func:`paged_get_device_error`)."""
    _lib.check(_lib.lib().paged_selftest_wait_timeout(int(limit_ns), _stream(stream)),
               "paged_selftest_wait_timeout")


def paged_selftest_read_stream(buf, sink, stream=None):
    """Read every byte of the device tensor ``buf`` once (read-only
    streaming bandwidth); ``sink`` is a device int32 tensor of one element
    that the kernel XOR-updates."""
    if not buf.is_cuda or not buf.is_contiguous():
        raise ValueError("buf must be a contiguous CUDA tensor")
    _need(sink, "sink", torch.int32, buf.device)
    _lib.check(_lib.lib().paged_selftest_read_stream(_ptr(buf), buf.numel() * buf.element_size(),
                                                     _ptr(sink), _stream(stream)),
               "paged_selftest_read_stream")


def _i64(a):
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


class BlockManager:
    """Host block manager (native): tables, slots and copy-on-write pairs."""

    def __init__(self, num_blocks, block_size, free_order=None):
        self._lib = _lib.lib()
        order = None
        if free_order is not None:
            order = _i64(free_order)
            if order.shape != (num_blocks,):
                raise ValueError("free_order must list every block once")
        self._h = self._lib.pkv_bm_create(num_blocks, block_size,
                                          None if order is None else order.ctypes.data)
        if not self._h:
            raise ValueError("bad block manager arguments")
        self.num_blocks, self.block_size = num_blocks, block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pkv_bm_destroy(h)
            self._h = None

    def admit(self, seq, num_tokens):
        rc = self._lib.pkv_bm_admit(self._h, seq, num_tokens)
        if rc == PKV_ERR_NOMEM:
            raise MemoryError("not enough free blocks (or host memory) to admit %d positions"
                              % num_tokens)
        _lib.check(rc, "admit")

    def fork(self, parent, child):
        _lib.check(self._lib.pkv_bm_fork(self._h, parent, child), "fork")

    def append(self, seqs):
        """Append one position to each sequence; returns (slots, pairs)."""
        s = _i64(seqs)
        n = s.shape[0]
        slots = np.empty(n, dtype=np.int64)
        pairs = np.empty((max(n, 1), 2), dtype=np.int64)
        npairs = ctypes.c_int64(0)
        rc = self._lib.pkv_bm_append(self._h, s.ctypes.data, n, slots.ctypes.data,
                                     pairs.ctypes.data, ctypes.byref(npairs))
        if rc == PKV_ERR_NOMEM:
            raise MemoryError("not enough free blocks (or host memory) for this step")
        _lib.check(rc, "append")
        return slots, pairs[: npairs.value].copy()

    def release(self, seq):
        _lib.check(self._lib.pkv_bm_release(self._h, seq), "release")

    def tables(self, seqs, max_blocks):
        s = _i64(seqs)
        tab = np.empty((s.shape[0], max_blocks), dtype=np.int32)
        lens = np.empty(s.shape[0], dtype=np.int32)
        _lib.check(self._lib.pkv_bm_tables(self._h, s.ctypes.data, s.shape[0], max_blocks,
                                           tab.ctypes.data, lens.ctypes.data), "tables")
        return tab, lens

    def slots(self, seq, start, count):
        """Slots of positions ``start .. start+count-1`` of a sequence."""
        out = np.empty(count, dtype=np.int64)
        _lib.check(self._lib.pkv_bm_slots(self._h, seq, start, count, out.ctypes.data), "slots")
        return out

    def num_free(self):
        return int(self._lib.pkv_bm_num_free(self._h))

    def seq_len(self, seq):
        return int(self._lib.pkv_bm_seq_len(self._h, seq))

    def num_seq_blocks(self, seq):
        return int(self._lib.pkv_bm_num_seq_blocks(self._h, seq))

    def refcount(self, block):
        return int(self._lib.pkv_bm_refcount(self._h, block))

    def check(self):
        return self._lib.pkv_bm_check(self._h) == 0

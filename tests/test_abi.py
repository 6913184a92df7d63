"""The C-ABI library loads and exports every declared symbol; host-side
argument checks return their codes without launching anything (no GPU)."""

import ctypes
import os
import re

import pytest

import paged_kv_cache_145_gb300 as pkv
from paged_kv_cache_145_gb300 import _lib

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                      "include", "pagedkv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w \*]*?\b([A-Za-z_]\w*)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "defined")))


@pytest.fixture(scope="module")
def lib():
    return _lib.lib()


def test_header_declares_expected_entry_points():
    names = declared_functions()
    for n in ("paged_kv_write", "paged_attention_decode", "paged_block_copy",
              "paged_attention_workspace_bytes", "paged_get_device_error", "paged_strerror"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _lib.SIGNATURES, name


def test_strerror_covers_codes(lib):
    for code in range(0, -10, -1):
        assert _lib.strerror(code) != "unknown error code"
    assert _lib.strerror(-99) == "unknown error code"


def fake_cache(**kw):
    c = dict(k_cache=0x10000, v_cache=0x20000, num_blocks=32, block_size=16, num_kv_heads=4,
             head_dim=64, dtype=_lib.PKV_F32, k_scale=0x80000, v_scale=0x90000, io_dtype=_lib.PKV_F32)
    c.update(kw)
    return _lib.pkv_cache(**c)


P = ctypes.c_void_p


def write(lib, cache, k=0x30000, v=0x40000, slots=0x50000, n=4):
    return lib.paged_kv_write(ctypes.byref(cache), P(k), P(v), P(slots), n, None)


def decode(lib, cache, heads=4, q=0x30000, out=0x40000, tables=0x50000, lens=0x60000,
           max_blocks=8, max_len=0, part=0, ws=0, ws_bytes=0, scale=0.125, n=4):
    return lib.paged_attention_decode(ctypes.byref(cache), P(q), P(tables), max_blocks, P(lens), n,
                                      heads, max_len, scale, P(out), P(ws), ws_bytes, part, None)


def test_write_argument_errors(lib):
    assert lib.paged_kv_write(None, P(1), P(1), P(1), 1, None) == -1
    assert write(lib, fake_cache(k_cache=0)) == -1
    assert write(lib, fake_cache(dtype=7)) == -3
    # FP8 pools need both scales and a 16-bit io type.
    assert write(lib, fake_cache(dtype=_lib.PKV_FP8_E4M3, io_dtype=_lib.PKV_F32)) == -3
    assert write(lib, fake_cache(dtype=_lib.PKV_FP8_E4M3, io_dtype=_lib.PKV_F16, k_scale=0)) == -1
    assert write(lib, fake_cache(num_blocks=0)) == -3
    assert write(lib, fake_cache(head_dim=3)) == -2        # 12-byte rows
    assert write(lib, fake_cache(k_cache=0x10008)) == -4
    assert write(lib, fake_cache(), k=0x30004) == -4
    assert write(lib, fake_cache(), slots=0x50004) == -4
    assert write(lib, fake_cache(), k=0) == -1
    assert write(lib, fake_cache(), n=-1) == -3
    assert write(lib, fake_cache(), n=0) == 0              # nothing to do


def test_decode_argument_errors(lib):
    c = fake_cache()
    assert decode(lib, c, heads=6) == -2                   # not a multiple of kv heads
    assert decode(lib, c, heads=4 * 3) == -2               # group of 3 unsupported
    assert decode(lib, fake_cache(head_dim=96)) == -2
    assert decode(lib, fake_cache(block_size=4)) == -2
    assert decode(lib, fake_cache(block_size=128)) == -2
    assert decode(lib, c, part=24) == -3                   # not a multiple of b
    assert decode(lib, c, part=16384) == -3
    assert decode(lib, c, part=8192 + 16) == -3           # just past the largest partition
    assert decode(lib, c, max_len=8 * 16 + 1) == -3        # beyond the table
    assert decode(lib, c, scale=float("nan")) == -3
    assert decode(lib, c, q=0x30002) == -4
    assert decode(lib, c, out=0) == -1
    assert decode(lib, c, n=70000) == -3
    assert decode(lib, c, n=0) == 0
    # 8 blocks * 16 = 128 positions > 1 partition of 64: workspace required.
    assert decode(lib, c, part=64) == -5
    need = lib.paged_attention_workspace_bytes(ctypes.byref(c), 4, 4, 128, 64)
    assert decode(lib, c, part=64, ws=0x70000, ws_bytes=need - 1) == -5
    assert decode(lib, c, part=64, ws=0x70004, ws_bytes=need) == -4


def test_block_copy_argument_errors(lib):
    c = fake_cache()
    assert lib.paged_block_copy(ctypes.byref(c), P(0), 3, None) == -1
    assert lib.paged_block_copy(ctypes.byref(c), P(0x50004), 3, None) == -4
    assert lib.paged_block_copy(ctypes.byref(c), P(0x50000), -1, None) == -3
    assert lib.paged_block_copy(ctypes.byref(c), P(0x50000), 0, None) == 0


def test_shared_decode_argument_errors(lib):
    # Group arguments are checked on the host before anything else.
    c = fake_cache()
    args = lambda starts, prefix, ng, mg, tail=0: (ctypes.byref(c), P(0x10000), P(0x20000), 4,
                                                    P(0x30000), 8, 8, 0, ctypes.c_float(0.1),
                                                    P(0x40000), starts, prefix, ng, mg, tail, P(0),
                                                    0, 0, None)
    assert lib.paged_attention_decode_shared(*args(P(0), P(0x50000), 2, 4)) == -1
    assert lib.paged_attention_decode_shared(*args(P(0x60000), P(0), 2, 4)) == -1
    assert lib.paged_attention_decode_shared(*args(P(0x60002), P(0x50000), 2, 4)) == -4
    assert lib.paged_attention_decode_shared(*args(P(0x60000), P(0x50000), -1, 4)) == -3
    assert lib.paged_attention_decode_shared(*args(P(0x60000), P(0x50000), 2, 0)) == -3
    assert lib.paged_attention_decode_shared(*args(P(0x60000), P(0x50000), 2, 9)) == -3
    assert lib.paged_attention_decode_shared(*args(P(0x60000), P(0x50000), 2, 4, -1)) == -3


def test_read_stream_argument_errors(lib):
    # Refused on the host, before any CUDA call: null pointers, a buffer or
    # size that is not a multiple of 16 bytes; an empty buffer launches nothing.
    assert lib.paged_selftest_read_stream(P(0), 64, P(0x60000), None) == -1
    assert lib.paged_selftest_read_stream(P(0x50000), 64, P(0), None) == -1
    assert lib.paged_selftest_read_stream(P(0x50004), 64, P(0x60000), None) == -4
    assert lib.paged_selftest_read_stream(P(0x50000), 40, P(0x60000), None) == -4
    assert lib.paged_selftest_read_stream(P(0x50000), 0, P(0x60000), None) == 0


def test_workspace_and_partition_sizes(lib):
    c = fake_cache(head_dim=128)
    ref = ctypes.byref(c)
    assert lib.paged_attention_partition_size(ref, 4, 4, 100, 0) == 512
    assert lib.paged_attention_partition_size(ref, 4, 4, 100, 48) == 48
    assert lib.paged_attention_partition_size(ref, 4, 4, 100, 40) == -3
    # One partition: no workspace.
    assert lib.paged_attention_workspace_bytes(ref, 4, 8, 512, 0) == 0
    # Three partitions: (m, l) pairs, then outputs from the next 256-byte boundary.
    S, H, D, P_ = 5, 8, 128, 3
    ml = S * H * P_ * 8
    expect = ((ml + 255) // 256) * 256 + S * H * P_ * D * 4
    assert lib.paged_attention_workspace_bytes(ref, S, H, 1100, 512) == expect


def test_binding_rejects_cpu_tensors():
    import torch
    with pytest.raises(ValueError):
        pkv.PagedKVCache(torch.zeros(2, 1, 16, 64), torch.zeros(2, 1, 16, 64))

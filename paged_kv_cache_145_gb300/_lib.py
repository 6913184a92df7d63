"""ctypes declarations of ``libpagedkv.so`` (the C ABI in include/pagedkv.h).

The library is loaded on first use.  If it has not been built, loading fails
loudly: there is no fallback implementation.
"""

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libpagedkv.so")

PKV_F32, PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2, 3

PKV_DEV_SLOT_RANGE = 1
PKV_DEV_TABLE_RANGE = 2
PKV_DEV_SEQ_LEN = 4
PKV_DEV_PAIR_RANGE = 8
PKV_DEV_TIMEOUT = 16
PKV_DEV_SHARING = 32
PKV_DEV_LAUNCH = 64

PKV_ERR_WORKSPACE = -5
PKV_ERR_NOMEM = -8
PKV_STATIC_WS_BYTES = 32 << 20
PKV_SWAP_OUT, PKV_SWAP_IN = 0, 1


class pkv_cache(ctypes.Structure):
    _fields_ = [
        ("k_cache", ctypes.c_void_p),
        ("v_cache", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int64),
        ("block_size", ctypes.c_int32),
        ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("dtype", ctypes.c_int32),
        ("k_scale", ctypes.c_void_p),
        ("v_scale", ctypes.c_void_p),
        ("io_dtype", ctypes.c_int32),
    ]


_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_CACHE = ctypes.POINTER(pkv_cache)

# name -> (restype, argtypes); every symbol the header declares.
SIGNATURES = {
    "paged_kv_write": (ctypes.c_int, [_CACHE, _P, _P, _P, _I64, _P]),
    "paged_attention_partition_size": (_I32, [_CACHE, _I32, _I32, _I32, _I32]),
    "paged_attention_workspace_bytes": (ctypes.c_size_t, [_CACHE, _I32, _I32, _I32, _I32]),
    "paged_attention_decode": (ctypes.c_int, [_CACHE, _P, _P, _I32, _P, _I32, _I32, _I32,
                                              ctypes.c_float, _P, _P, ctypes.c_size_t, _I32, _P]),
    "paged_attention_decode_shared": (ctypes.c_int, [_CACHE, _P, _P, _I32, _P, _I32, _I32, _I32,
                                                     ctypes.c_float, _P, _P, _P, _I32, _I32, _I32,
                                                     _P, ctypes.c_size_t, _I32, _P]),
    "paged_attention_decode_static_ws": (ctypes.c_int, [_CACHE, _P, _P, _I32, _P, _I32, _I32, _I32,
                                                        ctypes.c_float, _P, _I32, _P]),
    "paged_attention_prefill": (ctypes.c_int, [_CACHE, _P, _I64, _P, _I32, _I32, _P, _I32, _P,
                                               _I32, ctypes.c_float, _P, _P]),
    "paged_block_copy": (ctypes.c_int, [_CACHE, _P, _I64, _P]),
    "paged_block_swap": (ctypes.c_int, [_CACHE, _P, _P, _I64, _P, _I64, _I32, _P]),
    "paged_get_device_error": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_uint32)]),
    "paged_selftest_wait_timeout": (ctypes.c_int, [ctypes.c_uint64, _P]),
    "paged_selftest_read_stream": (ctypes.c_int, [_P, ctypes.c_size_t, _P, _P]),
    "paged_strerror": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_bm_create": (_P, [_I64, _I32, _P]),
    "pkv_bm_destroy": (None, [_P]),
    "pkv_bm_admit": (ctypes.c_int, [_P, _I64, _I64]),
    "pkv_bm_fork": (ctypes.c_int, [_P, _I64, _I64]),
    "pkv_bm_append": (ctypes.c_int, [_P, _P, _I64, _P, _P, ctypes.POINTER(_I64)]),
    "pkv_bm_release": (ctypes.c_int, [_P, _I64]),
    "pkv_bm_tables": (ctypes.c_int, [_P, _P, _I64, _I32, _P, _P]),
    "pkv_bm_slots": (ctypes.c_int, [_P, _I64, _I64, _I64, _P]),
    "pkv_bm_num_free": (_I64, [_P]),
    "pkv_bm_seq_len": (_I64, [_P, _I64]),
    "pkv_bm_num_seq_blocks": (_I64, [_P, _I64]),
    "pkv_bm_refcount": (_I32, [_P, _I64]),
    "pkv_bm_check": (ctypes.c_int, [_P]),
}

_lib = None


def lib():
    """The loaded library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                "libpagedkv.so is not built (expected at %s); run "
                "`python -m paged_kv_cache_145_gb300.build`" % LIB_PATH)
        handle = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def strerror(code):
    return lib().paged_strerror(int(code)).decode()


def check(code, what):
    if code != 0:
        raise RuntimeError("%s failed: %s (code %d)" % (what, strerror(code), code))

"""ctypes declarations of libtq.so (the C ABI in include/tq.h).

The library is built in-tree by ``turboquant_compressed_kv_tq_gb300.build``.
Loading fails loudly if it is missing: there is no other implementation to
fall back to.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

TQ_OK = 0
TQ_ERR_INVALID_ARG = 1
TQ_ERR_UNSUPPORTED = 2
TQ_ERR_CONFIG_MISMATCH = 3
TQ_ERR_CAPACITY = 4
TQ_ERR_OOM = 5
TQ_ERR_CUDA = 6
TQ_ERR_DEVICE_BOUNDS = 7

TQ_MODE_MSE = 0
TQ_MODE_PROD = 1
TQ_MODE_GROUP = 2

TQ_F32 = 0
TQ_BF16 = 1
TQ_F16 = 2

TQ_ENCODE_AUTO = 0
TQ_ENCODE_EXACT = 1

TQ_DEVERR_CAPACITY = 1
TQ_DEVERR_BLOCK = 2
TQ_DEVERR_SEQLEN = 4
TQ_DEVERR_TIMEOUT = 8

TQ_NOALLOC_SCRATCH_BYTES = 16 << 20


class TQError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} (status {status})")


class tq_codec_info_t(ctypes.Structure):
    _fields_ = [("head_dim", ctypes.c_int), ("bits", ctypes.c_int), ("mode", ctypes.c_int),
                ("group_size", ctypes.c_int), ("seed", ctypes.c_uint64),
                ("index_bits", ctypes.c_int), ("index_words", ctypes.c_int),
                ("sign_words", ctypes.c_int), ("record_bytes", ctypes.c_int),
                ("device", ctypes.c_int)]


class tq_decode_plan_info(ctypes.Structure):
    _fields_ = [("tensor_cores", ctypes.c_int), ("row_groups", ctypes.c_int), ("splits", ctypes.c_int),
                ("chunk_tokens", ctypes.c_int), ("tile_tokens", ctypes.c_int),
                ("smem_bytes", ctypes.c_size_t), ("workspace_bytes", ctypes.c_size_t),
                ("transposed", ctypes.c_int)]


class tq_cache_desc(ctypes.Structure):
    _fields_ = [("pool", ctypes.c_void_p), ("layer_stride", ctypes.c_int64),
                ("num_layers", ctypes.c_int), ("num_blocks", ctypes.c_int),
                ("block_tokens", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
                ("head_dim", ctypes.c_int), ("key_mode", ctypes.c_int), ("key_bits", ctypes.c_int),
                ("key_seed", ctypes.c_uint64), ("value_mode", ctypes.c_int),
                ("value_bits", ctypes.c_int), ("value_group", ctypes.c_int),
                ("value_seed", ctypes.c_uint64), ("subblock_bytes", ctypes.c_int64),
                ("stream_offset", ctypes.c_int64 * 7), ("encode_policy", ctypes.c_int)]


class tq_batch(ctypes.Structure):
    _fields_ = [("cache", ctypes.POINTER(tq_cache_desc)), ("block_table", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("batch", ctypes.c_int), ("capacity", ctypes.c_int),
                ("max_blocks", ctypes.c_int)]


class tq_split_state(ctypes.Structure):
    _fields_ = [("key_low", ctypes.c_void_p), ("value_low", ctypes.c_void_p), ("key_high", ctypes.c_void_p),
                ("value_high", ctypes.c_void_p), ("low", ctypes.POINTER(tq_cache_desc)),
                ("high", ctypes.POINTER(tq_cache_desc))]


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_ST = ctypes.c_int

SIGNATURES = {
    "tq_abi_version": (_I, []),
    "tq_launch_count": (_U64, []),
    "tq_status_string": (ctypes.c_char_p, [_ST]),
    "tq_codec_create": (_ST, [_I, _I, _I, _U64, ctypes.POINTER(_P)]),
    "tq_codec_create_group": (_ST, [_I, _I, _I, ctypes.POINTER(_P)]),
    "tq_bits_split": (_ST, [ctypes.c_double, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "tq_codec_pair_for_bits": (_ST, [_I, ctypes.c_double, _U64, ctypes.POINTER(_P), ctypes.POINTER(_P)]),
    "tq_codec_destroy": (None, [_P]),
    "tq_codec_info": (_ST, [_P, ctypes.POINTER(tq_codec_info_t)]),
    "tq_codec_build_host": (_ST, [_I, _I, _I, _U64, _P, _P, _P, _P]),
    "tq_codec_export": (_ST, [_P, _P, _P, _P, _P]),
    "tq_cache_desc_init": (_ST, [ctypes.POINTER(tq_cache_desc), _P, _P, _I, _I, _I, _I, _P, _SZ,
                                 ctypes.POINTER(_SZ)]),
    "tq_encode_append": (_ST, [_P, _P, ctypes.POINTER(tq_cache_desc), _I, _P, _P, _I, _I, _I, _P, _P,
                               _I, _P]),
    "tq_quantize": (_ST, [_P, _P, _I, _I64, _P, _P, _P, _P, _P]),
    "tq_decode_workspace_bytes": (_ST, [ctypes.POINTER(tq_cache_desc), _I, _I, _I, _I,
                                        ctypes.POINTER(_SZ)]),
    "tq_decode_attention": (_ST, [_P, _P, ctypes.POINTER(tq_cache_desc), _I, _P, _I, _I, _I, _I, _P,
                                  _P, _I, _I, _F, _P, _P, _SZ, _P]),
    "tq_decode_step": (_ST, [_P, _P, ctypes.POINTER(tq_cache_desc), _I, _P, _P, _I, _I, _P, _I, _I, _I, _I,
                             _P, _P, _I, _I, _F, _P, _P, _SZ, _P]),
    "tq_decode_plan": (_ST, [ctypes.POINTER(tq_cache_desc), _I, _I, _I, _I, _I,
                             ctypes.POINTER(tq_decode_plan_info)]),
    "tq_decode_attention_noalloc": (_ST, [_P, _P, ctypes.POINTER(tq_cache_desc), _I, _P, _I, _I, _I, _I,
                                          _P, _P, _I, _I, _F, _P, _P]),
    "tq_prefill_workspace_bytes": (_ST, [ctypes.POINTER(tq_cache_desc), _I, _I, _I, ctypes.POINTER(_SZ)]),
    "tq_prefill_attention": (_ST, [_P, _P, ctypes.POINTER(tq_cache_desc), _I, _P, _I, _I, _I, _I, _P,
                                   _P, _I, _F, _P, _P, _SZ, _P]),
    "tq_cache_copy_blocks": (_ST, [ctypes.POINTER(tq_cache_desc), ctypes.POINTER(tq_cache_desc), _P, _P, _I, _P]),
    "tq_decode_partials": (_ST, [_P, _P, ctypes.POINTER(tq_cache_desc), _I, _P, _I, _I, _I, _I, _P, _P, _P, _I,
                                 _I, _F, _P, _P, _P, _SZ, _P]),
    "tq_decode_merge": (_ST, [_P, _I, _P, _P, _I64, _P, _P]),
    "tq_encode_append_split": (_ST, [ctypes.POINTER(tq_split_state), _I, _P, _P, _P, _P, _I, _I, _I, _P, _P, _I,
                                     _P]),
    "tq_decode_workspace_bytes_split": (_ST, [ctypes.POINTER(tq_split_state), _I, _I, _I, _I,
                                              ctypes.POINTER(_SZ)]),
    "tq_decode_attention_split": (_ST, [ctypes.POINTER(tq_split_state), _I, _P, _I, _I, _I, _I, _P, _P, _I, _I, _F,
                                        _P, _P, _SZ, _P]),
    "tq_batch_filter": (_ST, [ctypes.POINTER(tq_batch), _P, _I, ctypes.POINTER(tq_batch), _P, _P, _P]),
    "tq_batch_extend": (_ST, [ctypes.POINTER(tq_batch), ctypes.POINTER(tq_batch), _P, _I, _P, _P]),
    "tq_batch_merge": (_ST, [ctypes.POINTER(tq_batch), ctypes.POINTER(tq_batch), _I, _P, _I, _P, _P]),
    "tq_batch_extract": (_ST, [ctypes.POINTER(tq_batch), _I, ctypes.POINTER(tq_batch), _P, _I, _P, _P]),
    "tq_device_error": (_ST, [ctypes.POINTER(ctypes.c_uint32)]),
    "tq_selftest_wait_timeout": (_ST, [ctypes.c_double, _P]),
}

_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libtq.so (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.LIB
            if not os.path.exists(path):
                raise RuntimeError(f"libtq.so is not built ({path}); run "
                                   "`python -c 'import __graft_entry__ as g; g.build()'`")
            L = ctypes.CDLL(path)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(L, name)
                f.restype = res
                f.argtypes = args
            _lib = L
    return _lib


def status_string(status: int) -> str:
    s = lib().tq_status_string(status)
    return s.decode() if s else "?"


def check(status: int, what: str) -> None:
    if status != TQ_OK:
        raise TQError(status, what)

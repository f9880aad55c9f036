"""GB300 TurboQuant compressed KV cache: Python binding of libtq.so.

The functions below carry the names of the C ABI (include/tq.h) and only
marshal arguments: tensors become device pointers, the current torch stream
becomes the cudaStream_t. Every step of encode and decode runs in the
library's CUDA kernels. PyTorch provides device memory and streams.
"""
from __future__ import annotations

import ctypes
from typing import Optional

import numpy as np

from . import _lib
from ._lib import (TQ_BF16, TQ_DEVERR_BLOCK, TQ_DEVERR_CAPACITY, TQ_DEVERR_SEQLEN, TQ_ENCODE_AUTO,
                   TQ_ENCODE_EXACT, TQ_F16, TQ_F32, TQ_MODE_GROUP, TQ_MODE_MSE, TQ_MODE_PROD, TQ_OK, TQError, check,
                   lib, library_path, status_string, tq_batch, tq_cache_desc, tq_codec_info_t, tq_split_state)

__all__ = [
    "tq_codec_create", "tq_codec_create_group", "tq_codec_destroy", "tq_codec_info",
    "tq_bits_split", "tq_codec_pair_for_bits",
    "tq_codec_build_host", "tq_codec_export", "tq_cache_desc_init", "tq_encode_append",
    "tq_quantize", "tq_decode_workspace_bytes", "tq_decode_attention", "tq_decode_attention_noalloc",
    "tq_decode_step", "tq_decode_plan",
    "tq_prefill_workspace_bytes", "tq_prefill_attention", "tq_cache_copy_blocks",
    "tq_decode_partials", "tq_decode_merge",
    "tq_encode_append_split", "tq_decode_workspace_bytes_split", "tq_decode_attention_split", "SplitCache",
    "tq_batch_filter", "tq_batch_extend", "tq_batch_merge", "tq_batch_extract", "Batch",
    "tq_device_error", "tq_selftest_wait_timeout",
    "tq_launch_count", "tq_abi_version", "Codec", "CompressedKVCache", "TQError",
    "TQ_MODE_MSE", "TQ_MODE_PROD", "TQ_MODE_GROUP", "TQ_F32", "TQ_BF16", "TQ_F16",
    "TQ_ENCODE_AUTO", "TQ_ENCODE_EXACT",
]


def _torch():
    import torch
    return torch


def _dtype_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.float32:
        return TQ_F32
    if t.dtype == torch.bfloat16:
        return TQ_BF16
    if t.dtype == torch.float16:
        return TQ_F16
    raise TypeError(f"unsupported dtype {t.dtype}")


def _ptr(t) -> Optional[int]:
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensor must be contiguous")
    return t.data_ptr()


def _stream(stream) -> Optional[int]:
    if stream is None:
        return _torch().cuda.current_stream().cuda_stream
    return stream if isinstance(stream, int) else stream.cuda_stream


# ----------------------------------------------------------------- raw ABI

def tq_abi_version() -> int:
    return lib().tq_abi_version()


def tq_launch_count() -> int:
    return int(lib().tq_launch_count())


def tq_codec_create(head_dim: int, bits: int, mode: int, seed: int) -> int:
    h = ctypes.c_void_p()
    check(lib().tq_codec_create(head_dim, bits, mode, seed, ctypes.byref(h)), "tq_codec_create")
    return h.value


def tq_codec_create_group(head_dim: int, bits: int, group_size: int) -> int:
    h = ctypes.c_void_p()
    check(lib().tq_codec_create_group(head_dim, bits, group_size, ctypes.byref(h)),
          "tq_codec_create_group")
    return h.value


def tq_bits_split(bits: float) -> tuple:
    """(key bits, value bits) of a possibly fractional width: floor/ceil, or b/b."""
    kb, vb = ctypes.c_int(), ctypes.c_int()
    check(lib().tq_bits_split(float(bits), ctypes.byref(kb), ctypes.byref(vb)), "tq_bits_split")
    return kb.value, vb.value


def tq_codec_pair_for_bits(head_dim: int, bits: float, seed: int) -> tuple:
    kh, vh = ctypes.c_void_p(), ctypes.c_void_p()
    check(lib().tq_codec_pair_for_bits(head_dim, float(bits), seed, ctypes.byref(kh), ctypes.byref(vh)),
          "tq_codec_pair_for_bits")
    return kh.value, vh.value


def tq_codec_destroy(handle: int) -> None:
    lib().tq_codec_destroy(handle)


def tq_codec_info(handle: int) -> dict:
    info = tq_codec_info_t()
    check(lib().tq_codec_info(handle, ctypes.byref(info)), "tq_codec_info")
    return {k: getattr(info, k) for k, _ in info._fields_}


def _tables(D: int, ib: int, with_s: bool):
    R = np.empty((D, D), np.float32)
    S = np.empty((D, D), np.float32) if with_s else None
    c = np.empty(1 << ib, np.float32)
    m = np.empty((1 << ib) - 1, np.float32)
    return R, S, c, m


def _np_ptr(a):
    return None if a is None else a.ctypes.data


def tq_codec_build_host(head_dim: int, bits: int, mode: int, seed: int):
    ib = bits - 1 if mode == TQ_MODE_PROD else bits
    R, S, c, m = _tables(head_dim, ib, mode == TQ_MODE_PROD)
    check(lib().tq_codec_build_host(head_dim, bits, mode, seed, _np_ptr(R), _np_ptr(S), _np_ptr(c),
                                    _np_ptr(m)), "tq_codec_build_host")
    return R, S, c, m


def tq_codec_export(handle: int):
    info = tq_codec_info(handle)
    R, S, c, m = _tables(info["head_dim"], info["index_bits"], info["mode"] == TQ_MODE_PROD)
    check(lib().tq_codec_export(handle, _np_ptr(R), _np_ptr(S), _np_ptr(c), _np_ptr(m)),
          "tq_codec_export")
    return R, S, c, m


def tq_cache_desc_init(key_codec: int, value_codec: int, num_layers: int, num_blocks: int,
                       block_tokens: int, num_kv_heads: int, pool=None):
    """Returns (desc, required_bytes). ``pool`` is a device tensor or None."""
    d = tq_cache_desc()
    req = ctypes.c_size_t()
    ptr = None if pool is None else pool.data_ptr()
    nbytes = 0 if pool is None else pool.numel() * pool.element_size()
    check(lib().tq_cache_desc_init(ctypes.byref(d), key_codec, value_codec, num_layers, num_blocks,
                                   block_tokens, num_kv_heads, ptr, nbytes, ctypes.byref(req)),
          "tq_cache_desc_init")
    return d, req.value


def tq_encode_append(key_codec: int, value_codec: int, desc: tq_cache_desc, layer: int, k, v,
                     seq_lens, block_table=None, max_blocks: int = 0, stream=None) -> None:
    batch, _, n_new, _ = k.shape
    check(lib().tq_encode_append(key_codec, value_codec, ctypes.byref(desc), layer, _ptr(k), _ptr(v),
                                 _dtype_code(k), batch, n_new, _ptr(seq_lens), _ptr(block_table),
                                 max_blocks, _stream(stream)), "tq_encode_append")


def tq_quantize(codec: int, x, idx, aux0=None, aux1=None, aux2=None, stream=None) -> None:
    n = x.shape[0]
    check(lib().tq_quantize(codec, _ptr(x), _dtype_code(x), n, _ptr(idx), _ptr(aux0), _ptr(aux1),
                            _ptr(aux2), _stream(stream)), "tq_quantize")


def tq_decode_workspace_bytes(desc: tq_cache_desc, batch: int, num_q_heads: int, q_len: int,
                              max_seq_len: int) -> int:
    out = ctypes.c_size_t()
    check(lib().tq_decode_workspace_bytes(ctypes.byref(desc), batch, num_q_heads, q_len, max_seq_len,
                                          ctypes.byref(out)), "tq_decode_workspace_bytes")
    return out.value


def tq_decode_attention(key_codec: int, value_codec: int, desc: tq_cache_desc, layer: int, q,
                        seq_lens, block_table, max_blocks: int, max_seq_len: int, out, workspace,
                        scale: float = 0.0, stream=None) -> None:
    batch, hq, lq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    check(lib().tq_decode_attention(key_codec, value_codec, ctypes.byref(desc), layer, _ptr(q),
                                    _dtype_code(q), batch, hq, lq, _ptr(seq_lens), _ptr(block_table),
                                    max_blocks, max_seq_len, scale, _ptr(out), _ptr(workspace),
                                    ws_bytes, _stream(stream)), "tq_decode_attention")


def tq_decode_plan(desc: tq_cache_desc, batch: int, num_q_heads: int, q_len: int, max_seq_len: int,
                   num_sms: int) -> dict:
    """The launch shape tq_decode_attention would use (host arithmetic; see include/tq.h)."""
    info = _lib.tq_decode_plan_info()
    check(lib().tq_decode_plan(ctypes.byref(desc), batch, num_q_heads, q_len, max_seq_len, num_sms,
                               ctypes.byref(info)), "tq_decode_plan")
    return {f: getattr(info, f) for f, _ in info._fields_}


def tq_decode_step(key_codec: int, value_codec: int, desc: tq_cache_desc, layer: int, k_new, v_new, q,
                   seq_lens, block_table, max_blocks: int, max_seq_len: int, out, workspace,
                   scale: float = 0.0, stream=None) -> None:
    """Append k_new / v_new [batch][kv heads][n_new][D] at seq_lens (the lengths before the step) and
    decode q over the grown sequences, in one call (see include/tq.h)."""
    batch, hq, lq, _ = q.shape
    n_new = k_new.shape[2]
    ws_bytes = workspace.numel() * workspace.element_size()
    check(lib().tq_decode_step(key_codec, value_codec, ctypes.byref(desc), layer, _ptr(k_new), _ptr(v_new),
                               _dtype_code(k_new), n_new, _ptr(q), _dtype_code(q), batch, hq, lq,
                               _ptr(seq_lens), _ptr(block_table), max_blocks, max_seq_len, scale, _ptr(out),
                               _ptr(workspace), ws_bytes, _stream(stream)), "tq_decode_step")


def tq_cache_copy_blocks(src: tq_cache_desc, dst: tq_cache_desc, src_blocks, dst_blocks, stream=None) -> None:
    n = src_blocks.numel()
    assert dst_blocks.numel() == n
    check(lib().tq_cache_copy_blocks(ctypes.byref(src), ctypes.byref(dst), _ptr(src_blocks), _ptr(dst_blocks), n,
                                     _stream(stream)), "tq_cache_copy_blocks")


def tq_prefill_workspace_bytes(desc: tq_cache_desc, batch: int, num_q_heads: int, q_len: int) -> int:
    out = ctypes.c_size_t()
    check(lib().tq_prefill_workspace_bytes(ctypes.byref(desc), batch, num_q_heads, q_len, ctypes.byref(out)),
          "tq_prefill_workspace_bytes")
    return out.value


def tq_prefill_attention(key_codec: int, value_codec: int, desc: tq_cache_desc, layer: int, q,
                         seq_lens, block_table, max_blocks: int, out, workspace, scale: float = 0.0,
                         stream=None) -> None:
    batch, hq, lq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    check(lib().tq_prefill_attention(key_codec, value_codec, ctypes.byref(desc), layer, _ptr(q),
                                     _dtype_code(q), batch, hq, lq, _ptr(seq_lens), _ptr(block_table),
                                     max_blocks, scale, _ptr(out), _ptr(workspace), ws_bytes,
                                     _stream(stream)), "tq_prefill_attention")


def tq_decode_attention_noalloc(key_codec: int, value_codec: int, desc: tq_cache_desc, layer: int, q,
                                seq_lens, block_table, max_blocks: int, max_seq_len: int, out,
                                scale: float = 0.0, stream=None) -> None:
    """tq_decode_attention with its scratch in the library's fixed device array
    (for callers that cannot allocate device memory); see include/tq.h."""
    batch, hq, lq, _ = q.shape
    check(lib().tq_decode_attention_noalloc(key_codec, value_codec, ctypes.byref(desc), layer, _ptr(q),
                                            _dtype_code(q), batch, hq, lq, _ptr(seq_lens),
                                            _ptr(block_table), max_blocks, max_seq_len, scale, _ptr(out),
                                            _stream(stream)), "tq_decode_attention_noalloc")


def tq_decode_partials(key_codec: int, value_codec: int, desc: tq_cache_desc, layer: int, q, seq_lens,
                       causal_end, block_table, max_blocks: int, max_seq_len: int, part_ml, part_acc, workspace,
                       scale: float = 0.0, stream=None) -> None:
    """Unnormalised softmax state of this shard of every sequence (see include/tq.h)."""
    batch, hq, lq, _ = q.shape
    ws_bytes = workspace.numel() * workspace.element_size()
    check(lib().tq_decode_partials(key_codec, value_codec, ctypes.byref(desc), layer, _ptr(q), _dtype_code(q),
                                   batch, hq, lq, _ptr(seq_lens), _ptr(causal_end), _ptr(block_table), max_blocks,
                                   max_seq_len, scale, _ptr(part_ml), _ptr(part_acc), _ptr(workspace), ws_bytes,
                                   _stream(stream)), "tq_decode_partials")


def tq_decode_merge(value_codec: int, parts_ml, parts_acc, out, stream=None) -> None:
    """Log-sum-exp merge of shards' states: parts_ml [P, ..., 2], parts_acc [P, ..., D] -> out [..., D]."""
    P = parts_ml.shape[0]
    rows = parts_ml[0].numel() // 2
    check(lib().tq_decode_merge(value_codec, P, _ptr(parts_ml), _ptr(parts_acc), rows, _ptr(out),
                                _stream(stream)), "tq_decode_merge")


class SplitCache:
    """Split (low/high) states: the low coordinates [0, DL) of every key and value
    in one cache, the high coordinates [DL, D) in another, each under its own
    codec pair; both caches share one block layout."""

    def __init__(self, key_low: "Codec", value_low: "Codec", key_high: "Codec", value_high: "Codec",
                 num_layers: int, num_blocks: int, block_tokens: int, num_kv_heads: int, device="cuda",
                 exact_encode: bool = False):
        self.low = CompressedKVCache(key_low, value_low, num_layers, num_blocks, block_tokens, num_kv_heads,
                                     device, exact_encode)
        self.high = CompressedKVCache(key_high, value_high, num_layers, num_blocks, block_tokens, num_kv_heads,
                                      device, exact_encode)
        self.low_dim = key_low.info["head_dim"]
        self.head_dim = self.low_dim + key_high.info["head_dim"]

    def state(self) -> tq_split_state:
        return tq_split_state(self.low.key.handle, self.low.value.handle, self.high.key.handle,
                              self.high.value.handle, ctypes.pointer(self.low.desc), ctypes.pointer(self.high.desc))

    def append(self, layer, k_low, v_low, k_high, v_high, seq_lens, block_table=None, max_blocks=0, stream=None):
        tq_encode_append_split(self, layer, k_low, v_low, k_high, v_high, seq_lens, block_table, max_blocks, stream)

    def workspace_bytes(self, batch, num_q_heads, q_len, max_seq_len):
        return tq_decode_workspace_bytes_split(self, batch, num_q_heads, q_len, max_seq_len)

    def decode(self, layer, q, seq_lens, block_table, max_blocks, max_seq_len, out, workspace, scale=0.0,
               stream=None):
        tq_decode_attention_split(self, layer, q, seq_lens, block_table, max_blocks, max_seq_len, out, workspace,
                                  scale, stream)


def tq_encode_append_split(sc: SplitCache, layer: int, k_low, v_low, k_high, v_high, seq_lens, block_table=None,
                           max_blocks: int = 0, stream=None) -> None:
    batch, _, n_new, _ = k_low.shape
    st = sc.state()
    check(lib().tq_encode_append_split(ctypes.byref(st), layer, _ptr(k_low), _ptr(v_low), _ptr(k_high),
                                       _ptr(v_high), _dtype_code(k_low), batch, n_new, _ptr(seq_lens),
                                       _ptr(block_table), max_blocks, _stream(stream)), "tq_encode_append_split")


def tq_decode_workspace_bytes_split(sc: SplitCache, batch: int, num_q_heads: int, q_len: int, max_seq_len: int) -> int:
    out = ctypes.c_size_t()
    st = sc.state()
    check(lib().tq_decode_workspace_bytes_split(ctypes.byref(st), batch, num_q_heads, q_len, max_seq_len,
                                                ctypes.byref(out)), "tq_decode_workspace_bytes_split")
    return out.value


def tq_decode_attention_split(sc: SplitCache, layer: int, q, seq_lens, block_table, max_blocks: int,
                              max_seq_len: int, out, workspace, scale: float = 0.0, stream=None) -> None:
    batch, hq, lq, _ = q.shape
    st = sc.state()
    ws_bytes = workspace.numel() * workspace.element_size()
    check(lib().tq_decode_attention_split(ctypes.byref(st), layer, _ptr(q), _dtype_code(q), batch, hq, lq,
                                          _ptr(seq_lens), _ptr(block_table), max_blocks, max_seq_len, scale,
                                          _ptr(out), _ptr(workspace), ws_bytes, _stream(stream)),
          "tq_decode_attention_split")


class Batch:
    """A batch of sequences in a paged cache: device block table [capacity][max_blocks]
    (-1 = no block) and sequence lengths [capacity], rows 0..batch-1 in use."""

    def __init__(self, cache: "CompressedKVCache", capacity: int, max_blocks: int, table=None, lens=None,
                 batch: int = 0):
        torch = _torch()
        dev = cache.pool.device
        self.cache = cache
        self.table = table if table is not None else torch.full((capacity, max_blocks), -1, dtype=torch.int32,
                                                                 device=dev)
        self.lens = lens if lens is not None else torch.zeros(capacity, dtype=torch.int32, device=dev)
        self.batch = batch
        assert self.table.shape == (capacity, max_blocks) and self.lens.shape == (capacity,)

    @property
    def capacity(self) -> int:
        return self.table.shape[0]

    @property
    def max_blocks(self) -> int:
        return self.table.shape[1]

    def view(self) -> tq_batch:
        return tq_batch(ctypes.pointer(self.cache.desc), _ptr(self.table), _ptr(self.lens), self.batch,
                        self.capacity, self.max_blocks)


def tq_batch_filter(batch: Batch, keep, out: Batch, freed, n_freed, stream=None) -> None:
    """Rows `keep` (host list) of `batch` become rows 0.. of `out` (same pool); the block ids of the
    other rows go to `freed` (device int32) and their count to n_freed (device int32 [1])."""
    keep_arr = (ctypes.c_int32 * max(1, len(keep)))(*[int(i) for i in keep])
    src, dst = batch.view(), out.view()
    check(lib().tq_batch_filter(ctypes.byref(src), keep_arr, len(keep), ctypes.byref(dst), _ptr(freed),
                                _ptr(n_freed), _stream(stream)), "tq_batch_filter")
    out.batch = dst.batch


def tq_batch_extend(dst: Batch, src: Batch, free_blocks=None, n_used=None, stream=None) -> None:
    """Append the sequences of `src` to `dst`, copying their blocks into dst's free blocks
    (free_blocks device int32, consumed from n_used[0]) unless both share a pool."""
    d, s_ = dst.view(), src.view()
    n_free = 0 if free_blocks is None else free_blocks.numel()
    check(lib().tq_batch_extend(ctypes.byref(d), ctypes.byref(s_), _ptr(free_blocks), n_free, _ptr(n_used),
                                _stream(stream)), "tq_batch_extend")
    dst.batch = d.batch


def tq_batch_merge(dst: Batch, srcs, free_blocks=None, n_used=None, stream=None) -> None:
    """tq_batch_extend of `dst` by each of `srcs` in order (one guard over all of them first)."""
    d = dst.view()
    arr = (tq_batch * max(1, len(srcs)))(*[b.view() for b in srcs])
    n_free = 0 if free_blocks is None else free_blocks.numel()
    check(lib().tq_batch_merge(ctypes.byref(d), arr, len(srcs), _ptr(free_blocks), n_free, _ptr(n_used),
                               _stream(stream)), "tq_batch_merge")
    dst.batch = d.batch


def tq_batch_extract(src: Batch, idx: int, dst: Batch, free_blocks=None, n_used=None, stream=None) -> None:
    """Sequence idx of `src` becomes the only sequence of `dst`."""
    s_, d = src.view(), dst.view()
    n_free = 0 if free_blocks is None else free_blocks.numel()
    check(lib().tq_batch_extract(ctypes.byref(s_), idx, ctypes.byref(d), _ptr(free_blocks), n_free,
                                 _ptr(n_used), _stream(stream)), "tq_batch_extract")
    dst.batch = d.batch


def tq_device_error() -> int:
    flags = ctypes.c_uint32()
    st = lib().tq_device_error(ctypes.byref(flags))
    if st not in (TQ_OK, 7):
        check(st, "tq_device_error")
    return flags.value


def tq_selftest_wait_timeout(seconds: float, stream=None) -> None:
    check(lib().tq_selftest_wait_timeout(float(seconds), _stream(stream)), "tq_selftest_wait_timeout")


# ----------------------------------------------------------------- helpers

class Codec:
    """Owns one codec handle."""

    def __init__(self, head_dim: int, bits: int, mode: int, seed: int = 0, group: int = 0,
                 _handle: int = 0):
        if _handle:
            self.handle = _handle
        elif mode == TQ_MODE_GROUP:
            self.handle = tq_codec_create_group(head_dim, bits, group)
        else:
            self.handle = tq_codec_create(head_dim, bits, mode, seed)
        self.info = tq_codec_info(self.handle)

    @classmethod
    def pair_for_bits(cls, head_dim: int, bits: float, seed: int = 0) -> tuple:
        """(key codec, value codec) for a possibly fractional bit width: MSE
        codecs of floor(bits) and ceil(bits) bits, seeds seed and seed + 1."""
        kh, vh = tq_codec_pair_for_bits(head_dim, bits, seed)
        return cls(0, 0, 0, _handle=kh), cls(0, 0, 0, _handle=vh)

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            try:
                tq_codec_destroy(h)
            except Exception:
                pass
            self.handle = None

    @property
    def record_bytes(self) -> int:
        return self.info["record_bytes"]

    def export(self):
        return tq_codec_export(self.handle)


class CompressedKVCache:
    """A device pool plus its descriptor (all layers), allocated through torch."""

    def __init__(self, key: Codec, value: Codec, num_layers: int, num_blocks: int,
                 block_tokens: int, num_kv_heads: int, device="cuda", exact_encode: bool = False):
        torch = _torch()
        self.key, self.value = key, value
        _, req = tq_cache_desc_init(key.handle, value.handle, num_layers, num_blocks, block_tokens,
                                    num_kv_heads, None)
        self.pool = torch.zeros(req, dtype=torch.uint8, device=device)
        self.desc, _ = tq_cache_desc_init(key.handle, value.handle, num_layers, num_blocks,
                                          block_tokens, num_kv_heads, self.pool)
        # TQ_ENCODE_EXACT: every append in the sequential fp32 order; AUTO lets
        # long appends rotate on the tensor cores
        self.desc.encode_policy = TQ_ENCODE_EXACT if exact_encode else TQ_ENCODE_AUTO
        self.num_layers, self.num_blocks = num_layers, num_blocks
        self.block_tokens, self.num_kv_heads = block_tokens, num_kv_heads

    @property
    def nbytes(self) -> int:
        return self.pool.numel()

    def append(self, layer, k, v, seq_lens, block_table=None, max_blocks=0, stream=None):
        tq_encode_append(self.key.handle, self.value.handle, self.desc, layer, k, v, seq_lens,
                         block_table, max_blocks, stream)

    def workspace_bytes(self, batch, num_q_heads, q_len, max_seq_len):
        return tq_decode_workspace_bytes(self.desc, batch, num_q_heads, q_len, max_seq_len)

    def copy_blocks_from(self, src: "CompressedKVCache", src_blocks, dst_blocks, stream=None):
        """Blocks src_blocks of `src` (every layer) become blocks dst_blocks of this cache."""
        tq_cache_copy_blocks(src.desc, self.desc, src_blocks, dst_blocks, stream)

    def prefill_workspace_bytes(self, batch, num_q_heads, q_len):
        return tq_prefill_workspace_bytes(self.desc, batch, num_q_heads, q_len)

    def prefill_attention(self, layer, q, seq_lens, block_table, max_blocks, out, workspace, scale=0.0,
                          stream=None):
        tq_prefill_attention(self.key.handle, self.value.handle, self.desc, layer, q, seq_lens, block_table,
                             max_blocks, out, workspace, scale, stream)

    def decode(self, layer, q, seq_lens, block_table, max_blocks, max_seq_len, out, workspace,
               scale=0.0, stream=None):
        tq_decode_attention(self.key.handle, self.value.handle, self.desc, layer, q, seq_lens,
                            block_table, max_blocks, max_seq_len, out, workspace, scale, stream)

    def decode_partials(self, layer, q, seq_lens, causal_end, block_table, max_blocks, max_seq_len, part_ml,
                        part_acc, workspace, scale=0.0, stream=None):
        """This cache holds one shard of each sequence: its unnormalised softmax state."""
        tq_decode_partials(self.key.handle, self.value.handle, self.desc, layer, q, seq_lens, causal_end,
                           block_table, max_blocks, max_seq_len, part_ml, part_acc, workspace, scale, stream)

    def decode_step(self, layer, k_new, v_new, q, seq_lens, block_table, max_blocks, max_seq_len, out,
                    workspace, scale=0.0, stream=None):
        """Append the step's tokens at seq_lens (lengths before the step) and decode, in one call."""
        tq_decode_step(self.key.handle, self.value.handle, self.desc, layer, k_new, v_new, q, seq_lens,
                       block_table, max_blocks, max_seq_len, out, workspace, scale, stream)

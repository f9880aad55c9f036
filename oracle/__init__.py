"""ctypes binding of the plain-C TurboQuant oracle (``tq_oracle.c``).

TEST INFRASTRUCTURE. Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference arm may import this package. The product
package never imports it.

Every function here only marshals numpy arrays into the C oracle; all of the
arithmetic is in ``tq_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "tq_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libtq_oracle.so")
_lock = threading.Lock()
_lib = None

MSE, PROD, GROUP = 0, 1, 2


def compile_source(src: str, out: str) -> str:
    """Compile one oracle source file into the shared library ``out`` (no FMA
    contraction, OpenMP); the include directory is this package's."""
    tmp = out + f".tmp{os.getpid()}"
    subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-std=c11", "-ffp-contract=off",
                           "-fopenmp", "-Wall", "-I", _HERE, src, "-o", tmp, "-lm"])
    os.replace(tmp, out)
    return out


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
            os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "tq_oracle.h"))):
        compile_source(_SRC, _SO)
    return _SO


def lib():
    """The loaded oracle. ``TQO_LIBRARY`` names another compiled copy of it to
    load instead (the planted-mistake tests point it at a mutant)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(os.environ.get("TQO_LIBRARY") or build()))
    return _lib


_P = ctypes.c_void_p
_I = ctypes.c_int
_I64 = ctypes.c_int64
_U64 = ctypes.c_uint64
_D = ctypes.c_double


def _declare(L):
    sig = {
        "tqo_splitmix64_at": (_U64, [_U64, _U64]),
        "tqo_normals": (None, [_U64, _I, _I64, _P]),
        "tqo_rotation_f64": (_I, [_I, _U64, _P]),
        "tqo_qjl_f64": (_I, [_I, _U64, _P]),
        "tqo_lloyd_max": (_I, [_I, _I, _P, _P]),
        "tqo_codec_tables": (_I, [_I, _I, _I, _U64, _P, _P, _P, _P]),
        "tqo_index_bits": (_I, [_I, _I]),
        "tqo_packed_words": (_I, [_I, _I]),
        "tqo_record_bytes": (_I, [_I, _I, _I, _I]),
        "tqo_bits_split": (None, [_D, ctypes.POINTER(_I), ctypes.POINTER(_I)]),
        "tqo_pack": (None, [_P, _I, _I, _P]),
        "tqo_unpack": (None, [_P, _I, _I, _P]),
        "tqo_f32_to_f16": (ctypes.c_uint16, [ctypes.c_float]),
        "tqo_f16_to_f32": (ctypes.c_float, [ctypes.c_uint16]),
        "tqo_encode_mse": (None, [_I64, _I, _P, _P, _P, _I, _P, _P]),
        "tqo_encode_prod": (None, [_I64, _I, _P, _P, _P, _P, _P, _I, _P, _P, _P, _P]),
        "tqo_encode_group": (None, [_I64, _I, _P, _I, _I, _P, _P, _P]),
        "tqo_dequant_mse": (None, [_I64, _I, _P, _P, _P, _P, _I, _P]),
        "tqo_dequant_prod": (None, [_I64, _I, _P, _P, _P, _P, _P, _P, _P, _I, _P]),
        "tqo_dequant_group": (None, [_I64, _I, _P, _P, _P, _I, _I, _P]),
        "tqo_attention_f64": (None, [_I, _I64, _I, _I, _P, _P, _P, _D, _P]),
        "tqo_decode_rotated": (None, [_I, _I64, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                      _I, _I, _I, _P, _P, _P, _P, _P, _P, _D, _P]),
        "tqo_decode_partial": (None, [_I, _I64, _I64, _I, _I, _P, _I, _I, _P, _P, _P, _P, _P, _P, _P,
                                      _I, _I, _I, _P, _P, _P, _P, _P, _D, _P, _P, _P]),
        "tqo_merge_partials": (None, [_I, _I, _I64, _P, _P, _P, _I, _P, _P]),
        "tqo_subblock_layout": (_I64, [_I, _I, _I, _I, _I, _I, _I, _P]),
        "tqo_pool_write": (None, [_P, _I, _I, _I, _P, _I, _I, _I, _I64, _I64, _I, _I, _I, _I, _I,
                                  _P, _P, _P, _P, _P, _P, _P, _P]),
        "tqo_num_threads": (_I, []),
        "tqo_set_num_threads": (None, [_I]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------- codec tables

def index_bits(bits: int, mode: int) -> int:
    return lib().tqo_index_bits(bits, mode)


def packed_words(D: int, ib: int) -> int:
    return lib().tqo_packed_words(D, ib)


def record_bytes(D: int, bits: int, mode: int, group: int = 0) -> int:
    return lib().tqo_record_bytes(D, bits, mode, group)


def bits_split(bits: float) -> tuple:
    kb, vb = ctypes.c_int(), ctypes.c_int()
    lib().tqo_bits_split(float(bits), ctypes.byref(kb), ctypes.byref(vb))
    return kb.value, vb.value


def normals(seed: int, stream: int, n: int) -> np.ndarray:
    out = np.empty(n, np.float64)
    lib().tqo_normals(seed, stream, n, _p(out))
    return out


def rotation_f64(D: int, seed: int) -> np.ndarray:
    out = np.empty((D, D), np.float64)
    assert lib().tqo_rotation_f64(D, seed, _p(out)) == 0
    return out


def qjl_f64(D: int, seed: int) -> np.ndarray:
    out = np.empty((D, D), np.float64)
    lib().tqo_qjl_f64(D, seed, _p(out))
    return out


def lloyd_max(D: int, b: int):
    L = 1 << b
    c = np.empty(L, np.float64)
    m = np.empty(L - 1, np.float64)
    it = lib().tqo_lloyd_max(D, b, _p(c), _p(m))
    assert it >= 0
    return c, m, it


class Codec:
    """fp32 codec tables as the oracle builds them."""

    def __init__(self, D: int, bits: int, mode: int, seed: int = 0, group: int = 0):
        self.D, self.bits, self.mode, self.seed, self.group = D, bits, mode, seed, group
        self.ib = index_bits(bits, mode)
        self.W = packed_words(D, self.ib)
        self.R = self.S = self.c = self.m = None
        if mode != GROUP:
            L = 1 << self.ib
            self.R = np.empty((D, D), np.float32)
            self.S = np.empty((D, D), np.float32) if mode == PROD else None
            self.c = np.empty(L, np.float32)
            self.m = np.empty(L - 1, np.float32)
            rc = lib().tqo_codec_tables(D, bits, mode, seed, _p(self.R), _p(self.S),
                                        _p(self.c), _p(self.m))
            assert rc == 0

    @property
    def record_bytes(self) -> int:
        return record_bytes(self.D, self.bits, self.mode, self.group)

    def encode(self, x: np.ndarray) -> dict:
        """x: [n, D] float32 -> record dict (numpy arrays)."""
        x = _c(x, np.float32).reshape(-1, self.D)
        n = x.shape[0]
        L = lib()
        if self.mode == MSE:
            idx = np.empty((n, self.W), np.uint32)
            norm = np.empty(n, np.float32)
            L.tqo_encode_mse(n, self.D, _p(x), _p(self.R), _p(self.m), self.ib, _p(idx), _p(norm))
            return {"idx": idx, "norm": norm}
        if self.mode == PROD:
            idx = np.empty((n, self.W), np.uint32)
            sgn = np.empty((n, self.D // 32), np.uint32)
            norm = np.empty(n, np.float32)
            rn = np.empty(n, np.float32)
            L.tqo_encode_prod(n, self.D, _p(x), _p(self.R), _p(self.S), _p(self.c), _p(self.m),
                              self.bits, _p(idx), _p(sgn), _p(norm), _p(rn))
            return {"idx": idx, "sgn": sgn, "norm": norm, "rnorm": rn}
        ng = self.D // self.group
        data = np.empty((n, self.W), np.uint32)
        sc = np.empty((n, ng), np.uint16)
        mn = np.empty((n, ng), np.uint16)
        L.tqo_encode_group(n, self.D, _p(x), self.bits, self.group, _p(data), _p(sc), _p(mn))
        return {"idx": data, "scale": sc, "min": mn}

    def dequant(self, rec: dict) -> np.ndarray:
        n = rec["idx"].shape[0]
        out = np.empty((n, self.D), np.float64)
        L = lib()
        if self.mode == MSE:
            L.tqo_dequant_mse(n, self.D, _p(rec["idx"]), _p(rec["norm"]), _p(self.R), _p(self.c),
                              self.ib, _p(out))
        elif self.mode == PROD:
            L.tqo_dequant_prod(n, self.D, _p(rec["idx"]), _p(rec["sgn"]), _p(rec["norm"]),
                               _p(rec["rnorm"]), _p(self.R), _p(self.S), _p(self.c), self.bits,
                               _p(out))
        else:
            L.tqo_dequant_group(n, self.D, _p(rec["idx"]), _p(rec["scale"]), _p(rec["min"]),
                                self.bits, self.group, _p(out))
        return out


def pack(codes: np.ndarray, D: int, b: int) -> np.ndarray:
    codes = _c(codes, np.uint8)
    out = np.empty(packed_words(D, b), np.uint32)
    lib().tqo_pack(_p(codes), D, b, _p(out))
    return out


def unpack(words: np.ndarray, D: int, b: int) -> np.ndarray:
    words = _c(words, np.uint32)
    out = np.empty(D, np.uint8)
    lib().tqo_unpack(_p(words), D, b, _p(out))
    return out


def f32_to_f16_bits(x: float) -> int:
    return int(lib().tqo_f32_to_f16(ctypes.c_float(x)))


def f16_bits_to_f32(h: int) -> float:
    return float(lib().tqo_f16_to_f32(ctypes.c_uint16(h)))


def attention_f64(q: np.ndarray, K: np.ndarray, V: np.ndarray, scale: float, Lq: int) -> np.ndarray:
    """q: [G, Lq, D]; K, V: [N, D] -> out [G, Lq, D] (fp64)."""
    q = _c(q, np.float64)
    K = _c(K, np.float64)
    V = _c(V, np.float64)
    G, _, D = q.shape
    N = K.shape[0]
    out = np.empty((G, Lq, D), np.float64)
    lib().tqo_attention_f64(D, N, G, Lq, _p(q), _p(K), _p(V), scale, _p(out))
    return out


def decode_rotated(q: np.ndarray, kc: Codec, krec: dict, vc: Codec, vrec: dict,
                   scale: float, Lq: int) -> np.ndarray:
    """Rotated-domain decode from records. q: [G, Lq, D] -> [G, Lq, D] fp64."""
    q = _c(q, np.float64)
    G, _, D = q.shape
    N = krec["idx"].shape[0]
    out = np.empty((G, Lq, D), np.float64)
    lib().tqo_decode_rotated(
        D, N, G, Lq, _p(q), kc.mode, kc.bits, _p(krec["idx"]), _p(krec.get("sgn")),
        _p(krec["norm"]), _p(krec.get("rnorm")), _p(kc.R), _p(kc.S), _p(kc.c),
        vc.mode, vc.bits, vc.group, _p(vrec["idx"]), _p(vrec.get("norm")),
        _p(vrec.get("scale")), _p(vrec.get("min")), _p(vc.R), _p(vc.c), scale, _p(out))
    return out


def decode_partial(q: np.ndarray, kc: Codec, krec: dict, vc: Codec, vrec: dict, scale: float, Lq: int,
                   causal_end: int = None):
    """Unnormalised softmax state of a shard of keys. q: [G, Lq, D]; returns
    (m [G*Lq], l [G*Lq], acc [G*Lq, D]) in fp64; causal_end defaults to the
    shard's own length (the queries are its newest tokens)."""
    q = _c(q, np.float64)
    G, _, D = q.shape
    N = krec["idx"].shape[0]
    E = N if causal_end is None else int(causal_end)
    m = np.empty(G * Lq, np.float64)
    l = np.empty(G * Lq, np.float64)
    acc = np.empty((G * Lq, D), np.float64)
    lib().tqo_decode_partial(
        D, N, E, G, Lq, _p(q), kc.mode, kc.bits, _p(krec["idx"]), _p(krec.get("sgn")),
        _p(krec["norm"]), _p(krec.get("rnorm")), _p(kc.R), _p(kc.S), _p(kc.c),
        vc.mode, vc.bits, vc.group, _p(vrec["idx"]), _p(vrec.get("norm")),
        _p(vrec.get("scale")), _p(vrec.get("min")), _p(vc.c), scale, _p(m), _p(l), _p(acc))
    return m, l, acc


def merge_partials(vc: Codec, m: np.ndarray, l: np.ndarray, acc: np.ndarray) -> np.ndarray:
    """Log-sum-exp merge of P parts: m, l [P, rows], acc [P, rows, D] -> [rows, D]."""
    m, l, acc = _c(m, np.float64), _c(l, np.float64), _c(acc, np.float64)
    P, rows, D = acc.shape
    out = np.empty((rows, D), np.float64)
    lib().tqo_merge_partials(D, P, rows, _p(m), _p(l), _p(acc), vc.mode, _p(vc.R), _p(out))
    return out


def decode_split(q: np.ndarray, low: tuple, high: tuple, scale: float, Lq: int) -> np.ndarray:
    """Decode over split states by the plain definition: each half's records
    dequantised by its own codec, the halves concatenated into whole vectors
    [k_low | k_high], [v_low | v_high], then plain softmax attention (fp64).
    low / high: (key codec, key records, value codec, value records); q [G, Lq, D]."""
    kcl, krl, vcl, vrl = low
    kch, krh, vch, vrh = high
    K = np.concatenate([kcl.dequant(krl), kch.dequant(krh)], axis=1)
    V = np.concatenate([vcl.dequant(vrl), vch.dequant(vrh)], axis=1)
    return attention_f64(q, K, V, scale, Lq)


def subblock_layout(kc: Codec, vc: Codec, BT: int):
    off = np.empty(7, np.int64)
    sub = lib().tqo_subblock_layout(kc.D, kc.mode, kc.bits, vc.mode, vc.bits, vc.group, BT,
                                    _p(off))
    return int(sub), [int(o) for o in off]


def pool_write(pool: np.ndarray, kc: Codec, vc: Codec, Hkv: int, BT: int, table, max_blocks: int,
               seq: int, h: int, t0: int, krec: dict, vrec: dict) -> None:
    """Write records (token-major) for tokens [t0, t0+n) into a uint8 layer pool."""
    assert pool.dtype == np.uint8 and pool.flags.c_contiguous
    n = krec["idx"].shape[0]
    tab = None if table is None else _c(table, np.int32)
    kr = {k: _c(v, v.dtype) for k, v in krec.items()}
    vr = {k: _c(v, v.dtype) for k, v in vrec.items()}
    lib().tqo_pool_write(_p(pool), kc.D, Hkv, BT, _p(tab), max_blocks, seq, h, t0, n,
                         kc.mode, kc.bits, vc.mode, vc.bits, vc.group,
                         _p(kr["idx"]), _p(kr.get("sgn")), _p(kr["norm"]), _p(kr.get("rnorm")),
                         _p(vr["idx"]), _p(vr.get("norm")), _p(vr.get("scale")),
                         _p(vr.get("min")))


def num_threads() -> int:
    return lib().tqo_num_threads()


def set_num_threads(n: int) -> None:
    lib().tqo_set_num_threads(int(n))

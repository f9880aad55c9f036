"""C-ABI checks that need no GPU: the library loads, exports every function
the header declares, and its host codec builder reproduces the oracle's fp32
tables bit for bit (two independent implementations of one construction)."""
import ctypes
import os
import re
import subprocess

import numpy as np
import pytest

from conftest import ROOT

import oracle as O
import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import _lib, build


@pytest.fixture(scope="module")
def libtq():
    build.build()
    return _lib.lib()


def _declared_functions():
    src = open(os.path.join(ROOT, "include", "tq.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(tq_\w+)\s*\(", src, flags=re.M))
    return sorted(names)


def test_header_symbols_exported(libtq):
    names = _declared_functions()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", _lib.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if l.strip()}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert hasattr(libtq, n)
        assert n in _lib.SIGNATURES, f"{n} not declared in the Python binding"


def test_abi_version_and_status_strings(libtq):
    assert tq.tq_abi_version() == 2
    for s in range(8):
        assert _lib.status_string(s)


def test_struct_layout_matches_header(libtq, tmp_path):
    # offsets the C compiler gives the descriptor must match the ctypes mirror
    fields = [f for f, _ in _lib.tq_cache_desc._fields_]
    src = tmp_path / "layout.c"
    src.write_text('#include <stddef.h>\n#include <stdio.h>\n#include "tq.h"\nint main(void) {\n'
                   '  printf("%zu\\n", sizeof(tq_cache_desc));\n' +
                   "".join(f'  printf("%zu\\n", offsetof(tq_cache_desc, {f}));\n' for f in fields) +
                   "  return 0;\n}\n")
    exe = tmp_path / "layout"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)])
    got = [int(v) for v in subprocess.check_output([str(exe)]).split()]
    assert got[0] == ctypes.sizeof(_lib.tq_cache_desc)
    assert got[1:] == [getattr(_lib.tq_cache_desc, f).offset for f in fields]


def test_unsupported_codecs_rejected_without_device(libtq):
    R = np.empty((96, 96), np.float32)
    st = libtq.tq_codec_build_host(96, 3, 0, 0, R.ctypes.data, None, None, None)
    assert st == _lib.TQ_ERR_UNSUPPORTED
    st = libtq.tq_codec_build_host(128, 1, 1, 0, None, None, None, None)   # prod needs >= 2 bits
    assert st == _lib.TQ_ERR_UNSUPPORTED


@pytest.mark.parametrize("D,bits,mode,seed", [
    (128, 3, 1, 0), (128, 3, 0, 1), (128, 4, 0, 0), (128, 4, 0, 1), (128, 3, 1, 42), (128, 4, 0, 43),
    (256, 3, 1, 42), (256, 3, 1, 0), (64, 2, 0, 7), (128, 2, 0, 3), (128, 1, 0, 5), (128, 5, 1, 9),
])
def test_library_tables_equal_oracle(libtq, D, bits, mode, seed):
    R, S, c, m = tq.tq_codec_build_host(D, bits, mode, seed)
    oc = O.Codec(D, bits, mode, seed)
    assert np.array_equal(R.view(np.uint32), oc.R.view(np.uint32))
    if mode == 1:
        assert np.array_equal(S.view(np.uint32), oc.S.view(np.uint32))
    assert np.array_equal(c.view(np.uint32), oc.c.view(np.uint32))
    assert np.array_equal(m.view(np.uint32), oc.m.view(np.uint32))


def test_cache_layout_matches_oracle_without_device(libtq):
    # tq_cache_desc_init needs codec handles (device); the layout arithmetic is
    # checked against the oracle through record sizes here and on the GPU.
    for (D, kb, km, vb, vm, g) in [(128, 3, 1, 3, 0, 0), (128, 3, 1, 4, 2, 64), (256, 3, 1, 2, 2, 32),
                                   (128, 4, 0, 4, 0, 0)]:
        assert O.record_bytes(D, kb, km, 0) + O.record_bytes(D, vb, vm, g) in (108, 128, 200, 136)


def test_bits_split_matches_oracle(libtq):
    # host-only arithmetic: the library's split of a fractional width against the oracle's
    widths = [1.0, 1.5, 2.0, 2.25, 2.5, 2.75, 3.0, 3.5, 3.9, 4.0, 3.0000005, 2.9999995, 3.00001,
              1.0000004, 3.999999, 2.0 + 1e-7]
    for b in widths:
        assert tq.tq_bits_split(b) == O.bits_split(b), b


def test_bits_split_rejects_out_of_range(libtq):
    kb, vb = ctypes.c_int(7), ctypes.c_int(7)
    for b in (0.5, 0.9999995, 4.5, 5.0, -3.0, float("nan"), float("inf")):
        st = libtq.tq_bits_split(b, ctypes.byref(kb), ctypes.byref(vb))
        assert st == _lib.TQ_ERR_UNSUPPORTED, b
        assert kb.value == 0 and vb.value == 0
    assert libtq.tq_bits_split(3.5, None, ctypes.byref(vb)) == _lib.TQ_ERR_INVALID_ARG
    kh, vh = ctypes.c_void_p(1), ctypes.c_void_p(1)
    # rejected before any device work, and both outputs cleared
    assert libtq.tq_codec_pair_for_bits(128, 4.5, 0, ctypes.byref(kh), ctypes.byref(vh)) == _lib.TQ_ERR_UNSUPPORTED
    assert not kh.value and not vh.value


# ------------------------------------------------------------------ decode planner (host arithmetic)

_KEYS = [("prod", 2), ("prod", 3), ("prod", 4), ("mse", 2), ("mse", 3), ("mse", 4)]
_VALUES = [("mse", 2, 0), ("mse", 3, 0), ("mse", 4, 0), ("group", 2, 32), ("group", 4, 32), ("group", 4, 64),
           ("group", 4, 128)]
_MODE = {"mse": 0, "prod": 1, "group": 2}
# the split kernel's dynamic shared memory must fit the 227 KB per-block opt-in
_SMEM_LIMIT = 227 * 1024


def _desc_from_oracle(D, key, value, BT, Hkv):
    """A cache descriptor whose layout fields come from the oracle's sub-block layout."""
    kc = O.Codec(D, key[1], _MODE[key[0]], 0)
    vc = O.Codec(D, value[1], _MODE[value[0]], 1, value[2])
    sub, off = O.subblock_layout(kc, vc, BT)
    d = _lib.tq_cache_desc()
    d.block_tokens, d.num_kv_heads, d.head_dim = BT, Hkv, D
    d.key_mode, d.key_bits = _MODE[key[0]], key[1]
    d.value_mode, d.value_bits, d.value_group = _MODE[value[0]], value[1], value[2]
    d.subblock_bytes = sub
    for k in range(7):
        d.stream_offset[k] = off[k]
    return d


def test_decode_plan_fits_shared_memory_for_every_codec_pair(libtq):
    # every tensor-core codec pair and block size: the stages, query fragments
    # and lookup tables fit; tiles divide blocks or gather whole blocks; the
    # splits cover the sequence
    for key in _KEYS:
        for value in _VALUES:
            for BT in (16, 64, 256, 4096):
                d = _desc_from_oracle(128, key, value, BT, 8)
                for (B, Hq, Lq, msl) in [(1, 64, 2, 262146), (32, 32, 1, 65536), (3, 8, 8, 700)]:
                    p = tq.tq_decode_plan(d, B, Hq, Lq, msl, 152)
                    assert p["tensor_cores"] == 1
                    assert 0 < p["smem_bytes"] <= _SMEM_LIMIT - 1024, (key, value, BT, p)
                    t = p["tile_tokens"]
                    # a tile lies inside one block or gathers at most four whole blocks
                    assert 16 <= t <= 64 and (BT % t == 0 or (t % BT == 0 and t // BT <= 4)), (key, value, BT, p)
                    assert p["chunk_tokens"] % t == 0
                    assert p["splits"] * p["chunk_tokens"] >= msl
                    assert p["row_groups"] == (Hq // 8 * Lq + 15) // 16


def test_decode_plan_of_the_bench_configuration(libtq):
    # keys prod 3-bit, values MSE 3-bit, 256-token blocks, GQA 8 x q_len 2 at
    # 256k on 152 SMs: 64-token tiles, 19 splits, 12 warps x 2 stages x 6912 B
    # + 8 KB query fragments + 16 KB value pair region + 32 KB key quad table
    # + 24 stage barriers and the tables' barrier
    d = _desc_from_oracle(128, ("prod", 3), ("mse", 3, 0), 256, 8)
    p = tq.tq_decode_plan(d, 1, 64, 2, 262146, 152)
    assert p["tile_tokens"] == 64 and p["splits"] == 19 and p["row_groups"] == 1
    assert p["smem_bytes"] == 12 * 2 * 6912 + 8192 + 16384 + 32768 + (12 * 2 + 1) * 8
    # a record pair too large for 64-token stages next to the tables: 32-token tiles
    d = _desc_from_oracle(128, ("prod", 4), ("group", 4, 32), 256, 8)
    assert tq.tq_decode_plan(d, 1, 64, 2, 4096, 152)["tile_tokens"] == 32


def test_decode_plan_rejects_bad_sizes(libtq):
    d = _desc_from_oracle(128, ("prod", 3), ("mse", 3, 0), 256, 8)
    info = _lib.tq_decode_plan_info()
    assert libtq.tq_decode_plan(ctypes.byref(d), 1, 64, 2, 1, 152, ctypes.byref(info)) == _lib.TQ_ERR_INVALID_ARG
    assert libtq.tq_decode_plan(ctypes.byref(d), 1, 63, 2, 100, 152, ctypes.byref(info)) == _lib.TQ_ERR_INVALID_ARG
    assert libtq.tq_decode_plan(ctypes.byref(d), 1, 64, 2, 100, 0, ctypes.byref(info)) == _lib.TQ_ERR_INVALID_ARG
    assert libtq.tq_decode_plan(ctypes.byref(d), 1, 8 * 65, 1, 100, 152, ctypes.byref(info)) == _lib.TQ_ERR_UNSUPPORTED


def test_selftest_wait_timeout_rejects_bad_deadlines_without_device(libtq):
    # the deadline is checked on the host before any CUDA call (none is possible here)
    for s in (0.0, -0.5, 1.01, float("nan"), float("inf")):
        assert libtq.tq_selftest_wait_timeout(s, None) == _lib.TQ_ERR_INVALID_ARG


def test_workspace_query_rejects_a_descriptor_without_heads(libtq):
    # checked on the host before any division by the head count or device call
    d = _desc_from_oracle(128, ("prod", 3), ("mse", 3, 0), 256, 8)
    d.num_kv_heads = 0
    n = ctypes.c_size_t(0)
    assert libtq.tq_decode_workspace_bytes(ctypes.byref(d), 1, 64, 2, 100, ctypes.byref(n)) == _lib.TQ_ERR_INVALID_ARG
    d.num_kv_heads = 8
    d.block_tokens = 24
    assert libtq.tq_decode_workspace_bytes(ctypes.byref(d), 1, 64, 2, 100, ctypes.byref(n)) == _lib.TQ_ERR_INVALID_ARG


def test_decode_plan_simt_shapes(libtq):
    # head_dims 64 and 256 with codec pairs the tensor-core kernels are not
    # built for take the SIMT kernels: no tensor-core shared memory
    for D, key, value in [(256, ("prod", 2), ("group", 4, 64)), (64, ("mse", 2), ("mse", 2, 0))]:
        d = _desc_from_oracle(D, key, value, 64, 2)
        p = tq.tq_decode_plan(d, 2, 16, 1, 8192, 152)
        assert p["tensor_cores"] == 0 and p["smem_bytes"] == 0
        assert p["splits"] * p["chunk_tokens"] >= 8192 and p["workspace_bytes"] > 0


@pytest.mark.parametrize("D", [64, 256])
def test_decode_plan_head_dim_64_256_codec_set(libtq, D):
    # the head_dim-64 and -256 tensor-core kernels: prod 3-bit keys with group
    # 2/4-bit or MSE 3/4-bit values, and MSE 4-bit keys and values; the rest
    # SIMT. At 64 the partial rows are 128 columns wide (the head_dim-128
    # layout); at 256 the stages hold 32 tokens (64-token stages do not fit).
    tc = {(("prod", 3), ("group", 2, 32)), (("prod", 3), ("group", 2, 64)), (("prod", 3), ("group", 4, 32)),
          (("prod", 3), ("group", 4, 64)), (("prod", 3), ("mse", 3, 0)), (("prod", 3), ("mse", 4, 0)),
          (("mse", 4), ("mse", 4, 0))}
    for key in (("prod", 2), ("prod", 3), ("prod", 4), ("mse", 2), ("mse", 3), ("mse", 4)):
        for value in (("group", 2, 32), ("group", 2, 64), ("group", 4, 32), ("group", 4, 64), ("mse", 2, 0),
                      ("mse", 3, 0), ("mse", 4, 0)):
            if D == 64 and value[0] == "group" and value[2] > 64:
                continue
            d = _desc_from_oracle(D, key, value, 64, 2)
            p = tq.tq_decode_plan(d, 2, 16, 2, 8192, 152)
            assert p["tensor_cores"] == ((key, value) in tc), (key, value, p)
            if p["tensor_cores"]:
                assert p["tile_tokens"] in ((32,) if D == 256 else (32, 64)), (key, value, p)
                assert 0 < p["smem_bytes"] <= _SMEM_LIMIT - 1024, (key, value, p)
                units, S = 2 * 2, p["splits"]   # 2 sequences x 2 KV heads x 1 row group
                r = lambda x: (x + 255) // 256 * 256
                q = r(units * 16 * D * 4)
                part = r(units * S * 16 * max(D, 128) * 4)
                ml = r(units * max(D // 128, 1) * S * 16 * 2 * 4)
                assert p["workspace_bytes"] == 2 * q + part + ml, (key, value, p)


@pytest.mark.parametrize("value", [("group", 2, 32), ("mse", 3, 1)])
def test_decode_plan_head_dim_256_tensor_cores(libtq, value):
    # prod 3-bit keys with group 2-bit or MSE 3-bit values at head_dim 256:
    # two CTAs (128-column value halves) per (unit, split), so 2 sequences x
    # 2 KV heads x 1 row group = 4 units x 2 halves = 8 CTAs per split; 19
    # splits cover 152 SMs; 200 or 204 record bytes per token need 32-token
    # tiles (64-token stages would not fit)
    d = _desc_from_oracle(256, ("prod", 3), value, 64, 2)
    p = tq.tq_decode_plan(d, 2, 16, 1, 8192, 152)
    assert p["tensor_cores"] == 1 and p["tile_tokens"] == 32
    assert p["splits"] == 19 and p["chunk_tokens"] == 448
    assert 0 < p["smem_bytes"] <= 227 * 1024 - 1024
    # fp32 q' and q'' rows (two arrays), partials for both halves, (max, sum)
    # rows for both halves
    units = 4
    q = units * 16 * 256 * 4
    part = units * 19 * 16 * 256 * 4
    ml = units * 2 * 19 * 16 * 2 * 4
    r = lambda x: (x + 255) // 256 * 256
    assert p["workspace_bytes"] == 2 * r(q) + r(part) + r(ml)


def test_decode_plan_split_rule(libtq):
    # splits: enough CTAs to cover the SMs, each split a multiple of the tile
    # and at most 16384 tokens, or 12288 where the units alone fill the SMs
    # (several waves of CTAs: shorter CTAs keep the last wave's tail short)
    d = _desc_from_oracle(128, ("prod", 3), ("mse", 3, 0), 256, 8)
    one = tq.tq_decode_plan(d, 1, 64, 2, 262146, 152)        # 8 units -> 19 splits of 13,824 tokens
    assert one["splits"] == 19 and one["chunk_tokens"] == 13824
    many = tq.tq_decode_plan(d, 32, 32, 1, 65536, 152)       # 256 units >= 152 SMs: split by length only
    assert many["splits"] == 6 and many["chunk_tokens"] == 12288
    few = tq.tq_decode_plan(d, 18, 64, 2, 65536, 152)        # 144 units < 152 SMs: 16384-token splits
    assert few["splits"] == 4 and few["chunk_tokens"] == 16384
    short = tq.tq_decode_plan(d, 1, 64, 2, 100, 152)         # a short sequence: one 32-token tile per split
    assert short["chunk_tokens"] == 32 and short["splits"] == 4


def test_decode_plan_transposed_for_few_rows(libtq):
    # head_dim 128 with at most 8 query rows per KV head and a codec pair of the
    # transposed kernel's set: the transposed form; 16 rows, other pairs, or
    # other head_dims: the 16-row form (or SIMT)
    few = {(("prod", 3), ("group", 4)), (("prod", 3), ("group", 2)), (("prod", 3), ("mse", 3)),
           (("prod", 3), ("mse", 4)), (("mse", 4), ("mse", 4))}   # any group size
    for key in _KEYS:
        for value in _VALUES:
            d = _desc_from_oracle(128, key, value, 64, 8)
            for Hq, Lq in ((32, 1), (64, 1), (16, 3), (64, 2)):
                p = tq.tq_decode_plan(d, 2, Hq, Lq, 4096, 152)
                rows = Hq // 8 * Lq
                want = 1 if rows <= 8 and (key, value[:2]) in few else 0
                assert p["transposed"] == want, (key, value, Hq, Lq, p)
    d = _desc_from_oracle(64, ("prod", 3), ("mse", 3, 0), 64, 8)
    assert tq.tq_decode_plan(d, 2, 32, 1, 4096, 152)["transposed"] == 0


def test_decode_plan_tile_balances_the_busiest_warp(libtq):
    # 64-token tiles unless 32-token tiles (each about 0.52 of a 64-token
    # tile's time) give the busiest of the 12 warps less work: at 256k a split
    # holds 216 tiles (18 per warp) or 432 half tiles (36 x 0.52 = 18.7); at
    # 32k, 27 tiles (3 for the busiest warp) or 54 half tiles (5 x 0.52 = 2.6)
    d = _desc_from_oracle(128, ("prod", 3), ("mse", 3, 0), 256, 8)
    assert tq.tq_decode_plan(d, 1, 64, 2, 262146, 152)["tile_tokens"] == 64
    d = _desc_from_oracle(128, ("mse", 4), ("mse", 4, 0), 256, 8)
    p = tq.tq_decode_plan(d, 1, 64, 2, 32768, 152)
    assert p["tile_tokens"] == 32 and p["splits"] == 19 and p["chunk_tokens"] == 1728
    # 32 sequences of up to 64k: splits of 12288 tokens, 192 tiles (16 for the
    # busiest warp) against 384 half tiles (32 x 0.52 = 16.6)
    d = _desc_from_oracle(128, ("prod", 3), ("group", 4, 64), 16, 8)
    assert tq.tq_decode_plan(d, 32, 32, 1, 65536, 152)["tile_tokens"] == 64


# ------------------------------------------------------------------ host-side argument checks

def _zero_args(fn):
    """One argument per ctypes argtype: NULL pointers, zero numbers."""
    args = []
    for t in fn.argtypes:
        if t in (ctypes.c_float, ctypes.c_double):
            args.append(0.0)
        elif t in (ctypes.c_int, ctypes.c_int64, ctypes.c_uint64, ctypes.c_size_t, ctypes.c_uint32):
            args.append(0)
        else:
            args.append(None)
    return args


@pytest.mark.parametrize("name", ["tq_encode_append", "tq_decode_attention", "tq_decode_step",
                                  "tq_decode_attention_noalloc", "tq_prefill_attention"])
def test_compute_calls_reject_missing_codecs_before_device_work(libtq, name):
    # a NULL codec is refused on the host, before any CUDA call (none is
    # possible here), with the header's status
    fn = getattr(libtq, name)
    d = _desc_from_oracle(128, ("prod", 3), ("mse", 3, 0), 256, 8)
    d.num_layers = 1
    args = _zero_args(fn)
    args[2] = ctypes.byref(d)
    args[3] = 0                       # layer
    assert fn(*args) == _lib.TQ_ERR_INVALID_ARG


def test_copy_blocks_mixed_configuration_guard_without_device(libtq):
    # the batch operations refuse caches of different configurations (the
    # pages raise on mixing them); the check is host arithmetic
    def desc(key=("prod", 3), value=("mse", 3, 0), BT=16, Hkv=2, D=128):
        d = _desc_from_oracle(D, key, value, BT, Hkv)
        d.num_layers = 2
        return d
    a = desc()
    f = libtq.tq_cache_copy_blocks
    assert f(ctypes.byref(a), ctypes.byref(desc()), None, None, 0, None) == _lib.TQ_OK   # nothing to copy
    for other in (desc(key=("prod", 4)), desc(key=("mse", 3)), desc(value=("mse", 4, 0)),
                  desc(value=("group", 4, 64)), desc(BT=32), desc(Hkv=4)):
        assert f(ctypes.byref(a), ctypes.byref(other), None, None, 0, None) == _lib.TQ_ERR_CONFIG_MISMATCH
    b = desc()
    b.num_layers = 3
    assert f(ctypes.byref(a), ctypes.byref(b), None, None, 0, None) == _lib.TQ_ERR_CONFIG_MISMATCH
    b = desc()
    b.key_seed = 5
    assert f(ctypes.byref(a), ctypes.byref(b), None, None, 0, None) == _lib.TQ_ERR_CONFIG_MISMATCH
    assert f(None, ctypes.byref(a), None, None, 0, None) == _lib.TQ_ERR_INVALID_ARG
    assert f(ctypes.byref(a), ctypes.byref(desc()), None, None, -1, None) == _lib.TQ_ERR_INVALID_ARG


def test_decode_plan_invariants_on_random_shapes(libtq):
    # seeded sweep: every plan covers the sequence with non-empty splits of
    # whole tiles (inside one block or gathering at most four), at most 16384
    # tokens each, inside the shared-memory budget
    rng = np.random.default_rng(11)
    for _ in range(300):
        key = _KEYS[rng.integers(len(_KEYS))]
        value = _VALUES[rng.integers(len(_VALUES))]
        BT = int(rng.choice([16, 32, 64, 128, 256, 1024]))
        Hkv = int(rng.choice([1, 2, 4, 8]))
        G = int(rng.choice([1, 2, 4, 8]))
        Lq = int(rng.integers(1, 65 // G + 1))
        B = int(rng.integers(1, 65))
        msl = int(rng.integers(Lq, 300001))
        sms = int(rng.choice([1, 20, 76, 148, 152]))
        d = _desc_from_oracle(128, key, value, BT, Hkv)
        p = tq.tq_decode_plan(d, B, Hkv * G, Lq, msl, sms)
        t, c, s = p["tile_tokens"], p["chunk_tokens"], p["splits"]
        case = (key, value, BT, Hkv, G, Lq, B, msl, sms, p)
        assert p["tensor_cores"] == 1 and (BT % t == 0 or (t % BT == 0 and t // BT <= 4)) and 16 <= t <= 64, case
        assert c % t == 0 and c <= max(16384, t), case
        assert s * c >= msl and (s - 1) * c < msl, case
        assert 0 < p["smem_bytes"] <= _SMEM_LIMIT - 1024, case
        assert p["row_groups"] == (G * Lq + 15) // 16 and p["workspace_bytes"] > 0, case


def test_prefill_workspace_follows_the_supported_codec_rule(libtq):
    # host arithmetic: the header's codec set for prefill attention (head_dim
    # 128; prod 3-bit keys with MSE 3/4-bit or group 4-bit values, or MSE
    # 4-bit keys and values) sizes a workspace; anything else is refused
    supported = {(("prod", 3), ("mse", 3, 0)), (("prod", 3), ("mse", 4, 0)), (("prod", 3), ("group", 4, 32)),
                 (("prod", 3), ("group", 4, 64)), (("prod", 3), ("group", 4, 128)), (("mse", 4), ("mse", 4, 0))}
    f = libtq.tq_prefill_workspace_bytes
    n = ctypes.c_size_t(0)
    for key in _KEYS:
        for value in _VALUES:
            d = _desc_from_oracle(128, key, value, 64, 8)
            st = f(ctypes.byref(d), 2, 64, 8192, ctypes.byref(n))
            if (key, value) in supported:
                # one 16-row fragment set per (sequence, KV head, row group), 256-byte rounded
                rows = (8 * 8192 + 15) // 16
                assert st == _lib.TQ_OK and n.value == (2 * 8 * rows * 2 * 8 * 32 * 16 + 255) // 256 * 256
            else:
                assert st == _lib.TQ_ERR_UNSUPPORTED, (key, value)
    d = _desc_from_oracle(256, ("prod", 3), ("group", 2, 32), 64, 2)
    assert f(ctypes.byref(d), 1, 16, 128, ctypes.byref(n)) == _lib.TQ_ERR_UNSUPPORTED
    d = _desc_from_oracle(128, ("prod", 3), ("mse", 3, 0), 64, 8)
    assert f(ctypes.byref(d), 1, 64, 0, ctypes.byref(n)) == _lib.TQ_ERR_INVALID_ARG
    assert f(ctypes.byref(d), 1, 60, 16, ctypes.byref(n)) == _lib.TQ_ERR_INVALID_ARG
    assert f(ctypes.byref(d), 1, 64, 16, None) == _lib.TQ_ERR_INVALID_ARG

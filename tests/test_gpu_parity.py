"""GPU path vs oracle: codec tables, bit-exact encode, paged append and decode
attention within the stated tolerance, on the workloads' shapes (reduced
where the oracle must stay fast), plus edge cases and error paths."""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle as O
import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import (GpuCase, compare_decode, oracle_codec, oracle_decode, raw_kv,
                         to_f32_np)

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    O.build()
    assert torch.cuda.is_available()


# ------------------------------------------------------------------ codecs

@pytest.mark.parametrize("D,bits,mode,seed", [(128, 3, 1, 0), (128, 3, 0, 1), (128, 4, 0, 0),
                                              (256, 3, 1, 42), (128, 4, 0, 43), (64, 2, 0, 5)])
def test_device_codec_tables_bit_exact(D, bits, mode, seed):
    c = tq.Codec(D, bits, mode, seed)
    R, S, cen, mid = c.export()
    oc = O.Codec(D, bits, mode, seed)
    assert np.array_equal(R.view(np.uint32), oc.R.view(np.uint32))
    if mode == 1:
        assert np.array_equal(S.view(np.uint32), oc.S.view(np.uint32))
    assert np.array_equal(cen.view(np.uint32), oc.c.view(np.uint32))
    assert np.array_equal(mid.view(np.uint32), oc.m.view(np.uint32))


@pytest.mark.parametrize("D,bits,seed,kb,vb", [(128, 3.5, 0, 3, 4), (128, 2.5, 7, 2, 3),
                                                (64, 3.0, 3, 3, 3), (256, 1.5, 11, 1, 2)])
def test_codec_pair_for_fractional_bits(D, bits, seed, kb, vb):
    # keys: MSE floor(b) bits with the seed; values: MSE ceil(b) bits with seed + 1
    kc, vc = tq.Codec.pair_for_bits(D, bits, seed)
    for c, b, s in ((kc, kb, seed), (vc, vb, seed + 1)):
        assert (c.info["head_dim"], c.info["bits"], c.info["mode"], c.info["seed"]) == (D, b, O.MSE, s)
        R, _, cen, mid = c.export()
        oc = O.Codec(D, b, O.MSE, s)
        assert np.array_equal(R.view(np.uint32), oc.R.view(np.uint32))
        assert np.array_equal(cen.view(np.uint32), oc.c.view(np.uint32))
        assert np.array_equal(mid.view(np.uint32), oc.m.view(np.uint32))


# ------------------------------------------------------------------ encode

def _vectors(n, D, dtype, seed, group=None):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, D, generator=g) * torch.exp(torch.randn(n, 1, generator=g) * 2)
    x[0] = 0                                       # zero vector
    x[1] = 1e-30                                   # norm underflows in fp32
    x[2, : (group or D)] = 0.5                     # constant group
    x[3] = torch.randn(D, generator=g) * 3e4       # large magnitude
    x[4, ::2] = -x[4, 1::2]                        # paired coordinates
    return x.to(dtype)


CODECS = [(1, 2), (1, 3), (1, 4), (1, 5), (0, 1), (0, 2), (0, 3), (0, 4)]


# every head_dim and codec in bf16; the f32 and f16 inputs on one shape
QUANT_CASES = [pytest.param(D, m, b, torch.bfloat16, id=f"bf16-d{D}-mode{m}-b{b}")
               for D in (64, 128, 256) for m, b in CODECS] + \
              [pytest.param(128, m, b, dt, id=f"{name}-d128-mode{m}-b{b}")
               for dt, name in ((torch.float32, "f32"), (torch.float16, "f16"))
               for m, b in CODECS if b in (3, 4)]


@pytest.mark.parametrize("D,mode,bits,dtype", QUANT_CASES)
def test_quantize_bit_exact(D, mode, bits, dtype):
    n = 3000 if D <= 128 else 1500
    x = _vectors(n, D, dtype, D * 100 + bits * 10 + mode)
    if dtype == torch.float16:
        x = x.clamp(-6e4, 6e4)
    c = tq.Codec(D, bits, mode, 7)
    ib = c.info["index_bits"]
    W = c.info["index_words"]
    xd = x.to(DEV)
    idx = torch.empty(n, W, dtype=torch.int32, device=DEV)
    norm = torch.empty(n, dtype=torch.float32, device=DEV)
    sgn = torch.empty(n, D // 32, dtype=torch.int32, device=DEV) if mode == 1 else None
    rn = torch.empty(n, dtype=torch.float32, device=DEV) if mode == 1 else None
    tq.tq_quantize(c.handle, xd, idx, norm, sgn, rn)
    torch.cuda.synchronize()
    oc = O.Codec(D, bits, mode, 7)
    rec = oc.encode(to_f32_np(x))
    assert np.array_equal(idx.cpu().numpy().view(np.uint32), rec["idx"])
    assert np.array_equal(norm.cpu().numpy().view(np.uint32), rec["norm"].view(np.uint32))
    if mode == 1:
        assert np.array_equal(sgn.cpu().numpy().view(np.uint32), rec["sgn"])
        assert np.array_equal(rn.cpu().numpy().view(np.uint32), rec["rnorm"].view(np.uint32))
    assert ib == oc.ib


@pytest.mark.parametrize("D,bits,group", [(128, 2, 32), (128, 4, 64), (256, 2, 32), (128, 4, 128),
                                          (64, 2, 32), (256, 4, 64)])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
def test_quantize_group_bit_exact(D, bits, group, dtype):
    n = 2000
    x = _vectors(n, D, dtype, D + bits + group, group)
    x = x.clamp(-6e4, 6e4)
    c = tq.Codec(D, bits, tq.TQ_MODE_GROUP, group=group)
    W = c.info["index_words"]
    idx = torch.empty(n, W, dtype=torch.int32, device=DEV)
    sc = torch.empty(n, D // group, dtype=torch.int16, device=DEV)
    mn = torch.empty(n, D // group, dtype=torch.int16, device=DEV)
    tq.tq_quantize(c.handle, x.to(DEV), idx, sc, mn)
    torch.cuda.synchronize()
    rec = O.Codec(D, bits, O.GROUP, group=group).encode(to_f32_np(x))
    assert np.array_equal(idx.cpu().numpy().view(np.uint32), rec["idx"])
    assert np.array_equal(sc.cpu().numpy().view(np.uint16), rec["scale"])
    assert np.array_equal(mn.cpu().numpy().view(np.uint16), rec["min"])


# ------------------------------------------------------------------ paged append

def _small_paged(name="small_paged", key=("prod", 3), value=("group", 4, 64), D=128, bt=16,
                 lens=(37, 100, 16, 1), append=2, Hkv=2, G=4, Lq=1):
    kspec = wl._spec(key[0], key[1], 11)
    vspec = wl._spec(value[0], value[1], 12, value[2] if len(value) > 2 else 0)
    return wl.Workload(name, 2, len(lens), Hkv, Hkv * G, D, tuple(lens), Lq, torch.bfloat16, 1.0, 99,
                       kspec, vspec, block_tokens=bt, shuffle_blocks=True, append_per_step=append,
                       prefill_chunk=64)


@pytest.mark.parametrize("value,key,D,chunk,lens", [
    (("group", 4, 64), ("prod", 3), 128, 24, (37, 100, 16, 1)),
    (("mse", 3), ("prod", 3), 128, 24, (37, 100, 16, 1)),
    (("group", 2, 32), ("prod", 3), 128, 24, (37, 100, 16, 1)),
    # chunks of >= 32 tokens take the register-blocked encoder (ragged tails included)
    (("mse", 3), ("prod", 3), 128, 300, (700, 45, 333)),
    (("group", 4, 64), ("mse", 4), 128, 257, (600, 33)),
    (("mse", 2), ("prod", 4), 64, 500, (530, 129)),
    (("group", 2, 32), ("prod", 3), 256, 100, (230, 64)),
    (("mse", 4), ("mse", 1), 256, 64, (100,)),
])
def test_append_into_paged_pool_bit_exact(value, key, D, chunk, lens):
    w = _small_paged(value=value, key=key, D=D, lens=lens)
    case = GpuCase(w, layers=[0, 1], seq_lens=w.seq_lens)
    case.prefill(chunk=chunk)       # several calls, crossing block boundaries
    # incremental appends of `append_per_step` tokens at the written end
    B = w.batch
    n_new = w.append_per_step
    for li, layer in enumerate(case.layers):
        k = torch.stack([wl.kv_chunk(w, layer, b, w.seq_lens[b], n_new, "k", DEV) for b in range(B)])
        v = torch.stack([wl.kv_chunk(w, layer, b, w.seq_lens[b], n_new, "v", DEV) for b in range(B)])
        sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
        case.cache.append(li, k, v, sl, case.table_d, case.max_blocks)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    kc, vc = oracle_codec(w.key, w.head_dim), oracle_codec(w.value, w.head_dim)
    sub, _ = O.subblock_layout(kc, vc, w.block_tokens)
    assert sub == case.cache.desc.subblock_bytes
    layer_bytes = case.cache.desc.layer_stride
    pool = case.cache.pool.cpu().numpy()
    for li, layer in enumerate(case.layers):
        want = np.zeros(layer_bytes, np.uint8)
        for b in range(B):
            n = w.seq_lens[b] + n_new
            K, V = raw_kv(w, layer, b, n, DEV)
            for h in range(w.num_kv_heads):
                O.pool_write(want, kc, vc, w.num_kv_heads, w.block_tokens, case.table.numpy(),
                             case.max_blocks, b, h, 0, kc.encode(K[h]), vc.encode(V[h]))
        got = pool[li * layer_bytes:(li + 1) * layer_bytes]
        assert np.array_equal(got, want)


# ------------------------------------------------------------------ decode

def _check_decode(w, layers, seq_lens=None, q_step=0):
    case = GpuCase(w, layers, seq_lens)
    case.prefill()
    errs = []
    for li, layer in enumerate(layers):
        q = wl.queries(w, layer, q_step, DEV)
        out = to_f32_np(case.decode(li, q))
        qn = to_f32_np(q).astype(np.float64)
        for b in range(w.batch):
            n = case.seq_lens[b]
            K, V = raw_kv(w, layer, b, n, DEV)
            for h in range(w.num_kv_heads):
                G = w.gqa
                ref = oracle_decode(w, K[h], V[h], qn[b, h * G:(h + 1) * G])
                errs.append(compare_decode(out[b, h * G:(h + 1) * G], ref))
    assert tq.tq_device_error() == 0
    return errs


def test_decode_tiny():
    _check_decode(wl.tiny(), [0])


@pytest.mark.parametrize("n", [512, 1024, 4096, 8192])
def test_decode_layer_d256(n):
    _check_decode(wl.layer_d256(n), [0])


@pytest.mark.parametrize("n", [1000, 4097])
def test_decode_layer_d256_mse_values(n):
    # the same layer with 3-bit MSE values (rotated back in the merge)
    w = dataclasses.replace(wl.layer_d256(4096), value=wl._spec("mse", 3, 1), seq_lens=(n,))
    _check_decode(w, [0])


def test_decode_stack_shape_reduced():
    w = dataclasses.replace(wl.stack_32k(), seq_lens=(3001,))
    _check_decode(w, [0, 63])


def test_decode_long_context_codecs_reduced():
    w = dataclasses.replace(wl.long_256k(), seq_lens=(9000,))
    _check_decode(w, [5])


def test_decode_paged_batch_reduced():
    base = wl.paged_batch()
    lens = tuple(int(x) // 24 for x in base.seq_lens[:6])
    w = dataclasses.replace(base, batch=6, seq_lens=lens)
    _check_decode(w, [0])


@pytest.mark.parametrize("n,lq", [(1, 1), (2, 2), (33, 2), (17, 4)])
def test_decode_short_sequences(n, lq):
    w = dataclasses.replace(_small_paged(lens=(n, n + 5), Lq=lq, G=8, bt=16), append_per_step=0)
    _check_decode(w, [0])


def test_decode_more_than_16_rows():
    w = dataclasses.replace(_small_paged(lens=(300,), Lq=3, G=8, bt=32), append_per_step=0)
    _check_decode(w, [1])


# ------------------------------------------------------------------ errors

def test_config_mismatch_and_capacity_errors():
    D = 128
    kc, vc = tq.Codec(D, 3, 1, 0), tq.Codec(D, 3, 0, 1)
    other = tq.Codec(D, 3, 1, 5)
    cache = tq.CompressedKVCache(kc, vc, 1, 4, 16, 1)
    k = torch.zeros(1, 1, 2, D, dtype=torch.bfloat16, device=DEV)
    sl = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(tq.TQError) as e:
        tq.tq_encode_append(other.handle, vc.handle, cache.desc, 0, k, k, sl, None, 4)
    assert e.value.status == 3
    big = torch.zeros(1, 1, 65, D, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(tq.TQError) as e:
        cache.append(0, big, big, sl, None, 4)
    assert e.value.status == 4
    with pytest.raises(tq.TQError) as e:
        tq.Codec(96, 3, 1, 0)
    assert e.value.status == 2


def test_device_flags_for_bad_block_and_seq_len():
    D = 128
    kc, vc = tq.Codec(D, 3, 1, 0), tq.Codec(D, 4, 0, 1)
    cache = tq.CompressedKVCache(kc, vc, 1, 4, 16, 1)
    assert tq.tq_device_error() == 0
    k = torch.ones(1, 1, 3, D, dtype=torch.bfloat16, device=DEV)
    table = torch.tensor([[0, 9]], dtype=torch.int32, device=DEV)   # block 9 is outside the pool
    sl = torch.tensor([15], dtype=torch.int32, device=DEV)
    cache.append(0, k, k, sl, table, 2)
    assert tq.tq_device_error() & tq.TQ_DEVERR_BLOCK
    before = cache.pool.clone()
    sl = torch.tensor([31], dtype=torch.int32, device=DEV)          # past the table's capacity
    cache.append(0, k, k, sl, table, 2)
    assert tq.tq_device_error() & tq.TQ_DEVERR_CAPACITY
    assert torch.equal(before, cache.pool)
    q = torch.ones(1, 2, 1, D, dtype=torch.bfloat16, device=DEV)
    out = torch.empty(1, 2, 1, D, dtype=torch.float32, device=DEV)
    ws = torch.empty(cache.workspace_bytes(1, 2, 1, 32), dtype=torch.uint8, device=DEV)
    sl = torch.tensor([40], dtype=torch.int32, device=DEV)          # longer than the table
    cache.decode(0, q, sl, torch.tensor([[0, 1]], dtype=torch.int32, device=DEV), 2, 32, out, ws)
    assert tq.tq_device_error() & tq.TQ_DEVERR_SEQLEN
    assert tq.tq_device_error() == 0


def test_empty_batch_is_noop():
    D = 128
    kc, vc = tq.Codec(D, 3, 1, 0), tq.Codec(D, 4, 0, 1)
    cache = tq.CompressedKVCache(kc, vc, 1, 4, 16, 1)
    n0 = tq.tq_launch_count()
    k = torch.zeros(0, 1, 2, D, dtype=torch.bfloat16, device=DEV)
    cache.append(0, k, k, torch.zeros(0, dtype=torch.int32, device=DEV), None, 4)
    assert tq.tq_launch_count() == n0


KEYS = [("prod", 2), ("prod", 3), ("prod", 4), ("mse", 2), ("mse", 3), ("mse", 4)]
VALUES = [("mse", 2), ("mse", 3), ("mse", 4), ("group", 2, 32), ("group", 4, 32), ("group", 4, 64), ("group", 4, 128)]


@pytest.mark.parametrize("key", KEYS)
@pytest.mark.parametrize("value", VALUES)
def test_decode_codec_combinations(key, value):
    # every tensor-core kernel instantiation: ragged length, two query positions
    w = dataclasses.replace(_small_paged(key=key, value=value, lens=(203,), Lq=2, G=8, bt=64, Hkv=2),
                            append_per_step=0)
    _check_decode(w, [0])


@pytest.mark.parametrize("bt", [16, 32, 128])
def test_decode_block_sizes(bt):
    w = dataclasses.replace(_small_paged(lens=(300, 77, 1000), Lq=1, G=4, bt=bt), append_per_step=0)
    _check_decode(w, [1])


def test_decode_head_dim_64():
    w = dataclasses.replace(_small_paged(key=("prod", 3), value=("mse", 4), D=64, lens=(150,), Lq=2, G=4),
                            append_per_step=0)
    _check_decode(w, [0])

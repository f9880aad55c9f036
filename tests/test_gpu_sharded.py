"""Sequence-sharded decode on one GPU: tq_decode_partials over each shard of
a sequence's tokens (each shard in a cache of its own, as on separate GPUs),
tq_decode_merge of the shards' states; compared with tq_decode_attention over
the whole sequence and with the oracle (its decode of the whole sequence, and
its partial state of each shard through the invariants m + ln l and acc / l).
"""
import math

import numpy as np
import pytest
import torch

import oracle as O
import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import sharded
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import compare_decode, oracle_codec, raw_kv, to_f32_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _cache_of(w, layer, b, start, count, kc, vc):
    nblk = max(1, (count + w.block_tokens - 1) // w.block_tokens)
    cache = tq.CompressedKVCache(kc, vc, 1, nblk, w.block_tokens, w.num_kv_heads, DEV, exact_encode=True)
    if count:
        k = wl.kv_chunk(w, layer, b, start, count, "k", DEV).unsqueeze(0)
        v = wl.kv_chunk(w, layer, b, start, count, "v", DEV).unsqueeze(0)
        cache.append(0, k, v, torch.zeros(1, dtype=torch.int32, device=DEV), None, nblk)
    return cache, nblk


CASES = [
    # head_dim, key, value, KV heads, GQA, q_len, tokens, shard cuts
    (128, ("prod", 3), ("mse", 3), 2, 8, 2, 5003, (0, 1700, 3333, 5003)),   # the long-context codecs
    (128, ("mse", 4), ("mse", 4), 2, 8, 2, 700, (0, 699, 700)),             # last shard shorter than q_len
    (128, ("prod", 3), ("group", 4, 64), 2, 4, 1, 900, (0, 0, 450, 900)),   # an empty shard
    (256, ("prod", 3), ("group", 2, 32), 2, 8, 1, 1000, (0, 600, 1000)),    # head_dim 256, group values
    (256, ("prod", 3), ("mse", 3), 2, 8, 2, 3000, (0, 1000, 3000)),         # head_dim 256, MSE values
    (256, ("prod", 2), ("group", 4, 64), 1, 4, 1, 800, (0, 400, 800)),      # head_dim 256 on the SIMT kernels
    (64, ("prod", 3), ("mse", 3), 2, 8, 2, 2000, (0, 900, 2000)),          # head_dim 64, MSE values
    (64, ("mse", 2), ("mse", 2), 2, 4, 1, 700, (0, 350, 700)),             # head_dim 64 on the SIMT kernels
    (128, ("prod", 3), ("mse", 3), 1, 8, 2, 160000, (0, 10000, 160000)),    # one head: a shard of > 128 splits
]


@pytest.mark.parametrize("D,key,value,Hkv,G,Lq,N,cuts", CASES)
def test_sharded_decode_equals_whole_decode(D, key, value, Hkv, G, Lq, N, cuts):
    kspec = wl._spec(key[0], key[1], 3)
    vspec = wl._spec(value[0], value[1], 4, value[2] if len(value) > 2 else 0)
    w = wl.Workload("sharded", 1, 1, Hkv, Hkv * G, D, (N,), Lq, torch.bfloat16, 1.0, 13, kspec, vspec,
                    block_tokens=64)
    kc = tq.Codec(D, kspec.bits, kspec.mode, kspec.seed, kspec.group_size)
    vc = tq.Codec(D, vspec.bits, vspec.mode, vspec.seed, vspec.group_size)
    q = wl.queries(w, 0, 0, DEV)
    Hq = Hkv * G
    # the whole sequence in one cache
    whole, nblk = _cache_of(w, 0, 0, 0, N, kc, vc)
    ws = torch.empty(whole.workspace_bytes(1, Hq, Lq, N), dtype=torch.uint8, device=DEV)
    ref_gpu = torch.empty(1, Hq, Lq, D, dtype=torch.float32, device=DEV)
    whole.decode(0, q, torch.tensor([N], dtype=torch.int32, device=DEV), None, nblk, N, ref_gpu, ws)
    # shards, each in a cache of its own
    P = len(cuts) - 1
    ml = torch.empty(P, 1, Hq, Lq, 2, dtype=torch.float32, device=DEV)
    acc = torch.empty(P, 1, Hq, Lq, D, dtype=torch.float32, device=DEV)
    caches = []
    for p, (s, e) in enumerate(zip(cuts[:-1], cuts[1:])):
        c = e - s
        cache, nb = _cache_of(w, 0, 0, s, c, kc, vc)
        caches.append(cache)
        msl = max(Lq, c)
        wsp = torch.empty(cache.workspace_bytes(1, Hq, Lq, msl), dtype=torch.uint8, device=DEV)
        cache.decode_partials(0, q, torch.tensor([c], dtype=torch.int32, device=DEV),
                              torch.tensor([N - s], dtype=torch.int32, device=DEV), None, nb, msl,
                              ml[p], acc[p], wsp)
    out = torch.empty(1, Hq, Lq, D, dtype=torch.float32, device=DEV)
    tq.tq_decode_merge(vc.handle, ml, acc, out)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    got, whole_out = to_f32_np(out), to_f32_np(ref_gpu)
    assert np.abs(got - whole_out).max() <= 1e-4 * max(1.0, np.abs(whole_out).max())
    # against the oracle: the whole decode, and each shard's state
    okc, ovc = oracle_codec(kspec, D), oracle_codec(vspec, D)
    qn = to_f32_np(q).astype(np.float64)
    mln, accn = to_f32_np(ml).astype(np.float64), to_f32_np(acc).astype(np.float64)
    K, V = raw_kv(w, 0, 0, N)
    for h in range(Hkv):
        rows = slice(h * G, (h + 1) * G)
        kr, vr = okc.encode(K[h]), ovc.encode(V[h])
        ref = O.decode_rotated(qn[0, rows], okc, kr, ovc, vr, 1 / math.sqrt(D), Lq)
        compare_decode(got[0, rows], ref)
        for p, (s, e) in enumerate(zip(cuts[:-1], cuts[1:])):
            m, l, a = O.decode_partial(qn[0, rows], okc, {k: v[s:e] for k, v in kr.items()}, ovc,
                                       {k: v[s:e] for k, v in vr.items()}, 1 / math.sqrt(D), Lq, N - s)
            gm, gl = mln[p, 0, rows, :, 0].reshape(-1), mln[p, 0, rows, :, 1].reshape(-1)
            ga = accn[p, 0, rows].reshape(-1, D)
            seen = l > 0
            assert np.array_equal(seen, gl > 0) and np.all(gm[~seen] == -np.inf) and not ga[~seen].any()
            if seen.any():
                lse, glse = m[seen] + np.log(l[seen]), gm[seen] + np.log(gl[seen])
                assert np.abs(glse - lse).max() <= 2e-3
                na, ga_n = a[seen] / l[seen, None], ga[seen] / gl[seen, None]
                assert np.abs(ga_n - na).max() <= 2e-3 * max(1.0, np.abs(na).max())


def test_sharded_decode_argument_errors():
    kc, vc = tq.Codec(128, 3, tq.TQ_MODE_PROD, 0), tq.Codec(128, 3, tq.TQ_MODE_MSE, 1)
    cache = tq.CompressedKVCache(kc, vc, 1, 4, 64, 1, DEV)
    q = torch.zeros(1, 8, 2, 128, dtype=torch.bfloat16, device=DEV)
    ml = torch.empty(1, 8, 2, 2, dtype=torch.float32, device=DEV)
    acc = torch.empty(1, 8, 2, 128, dtype=torch.float32, device=DEV)
    ws = torch.empty(cache.workspace_bytes(1, 8, 2, 64), dtype=torch.uint8, device=DEV)
    sl = torch.zeros(1, dtype=torch.int32, device=DEV)
    with pytest.raises(tq.TQError) as e:     # no partial-state buffers
        tq.tq_decode_partials(kc.handle, vc.handle, cache.desc, 0, q, sl, None, None, 4, 64, ml, None, ws)
    assert e.value.status == 1
    with pytest.raises(tq.TQError) as e:     # misaligned accumulator
        tq.tq_decode_partials(kc.handle, vc.handle, cache.desc, 0, q, sl, None, None, 4, 64, ml,
                              acc.view(-1)[1:], ws)
    assert e.value.status == 1
    out = torch.empty(16, 128, dtype=torch.float32, device=DEV)
    with pytest.raises(tq.TQError) as e:     # no parts
        tq._lib.check(tq.lib().tq_decode_merge(vc.handle, 0, ml.data_ptr(), acc.data_ptr(), 16, out.data_ptr(),
                                               None), "tq_decode_merge")
    assert e.value.status == 1

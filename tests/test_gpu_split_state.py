"""Split (low/high) states on the GPU through the C ABI: the two halves'
pools are bit-identical to the oracle's pool writes of each half's records,
and decode over the split state matches the oracle's decode of the same
records (dequantise each half, concatenate, attend) within the decode
tolerance."""
import math

import numpy as np
import pytest
import torch

import oracle as O
import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import compare_decode, to_f32_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


_MODES = {"mse": (tq.TQ_MODE_MSE, O.MSE), "prod": (tq.TQ_MODE_PROD, O.PROD), "group": (tq.TQ_MODE_GROUP, O.GROUP)}


def _codecs(D, spec, seed):
    mode, bits = spec[0], spec[1]
    group = spec[2] if len(spec) > 2 else 0
    g = tq.Codec(D, bits, _MODES[mode][0], seed, group)
    o = O.Codec(D, bits, _MODES[mode][1], seed, group)
    return g, o


CASES = [
    # low (D, key, value), high (D, key, value), KV heads, GQA, q_len, lengths, block tokens
    ((64, ("prod", 3), ("mse", 3)), (64, ("mse", 4), ("mse", 4)), 2, 8, 2, (700, 1333), 64),
    ((128, ("prod", 3), ("mse", 2)), (128, ("prod", 4), ("group", 4, 64)), 1, 4, 1, (2050,), 256),
    ((64, ("mse", 2), ("group", 2, 32)), (128, ("mse", 4), ("mse", 4)), 2, 4, 2, (513, 96, 1000), 16),
]


@pytest.mark.parametrize("low,high,Hkv,G,Lq,lens,BT", CASES)
def test_split_state_encode_and_decode(low, high, Hkv, G, Lq, lens, BT):
    DL, DH = low[0], high[0]
    D = DL + DH
    B = len(lens)
    kl, okl = _codecs(DL, low[1], 11)
    vl, ovl = _codecs(DL, low[2], 12)
    kh, okh = _codecs(DH, high[1], 21)
    vh, ovh = _codecs(DH, high[2], 22)
    w = wl.Workload("split", 1, B, Hkv, Hkv * G, D, tuple(lens), Lq, torch.bfloat16, 1.0, 17,
                    wl._spec("mse", 2), wl._spec("mse", 2), block_tokens=BT, shuffle_blocks=True)
    table, nblocks = wl.block_table(w, list(lens))
    max_blocks = table.shape[1]
    sc = tq.SplitCache(kl, vl, kh, vh, 1, nblocks, BT, Hkv, DEV, exact_encode=True)
    table_d = table.to(DEV)
    K = [wl.kv_chunk(w, 0, b, 0, n, "k", DEV) for b, n in enumerate(lens)]   # [Hkv, n, D]
    V = [wl.kv_chunk(w, 0, b, 0, n, "v", DEV) for b, n in enumerate(lens)]
    for b in range(B):
        k, v = K[b].unsqueeze(0), V[b].unsqueeze(0)
        sc.append(0, k[..., :DL].contiguous(), v[..., :DL].contiguous(), k[..., DL:].contiguous(),
                  v[..., DL:].contiguous(), torch.zeros(1, dtype=torch.int32, device=DEV),
                  table_d[b:b + 1].contiguous(), max_blocks)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    # pools: the oracle's records of each half at the same blocks
    for cache, okc, ovc, a, Dh in ((sc.low, okl, ovl, 0, DL), (sc.high, okh, ovh, DL, DH)):
        want = np.zeros(cache.pool.numel(), np.uint8)
        recs = {}
        for b in range(B):
            Kn, Vn = to_f32_np(K[b])[..., a:a + Dh], to_f32_np(V[b])[..., a:a + Dh]
            for h in range(Hkv):
                kr, vr = okc.encode(Kn[h]), ovc.encode(Vn[h])
                recs[(b, h)] = (kr, vr)
                O.pool_write(want, okc, ovc, Hkv, BT, table.numpy(), max_blocks, b, h, 0, kr, vr)
        assert np.array_equal(cache.pool.cpu().numpy(), want)
        cache.recs = recs
    # decode
    q = wl.queries(w, 0, 0, DEV)
    msl = max(lens)
    ws = torch.empty(sc.workspace_bytes(B, Hkv * G, Lq, msl), dtype=torch.uint8, device=DEV)
    out = torch.full((B, Hkv * G, Lq, D), float("nan"), dtype=torch.float32, device=DEV)
    sc.decode(0, q, torch.tensor(lens, dtype=torch.int32, device=DEV), table_d, max_blocks, msl, out, ws)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    got, qn = to_f32_np(out), to_f32_np(q).astype(np.float64)
    for b in range(B):
        for h in range(Hkv):
            lo_r, hi_r = sc.low.recs[(b, h)], sc.high.recs[(b, h)]
            ref = O.decode_split(qn[b, h * G:(h + 1) * G], (okl, lo_r[0], ovl, lo_r[1]),
                                 (okh, hi_r[0], ovh, hi_r[1]), 1 / math.sqrt(D), Lq)
            compare_decode(got[b, h * G:(h + 1) * G], ref)


def test_split_state_refuses_mismatched_halves():
    kl, vl = tq.Codec(64, 3, tq.TQ_MODE_PROD, 1), tq.Codec(64, 3, tq.TQ_MODE_MSE, 2)
    kh, vh = tq.Codec(64, 4, tq.TQ_MODE_MSE, 3), tq.Codec(64, 4, tq.TQ_MODE_MSE, 4)
    sc = tq.SplitCache(kl, vl, kh, vh, 1, 8, 16, 2, DEV)
    other = tq.CompressedKVCache(kh, vh, 1, 4, 16, 2, DEV)     # another block count
    sc.high = other
    q = torch.zeros(1, 8, 1, 128, dtype=torch.bfloat16, device=DEV)
    with pytest.raises(tq.TQError) as e:
        sc.workspace_bytes(1, 8, 1, 16)
    assert e.value.status == 3

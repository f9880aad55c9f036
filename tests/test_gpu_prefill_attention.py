"""Prefill attention over the compressed cache versus the oracle.

A chunk of q_len query positions, already appended, attends to its
sequence's compressed prefix and causally to itself; the oracle decodes its
own records of the same inputs (rotated-domain decode with q_len rows per
query head). Same tolerance as decode: max |gpu - oracle| <= 2e-3 and cosine
>= 0.9999 per output row.
"""
import numpy as np
import pytest
import torch

import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import GpuCase, compare_decode, oracle_decode, raw_kv, to_f32_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _run(key, value, lens, q_len, Hkv, G, BT, shuffle=False, scales=None, seed=31):
    kspec = wl._spec(key[0], key[1], 0)
    vspec = wl._spec(value[0], value[1], 1, value[2] if len(value) > 2 else 0)
    w = wl.Workload("prefill_attn", 1, len(lens), Hkv, Hkv * G, 128, tuple(lens), q_len, torch.bfloat16, 1.0,
                    seed, kspec, vspec, block_tokens=BT, shuffle_blocks=shuffle, append_per_step=0,
                    prefill_chunk=512, head_scale_range=scales)
    case = GpuCase(w, layers=[0])
    case.prefill()
    q = wl.queries(w, 0, 0, DEV)
    B = len(lens)
    ws = torch.empty(case.cache.prefill_workspace_bytes(B, w.num_q_heads, q_len), dtype=torch.uint8, device=DEV)
    out = torch.full((B, w.num_q_heads, q_len, 128), float("nan"), dtype=torch.float32, device=DEV)
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    case.cache.prefill_attention(0, q, sl, case.table_d, case.max_blocks, out, ws)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    out = to_f32_np(out)
    assert np.isfinite(out).all()
    qn = to_f32_np(q).astype(np.float64)
    for b in range(B):
        K, V = raw_kv(w, 0, b, lens[b], DEV)
        for h in range(Hkv):
            ref = oracle_decode(w, K[h], V[h], qn[b, h * G:(h + 1) * G])
            compare_decode(out[b, h * G:(h + 1) * G], ref)
    return case, q, out


@pytest.mark.parametrize("key,value,lens,q_len,Hkv,G,BT,shuffle", [
    # the long-context codecs: 700 cached + a 300-token chunk, GQA 8, 256-token blocks
    (("prod", 3), ("mse", 3), (1000,), 300, 2, 8, 256, False),
    # ragged chunk (not a multiple of 16), two sequences
    (("prod", 3), ("mse", 3), (1500, 777), 129, 2, 8, 64, False),
    # the paged-batch codecs: group values, 16-token blocks in a shuffled order, GQA 4
    (("prod", 3), ("group", 4, 64), (333, 1200, 90), 40, 2, 4, 16, True),
    # prod keys with 4-bit values, no GQA
    (("prod", 3), ("mse", 4), (640,), 200, 2, 1, 32, False),
    # the whole sequence is the chunk: causal self-attention only
    (("prod", 3), ("mse", 3), (256,), 256, 1, 8, 64, False),
    # degenerate chunks that decode also covers
    (("prod", 3), ("mse", 3), (900,), 1, 2, 8, 64, False),
    (("prod", 3), ("mse", 3), (900,), 2, 2, 8, 64, False),
])
def test_prefill_attention_matches_oracle(key, value, lens, q_len, Hkv, G, BT, shuffle):
    _run(key, value, lens, q_len, Hkv, G, BT, shuffle)


def test_prefill_attention_mse4_with_head_scales():
    # the 64-layer stack's codecs (4-bit MSE keys and values, per-head scales)
    _run(("mse", 4), ("mse", 4), (2048,), 384, 2, 8, 256, scales=(0.5, 2.0))


def test_prefill_equals_decode_for_short_chunks():
    # for q_len within decode's range the two entry points compute the same function
    case, q, out = _run(("prod", 3), ("mse", 3), (1200,), 2, 2, 8, 256)
    w = case.w
    dec = to_f32_np(case.decode(0, q))
    assert np.abs(dec - out).max() <= 1e-3


def test_prefill_attention_unsupported_codecs():
    kc, vc = tq.Codec(128, 4, tq.TQ_MODE_PROD, 0), tq.Codec(128, 2, tq.TQ_MODE_MSE, 1)
    cache = tq.CompressedKVCache(kc, vc, 1, 4, 16, 1, DEV)
    with pytest.raises(tq.TQError) as e:
        cache.prefill_workspace_bytes(1, 8, 32)
    assert e.value.status == 2


def test_prefill_attention_stress_vectors():
    # values with zero rows (zero norms), one-hot and constant rows and scales
    # 2^-12 .. 2^12 (value norms up to ~5e4: P' = p * norm must stay inside
    # fp16 while the running maximum lags by its gap); N(0, 1) keys (keys at
    # 2^12 would make the softmax an argmax whose near-ties the fp16 query
    # operand cannot resolve, whichever kernel computes it)
    w = wl.Workload("prefill_stress", 1, 1, 2, 16, 128, (700,), 300, torch.bfloat16, 1.0, 3,
                    wl._spec("prod", 3, 0), wl._spec("mse", 3, 1), block_tokens=64, append_per_step=0,
                    prefill_chunk=512)
    D, Hkv, N, Lq, G = 128, 2, 700, 300, 8
    K = wl.kv_chunk(w, 0, 0, 0, N, "k", DEV).unsqueeze(0)
    V = wl.encoder_stress(82, 1, Hkv, N, D, torch.bfloat16, DEV)
    case = GpuCase(w, layers=[0])
    zero = torch.zeros(1, dtype=torch.int32, device=DEV)
    case.cache.append(0, K, V, zero, case.table_d, case.max_blocks)
    q = wl.queries(w, 0, 0, DEV)
    ws = torch.empty(case.cache.prefill_workspace_bytes(1, w.num_q_heads, Lq), dtype=torch.uint8, device=DEV)
    out = torch.full((1, w.num_q_heads, Lq, D), float("nan"), dtype=torch.float32, device=DEV)
    sl = torch.tensor([N], dtype=torch.int32, device=DEV)
    case.cache.prefill_attention(0, q, sl, case.table_d, case.max_blocks, out, ws)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    out = to_f32_np(out)
    assert np.isfinite(out).all()
    qn = to_f32_np(q).astype(np.float64)
    Kn, Vn = to_f32_np(K[0]), to_f32_np(V[0])
    for h in range(Hkv):
        ref = oracle_decode(w, Kn[h], Vn[h], qn[0, h * G:(h + 1) * G]).reshape(-1, D)
        got = out[0, h * G:(h + 1) * G].reshape(-1, D).astype(np.float64)
        scale = max(1.0, float(np.abs(ref).max()))
        assert np.abs(got - ref).max() / scale <= 2e-3
        # rows whose weight sits on a zero or 2^-100 value are zero to fp32
        live = np.linalg.norm(ref, axis=-1) > 1e-3 * scale
        assert live.sum() >= len(live) // 2
        compare_decode(got[live] / scale, ref[live] / scale)

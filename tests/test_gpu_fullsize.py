"""Decode parity at the workloads' full sizes.

The long-context case runs in the decode launch configuration the benchmark
times (262,144 cached tokens, 256-token blocks, contiguous cache with no block
table, prefill in 8192-token chunks, a 2-token append through the
short-append kernel, then query length 2). The oracle cannot decode every
output at these sizes in seconds, so each test compares sampled (sequence, KV
head) outputs element by element against the oracle's decode of its own
records, and checks the rest by properties that hold at any size (the device
error word stays clear, every output is finite).

Most caches are written with the exact encode policy, so the GPU and the
oracle decode identical records and the comparison measures the decode alone
(the tensor-core prefill may differ from the oracle's codes inside the fp32
tie band, which tests/test_gpu_encode_tc.py checks on its own). The benchmark
itself prefills with the tensor-core encoder: its test reads the records the
GPU wrote back to the host and holds the GPU decode of them to the decode
tolerance against the oracle's decode of the same records.
"""
import numpy as np
import pytest
import torch

import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
import oracle as O
from parity_util import GpuCase, compare_decode, oracle_codec, oracle_decode, read_records_blocks, to_f32_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _head_kv(w, layer, seq, n, h):
    """Raw K, V [n, D] (float32) of one head, regenerated from the seeded chunks."""
    k = wl.kv_chunk(w, layer, seq, 0, n, "k", DEV)[h]
    v = wl.kv_chunk(w, layer, seq, 0, n, "v", DEV)[h]
    return to_f32_np(k), to_f32_np(v)


def _long_context_cache(layer, exact_encode):
    """One layer of the 256k workload, prefilled in 8192-token chunks and
    grown by one 2-token append, as the benchmark builds it."""
    w = wl.long_256k()
    D, Hkv, Hq, Lq, BT = w.head_dim, w.num_kv_heads, w.num_q_heads, w.q_len, w.block_tokens
    N0, A, C = w.seq_lens[0], w.append_per_step, w.prefill_chunk
    cap = N0 + A
    nblk = (cap + BT - 1) // BT
    kc = tq.Codec(D, w.key.bits, w.key.mode, w.key.seed)
    vc = tq.Codec(D, w.value.bits, w.value.mode, w.value.seed)
    cache = tq.CompressedKVCache(kc, vc, 1, nblk, BT, Hkv, DEV, exact_encode=exact_encode)
    starts = torch.arange(0, N0, C, dtype=torch.int32, device=DEV)
    for c in range(N0 // C):
        k = wl.kv_chunk(w, layer, 0, c * C, C, "k", DEV).unsqueeze(0)
        v = wl.kv_chunk(w, layer, 0, c * C, C, "v", DEV).unsqueeze(0)
        cache.append(0, k, v, starts[c:c + 1], None, nblk)
    kn = wl.kv_chunk(w, layer, 0, N0, A, "k", DEV).unsqueeze(0)
    vn = wl.kv_chunk(w, layer, 0, N0, A, "v", DEV).unsqueeze(0)
    cache.append(0, kn, vn, torch.tensor([N0], dtype=torch.int32, device=DEV), None, nblk)
    q = wl.queries(w, layer, 0, DEV)
    sl = torch.tensor([cap], dtype=torch.int32, device=DEV)
    ws = torch.empty(cache.workspace_bytes(1, Hq, Lq, cap), dtype=torch.uint8, device=DEV)
    out = torch.empty(1, Hq, Lq, D, dtype=torch.float32, device=DEV)
    cache.decode(0, q, sl, None, nblk, cap, out, ws)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    out = to_f32_np(out)
    assert np.isfinite(out).all()
    return w, cache, nblk, cap, to_f32_np(q).astype(np.float64), out


def test_long_context_full_size_bench_configuration():
    layer = 37
    w, cache, nblk, cap, qn, out = _long_context_cache(layer, exact_encode=True)
    G = w.gqa
    for h in (0, 5):
        K, V = _head_kv(w, layer, 0, cap, h)
        ref = oracle_decode(w, K, V, qn[0, h * G:(h + 1) * G])
        compare_decode(out[0, h * G:(h + 1) * G], ref)


def test_long_context_tensor_core_prefill_decode_tolerance():
    # the benchmark's own composition: prefill on the tensor-core encoder
    # (the default policy), then decode; the oracle decodes the records the
    # GPU wrote, so every difference left is the decode's
    layer = 11
    w, cache, nblk, cap, qn, out = _long_context_cache(layer, exact_encode=False)
    assert cache.desc.encode_policy == tq.TQ_ENCODE_AUTO
    kc, vc = oracle_codec(w.key, w.head_dim), oracle_codec(w.value, w.head_dim)
    pool = cache.pool.cpu().numpy()
    G = w.gqa
    for h in (0, 3, 6):
        krec, vrec = read_records_blocks(pool, kc, vc, w.num_kv_heads, w.block_tokens, None, nblk, 0, h, cap)
        ref = O.decode_rotated(qn[0, h * G:(h + 1) * G], kc, krec, vc, vrec, 1 / np.sqrt(w.head_dim), w.q_len)
        compare_decode(out[0, h * G:(h + 1) * G], ref)


def test_stack_32k_full_size_all_heads():
    # 32,768 tokens, 4-bit MSE keys and values, per-head scales, q_len 2
    w = wl.stack_32k()
    layer = 17
    case = GpuCase(w, layers=[layer])
    case.prefill()
    assert tq.tq_device_error() == 0
    q = wl.queries(w, layer, 0, DEV)
    out = to_f32_np(case.decode(0, q))
    assert np.isfinite(out).all()
    qn = to_f32_np(q).astype(np.float64)
    G = w.gqa
    for h in range(w.num_kv_heads):
        K, V = _head_kv(w, layer, 0, case.seq_lens[0], h)
        compare_decode(out[0, h * G:(h + 1) * G], oracle_decode(w, K, V, qn[0, h * G:(h + 1) * G]))


def test_paged_batch_full_size_sampled_sequences():
    # 32 ragged sequences (4k..64k tokens) in 16-token blocks handed out in a
    # shuffled order; one batched append of a token per sequence, then one
    # batched decode step with q_len 1
    w = wl.paged_batch()
    layer = 3
    case = GpuCase(w, layers=[layer])
    case.prefill()
    B = w.batch
    k = torch.stack([wl.kv_chunk(w, layer, b, w.seq_lens[b], 1, "k", DEV) for b in range(B)])
    v = torch.stack([wl.kv_chunk(w, layer, b, w.seq_lens[b], 1, "v", DEV) for b in range(B)])
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
    case.cache.append(0, k, v, sl, case.table_d, case.max_blocks)
    case.seq_lens = [n + 1 for n in w.seq_lens]
    q = wl.queries(w, layer, 0, DEV)
    out = to_f32_np(case.decode(0, q))
    assert tq.tq_device_error() == 0
    assert np.isfinite(out).all()
    qn = to_f32_np(q).astype(np.float64)
    G = w.gqa
    for b in (0, 13, 31):
        for h in (0, 7):
            K, V = _head_kv(w, layer, b, case.seq_lens[b], h)
            compare_decode(out[b, h * G:(h + 1) * G], oracle_decode(w, K, V, qn[b, h * G:(h + 1) * G]))

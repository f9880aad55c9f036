"""Decode parity at the edges of the decode's tiling.

Token counts around the 64-token tiles and 128-token blocks (only the query
positions, a tile minus one, exactly one tile, one over) for every codec pair
of the prefill kernels, 128- to 512-token blocks in a shuffled order, causal
query lengths above one, more than 16 query rows (two row groups), a sequence
long enough for many token splits (past one merge chunk), head_dims 64 and 256
on the tensor-core path (64 in the head_dim-128 layout, 256 as two 128-column
value halves per unit), up to 8 query rows per KV head (the transposed
kernel), per-head scales, and inputs with zero,
tiny and one-hot vectors (zero-norm values, zero keys). Every output row is
compared with the oracle's decode of the same raw inputs (the max abs error
and cosine bounds of the decode parity rule); the last case checks that two
block sizes of one cache decode alike.
"""
import dataclasses
import math

import numpy as np
import pytest
import torch

import oracle as O
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


def _workload(key, value, lens, Lq, Hkv, G, bt, shuffle=False, scales=None, seed=5, D=128):
    kspec = wl._spec(key[0], key[1], 21)
    vspec = wl._spec(value[0], value[1], 22, value[2] if len(value) > 2 else 0)
    return wl.Workload("decode_tc", 1, len(lens), Hkv, Hkv * G, D, tuple(lens), Lq, torch.bfloat16, 1.0,
                       seed, kspec, vspec, block_tokens=bt, shuffle_blocks=shuffle, append_per_step=0,
                       prefill_chunk=1024, head_scale_range=scales)


def _check(w):
    case = GpuCase(w, layers=[0])
    case.prefill()
    q = wl.queries(w, 0, 0, DEV)
    out = to_f32_np(case.decode(0, q))
    assert tq.tq_device_error() == 0
    assert np.isfinite(out).all()
    qn = to_f32_np(q).astype(np.float64)
    G = w.gqa
    for b in range(w.batch):
        K, V = raw_kv(w, 0, b, w.seq_lens[b], DEV)
        for h in range(w.num_kv_heads):
            compare_decode(out[b, h * G:(h + 1) * G], oracle_decode(w, K[h], V[h], qn[b, h * G:(h + 1) * G]))


@pytest.mark.parametrize("key,value", [(("prod", 3), ("mse", 3)), (("prod", 3), ("mse", 4)),
                                       (("prod", 3), ("group", 4, 64)), (("mse", 4), ("mse", 4))])
def test_tile_edges_every_codec_pair(key, value):
    # one sequence per tile edge (the shortest holds just the
    # two query positions), GQA 8
    _check(_workload(key, value, (2, 127, 128, 129, 700), 2, 2, 8, 128))


@pytest.mark.parametrize("bt", [16, 32, 128, 256, 512])
def test_block_sizes_shuffled_pages(bt):
    _check(_workload(("prod", 3), ("mse", 3), (300, 1000, 2049), 1, 2, 4, bt, shuffle=True))


def test_two_row_groups_causal():
    # G 8 x q_len 4 = 32 rows per KV head; the newest 4 tokens are causal
    _check(_workload(("prod", 3), ("mse", 3), (513, 1280), 4, 2, 8, 256))


def test_many_splits_long_sequence():
    # one KV head: the plan spreads 40,000 tokens over many token splits
    _check(_workload(("prod", 3), ("mse", 3), (40000,), 2, 1, 8, 256))


def test_splits_beyond_one_merge_chunk():
    # one KV head at 150,000 tokens: more than 128 token splits, so the merge
    # goes past the 32 splits whose loads it issues at once and past its first
    # chunk of 128 split weights
    w = _workload(("prod", 3), ("mse", 3), (150000,), 2, 1, 8, 256)
    case = GpuCase(w, layers=[0])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    plan = tq.tq_decode_plan(case.cache.desc, 1, w.num_q_heads, w.q_len, w.seq_lens[0], sms)
    assert plan["splits"] > 128, plan
    case.prefill()
    q = wl.queries(w, 0, 0, DEV)
    out = to_f32_np(case.decode(0, q))
    assert tq.tq_device_error() == 0
    qn = to_f32_np(q).astype(np.float64)
    K, V = raw_kv(w, 0, 0, w.seq_lens[0], DEV)
    compare_decode(out[0], oracle_decode(w, K[0], V[0], qn[0]))


def _plan(w):
    case = GpuCase(w, layers=[0])
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    return case, tq.tq_decode_plan(case.cache.desc, w.batch, w.num_q_heads, w.q_len, max(w.seq_lens), sms)


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("key,value", [(("prod", 3), ("group", 2, 32)), (("prod", 3), ("mse", 3)),
                                       (("prod", 3), ("group", 2, 64)), (("prod", 3), ("group", 4, 64)),
                                       (("prod", 3), ("mse", 4)), (("mse", 4), ("mse", 4))])
def test_head_dim_64_256_tile_edges(D, key, value):
    # every codec pair of the tensor-core kernels at head_dim 64 (the
    # head_dim-128 layout, 64-token tiles) and 256 (two value halves, 32-token
    # tiles): sequences around the tiles, 64-token blocks, q_len 2 x GQA 8
    w = _workload(key, value, (2, 31, 32, 33, 63, 64, 65, 700), 2, 2, 8, 64, D=D)
    _, plan = _plan(w)
    assert plan["tensor_cores"] == 1, plan
    _check(w)


def test_head_dim_64_many_splits_shuffled_small_blocks():
    # one KV head over 30000 tokens in 16-token blocks (four per stage) in a
    # shuffled order, 32 rows (two row groups)
    w = _workload(("prod", 3), ("mse", 3), (30000, 777), 4, 1, 8, 16, shuffle=True, D=64)
    _, plan = _plan(w)
    assert plan["tensor_cores"] == 1 and plan["splits"] > 32, plan
    _check(w)


def test_head_dim_256_two_row_groups_shuffled():
    # 32 rows per KV head (two row groups), 16-token blocks in a shuffled order
    w = _workload(("prod", 3), ("mse", 3), (513, 1280), 4, 2, 8, 16, shuffle=True, D=256)
    _check(w)


def test_head_dim_256_many_splits():
    # one KV head: more splits than the merge loads at once
    w = _workload(("prod", 3), ("group", 2, 32), (20000,), 1, 1, 8, 256, D=256)
    _, plan = _plan(w)
    assert plan["tensor_cores"] == 1 and plan["splits"] > 32, plan
    _check(w)


@pytest.mark.parametrize("key,value", [(("prod", 3), ("group", 4, 64)), (("prod", 3), ("group", 2, 32)),
                                       (("prod", 3), ("mse", 3)), (("prod", 3), ("mse", 4)), (("mse", 4), ("mse", 4))])
@pytest.mark.parametrize("G,Lq", [(1, 1), (4, 1), (2, 3), (4, 2), (8, 1)])
def test_few_rows_transposed_kernel(key, value, G, Lq):
    # at most 8 query rows per KV head: the split kernel's transposed form
    # (tokens on the MMA's M, rows on N), causal for q_len > 1, around the tiles
    w = _workload(key, value, (3, 31, 64, 65, 700), Lq, 2, G, 64)
    _, plan = _plan(w)
    assert plan["tensor_cores"] == 1 and plan["transposed"] == 1, plan
    _check(w)


@pytest.mark.parametrize("G,Lq,bt", [(8, 2, 16), (4, 1, 16), (8, 2, 256), (4, 1, 64)])
def test_splits_with_partial_warp_rounds(G, Lq, bt):
    # The 12 warps of a split take its tiles in turn; sequence lengths whose
    # splits end in a partial round (some warps a tile short), a lone partial
    # tile and a split of two tokens; 16-token blocks in a shuffled order (a
    # tile gathers several blocks); 16 query rows per KV head (the 16-row
    # form) or 4 (transposed)
    w = _workload(("prod", 3), ("mse", 3), (20000, 1000, 150, 2), Lq, 2, G, bt, shuffle=True)
    _, plan = _plan(w)
    assert plan["tensor_cores"] == 1 and plan["transposed"] == (1 if G * Lq <= 8 else 0), plan
    tile, chunk = plan["tile_tokens"], plan["chunk_tokens"]
    tiles = {-(-min(chunk, n - t0) // tile) for n in w.seq_lens for t0 in range(0, n, chunk)}
    assert any(t % 12 for t in tiles) and 1 in tiles, (plan, tiles)
    _check(w)


def test_head_scales_mse4():
    _check(_workload(("mse", 4), ("mse", 4), (5000,), 2, 2, 8, 256, scales=(0.5, 2.0)))


def test_group_values_one_query_row_per_head():
    _check(_workload(("prod", 3), ("group", 4, 64), (129, 3000), 1, 2, 1, 128, shuffle=True))


@pytest.mark.parametrize("key,value", [(("prod", 3), ("mse", 3)), (("mse", 4), ("mse", 4)), (("mse", 2), ("mse", 3))])
def test_stress_vectors(key, value):
    # keys and values with zero rows (zero norms), one-hot rows, constant rows
    # and scales 2^-12 .. 2^12: the decode of those records against the oracle's
    w = _workload(key, value, (900,), 2, 2, 4, 256)
    D, Hkv, N = w.head_dim, w.num_kv_heads, w.seq_lens[0]
    K = wl.encoder_stress(71, 1, Hkv, N, D, torch.bfloat16, DEV)
    V = wl.encoder_stress(72, 1, Hkv, N, D, torch.bfloat16, DEV)
    case = GpuCase(w, layers=[0])
    zero = torch.zeros(1, dtype=torch.int32, device=DEV)
    case.cache.append(0, K, V, zero, case.table_d, case.max_blocks)
    torch.cuda.synchronize()
    q = wl.queries(w, 0, 0, DEV)
    out = to_f32_np(case.decode(0, q))
    assert tq.tq_device_error() == 0
    assert np.isfinite(out).all()
    qn = to_f32_np(q).astype(np.float64)
    Kn, Vn = to_f32_np(K[0]), to_f32_np(V[0])
    G = w.gqa
    for h in range(Hkv):
        ref = oracle_decode(w, Kn[h], Vn[h], qn[0, h * G:(h + 1) * G]).reshape(-1, D)
        got = out[0, h * G:(h + 1) * G].reshape(-1, D).astype(np.float64)
        # value rows at 2^12 make outputs of that magnitude: compare relative to it
        scale = max(1.0, float(np.abs(ref).max()))
        assert np.abs(got - ref).max() / scale <= 2e-3
        # 2^12-scaled keys concentrate a row's weight on one token, whose value
        # may be a zero or 2^-100 vector: such rows are zero to fp32, and a
        # cosine says nothing about them; every other row meets the bound
        norm = np.linalg.norm(ref, axis=-1)
        live = norm > 1e-3 * scale
        assert live.sum() >= len(live) // 2
        compare_decode(got[live] / scale, ref[live] / scale)


def test_block_size_does_not_change_the_result():
    # the same tokens cached in 128-token and in 64-token blocks decode alike
    # (the token splits and block lookups differ)
    w = _workload(("prod", 3), ("mse", 3), (1500,), 2, 2, 8, 128)
    case = GpuCase(w, layers=[0])
    case.prefill()
    q = wl.queries(w, 0, 0, DEV)
    out_tc = to_f32_np(case.decode(0, q))
    w64 = dataclasses.replace(w, block_tokens=64)
    case64 = GpuCase(w64, layers=[0])
    case64.prefill()
    out_mma = to_f32_np(case64.decode(0, q))
    assert tq.tq_device_error() == 0
    assert np.abs(out_tc - out_mma).max() <= 2e-3

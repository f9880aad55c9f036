"""tq_decode_step (append + decode attention in one call) on the GPU.

Against the two calls it stands for (tq_encode_append, then
tq_decode_attention over the grown sequences): the same cache bytes and the
same output bits, for the fused launch (rotated codecs, head_dim 128,
n_new <= 8) and for the paths that run the two calls in order. Against the
oracle: the outputs of the fused step, from the raw inputs.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import _lib
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import GpuCase, compare_decode, oracle_decode, raw_kv, to_f32_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _workload(key, value, D=128, lens=(37, 100, 16, 3), n_new=2, Lq=2, G=4, Hkv=2, bt=16):
    kspec = wl._spec(key[0], key[1], 11)
    vspec = wl._spec(value[0], value[1], 12, value[2] if len(value) > 2 else 0)
    return wl.Workload("decode_step", 2, len(lens), Hkv, Hkv * G, D, tuple(lens), Lq, torch.bfloat16, 1.0, 99,
                       kspec, vspec, block_tokens=bt, shuffle_blocks=True, append_per_step=n_new,
                       prefill_chunk=64)


def _run(w, fused_call: bool):
    """Prefill two layers, then one step per layer; returns the case and the outputs."""
    case = GpuCase(w, [0, 3])
    case.prefill()
    B, n_new = w.batch, w.append_per_step
    msl = max(w.seq_lens) + n_new
    outs = []
    for li, layer in enumerate(case.layers):
        k = torch.stack([wl.kv_chunk(w, layer, b, w.seq_lens[b], n_new, "k", DEV) for b in range(B)])
        v = torch.stack([wl.kv_chunk(w, layer, b, w.seq_lens[b], n_new, "v", DEV) for b in range(B)])
        q = wl.queries(w, layer, 0, DEV)
        sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
        ws = torch.empty(case.cache.workspace_bytes(B, w.num_q_heads, w.q_len, msl), dtype=torch.uint8,
                         device=DEV)
        out = torch.full((B, w.num_q_heads, w.q_len, w.head_dim), float("nan"), dtype=torch.float32, device=DEV)
        if fused_call:
            case.cache.decode_step(li, k, v, q, sl, case.table_d, case.max_blocks, msl, out, ws)
        else:
            case.cache.append(li, k, v, sl, case.table_d, case.max_blocks)
            case.cache.decode(li, q, sl + n_new, case.table_d, case.max_blocks, msl, out, ws)
        outs.append(out)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    return case, outs


CASES = [
    # fused: one launch for the append and the query prep
    pytest.param(("prod", 3), ("mse", 3), 128, (37, 100, 16, 3), 2, 2, 4, id="prod3-mse3-fused"),
    pytest.param(("mse", 4), ("mse", 4), 128, (37, 100, 16, 3), 2, 2, 4, id="mse4-mse4-fused"),
    pytest.param(("prod", 2), ("mse", 2), 128, (70, 5), 1, 1, 8, id="prod2-mse2-fused-q1"),
    pytest.param(("prod", 4), ("mse", 4), 128, (0, 129, 64), 5, 5, 4, id="prod4-mse4-fused-nv8-empty-seq"),
    pytest.param(("prod", 3), ("mse", 3), 128, (300, 17, 64), 8, 8, 8, id="prod3-mse3-fused-n8-64rows"),
    pytest.param(("mse", 2), ("mse", 3), 128, (1000, 48), 2, 2, 8, id="mse2-mse3-fused-quad-pair"),
    # the two calls in order
    pytest.param(("prod", 3), ("group", 4, 64), 128, (37, 100, 16, 3), 2, 2, 4, id="group-values-unfused"),
    pytest.param(("prod", 3), ("mse", 3), 128, (37, 100), 12, 2, 4, id="n12-unfused"),
    pytest.param(("prod", 3), ("mse", 3), 64, (37, 100), 2, 2, 4, id="d64-unfused"),
    pytest.param(("prod", 3), ("group", 2, 32), 256, (37, 100, 5), 2, 2, 8, id="d256-group2-unfused"),
    pytest.param(("prod", 3), ("mse", 3), 256, (70, 300), 1, 1, 8, id="d256-mse3-unfused"),
]


@pytest.mark.parametrize("key,value,D,lens,n_new,Lq,G", CASES)
def test_decode_step_equals_append_then_decode(key, value, D, lens, n_new, Lq, G):
    w = _workload(key, value, D=D, lens=lens, n_new=n_new, Lq=Lq, G=G)
    case_a, out_a = _run(w, fused_call=False)
    case_b, out_b = _run(w, fused_call=True)
    assert torch.equal(case_a.cache.pool, case_b.cache.pool), "cache bytes differ"
    for a, b in zip(out_a, out_b):
        assert not torch.isnan(b).any()
        assert torch.equal(a, b), f"outputs differ: max {float((a - b).abs().max()):.3e}"


@pytest.mark.parametrize("key,value,lens,n_new,G", [
    (("prod", 3), ("mse", 3), (37, 300, 3), 2, 8),
    (("mse", 4), ("mse", 4), (1, 64), 5, 4),
])
def test_decode_step_matches_oracle(key, value, lens, n_new, G):
    w = _workload(key, value, lens=lens, n_new=n_new, Lq=n_new, G=G)
    case, outs = _run(w, fused_call=True)
    for li, layer in enumerate(case.layers):
        q = wl.queries(w, layer, 0, DEV)
        qn = to_f32_np(q).astype(np.float64)
        out = to_f32_np(outs[li])
        for b in range(w.batch):
            K, V = raw_kv(w, layer, b, w.seq_lens[b] + n_new, DEV)
            for h in range(w.num_kv_heads):
                ref = oracle_decode(w, K[h], V[h], qn[b, h * G:(h + 1) * G])
                compare_decode(out[b, h * G:(h + 1) * G], ref)


def test_decode_step_argument_errors():
    w = _workload(("prod", 3), ("mse", 3))
    case = GpuCase(w, [0])
    B = w.batch
    k = torch.zeros(B, w.num_kv_heads, 2, w.head_dim, dtype=torch.bfloat16, device=DEV)
    q = torch.zeros(B, w.num_q_heads, 2, w.head_dim, dtype=torch.bfloat16, device=DEV)
    sl = torch.tensor(w.seq_lens, dtype=torch.int32, device=DEV)
    out = torch.empty(B, w.num_q_heads, 2, w.head_dim, dtype=torch.float32, device=DEV)
    msl = max(w.seq_lens) + 2
    need = case.cache.workspace_bytes(B, w.num_q_heads, 2, msl)
    small = torch.empty(max(need - 256, 256), dtype=torch.uint8, device=DEV)
    with pytest.raises(tq.TQError) as e:
        case.cache.decode_step(0, k, k, q, sl, case.table_d, case.max_blocks, msl, out, small)
    assert e.value.status == _lib.TQ_ERR_CAPACITY
    ws = torch.empty(need, dtype=torch.uint8, device=DEV)
    with pytest.raises(tq.TQError) as e:
        case.cache.decode_step(5, k, k, q, sl, case.table_d, case.max_blocks, msl, out, ws)
    assert e.value.status == _lib.TQ_ERR_INVALID_ARG
    # n_new = 0: a plain decode over the cache as it is
    case.prefill()
    z = torch.zeros(B, w.num_kv_heads, 0, w.head_dim, dtype=torch.bfloat16, device=DEV)
    case.cache.decode_step(0, z, z, q, sl, case.table_d, case.max_blocks, msl, out, ws)
    ref = case.decode(0, q, msl)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert tq.tq_device_error() == 0

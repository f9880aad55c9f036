"""Batch cache operations on the paged layout (block copies + block tables).

merge / extend copy sequences' blocks into a batch pool and add table rows,
extract copies one sequence's blocks into a cache of its own, filter keeps a
subset of table rows. Expected pools are written by the oracle from its own
records of the same inputs (bit-exact); decode over the merged or filtered
batch is compared with decode over the original caches.
"""
import numpy as np
import pytest
import torch

import oracle as O
import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import raw_kv, to_f32_np

pytestmark = pytest.mark.gpu

DEV = "cuda"
D, HKV, BT, G = 128, 2, 16, 4


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _workload(lens, key=("prod", 3), value=("mse", 3)):
    return wl.Workload("cache_ops", 2, len(lens), HKV, HKV * G, D, tuple(lens), 1, torch.bfloat16, 1.0, 77,
                       wl._spec(key[0], key[1], 5), wl._spec(value[0], value[1], 6), block_tokens=BT,
                       prefill_chunk=64)


def _single_cache(w, b, kc, vc):
    """Sequence b of w alone in a contiguous cache (identity table), 2 layers."""
    n = w.seq_lens[b]
    nblk = (n + BT - 1) // BT
    cache = tq.CompressedKVCache(kc, vc, w.num_layers, nblk, BT, HKV, DEV, exact_encode=True)
    zero = torch.zeros(1, dtype=torch.int32, device=DEV)
    for layer in range(w.num_layers):
        k = wl.kv_chunk(w, layer, b, 0, n, "k", DEV).unsqueeze(0)
        v = wl.kv_chunk(w, layer, b, 0, n, "v", DEV).unsqueeze(0)
        cache.append(layer, k, v, zero, None, nblk)
    return cache, nblk


def _decode(cache, w, layer, q, lens, table, max_blocks):
    sl = torch.tensor(lens, dtype=torch.int32, device=DEV)
    msl = max(lens)
    ws = torch.empty(cache.workspace_bytes(len(lens), w.num_q_heads, 1, msl), dtype=torch.uint8, device=DEV)
    out = torch.empty(len(lens), w.num_q_heads, 1, D, dtype=torch.float32, device=DEV)
    cache.decode(layer, q, sl, table, max_blocks, msl, out, ws)
    torch.cuda.synchronize()
    return to_f32_np(out)


def test_merge_extract_filter_extend():
    w = _workload((37, 100, 16))
    kc, vc = tq.Codec(D, 3, tq.TQ_MODE_PROD, 5), tq.Codec(D, 3, tq.TQ_MODE_MSE, 6)
    singles = [_single_cache(w, b, kc, vc) for b in range(w.batch)]

    # merge: every sequence's blocks into one pool, handed out in a shuffled order
    nblk = [n for _, n in singles]
    total = sum(nblk)
    max_blocks = max(nblk)
    g = torch.Generator().manual_seed(3)
    phys = torch.randperm(total, generator=g).to(torch.int32)
    table = torch.zeros(w.batch, max_blocks, dtype=torch.int32)
    batch = tq.CompressedKVCache(kc, vc, w.num_layers, total, BT, HKV, DEV)
    o = 0
    for b, (cache, n) in enumerate(singles):
        table[b, :n] = phys[o:o + n]
        batch.copy_blocks_from(cache, torch.arange(n, dtype=torch.int32, device=DEV), phys[o:o + n].to(DEV))
        o += n
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0

    # the merged pool equals the oracle's pool of the same records at those blocks
    okc, ovc = O.Codec(D, 3, O.PROD, 5), O.Codec(D, 3, O.MSE, 6)
    layer_bytes = batch.desc.layer_stride
    got = batch.pool.cpu().numpy()
    for layer in range(w.num_layers):
        want = np.zeros(layer_bytes, np.uint8)
        for b in range(w.batch):
            K, V = raw_kv(w, layer, b, w.seq_lens[b], DEV)
            for h in range(HKV):
                O.pool_write(want, okc, ovc, HKV, BT, table.numpy(), max_blocks, b, h, 0,
                             okc.encode(K[h]), ovc.encode(V[h]))
        assert np.array_equal(got[layer * layer_bytes:(layer + 1) * layer_bytes], want)

    # decode over the batch equals decode over each original cache
    q = wl.queries(w, 1, 0, DEV)
    table_d = table.to(DEV)
    merged = _decode(batch, w, 1, q, list(w.seq_lens), table_d, max_blocks)
    for b, (cache, n) in enumerate(singles):
        alone = _decode(cache, w, 1, q[b:b + 1].contiguous(), [w.seq_lens[b]], None, n)
        assert np.abs(merged[b] - alone[0]).max() <= 1e-5

    # filter: keep sequences 2 and 0 (table rows only, no copy)
    keep = [2, 0]
    sub = _decode(batch, w, 1, q[keep].contiguous(), [w.seq_lens[b] for b in keep],
                  table[keep].contiguous().to(DEV), max_blocks)
    for i, b in enumerate(keep):
        assert np.abs(sub[i] - merged[b]).max() <= 1e-5

    # extract: sequence 1 back into a cache of its own, identical bytes
    n1 = nblk[1]
    alone = tq.CompressedKVCache(kc, vc, w.num_layers, n1, BT, HKV, DEV)
    alone.copy_blocks_from(batch, table[1, :n1].to(DEV), torch.arange(n1, dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert torch.equal(alone.pool, singles[1][0].pool)

    # extend: a second batch's sequences appended into spare blocks of a larger pool
    w2 = _workload((50,))
    other, n_o = _single_cache(w2, 0, kc, vc)
    big = tq.CompressedKVCache(kc, vc, w.num_layers, total + n_o, BT, HKV, DEV)
    big.copy_blocks_from(batch, torch.arange(total, dtype=torch.int32, device=DEV),
                         torch.arange(total, dtype=torch.int32, device=DEV))
    big.copy_blocks_from(other, torch.arange(n_o, dtype=torch.int32, device=DEV),
                         torch.arange(total, total + n_o, dtype=torch.int32, device=DEV))
    mb = max(max_blocks, n_o)
    table2 = torch.zeros(w.batch + 1, mb, dtype=torch.int32)
    table2[:w.batch, :max_blocks] = table
    table2[w.batch, :n_o] = torch.arange(total, total + n_o, dtype=torch.int32)
    q2 = torch.cat([q, wl.queries(w2, 1, 0, DEV)])
    ext = _decode(big, w, 1, q2, list(w.seq_lens) + [50], table2.to(DEV), mb)
    assert np.abs(ext[:w.batch] - merged).max() <= 1e-5
    assert np.abs(ext[w.batch] - _decode(other, w2, 1, q2[w.batch:].contiguous(), [50], None, n_o)[0]).max() <= 1e-5
    assert tq.tq_device_error() == 0


def test_copy_refuses_mixed_configurations():
    kc, vc = tq.Codec(D, 3, tq.TQ_MODE_PROD, 5), tq.Codec(D, 3, tq.TQ_MODE_MSE, 6)
    kc2 = tq.Codec(D, 3, tq.TQ_MODE_PROD, 9)   # another seed
    a = tq.CompressedKVCache(kc, vc, 1, 4, BT, HKV, DEV)
    b = tq.CompressedKVCache(kc2, vc, 1, 4, BT, HKV, DEV)
    ids = torch.arange(2, dtype=torch.int32, device=DEV)
    with pytest.raises(tq.TQError) as e:
        b.copy_blocks_from(a, ids, ids)
    assert e.value.status == 3


def test_copy_flags_out_of_range_blocks():
    kc, vc = tq.Codec(D, 3, tq.TQ_MODE_PROD, 5), tq.Codec(D, 3, tq.TQ_MODE_MSE, 6)
    a = tq.CompressedKVCache(kc, vc, 1, 4, BT, HKV, DEV)
    b = tq.CompressedKVCache(kc, vc, 1, 4, BT, HKV, DEV)
    b.pool.fill_(7)
    before = b.pool.clone()
    b.copy_blocks_from(a, torch.tensor([0, 9], dtype=torch.int32, device=DEV),
                       torch.tensor([5, 1], dtype=torch.int32, device=DEV))
    torch.cuda.synchronize()
    assert tq.tq_device_error() & tq._lib.TQ_DEVERR_BLOCK
    assert torch.equal(b.pool, before)       # both pairs had an id out of range: nothing written

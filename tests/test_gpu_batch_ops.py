"""The batch operations of the library (tq_batch_merge / filter / extend /
extract), the BatchTurboQuantKVCache operations of "omlx/turboquant_kv.py" on
the paged layout, through the C ABI.

Expected pools are written by the oracle from its own records of the same
inputs, at the blocks the library's table rows name (bit-exact); decode over
each resulting batch is compared with the oracle and with decode over the
original caches; block tables, lengths and freed block lists are checked
entry by entry.
"""
import numpy as np
import pytest
import torch

import oracle as O
import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import compare_decode, oracle_decode, raw_kv, to_f32_np

pytestmark = pytest.mark.gpu

DEV = "cuda"
D, HKV, BT, G = 128, 2, 16, 4


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _workload(lens, seed=77):
    return wl.Workload("batch_ops", 2, len(lens), HKV, HKV * G, D, tuple(lens), 1, torch.bfloat16, 1.0, seed,
                       wl._spec("prod", 3, 5), wl._spec("mse", 3, 6), block_tokens=BT, prefill_chunk=64)


def _codecs():
    return tq.Codec(D, 3, tq.TQ_MODE_PROD, 5), tq.Codec(D, 3, tq.TQ_MODE_MSE, 6)


def _single(w, b, kc, vc):
    """Sequence b of w alone in a cache of its own, as a one-row batch."""
    n = w.seq_lens[b]
    nblk = (n + BT - 1) // BT
    cache = tq.CompressedKVCache(kc, vc, w.num_layers, nblk, BT, HKV, DEV, exact_encode=True)
    zero = torch.zeros(1, dtype=torch.int32, device=DEV)
    for layer in range(w.num_layers):
        k = wl.kv_chunk(w, layer, b, 0, n, "k", DEV).unsqueeze(0)
        v = wl.kv_chunk(w, layer, b, 0, n, "v", DEV).unsqueeze(0)
        cache.append(layer, k, v, zero, None, nblk)
    table = torch.arange(nblk, dtype=torch.int32, device=DEV).view(1, nblk)
    lens = torch.tensor([n], dtype=torch.int32, device=DEV)
    return tq.Batch(cache, 1, nblk, table, lens, batch=1)


def _decode(bt: tq.Batch, num_q_heads, layer, q):
    lens = bt.lens[:bt.batch].cpu().tolist()
    msl = max(lens)
    ws = torch.empty(bt.cache.workspace_bytes(bt.batch, num_q_heads, 1, msl), dtype=torch.uint8, device=DEV)
    out = torch.empty(bt.batch, num_q_heads, 1, D, dtype=torch.float32, device=DEV)
    bt.cache.decode(layer, q, bt.lens[:bt.batch].contiguous(), bt.table[:bt.batch].contiguous(), bt.max_blocks,
                    msl, out, ws)
    torch.cuda.synchronize()
    return to_f32_np(out)


def _oracle_pool(bt: tq.Batch, sources):
    """The oracle's pool of a batch: each row's sequence (workload, index) written
    at the blocks its table row names."""
    okc, ovc = O.Codec(D, 3, O.PROD, 5), O.Codec(D, 3, O.MSE, 6)
    cache = bt.cache
    table = bt.table.cpu().numpy()
    want = np.zeros(cache.pool.numel(), np.uint8)
    stride = cache.desc.layer_stride
    for layer in range(cache.num_layers):
        view = want[layer * stride:(layer + 1) * stride]
        for r, (w, b) in enumerate(sources):
            K, V = raw_kv(w, layer, b, w.seq_lens[b], DEV)
            for h in range(HKV):
                O.pool_write(view, okc, ovc, HKV, BT, table, bt.max_blocks, r, h, 0, okc.encode(K[h]),
                             ovc.encode(V[h]))
    return want


def test_batch_merge_filter_extract_extend():
    w = _workload((37, 100, 16))
    kc, vc = _codecs()
    singles = [_single(w, b, kc, vc) for b in range(w.batch)]
    nblk = [s.max_blocks for s in singles]
    spare = 9
    big = tq.CompressedKVCache(kc, vc, w.num_layers, sum(nblk) + spare, BT, HKV, DEV)
    g = torch.Generator().manual_seed(3)
    free = torch.randperm(big.num_blocks, generator=g).to(torch.int32).to(DEV)
    used = torch.zeros(1, dtype=torch.int32, device=DEV)
    mb = max(nblk) + 2
    batch = tq.Batch(big, 8, mb)

    # ---- merge: each sequence's blocks go to the next free blocks, in order
    tq.tq_batch_merge(batch, singles, free, used)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0 and batch.batch == 3
    assert int(used[0]) == sum(nblk)
    tab, fl = batch.table.cpu(), free.cpu()
    o = 0
    for b, n in enumerate(nblk):
        assert torch.equal(tab[b, :n], fl[o:o + n]) and bool((tab[b, n:] == -1).all())
        o += n
    assert batch.lens[:3].cpu().tolist() == list(w.seq_lens)
    assert np.array_equal(big.pool.cpu().numpy(), _oracle_pool(batch, [(w, b) for b in range(3)]))
    q = wl.queries(w, 1, 0, DEV)
    merged = _decode(batch, w.num_q_heads, 1, q)
    qn = to_f32_np(q).astype(np.float64)
    for b in range(3):
        K, V = raw_kv(w, 1, b, w.seq_lens[b], DEV)
        for h in range(HKV):
            compare_decode(merged[b, h * G:(h + 1) * G], oracle_decode(w, K[h], V[h], qn[b, h * G:(h + 1) * G]))
        alone = _decode(singles[b], w.num_q_heads, 1, q[b:b + 1].contiguous())
        assert np.abs(merged[b] - alone[0]).max() <= 1e-5

    # ---- filter: keep rows 2 and 0 (same pool, rows only); row 1's blocks are freed
    kept = tq.Batch(big, 8, mb)
    freed = torch.full((8 * mb,), -7, dtype=torch.int32, device=DEV)
    n_freed = torch.full((1,), -1, dtype=torch.int32, device=DEV)
    tq.tq_batch_filter(batch, [2, 0], kept, freed, n_freed)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0 and kept.batch == 2
    assert torch.equal(kept.table[:2].cpu(), tab[[2, 0]]) and kept.lens[:2].cpu().tolist() == [16, 37]
    assert int(n_freed[0]) == nblk[1]
    assert torch.equal(freed[:nblk[1]].cpu(), tab[1, :nblk[1]])
    sub = _decode(kept, w.num_q_heads, 1, q[[2, 0]].contiguous())
    assert np.abs(sub[0] - merged[2]).max() <= 1e-5 and np.abs(sub[1] - merged[0]).max() <= 1e-5

    # ---- extract: sequence 1 into a cache of its own: the same bytes as the original
    alone_cache = tq.CompressedKVCache(kc, vc, w.num_layers, nblk[1], BT, HKV, DEV)
    alone = tq.Batch(alone_cache, 1, nblk[1])
    used1 = torch.zeros(1, dtype=torch.int32, device=DEV)
    tq.tq_batch_extract(batch, 1, alone, torch.arange(nblk[1], dtype=torch.int32, device=DEV), used1)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0 and alone.batch == 1 and int(used1[0]) == nblk[1]
    assert torch.equal(alone_cache.pool, singles[1].cache.pool)
    assert torch.equal(alone.table[0].cpu(), torch.arange(nblk[1], dtype=torch.int32))

    # ---- extend: another batch's sequence appended into the remaining free blocks
    w2 = _workload((50,), seed=91)
    other = _single(w2, 0, kc, vc)
    tq.tq_batch_extend(batch, other, free, used)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0 and batch.batch == 4
    n_o = other.max_blocks
    assert int(used[0]) == sum(nblk) + n_o
    assert torch.equal(batch.table[3, :n_o].cpu(), fl[sum(nblk):sum(nblk) + n_o])
    assert np.array_equal(big.pool.cpu().numpy(),
                          _oracle_pool(batch, [(w, 0), (w, 1), (w, 2), (w2, 0)]))
    q2 = torch.cat([q, wl.queries(w2, 1, 0, DEV)])
    ext = _decode(batch, w.num_q_heads, 1, q2)
    assert np.abs(ext[:3] - merged).max() <= 1e-5
    assert np.abs(ext[3] - _decode(other, w.num_q_heads, 1, q2[3:].contiguous())[0]).max() <= 1e-5


def test_batch_extend_within_one_pool_moves_rows_only():
    w = _workload((40, 20))
    kc, vc = _codecs()
    nb = [3, 2]
    cache = tq.CompressedKVCache(kc, vc, w.num_layers, 8, BT, HKV, DEV, exact_encode=True)
    a = tq.Batch(cache, 4, 4)
    b = tq.Batch(cache, 2, 4)
    a.table[0, :3] = torch.tensor([5, 1, 7], dtype=torch.int32)
    a.lens[0] = 40
    a.batch = 1
    b.table[0, :2] = torch.tensor([0, 6], dtype=torch.int32)
    b.table[0, 2] = 3                      # a block reserved past the sequence's tokens
    b.lens[0] = 20
    b.batch = 1
    before = cache.pool.clone()
    tq.tq_batch_extend(a, b)
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0 and a.batch == 2
    assert a.table[1].cpu().tolist() == [0, 6, 3, -1] and int(a.lens[1]) == 20
    assert torch.equal(cache.pool, before)   # nothing copied


def test_batch_guard_and_argument_errors():
    kc, vc = _codecs()
    kc2 = tq.Codec(D, 3, tq.TQ_MODE_PROD, 9)             # another seed: another configuration
    c1 = tq.CompressedKVCache(kc, vc, 1, 4, BT, HKV, DEV)
    c2 = tq.CompressedKVCache(kc2, vc, 1, 4, BT, HKV, DEV)
    a, b = tq.Batch(c1, 4, 4), tq.Batch(c2, 4, 4)
    b.batch = 1
    b.lens[0] = 5
    good = tq.Batch(c1, 2, 4)
    good.batch = 1
    good.lens[0] = 5
    good.table[0, 0] = 0
    free = torch.arange(4, dtype=torch.int32, device=DEV)
    used = torch.zeros(1, dtype=torch.int32, device=DEV)
    n0 = tq.tq_launch_count()
    # mixed configurations are refused before anything runs, for every source
    with pytest.raises(tq.TQError) as e:
        tq.tq_batch_merge(a, [good, b], free, used)
    assert e.value.status == 3 and a.batch == 0
    with pytest.raises(tq.TQError) as e:
        tq.tq_batch_extend(a, b, free, used)
    assert e.value.status == 3
    # filter: repeated or out-of-range rows, and an output of another pool
    a.batch = 3
    out = tq.Batch(c1, 4, 4)
    freed = torch.zeros(16, dtype=torch.int32, device=DEV)
    nf = torch.zeros(1, dtype=torch.int32, device=DEV)
    for keep in ([0, 0], [3], [-1]):
        with pytest.raises(tq.TQError) as e:
            tq.tq_batch_filter(a, keep, out, freed, nf)
        assert e.value.status == 1
    with pytest.raises(tq.TQError) as e:
        tq.tq_batch_filter(a, [0], tq.Batch(c2, 4, 4), freed, nf)
    assert e.value.status == 3
    # capacity of the destination rows
    small = tq.Batch(c1, 1, 4)
    small.batch = 1
    with pytest.raises(tq.TQError) as e:
        tq.tq_batch_extend(small, good)
    assert e.value.status == 4
    # extract index out of range
    with pytest.raises(tq.TQError) as e:
        tq.tq_batch_extract(good, 1, tq.Batch(c1, 1, 4), free, used)
    assert e.value.status == 1
    assert tq.tq_launch_count() == n0        # nothing was launched


def test_batch_free_list_exhaustion_is_flagged():
    w = _workload((40,))
    kc, vc = _codecs()
    src = _single(w, 0, kc, vc)              # 3 blocks
    dst_cache = tq.CompressedKVCache(kc, vc, w.num_layers, 4, BT, HKV, DEV)
    dst = tq.Batch(dst_cache, 1, 4)
    used = torch.zeros(1, dtype=torch.int32, device=DEV)
    tq.tq_batch_extend(dst, src, torch.tensor([2, 0], dtype=torch.int32, device=DEV), used)
    torch.cuda.synchronize()
    assert tq.tq_device_error() & tq._lib.TQ_DEVERR_CAPACITY
    # the sequence keeps the tokens of the blocks it received
    assert dst.table[0].cpu().tolist() == [2, 0, -1, -1] and int(dst.lens[0]) == 32 and int(used[0]) == 2

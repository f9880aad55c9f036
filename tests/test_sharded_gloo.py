"""The host logic of the sequence-sharded decode on two gloo ranks (CPU).

Each rank owns a contiguous range of every sequence's tokens
(turboquant_compressed_kv_tq_gb300.sharded: shard ranges, causal ends, the
all-gather of the per-row states). Here the per-shard state comes from the
oracle on the host, so that the exchange and the ordering are what is
tested: the merge of the gathered states must equal the oracle's decode of
the whole sequence, on every rank. The GPU kernels of the same scheme are
checked in tests/test_gpu_sharded.py.
"""
import math
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from turboquant_compressed_kv_tq_gb300 import sharded


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _case(seed=11):
    rng = np.random.default_rng(seed)
    D, G, Lq = 64, 4, 2
    lens = [23, 2, 50]                     # the middle sequence is shorter than the ranks' count x Lq
    K = [rng.standard_normal((n, D)).astype(np.float32) for n in lens]
    V = [rng.standard_normal((n, D)).astype(np.float32) for n in lens]
    q = [rng.standard_normal((G, Lq, D)) for _ in lens]
    return D, G, Lq, lens, K, V, q


def _worker(rank, world, port, outq):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch
    import torch.distributed as dist
    import oracle as O
    from turboquant_compressed_kv_tq_gb300 import sharded as sh
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        D, G, Lq, lens, K, V, q = _case()
        kc, vc = O.Codec(D, 3, O.PROD, 1), O.Codec(D, 3, O.MSE, 2)
        starts, counts, ends = sh.shard_ranges(lens, world, rank)
        B = len(lens)
        ml = torch.zeros(B, G, Lq, 2, dtype=torch.float64)
        acc = torch.zeros(B, G, Lq, D, dtype=torch.float64)
        for b in range(B):
            s, c = starts[b], counts[b]
            kr, vr = kc.encode(K[b][s:s + c]), vc.encode(V[b][s:s + c])
            m, l, a = O.decode_partial(q[b], kc, kr, vc, vr, 1 / math.sqrt(D), Lq, ends[b])
            ml[b, ..., 0] = torch.from_numpy(m.reshape(G, Lq))
            ml[b, ..., 1] = torch.from_numpy(l.reshape(G, Lq))
            acc[b] = torch.from_numpy(a.reshape(G, Lq, D))
        ml_all, acc_all = sh.gather_states(ml, acc)
        errs = []
        for b in range(B):
            got = O.merge_partials(vc, ml_all[:, b, ..., 0].reshape(world, -1).numpy(),
                                   ml_all[:, b, ..., 1].reshape(world, -1).numpy(),
                                   acc_all[:, b].reshape(world, G * Lq, D).numpy())
            ref = O.decode_rotated(q[b], kc, kc.encode(K[b]), vc, vc.encode(V[b]), 1 / math.sqrt(D), Lq)
            errs.append(float(np.abs(got - ref.reshape(G * Lq, D)).max()))
        outq.put((rank, counts, max(errs)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_merge_equals_unsharded_decode():
    ctx = mp.get_context("spawn")
    outq = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, outq)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(outq.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, c0, e0), (_, c1, e1) = res
    assert [a + b for a, b in zip(c0, c1)] == [23, 2, 50]
    assert e0 <= 1e-11 and e1 <= 1e-11


def test_shard_ranges_cover_each_sequence_once():
    for n in (0, 1, 2, 7, 100, 262146):
        for world in (1, 2, 3, 8):
            spans = [sharded.shard_range(n, world, r) for r in range(world)]
            pos = 0
            for s, c in spans:
                assert s == pos and c >= 0
                pos += c
            assert pos == n
            assert max(c for _, c in spans) - min(c for _, c in spans) <= 1
    starts, counts, ends = sharded.shard_ranges([10, 3], 4, 3)
    assert starts == [8, 3] and counts == [2, 0] and ends == [2, 0]
    with pytest.raises(ValueError):
        sharded.shard_range(5, 2, 2)

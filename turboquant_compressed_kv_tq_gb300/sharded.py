"""Sequence-sharded decode across ranks (one process per GPU).

When a KV cache is split by token position over several GPUs
("turboquant/validate_moe_phase2.py", TEST 3: with tensor parallelism each GPU
holds a shard of the KV cache), every rank keeps a contiguous range of each
sequence's tokens in its own compressed cache. A decode step is then:

  1. each rank: ``tq_decode_partials`` over its shard, with the causal end of
     the queries expressed in its local token indices;
  2. one all-gather of the per-row states (max, sum, accumulator) -- the only
     exchange, ``rows * (head_dim + 2)`` floats per rank;
  3. every rank (or only the consumer): ``tq_decode_merge`` of the gathered
     states, which also applies the inverse value rotation.

This module holds the host logic of that scheme (which tokens a rank owns,
the causal ends, the gather); the arithmetic runs in the library's kernels.
"""
from __future__ import annotations

from typing import List, Sequence, Tuple


def shard_range(n_tokens: int, world: int, rank: int) -> Tuple[int, int]:
    """(first token, token count) of `rank`'s contiguous shard of a sequence of
    n_tokens tokens over `world` ranks; the first n_tokens % world ranks hold
    one token more."""
    if world <= 0 or not 0 <= rank < world or n_tokens < 0:
        raise ValueError("bad shard arguments")
    base, extra = divmod(n_tokens, world)
    start = rank * base + min(rank, extra)
    return start, base + (1 if rank < extra else 0)


def shard_ranges(seq_lens: Sequence[int], world: int, rank: int) -> Tuple[List[int], List[int], List[int]]:
    """Per sequence: this rank's (first token, token count) and the causal end
    of the queries in its local indices (global length - first token)."""
    starts, counts, ends = [], [], []
    for n in seq_lens:
        s, c = shard_range(int(n), world, rank)
        starts.append(s)
        counts.append(c)
        ends.append(int(n) - s)
    return starts, counts, ends


def gather_states(part_ml, part_acc, group=None):
    """All-gather every rank's (max, sum) and accumulator tensors, stacked in
    rank order: [world, ...] each."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = []
    for t in (part_ml.contiguous(), part_acc.contiguous()):
        # ranks' tensors concatenated along the first dimension, then split by rank
        g = torch.empty((world * t.shape[0],) + tuple(t.shape[1:]), dtype=t.dtype, device=t.device)
        dist.all_gather_into_tensor(g, t, group=group)
        out.append(g.view((world,) + tuple(t.shape)))
    return out[0], out[1]


def sharded_decode(cache, layer: int, q, local_lens, causal_end, block_table, max_blocks: int, max_seq_len: int,
                   out, workspace, group=None, scale: float = 0.0) -> None:
    """One sharded decode step of one layer on this rank: partial states of the
    local shard, one all-gather, then the merge into `out` [batch, Hq, Lq, D]."""
    import torch
    from . import tq_decode_merge
    B, Hq, Lq, D = q.shape
    ml = torch.empty(B, Hq, Lq, 2, dtype=torch.float32, device=q.device)
    acc = torch.empty(B, Hq, Lq, D, dtype=torch.float32, device=q.device)
    cache.decode_partials(layer, q, local_lens, causal_end, block_table, max_blocks, max_seq_len, ml, acc,
                          workspace, scale)
    ml_all, acc_all = gather_states(ml, acc, group)
    tq_decode_merge(cache.value.handle, ml_all, acc_all, out)

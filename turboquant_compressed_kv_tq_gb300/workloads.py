"""Seeded synthetic workloads: shapes, value distributions and generators.

This module holds no codec arithmetic. It only says which inputs the
validation and benchmark workloads use and draws them reproducibly, so that the
GPU path and the CPU oracle can be fed byte-identical inputs.

Workload shapes follow the pages:

* ``tiny`` -- the synthetic validation of "turboquant/validate_moe_phase2.py"
  (keys ``torch.randn(...) * 0.02``, seed 42), at head_dim 128 with one KV
  head and GQA 4.
* ``layer_d256`` -- the same script's head_dim 256, 2 KV heads, 16 query heads,
  N in {512, 1024, 4096, 8192}; keys 3-bit prod, values 2-bit group quant.
* ``stack_32k`` / ``long_256k`` -- the 64-layer, 8-KV-head, head_dim 128
  stack of "lightning-mlx/plan.md" (memory math and bandwidth-bound decode
  analysis), decoding with query length 2 (speculative verify of two tokens).
* ``paged_batch`` -- continuous batching of 32 ragged sequences through a
  paged cache of 16-token blocks ("omlx/turboquant_kv.py",
  BatchTurboQuantKVCache), 32 query heads.

Generators: every tensor is drawn by ``torch.Generator`` from a seed derived
from (workload seed, layer, chunk, tensor tag), on the device the caller
names.  Re-drawing the same (seed, shape, device) gives the same values, so a
test can regenerate any slice of a large workload on the device and copy it
to the host for the oracle.
"""
from __future__ import annotations

import dataclasses
import hashlib
from typing import Optional, Sequence

import torch

MODE_MSE = 0
MODE_PROD = 1
MODE_GROUP = 2

_MODE_NAMES = {"mse": MODE_MSE, "prod": MODE_PROD, "group": MODE_GROUP}


@dataclasses.dataclass(frozen=True)
class CodecSpec:
    mode: int
    bits: int
    seed: int = 0
    group_size: int = 0


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    num_layers: int
    batch: int
    num_kv_heads: int
    num_q_heads: int
    head_dim: int
    seq_lens: Sequence[int]          # cached tokens per sequence after the step's append
    q_len: int
    dtype: torch.dtype               # dtype of K, V and q inputs
    std: float                       # per-coordinate standard deviation
    input_seed: int
    key: CodecSpec
    value: CodecSpec
    block_tokens: int = 256          # paged-pool block size (tokens)
    head_scale_range: Optional[tuple] = None   # per-(layer, head) scale ~ U[lo, hi]
    shuffle_blocks: bool = False     # physical blocks assigned in a shuffled order
    prefill_chunk: int = 8192
    decode_steps: int = 1
    append_per_step: int = 0         # tokens appended per decode step

    @property
    def gqa(self) -> int:
        return self.num_q_heads // self.num_kv_heads


def _spec(mode: str, bits: int, seed: int = 0, group: int = 0) -> CodecSpec:
    return CodecSpec(_MODE_NAMES[mode], bits, seed, group)


def tiny() -> Workload:
    return Workload("tiny", 1, 1, 1, 4, 128, (512,), 1, torch.float32, 0.02, 42,
                    _spec("prod", 3, 42), _spec("mse", 4, 43), block_tokens=64)


def layer_d256(n: int = 8192) -> Workload:
    assert n in (512, 1024, 4096, 8192)
    return Workload(f"layer_d256_n{n}", 1, 1, 2, 16, 256, (n,), 1, torch.bfloat16, 0.02,
                    42, _spec("prod", 3, 42), _spec("group", 2, 0, 32), block_tokens=64)


def stack_32k() -> Workload:
    return Workload("stack_32k", 64, 1, 8, 64, 128, (32768,), 2, torch.bfloat16, 1.0, 3,
                    _spec("mse", 4, 0), _spec("mse", 4, 1), block_tokens=256,
                    head_scale_range=(0.5, 2.0))


def long_256k(steps: int = 256) -> Workload:
    return Workload("long_256k", 64, 1, 8, 64, 128, (262144,), 2, torch.bfloat16, 1.0, 4,
                    _spec("prod", 3, 0), _spec("mse", 3, 1), block_tokens=256,
                    decode_steps=steps, append_per_step=2)


def paged_batch(seed: int = 5) -> Workload:
    g = torch.Generator().manual_seed(seed)
    lens = torch.randint(4096, 65537, (32,), generator=g).tolist()
    return Workload("paged_batch", 64, 32, 8, 32, 128, tuple(lens), 1, torch.bfloat16, 1.0,
                    seed, _spec("prod", 3, 0), _spec("group", 4, 0, 64), block_tokens=16,
                    shuffle_blocks=True, append_per_step=1)


WORKLOADS = {
    "tiny": tiny,
    "layer_d256": layer_d256,
    "stack_32k": stack_32k,
    "long_256k": long_256k,
    "paged_batch": paged_batch,
}


def derive_seed(*parts) -> int:
    """A 63-bit seed from any tuple of ints/strings (stable across machines)."""
    h = hashlib.sha256(repr(tuple(parts)).encode()).digest()
    return int.from_bytes(h[:8], "little") & ((1 << 63) - 1)


def _normal(shape, seed: int, dtype: torch.dtype, device, std: float) -> torch.Tensor:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    x = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def head_scales(w: Workload, layer: int) -> Optional[torch.Tensor]:
    """Per-(layer, kv head) scale ~ U[lo, hi] (CPU float32), or None."""
    if w.head_scale_range is None:
        return None
    lo, hi = w.head_scale_range
    g = torch.Generator().manual_seed(derive_seed(w.input_seed, "head_scale", layer))
    return lo + (hi - lo) * torch.rand(w.num_kv_heads, generator=g)


def kv_chunk(w: Workload, layer: int, seq: int, t0: int, n: int, which: str, device="cpu"):
    """Keys or values of tokens [t0, t0+n) of sequence ``seq``: [Hkv, n, D].

    Tokens are drawn in fixed chunks of ``w.prefill_chunk`` so any slice can be
    regenerated alone; ``which`` is "k" or "v".
    """
    out = []
    c = w.prefill_chunk
    t = t0
    while t < t0 + n:
        ci = t // c
        lo = ci * c
        hi = min(lo + c, t0 + n)
        full = _normal((w.num_kv_heads, c, w.head_dim),
                       derive_seed(w.input_seed, which, layer, seq, ci), torch.float32,
                       device, w.std)
        out.append(full[:, t - lo: hi - lo])
        t = hi
    x = torch.cat(out, dim=1) if len(out) > 1 else out[0]
    s = head_scales(w, layer)
    if s is not None:
        x = x * s.to(x.device).view(-1, 1, 1)
    return x.to(w.dtype).contiguous()


def queries(w: Workload, layer: int, step: int = 0, device="cpu") -> torch.Tensor:
    """Decode queries [B, Hq, Lq, D]."""
    q = _normal((w.batch, w.num_q_heads, w.q_len, w.head_dim),
                derive_seed(w.input_seed, "q", layer, step), torch.float32, device, w.std)
    s = head_scales(w, layer)
    if s is not None:
        q = q * s.repeat_interleave(w.gqa).to(q.device).view(1, -1, 1, 1)
    return q.to(w.dtype).contiguous()


def block_table(w: Workload, capacity_tokens: Sequence[int], device="cpu"):
    """Block table [B, max_blocks] int32 for per-sequence capacities.

    Physical blocks are numbered densely; with ``shuffle_blocks`` they are
    handed out in a seeded random order (a fragmented pool).
    Returns (table, num_physical_blocks).
    """
    bt = w.block_tokens
    nblk = [(c + bt - 1) // bt for c in capacity_tokens]
    maxb = max(nblk)
    total = sum(nblk)
    if w.shuffle_blocks:
        g = torch.Generator().manual_seed(derive_seed(w.input_seed, "blocks"))
        phys = torch.randperm(total, generator=g)
    else:
        phys = torch.arange(total)
    table = torch.zeros(len(nblk), maxb, dtype=torch.int32)
    o = 0
    for b, k in enumerate(nblk):
        table[b, :k] = phys[o:o + k].to(torch.int32)
        o += k
    return table.to(device), total


def encoder_stress(seed: int, batch: int, num_kv_heads: int, n: int, head_dim: int,
                   dtype=torch.bfloat16, device="cpu") -> torch.Tensor:
    """Vectors [batch, Hkv, n, D] that stress an encoder's arithmetic.

    Mostly N(0,1) rows times a per-row scale 2^u, u ~ U[-12, 12]; among them
    all-zero rows, one-hot rows, constant rows, rows with one dominant
    coordinate and a tail 2^-20 below it, and rows at 2^-100 (tiny but normal
    in bf16). Seeded; drawn on the host, then moved to ``device``.
    """
    g = torch.Generator().manual_seed(derive_seed(seed, "stress", batch, num_kv_heads, n, head_dim))
    x = torch.randn(batch, num_kv_heads, n, head_dim, generator=g, dtype=torch.float32)
    u = torch.randint(-12, 13, (batch, num_kv_heads, n, 1), generator=g).to(torch.float32)
    x = x * torch.pow(2.0, u)
    kind = torch.randint(0, 40, (batch, num_kv_heads, n), generator=g)
    spike = torch.randint(0, head_dim, (batch, num_kv_heads, n), generator=g)
    onehot = torch.nn.functional.one_hot(spike, head_dim).to(torch.float32)
    x = torch.where((kind == 0).unsqueeze(-1), torch.zeros_like(x), x)
    x = torch.where((kind == 1).unsqueeze(-1), onehot * 3.0, x)
    x = torch.where((kind == 2).unsqueeze(-1), torch.full_like(x, -0.75), x)
    x = torch.where((kind == 3).unsqueeze(-1), onehot * 5.0 + x * 2.0 ** -20, x)
    x = torch.where((kind == 4).unsqueeze(-1), x * 2.0 ** -100, x)
    return x.to(dtype).to(device).contiguous()

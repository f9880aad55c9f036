"""Shared helpers for GPU-vs-oracle parity tests.

Inputs come from the seeded workload generators; expected values come only
from the oracle. The GPU side is driven through the C ABI binding.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle as O
import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl

ATOL = 2e-3        # max |gpu - oracle| on decode outputs
COS_MIN = 0.9999   # min cosine(gpu row, oracle row)


def oracle_codec(spec: wl.CodecSpec, D: int) -> O.Codec:
    return O.Codec(D, spec.bits, spec.mode, spec.seed, spec.group_size)


def gpu_codec(spec: wl.CodecSpec, D: int) -> tq.Codec:
    return tq.Codec(D, spec.bits, spec.mode, spec.seed, spec.group_size)


def to_f32_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float32).numpy()


def compare_decode(gpu: np.ndarray, ref: np.ndarray, atol: float = ATOL, cos_min: float = COS_MIN):
    gpu = gpu.reshape(-1, gpu.shape[-1]).astype(np.float64)
    ref = ref.reshape(-1, ref.shape[-1])
    err = np.abs(gpu - ref).max()
    cos = (gpu * ref).sum(-1) / np.maximum(np.linalg.norm(gpu, axis=-1) * np.linalg.norm(ref, axis=-1),
                                           1e-300)
    assert err <= atol, f"max abs error {err:.3e} > {atol}"
    assert cos.min() >= cos_min, f"min cosine {cos.min():.7f} < {cos_min}"
    return err, cos.min()


class GpuCase:
    """One workload slice on the GPU: codecs, pool, block table, inputs."""

    def __init__(self, w: wl.Workload, layers, seq_lens=None, device="cuda", exact_encode=True):
        self.w = w
        self.layers = list(layers)
        self.D = w.head_dim
        self.seq_lens = list(seq_lens if seq_lens is not None else w.seq_lens)
        self.kc = gpu_codec(w.key, self.D)
        self.vc = gpu_codec(w.value, self.D)
        cap = [n + w.append_per_step for n in self.seq_lens]
        self.table, nblocks = wl.block_table(w, cap)
        self.max_blocks = self.table.shape[1]
        self.cache = tq.CompressedKVCache(self.kc, self.vc, len(self.layers), nblocks,
                                          w.block_tokens, w.num_kv_heads, device,
                                          exact_encode=exact_encode)
        self.table_d = self.table.to(device)
        self.device = device

    def prefill(self, chunk=None):
        """Encode every sequence's tokens, layer by layer, in chunks."""
        w = self.w
        chunk = chunk or w.prefill_chunk
        B = w.batch
        for li, layer in enumerate(self.layers):
            done = [0] * B
            while any(done[b] < self.seq_lens[b] for b in range(B)):
                # one append call per step over the sequences that still have tokens
                n = min(chunk, max(self.seq_lens[b] - done[b] for b in range(B)))
                for b in range(B):
                    nb = min(n, self.seq_lens[b] - done[b])
                    if nb <= 0:
                        continue
                    k = wl.kv_chunk(w, layer, b, done[b], nb, "k", self.device).unsqueeze(0)
                    v = wl.kv_chunk(w, layer, b, done[b], nb, "v", self.device).unsqueeze(0)
                    sl = torch.tensor([done[b]], dtype=torch.int32, device=self.device)
                    self.cache.append(li, k, v, sl, self.table_d[b:b + 1].contiguous(), self.max_blocks)
                    done[b] += nb
        torch.cuda.synchronize()

    def decode(self, li, q, max_seq_len=None):
        w = self.w
        B = q.shape[0]
        sl = torch.tensor(self.seq_lens, dtype=torch.int32, device=self.device)
        msl = max_seq_len or max(self.seq_lens)
        ws = torch.empty(self.cache.workspace_bytes(B, w.num_q_heads, w.q_len, msl), dtype=torch.uint8,
                         device=self.device)
        out = torch.empty(B, w.num_q_heads, w.q_len, self.D, dtype=torch.float32, device=self.device)
        self.cache.decode(li, q, sl, self.table_d, self.max_blocks, msl, out, ws)
        torch.cuda.synchronize()
        return out


def raw_kv(w: wl.Workload, layer: int, seq: int, n_tokens: int, device="cuda"):
    """The exact K, V values [Hkv, N, D] (float32 numpy) the GPU side encodes."""
    K = to_f32_np(wl.kv_chunk(w, layer, seq, 0, n_tokens, "k", device))
    V = to_f32_np(wl.kv_chunk(w, layer, seq, 0, n_tokens, "v", device))
    return K, V


def oracle_decode(w: wl.Workload, K: np.ndarray, V: np.ndarray, q: np.ndarray, scale=None):
    """Expected output rows [G, Lq, D] of one (sequence, kv head) from raw inputs.

    K, V: [N, D] float32; q: [G, Lq, D] float64 queries of that kv head's group.
    """
    D = w.head_dim
    kc, vc = oracle_codec(w.key, D), oracle_codec(w.value, D)
    kr, vr = kc.encode(K), vc.encode(V)
    return O.decode_rotated(q, kc, kr, vc, vr, scale or 1 / math.sqrt(D), w.q_len)


def read_records(layer_pool: np.ndarray, kc: O.Codec, vc: O.Codec, Hkv: int, BT: int, table, max_blocks: int,
                 seq: int, h: int, t0: int, n: int):
    """Key and value records of tokens [t0, t0+n) of (seq, head h) from a layer pool.

    The sub-block layout is the oracle's (subblock_layout); ``table`` is the
    block table (numpy) or None for the identity.
    """
    sub, off = O.subblock_layout(kc, vc, BT)
    Wk, Wv, Ws = kc.W, vc.W, kc.D // 32
    ng = vc.D // vc.group if vc.mode == O.GROUP else 0
    rows = {"k_idx": [], "k_sgn": [], "k_norm": [], "k_rnorm": [], "v_idx": [], "v_norm": [],
            "v_scale": [], "v_min": []}
    for t in range(t0, t0 + n):
        lb, slot = t // BT, t % BT
        pb = int(table[seq, lb]) if table is not None else seq * max_blocks + lb
        base = (pb * Hkv + h) * sub

        def take(o, count, dt):
            size = np.dtype(dt).itemsize * count
            a = base + o + slot * size
            return layer_pool[a:a + size].view(dt)
        rows["k_idx"].append(take(off[0], Wk, np.uint32))
        rows["k_norm"].append(take(off[2], 1, np.float32))
        if kc.mode == O.PROD:
            rows["k_sgn"].append(take(off[1], Ws, np.uint32))
            rows["k_rnorm"].append(take(off[3], 1, np.float32))
        rows["v_idx"].append(take(off[4], Wv, np.uint32))
        if vc.mode == O.GROUP:
            rows["v_scale"].append(take(off[5], ng, np.uint16))
            rows["v_min"].append(take(off[6], ng, np.uint16))
        else:
            rows["v_norm"].append(take(off[5], 1, np.float32))
    out = {k: np.stack(v) for k, v in rows.items() if v}
    krec = {"idx": out["k_idx"], "norm": out["k_norm"][:, 0]}
    if kc.mode == O.PROD:
        krec["sgn"], krec["rnorm"] = out["k_sgn"], out["k_rnorm"][:, 0]
    vrec = {"idx": out["v_idx"]}
    if vc.mode == O.GROUP:
        vrec["scale"], vrec["min"] = out["v_scale"], out["v_min"]
    else:
        vrec["norm"] = out["v_norm"][:, 0]
    return krec, vrec


def read_records_blocks(layer_pool: np.ndarray, kc: O.Codec, vc: O.Codec, Hkv: int, BT: int, table,
                        max_blocks: int, seq: int, h: int, n: int):
    """Records of tokens [0, n) of (seq, head h), gathered a whole block at a
    time (the same layout as ``read_records``; fast enough for full-size
    sequences)."""
    sub, off = O.subblock_layout(kc, vc, BT)
    Wk, Wv, Ws = kc.W, vc.W, kc.D // 32
    ng = vc.D // vc.group if vc.mode == O.GROUP else 0
    fields = [(0, Wk, np.uint32, "k_idx"), (2, 1, np.float32, "k_norm"), (4, Wv, np.uint32, "v_idx")]
    if kc.mode == O.PROD:
        fields += [(1, Ws, np.uint32, "k_sgn"), (3, 1, np.float32, "k_rnorm")]
    if vc.mode == O.GROUP:
        fields += [(5, ng, np.uint16, "v_scale"), (6, ng, np.uint16, "v_min")]
    else:
        fields += [(5, 1, np.float32, "v_norm")]
    parts = {name: [] for *_, name in fields}
    nblk = (n + BT - 1) // BT
    for lb in range(nblk):
        pb = int(table[seq, lb]) if table is not None else seq * max_blocks + lb
        base = (pb * Hkv + h) * sub
        take = min(BT, n - lb * BT)
        for k, count, dt, name in fields:
            size = np.dtype(dt).itemsize * count
            a = base + off[k]
            parts[name].append(layer_pool[a:a + BT * size].view(dt).reshape(BT, count)[:take])
    out = {name: np.concatenate(v) for name, v in parts.items()}
    krec = {"idx": out["k_idx"], "norm": out["k_norm"][:, 0]}
    if kc.mode == O.PROD:
        krec["sgn"], krec["rnorm"] = out["k_sgn"], out["k_rnorm"][:, 0]
    vrec = {"idx": out["v_idx"]}
    if vc.mode == O.GROUP:
        vrec["scale"], vrec["min"] = out["v_scale"], out["v_min"]
    else:
        vrec["norm"] = out["v_norm"][:, 0]
    return krec, vrec

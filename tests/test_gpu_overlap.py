"""Back-to-back decode steps whose kernels overlap (programmatic dependent launch).

The bench's step pattern -- for each layer, append two tokens then decode,
all through one shared workspace -- runs once with every call queued back to
back (the append, query-prep and split kernels overlap their neighbours) and
once with a device synchronisation after every call (no overlap possible).
The outputs must be bit-identical, and the last step matches the oracle
(caches encoded with the exact policy, so both sides decode the same records).
"""
import dataclasses

import numpy as np
import pytest
import torch

import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import compare_decode, oracle_decode, raw_kv, to_f32_np

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


def _run_steps(w, layers, steps, sync_each, fused=False):
    D, Hkv, Hq, Lq, BT = w.head_dim, w.num_kv_heads, w.num_q_heads, w.q_len, w.block_tokens
    N0, A = w.seq_lens[0], w.append_per_step
    cap = N0 + A * steps
    nblk = (cap + BT - 1) // BT
    kc = tq.Codec(D, w.key.bits, w.key.mode, w.key.seed)
    vc = tq.Codec(D, w.value.bits, w.value.mode, w.value.seed)
    cache = tq.CompressedKVCache(kc, vc, layers, nblk, BT, Hkv, DEV, exact_encode=True)
    zero = torch.zeros(1, dtype=torch.int32, device=DEV)
    for layer in range(layers):
        k = wl.kv_chunk(w, layer, 0, 0, N0, "k", DEV).unsqueeze(0)
        v = wl.kv_chunk(w, layer, 0, 0, N0, "v", DEV).unsqueeze(0)
        cache.append(layer, k, v, zero, None, nblk)
    torch.cuda.synchronize()
    ins = []
    for s in range(steps):
        kn = torch.stack([wl.kv_chunk(w, l, 0, N0 + A * s, A, "k", DEV) for l in range(layers)]).unsqueeze(1)
        vn = torch.stack([wl.kv_chunk(w, l, 0, N0 + A * s, A, "v", DEV) for l in range(layers)]).unsqueeze(1)
        q = torch.stack([wl.queries(w, l, s, DEV)[0] for l in range(layers)]).unsqueeze(1)
        ins.append((kn.contiguous(), vn.contiguous(), q.contiguous()))
    pre = torch.tensor([N0 + A * s for s in range(steps)], dtype=torch.int32, device=DEV)
    post = pre + A
    ws = torch.empty(cache.workspace_bytes(1, Hq, Lq, cap), dtype=torch.uint8, device=DEV)
    outs = torch.empty(steps, layers, 1, Hq, Lq, D, dtype=torch.float32, device=DEV)
    torch.cuda.synchronize()
    for s in range(steps):
        kn, vn, q = ins[s]
        for layer in range(layers):
            if fused:   # tq_decode_step: the append inside the decode's first launch
                cache.decode_step(layer, kn[layer], vn[layer], q[layer], pre[s:s + 1], None, nblk, cap,
                                  outs[s, layer], ws)
                continue
            cache.append(layer, kn[layer], vn[layer], pre[s:s + 1], None, nblk)
            if sync_each:
                torch.cuda.synchronize()
            cache.decode(layer, q[layer], post[s:s + 1], None, nblk, cap, outs[s, layer], ws)
            if sync_each:
                torch.cuda.synchronize()
    torch.cuda.synchronize()
    assert tq.tq_device_error() == 0
    return to_f32_np(outs), [to_f32_np(t[2]) for t in ins]


def test_overlapped_steps_equal_serialised_steps():
    w = dataclasses.replace(wl.long_256k(), seq_lens=(20000,), prefill_chunk=4096)
    layers, steps = 4, 3
    fast, qs = _run_steps(w, layers, steps, sync_each=False)
    slow, _ = _run_steps(w, layers, steps, sync_each=True)
    assert np.array_equal(fast.view(np.uint32), slow.view(np.uint32))
    # the last step of two layers against the oracle
    G = w.gqa
    n = w.seq_lens[0] + w.append_per_step * steps
    for layer in (0, layers - 1):
        K, V = raw_kv(w, layer, 0, n, DEV)
        qn = qs[steps - 1][layer].astype(np.float64)
        for h in (0, 3):
            ref = oracle_decode(w, K[h], V[h], qn[0, h * G:(h + 1) * G])
            compare_decode(fast[steps - 1, layer, 0, h * G:(h + 1) * G], ref)


@pytest.mark.parametrize("layers,steps", [(4, 3), (1, 5)])
def test_overlapped_fused_steps_equal_serialised_steps(layers, steps):
    """The same steps through tq_decode_step, back to back: bit-identical to the
    separate calls with a device synchronisation after each (one layer: each
    step's append follows the previous step's decode of the same cache)."""
    w = dataclasses.replace(wl.long_256k(), seq_lens=(20000,), prefill_chunk=4096)
    fused, _ = _run_steps(w, layers, steps, sync_each=False, fused=True)
    slow, _ = _run_steps(w, layers, steps, sync_each=True)
    assert np.array_equal(fused.view(np.uint32), slow.view(np.uint32))

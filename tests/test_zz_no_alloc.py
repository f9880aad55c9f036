"""Decode attention for callers that cannot allocate device memory.

Hosts that own all GPU memory without exposing an allocator, and serving loops
that must not allocate while running, call tq_decode_attention_noalloc, which
keeps its scratch in a fixed device array inside the library instead of a
caller-provided workspace. These tests check it through the C ABI against the
regular entry point (caller workspace) on two calls in a row: both run the
same kernels with the same launch shape, so the outputs must be bit-identical,
and the device's free memory must not change across a call. A request too
large for the fixed array is refused with a clear status.

This file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import dataclasses

import pytest
import torch

import turboquant_compressed_kv_tq_gb300 as tq
from turboquant_compressed_kv_tq_gb300 import workloads as wl
from parity_util import GpuCase

pytestmark = pytest.mark.gpu

DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def _lib_built():
    from turboquant_compressed_kv_tq_gb300 import build
    build.build()
    assert torch.cuda.is_available()


@pytest.mark.parametrize("shape", ["long_256k", "layer_d256", "d64"])
def test_noalloc_matches_workspace_entry_on_two_calls(shape):
    # the bench's codecs and head layout (8 KV heads, GQA 8, two query
    # positions); the head_dim-256 layer (its query rows in the scratch); the
    # same codecs at head_dim 64 (the head_dim-128 layout's wider partials)
    if shape == "long_256k":
        w = dataclasses.replace(wl.long_256k(), seq_lens=(5003,))
    elif shape == "layer_d256":
        w = dataclasses.replace(wl.layer_d256(4096), num_layers=2, seq_lens=(3001,))
    else:
        w = dataclasses.replace(wl.long_256k(), head_dim=64, num_layers=2, seq_lens=(7000,))
    case = GpuCase(w, layers=[0, 1])
    case.prefill()
    sl = torch.tensor(case.seq_lens, dtype=torch.int32, device=DEV)
    msl = max(case.seq_lens)
    assert case.cache.workspace_bytes(1, w.num_q_heads, w.q_len, msl) <= tq._lib.TQ_NOALLOC_SCRATCH_BYTES
    free_after = []
    for li, layer in enumerate(case.layers):          # two calls in a row, different inputs
        q = wl.queries(w, layer, 0, DEV)
        ref = case.decode(li, q)                        # regular entry, caller workspace
        out = torch.full_like(ref, float("nan"))
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        tq.tq_decode_attention_noalloc(case.kc.handle, case.vc.handle, case.cache.desc, li, q, sl,
                                       case.table_d, case.max_blocks, msl, out)
        torch.cuda.synchronize()
        free_after.append(torch.cuda.mem_get_info()[0])
        # the same kernels with the same launch shape: bit-identical outputs
        assert torch.equal(out, ref)
        # the call reserved nothing on the device: its array was reserved when
        # the codecs were created
        assert free_after[-1] == free_before
    assert tq.tq_device_error() == 0


def test_noalloc_refuses_requests_beyond_its_scratch():
    D, Hkv, batch, q_len, hq = 128, 8, 64, 8, 64
    kc, vc = tq.Codec(D, 3, tq.TQ_MODE_PROD, 0), tq.Codec(D, 3, tq.TQ_MODE_MSE, 1)
    cache = tq.CompressedKVCache(kc, vc, 1, batch, 16, Hkv)
    assert cache.workspace_bytes(batch, hq, q_len, 16) > tq._lib.TQ_NOALLOC_SCRATCH_BYTES
    q = torch.zeros(batch, hq, q_len, D, dtype=torch.bfloat16, device=DEV)
    out = torch.zeros(batch, hq, q_len, D, dtype=torch.float32, device=DEV)
    sl = torch.full((batch,), 16, dtype=torch.int32, device=DEV)
    with pytest.raises(tq.TQError) as e:
        tq.tq_decode_attention_noalloc(kc.handle, vc.handle, cache.desc, 0, q, sl, None, 1, 16, out)
    assert e.value.status == 4
    assert not out.any()                               # nothing was launched

"""The seeded input generators on the CPU: any slice of a workload can be drawn
alone and equals the same tokens drawn as part of a larger slice; the draws
have the stated distributions; block tables are permutations of the pool."""
import math

import pytest
import torch

from turboquant_compressed_kv_tq_gb300 import workloads as wl


def _small(**kw):
    base = dict(name="t", num_layers=2, batch=2, num_kv_heads=2, num_q_heads=8, head_dim=64,
                seq_lens=(300, 41), q_len=2, dtype=torch.float32, std=1.0, input_seed=7,
                key=wl._spec("prod", 3, 0), value=wl._spec("mse", 3, 1), prefill_chunk=128)
    base.update(kw)
    return wl.Workload(**base)


@pytest.mark.parametrize("cuts", [(0, 300), (0, 128, 300), (0, 5, 127, 129, 256, 300), (17, 200, 255, 299)])
def test_kv_chunk_slices_agree_across_chunk_boundaries(cuts):
    w = _small()
    whole = wl.kv_chunk(w, 1, 0, cuts[0], cuts[-1] - cuts[0], "k")
    parts = [wl.kv_chunk(w, 1, 0, a, b - a, "k") for a, b in zip(cuts[:-1], cuts[1:])]
    assert torch.equal(whole, torch.cat(parts, dim=1))
    assert whole.shape == (w.num_kv_heads, cuts[-1] - cuts[0], w.head_dim)


def test_draws_are_deterministic_and_separated():
    w = _small()
    a = wl.kv_chunk(w, 0, 0, 0, 64, "k")
    assert torch.equal(a, wl.kv_chunk(w, 0, 0, 0, 64, "k"))
    for other in (wl.kv_chunk(w, 0, 0, 0, 64, "v"), wl.kv_chunk(w, 1, 0, 0, 64, "k"),
                  wl.kv_chunk(w, 0, 1, 0, 64, "k"), wl.kv_chunk(_small(input_seed=8), 0, 0, 0, 64, "k")):
        assert not torch.equal(a, other)
    q0, q1 = wl.queries(w, 0, 0), wl.queries(w, 0, 1)
    assert q0.shape == (w.batch, w.num_q_heads, w.q_len, w.head_dim)
    assert torch.equal(q0, wl.queries(w, 0, 0)) and not torch.equal(q0, q1)


def test_derive_seed_is_stable_and_63_bit():
    s = wl.derive_seed(4, "k", 0, 0, 0)
    assert s == wl.derive_seed(4, "k", 0, 0, 0)
    assert 0 <= s < 2 ** 63
    assert len({wl.derive_seed(4, t, l, 0, c) for t in "kv" for l in range(4) for c in range(4)}) == 32


def test_tiny_workload_distribution():
    w = wl.tiny()
    x = wl.kv_chunk(w, 0, 0, 0, w.seq_lens[0], "k")
    assert x.dtype == torch.float32 and x.shape == (1, 512, 128)
    n = x.numel()
    # N(0, 0.02^2): mean within 5 standard errors, std within 2 %
    assert abs(float(x.mean())) < 5 * 0.02 / math.sqrt(n)
    assert abs(float(x.std()) / 0.02 - 1) < 0.02


def test_head_scales_apply_per_kv_head():
    w = _small(head_scale_range=(0.5, 2.0))
    s = wl.head_scales(w, 1)
    assert s.shape == (w.num_kv_heads,) and bool(((s >= 0.5) & (s <= 2.0)).all())
    plain = wl.kv_chunk(_small(), 1, 0, 0, 32, "v")
    scaled = wl.kv_chunk(w, 1, 0, 0, 32, "v")
    assert torch.allclose(scaled, plain * s.view(-1, 1, 1))
    qs = wl.queries(w, 1) / wl.queries(_small(), 1)
    assert torch.allclose(qs[0, :, 0, 0], s.repeat_interleave(w.gqa))


@pytest.mark.parametrize("shuffle", [False, True])
def test_block_table_is_a_permutation_of_the_pool(shuffle):
    w = _small(block_tokens=16, shuffle_blocks=shuffle)
    caps = (300, 41, 16, 1)
    table, total = wl.block_table(w, caps)
    need = [(c + 15) // 16 for c in caps]
    assert total == sum(need) and table.shape == (len(caps), max(need)) and table.dtype == torch.int32
    used = torch.cat([table[b, :k] for b, k in enumerate(need)])
    assert sorted(used.tolist()) == list(range(total))
    if not shuffle:
        assert used.tolist() == list(range(total))


def test_paged_batch_lengths_and_stress_rows():
    w = wl.paged_batch()
    assert len(w.seq_lens) == 32 and all(4096 <= n <= 65536 for n in w.seq_lens)
    x = wl.encoder_stress(3, 2, 2, 400, 128, dtype=torch.float32)
    rows = x.reshape(-1, 128)
    nz = (rows != 0).sum(-1)
    assert bool((nz == 0).any())                              # all-zero rows
    assert bool(((nz == 1) & (rows.abs().amax(-1) == 3.0)).any())  # one-hot rows
    assert bool((rows == -0.75).all(-1).any())                # constant rows
    assert bool((rows.abs().amax(-1) < 2.0 ** -80).logical_and(nz > 0).any())  # 2^-100-scaled rows

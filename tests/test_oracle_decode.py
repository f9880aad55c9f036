"""Pins of the oracle's decode attention and of the paged-pool layout."""
import math

import numpy as np
import pytest
from scipy import special

import oracle as O


def _brute(q, K, V, scale, Lq):
    G, _, D = q.shape
    N = K.shape[0]
    out = np.zeros_like(q)
    for g in range(G):
        for l in range(Lq):
            nv = N - Lq + l + 1
            p = special.softmax(K[:nv] @ q[g, l] * scale)
            out[g, l] = p @ V[:nv]
    return out


@pytest.mark.parametrize("Lq", [1, 2, 3, 9])
def test_attention_equals_brute_force(oracle_lib, Lq):
    rng = np.random.default_rng(Lq)
    G, N, D = 3, 9, 16
    q = rng.standard_normal((G, Lq, D))
    K = rng.standard_normal((N, D))
    V = rng.standard_normal((N, D))
    got = O.attention_f64(q, K, V, 0.3, Lq)
    assert np.abs(got - _brute(q, K, V, 0.3, Lq)).max() < 1e-13
    if Lq == N:
        # a chunk that is the whole sequence: its first query sees one token
        assert np.array_equal(got[:, 0], np.broadcast_to(V[0], (G, D)))


def test_attention_single_token_is_value(oracle_lib):
    D = 8
    q = np.ones((1, 1, D))
    K = np.zeros((1, D))
    V = np.arange(D, dtype=np.float64)[None]
    assert np.array_equal(O.attention_f64(q, K, V, 1.0, 1)[0, 0], V[0])


CASES = [
    # D, key (mode, bits), value (mode, bits, group), G, Lq, N
    (128, (O.PROD, 3), (O.MSE, 4, 0), 4, 1, 70),
    (128, (O.MSE, 4), (O.MSE, 4, 0), 8, 2, 64),
    (128, (O.PROD, 3), (O.MSE, 3, 0), 8, 2, 50),
    (256, (O.PROD, 3), (O.GROUP, 2, 32), 8, 1, 40),
    (128, (O.PROD, 3), (O.GROUP, 4, 64), 4, 1, 45),
    # a prefill chunk that is the whole sequence (every query causal)
    (128, (O.PROD, 3), (O.MSE, 3, 0), 2, 24, 24),
]


def _setup(D, kspec, vspec, G, Lq, N, seed=0):
    rng = np.random.default_rng(seed)
    kc = O.Codec(D, kspec[1], kspec[0], 3)
    vc = O.Codec(D, vspec[1], vspec[0], 4, vspec[2])
    K = rng.standard_normal((N, D)).astype(np.float32)
    V = rng.standard_normal((N, D)).astype(np.float32)
    q = rng.standard_normal((G, Lq, D))
    return kc, vc, K, V, q


@pytest.mark.parametrize("case", CASES)
def test_rotated_decode_equals_dequantise_then_attend(oracle_lib, case):
    D, ks, vs, G, Lq, N = case
    kc, vc, K, V, q = _setup(*case)
    kr, vr = kc.encode(K), vc.encode(V)
    scale = 1 / math.sqrt(D)
    plain = O.attention_f64(q, kc.dequant(kr), vc.dequant(vr), scale, Lq)
    rot = O.decode_rotated(q, kc, kr, vc, vr, scale, Lq)
    assert np.abs(plain - rot).max() < 1e-9 * max(1.0, np.abs(plain).max())


@pytest.mark.parametrize("case", CASES[1:3])
def test_query_zero_of_two_ignores_newest_token(oracle_lib, case):
    D, ks, vs, G, Lq, N = case
    kc, vc, K, V, q = _setup(*case)
    kr, vr = kc.encode(K), vc.encode(V)
    base = O.decode_rotated(q, kc, kr, vc, vr, 0.1, Lq)
    K2, V2 = K.copy(), V.copy()
    K2[-1] *= -3
    V2[-1] += 5
    alt = O.decode_rotated(q, kc, kc.encode(K2), vc, vc.encode(V2), 0.1, Lq)
    assert np.array_equal(base[:, 0], alt[:, 0])
    assert not np.allclose(base[:, 1], alt[:, 1])


def test_quality_close_to_exact_attention(oracle_lib):
    # validation-style quality check (cosine of attention outputs)
    D, G, N = 128, 4, 512
    rng = np.random.default_rng(42)
    K = (rng.standard_normal((N, D)) * 0.02).astype(np.float32)
    V = (rng.standard_normal((N, D)) * 0.02).astype(np.float32)
    q = rng.standard_normal((G, 1, D)) * 0.02
    kc, vc = O.Codec(D, 3, O.PROD, 42), O.Codec(D, 4, O.MSE, 43)
    got = O.decode_rotated(q, kc, kc.encode(K), vc, vc.encode(V), 1 / math.sqrt(D), 1)
    ref = O.attention_f64(q, K.astype(np.float64), V.astype(np.float64), 1 / math.sqrt(D), 1)
    cos = (got * ref).sum(-1) / np.linalg.norm(got, axis=-1) / np.linalg.norm(ref, axis=-1)
    assert cos.min() > 0.99


def test_subblock_layout_and_pool_write(oracle_lib):
    D, BT, Hkv = 128, 16, 2
    kc, vc = O.Codec(D, 3, O.PROD, 0), O.Codec(D, 4, O.GROUP, group=64)
    sub, off = O.subblock_layout(kc, vc, BT)
    assert sub == BT * (kc.record_bytes + vc.record_bytes)
    assert kc.record_bytes == 56 and vc.record_bytes == 72
    assert all(o % 16 == 0 for o in off if o >= 0)
    rng = np.random.default_rng(0)
    K = rng.standard_normal((40, D)).astype(np.float32)
    V = rng.standard_normal((40, D)).astype(np.float32)
    kr, vr = kc.encode(K), vc.encode(V)
    table = np.array([[5, 2, 7]], np.int32)
    pool = np.zeros(8 * Hkv * sub, np.uint8)
    O.pool_write(pool, kc, vc, Hkv, BT, table, 3, 0, 1, 0, kr, vr)
    # token 37 -> logical block 2 -> physical 7, slot 5, head 1
    base = (7 * Hkv + 1) * sub
    t, slot = 37, 5
    got = pool[base + off[0] + slot * 32: base + off[0] + slot * 32 + 32].view(np.uint32)
    assert np.array_equal(got, kr["idx"][t])
    assert pool[base + off[2] + 4 * slot: base + off[2] + 4 * slot + 4].view(np.float32)[0] == kr["norm"][t]
    assert np.array_equal(pool[base + off[6] + 4 * slot: base + off[6] + 4 * slot + 4].view(np.uint16),
                          vr["min"][t])
    # head 0 and unused blocks untouched
    assert not pool[(7 * Hkv) * sub:(7 * Hkv + 1) * sub].any()
    assert not pool[0:(2 * Hkv) * sub].any()


# ------------------------------------------------------------------ sequence-sharded decode

def _slice_rec(rec, a, b):
    return {k: v[a:b] for k, v in rec.items()}


@pytest.mark.parametrize("case", CASES[:5])
def test_partial_state_equals_dequantised_brute_force(oracle_lib, case):
    # (m, l, acc) of a shard computed independently: scores from the
    # dequantised keys, values in the rotated domain (MSE) or as dequantised
    # (group)
    D, ks, vs, G, Lq, N = case
    kc, vc, K, V, q = _setup(*case)
    kr, vr = kc.encode(K), vc.encode(V)
    scale = 1 / math.sqrt(D)
    a, b = N // 3, N - 5
    E = N - a                                  # the shard's causal end: the global end, locally
    m, l, acc = O.decode_partial(q, kc, _slice_rec(kr, a, b), vc, _slice_rec(vr, a, b), scale, Lq, E)
    Kh, Vh = kc.dequant(kr)[a:b], vc.dequant(vr)[a:b]
    # V_hat = (n c_hat) @ R_v: the rotated-domain value is V_hat R_v^-1 (the
    # fp32 table is orthogonal only to ~1e-7, so its transpose is not exact)
    Vr = Vh @ np.linalg.inv(vc.R.astype(np.float64)) if vc.mode == O.MSE else Vh
    for g in range(G):
        for lq in range(Lq):
            r = g * Lq + lq
            nv = min(b - a, E - Lq + lq + 1)
            s = scale * (Kh[:nv] @ q[g, lq])
            mm = s.max()
            p = np.exp(s - mm)
            assert abs(m[r] - mm) <= 1e-12 * max(1.0, abs(mm))
            assert abs(l[r] - p.sum()) <= 1e-11 * p.sum()
            assert np.abs(acc[r] - p @ Vr[:nv]).max() <= 1e-10 * max(1.0, np.abs(acc[r]).max())


@pytest.mark.parametrize("case", CASES)
def test_merged_shards_equal_the_unsharded_decode(oracle_lib, case):
    D, ks, vs, G, Lq, N = case
    kc, vc, K, V, q = _setup(*case)
    kr, vr = kc.encode(K), vc.encode(V)
    scale = 1 / math.sqrt(D)
    ref = O.decode_rotated(q, kc, kr, vc, vr, scale, Lq).reshape(G * Lq, D)
    # one part with its own end is the plain decode
    m, l, acc = O.decode_partial(q, kc, kr, vc, vr, scale, Lq)
    one = O.merge_partials(vc, m[None], l[None], acc[None])
    assert np.abs(one - ref).max() <= 1e-12 * max(1.0, np.abs(ref).max())
    # three shards, the last one shorter than the query chunk when Lq is large
    cuts = [0, N // 2, N - 1, N] if Lq > 2 else [0, 7, N // 2, N]
    parts = [O.decode_partial(q, kc, _slice_rec(kr, a, b), vc, _slice_rec(vr, a, b), scale, Lq, N - a)
             for a, b in zip(cuts[:-1], cuts[1:])]
    m = np.stack([p[0] for p in parts])
    l = np.stack([p[1] for p in parts])
    acc = np.stack([p[2] for p in parts])
    got = O.merge_partials(vc, m, l, acc)
    assert np.abs(got - ref).max() <= 1e-11 * max(1.0, np.abs(ref).max())
    # the order of the parts does not matter
    rev = O.merge_partials(vc, m[::-1], l[::-1], acc[::-1])
    assert np.abs(rev - ref).max() <= 1e-11 * max(1.0, np.abs(ref).max())


def test_shard_with_no_visible_key_is_neutral(oracle_lib):
    D, ks, vs, G, Lq, N = CASES[5]           # a whole-sequence chunk: query 0 sees token 0 only
    kc, vc, K, V, q = _setup(*CASES[5])
    kr, vr = kc.encode(K), vc.encode(V)
    m, l, acc = O.decode_partial(q, kc, _slice_rec(kr, 1, N), vc, _slice_rec(vr, 1, N), 0.1, Lq, N - 1)
    # rows of query 0 see no key of the shard [1, N)
    rows0 = [g * Lq for g in range(G)]
    assert np.all(m[rows0] == -np.inf) and np.all(l[rows0] == 0) and not acc[rows0].any()
    m0, l0, a0 = O.decode_partial(q, kc, _slice_rec(kr, 0, 1), vc, _slice_rec(vr, 0, 1), 0.1, Lq, N)
    both = O.merge_partials(vc, np.stack([m, m0]), np.stack([l, l0]), np.stack([acc, a0]))
    ref = O.decode_rotated(q, kc, kr, vc, vr, 0.1, Lq).reshape(G * Lq, D)
    assert np.abs(both - ref).max() <= 1e-11 * max(1.0, np.abs(ref).max())
    # an all-empty merge gives zeros rather than NaN
    empty = O.merge_partials(vc, np.full((2, G * Lq), -np.inf), np.zeros((2, G * Lq)), np.zeros((2, G * Lq, D)))
    assert not empty.any()

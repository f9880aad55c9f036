"""Pins of the oracle's decode over split (low/high) states.

The oracle decodes a split state by the plain definition (each half
dequantised by its own codec, the halves concatenated, plain attention). Here
that is checked against an independent route in the rotated domain of each
half (the form the GPU kernel computes), against the causal rule, and against
what a mixed width means for the reconstruction error.
"""
import math

import numpy as np
import pytest

import oracle as O


def _half(D, kspec, vspec, seed):
    kc = O.Codec(D, kspec[1], kspec[0], seed)
    vc = O.Codec(D, vspec[1], vspec[0], seed + 1, vspec[2] if len(vspec) > 2 else 0)
    return kc, vc


def _rotated_split(q, halves, scale, Lq):
    """softmax(sum of the halves' rotated-domain scores) . [V_low | V_high]."""
    G, _, D = q.shape
    N = halves[0][1]["idx"].shape[0]
    out = np.zeros((G, Lq, D))
    d0 = 0
    parts = []
    for kc, kr, vc, vr in halves:
        Dh = kc.D
        codes_k = np.stack([O.unpack(w, Dh, kc.ib) for w in kr["idx"]]).astype(np.int64)
        ck = kc.c.astype(np.float64)[codes_k] * kr["norm"].astype(np.float64)[:, None]       # n c[idx]
        sig = None
        if kc.mode == O.PROD:
            bits = np.stack([O.unpack(w, Dh, 1) for w in kr["sgn"]]).astype(np.float64)
            sig = (2 * bits - 1) * (math.sqrt(math.pi / 2) / Dh * kr["rnorm"].astype(np.float64)
                                    * kr["norm"].astype(np.float64))[:, None]
        if vc.mode == O.GROUP:
            vv = vc.dequant(vr)
        else:
            codes_v = np.stack([O.unpack(w, Dh, vc.ib) for w in vr["idx"]]).astype(np.int64)
            vv = vc.c.astype(np.float64)[codes_v] * vr["norm"].astype(np.float64)[:, None]    # rotated domain
        parts.append((kc, ck, sig, vc, vv, d0, Dh))
        d0 += Dh
    for g in range(G):
        for l in range(Lq):
            nv = N - Lq + l + 1
            s = np.zeros(nv)
            for kc, ck, sig, vc, vv, a, Dh in parts:
                q1 = kc.R.astype(np.float64) @ q[g, l, a:a + Dh]
                s += ck[:nv] @ q1
                if sig is not None:
                    s += sig[:nv] @ (kc.S.astype(np.float64) @ q1)
            p = np.exp(scale * s - (scale * s).max())
            p /= p.sum()
            for kc, ck, sig, vc, vv, a, Dh in parts:
                o = p @ vv[:nv]
                out[g, l, a:a + Dh] = o @ vc.R.astype(np.float64) if vc.mode != O.GROUP else o
    return out


CASES = [
    # (low D, key, value), (high D, key, value), G, Lq, N
    ((64, (O.PROD, 3), (O.MSE, 3)), (64, (O.MSE, 4), (O.MSE, 4)), 4, 2, 37),
    ((128, (O.PROD, 3), (O.MSE, 2)), (128, (O.PROD, 4), (O.GROUP, 4, 64)), 2, 1, 25),
    ((64, (O.MSE, 2), (O.GROUP, 2, 32)), (128, (O.MSE, 4), (O.MSE, 4)), 3, 3, 19),
]


@pytest.mark.parametrize("low,high,G,Lq,N", CASES)
def test_split_decode_equals_rotated_domain_route(oracle_lib, low, high, G, Lq, N):
    rng = np.random.default_rng(N)
    D = low[0] + high[0]
    halves = []
    X = rng.standard_normal((2, N, D)).astype(np.float32)
    q = rng.standard_normal((G, Lq, D))
    for (Dh, ks, vs), a, seed in ((low, 0, 5), (high, low[0], 9)):
        kc, vc = _half(Dh, ks, vs, seed)
        halves.append((kc, kc.encode(X[0][:, a:a + Dh]), vc, vc.encode(X[1][:, a:a + Dh])))
    scale = 1 / math.sqrt(D)
    got = O.decode_split(q, halves[0], halves[1], scale, Lq)
    ref = _rotated_split(q, halves, scale, Lq)
    assert np.abs(got - ref).max() < 1e-9 * max(1.0, np.abs(ref).max())
    # the causal rule: query 0 of Lq > 1 never sees the newest token
    if Lq > 1:
        X2 = X.copy()
        X2[:, -1] *= -4
        halves2 = []
        for (Dh, ks, vs), a, seed in ((low, 0, 5), (high, low[0], 9)):
            kc, vc = _half(Dh, ks, vs, seed)
            halves2.append((kc, kc.encode(X2[0][:, a:a + Dh]), vc, vc.encode(X2[1][:, a:a + Dh])))
        alt = O.decode_split(q, halves2[0], halves2[1], scale, Lq)
        assert np.array_equal(alt[:, 0], got[:, 0]) and not np.allclose(alt[:, -1], got[:, -1])


def test_mixed_width_reconstruction_error_is_the_halves_average(oracle_lib):
    # 2-bit low half and 4-bit high half of unit-variance vectors: the relative
    # reconstruction error is the average of the two halves' Lloyd-Max
    # distortions (each half carries about half of the energy), between the
    # uniform 2-bit and 4-bit errors; the average width is 3 bits
    D, n = 128, 3000
    rng = np.random.default_rng(1)
    X = rng.standard_normal((n, D)).astype(np.float32)

    def rel_err(kc, x):
        xh = kc.dequant(kc.encode(x))
        return float(((xh - x) ** 2).sum() / (x.astype(np.float64) ** 2).sum())

    lo, hi = O.Codec(64, 2, O.MSE, 3), O.Codec(64, 4, O.MSE, 4)
    e_lo, e_hi = rel_err(lo, X[:, :64]), rel_err(hi, X[:, 64:])
    xs = np.concatenate([lo.dequant(lo.encode(X[:, :64])), hi.dequant(hi.encode(X[:, 64:]))], axis=1)
    e_split = float(((xs - X) ** 2).sum() / (X.astype(np.float64) ** 2).sum())
    assert abs(e_split - 0.5 * (e_lo + e_hi)) < 0.05 * e_split
    e2 = rel_err(O.Codec(D, 2, O.MSE, 3), X)
    e4 = rel_err(O.Codec(D, 4, O.MSE, 3), X)
    assert e4 < e_split < e2
    assert (64 * lo.bits + 64 * hi.bits) / D == 3

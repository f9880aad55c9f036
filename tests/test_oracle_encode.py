"""Pins of the oracle's bit packing, fp16 conversion and encoders.

Each encoder is checked against properties fixed by the definitions rather
than by re-running its own formula: nearest-centroid coding in fp64 away from
the fp32 error bound, norms, the residual norm and sign sketch, group
reconstruction bounds, the expected distortion and the unbiasedness and exact
variance of the QJL inner-product estimator over seeds.
"""
import math

import numpy as np
import pytest
from scipy import integrate

from conftest import read_golden

import oracle as O

U32 = 2.0 ** -24


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("b", range(1, 9))
def test_pack_roundtrip(oracle_lib, D, b):
    rng = np.random.default_rng(D * 10 + b)
    W = O.packed_words(D, b)
    assert W == -(-D * b // 32)
    for codes in (rng.integers(0, 1 << b, D), np.full(D, (1 << b) - 1), np.zeros(D)):
        w = O.pack(codes, D, b)
        assert np.array_equal(O.unpack(w, D, b), codes.astype(np.uint8))
        # every code is recoverable from the bit stream at position i*b
        bits = np.unpackbits(w.view(np.uint8), bitorder="little")
        for i in (0, D // 2, D - 1):
            v = sum(int(bits[i * b + k]) << k for k in range(b))
            assert v == codes[i]


def test_pack_hand_example(oracle_lib):
    want = [int(v, 16) for _, v in read_golden("pack_3bit_example.txt")]
    assert [int(x) for x in O.pack(np.arange(32) % 8, 32, 3)] == want


def test_packed_width_and_head_dim_inference(oracle_lib):
    for D, bits, mode, W, Dinf in read_golden("packed_width.txt"):
        D, bits, W, Dinf = int(D), int(bits), int(W), int(Dinf)
        m = O.PROD if mode == "prod" else O.MSE
        ib = O.index_bits(bits, m)
        assert O.packed_words(D, ib) == W
        assert W * 32 // max(ib, 1) == Dinf == D


def test_fp16_conversion_matches_ieee(oracle_lib):
    rng = np.random.default_rng(1)
    xs = np.concatenate([
        rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 20000),
        np.array([0.0, -0.0, 65504.0, 65519.0, 65520.0, 1e9, -1e9, 2.0 ** -24, 2.0 ** -25,
                  1.5 * 2.0 ** -25, 2.0 ** -14, 2.0 ** -14 * (1 - 2.0 ** -11), 1.0 + 2.0 ** -11,
                  1.0 + 3 * 2.0 ** -11, np.inf, -np.inf], np.float32)])
    for x in xs:
        h = O.f32_to_f16_bits(float(x))
        with np.errstate(over="ignore"):   # values past the binary16 range round to infinity
            ref = int(np.float32(x).astype(np.float16).view(np.uint16))
        assert h == ref, x
        assert O.f16_bits_to_f32(h) == float(np.uint16(h).view(np.float16).astype(np.float32))


def _ambiguity(R, x, n):
    # fp32 sequential-fma dot product error bound, relative to the unit domain
    D = len(x)
    g = D * U32 / (1 - D * U32)
    return (g * np.abs(R) @ np.abs(x)) / n + 4 * U32


@pytest.mark.parametrize("D,b", [(128, 2), (128, 3), (128, 4), (256, 2), (64, 1)])
def test_mse_encode_is_nearest_centroid(oracle_lib, D, b):
    cd = O.Codec(D, b, O.MSE, 3)
    rng = np.random.default_rng(b)
    x = (rng.standard_normal((300, D)) * rng.uniform(0.01, 5, (300, 1))).astype(np.float32)
    x[0] = 0.0
    rec = cd.encode(x)
    R = cd.R.astype(np.float64)
    c = cd.c.astype(np.float64)
    checked = 0
    for v in range(len(x)):
        xv = x[v].astype(np.float64)
        n = np.linalg.norm(xv)
        assert abs(rec["norm"][v] - n) <= (D + 2) * U32 * n + 1e-45
        codes = O.unpack(rec["idx"][v], D, b).astype(int)
        if n == 0:
            assert np.all(codes == (1 << b) // 2 - 1)   # y = 0 sits below the zero midpoint
            continue
        y = R @ xv / n
        amb = _ambiguity(R, xv, n)
        near = np.argmin(np.abs(y[:, None] - c[None, :]), axis=1)
        dist_mid = np.min(np.abs(y[:, None] - cd.m.astype(np.float64)[None, :]), axis=1)
        ok = dist_mid > amb
        assert np.array_equal(codes[ok], near[ok])
        checked += ok.sum()
    assert checked > 0.99 * 299 * D


def test_prod_encode_residual_and_signs(oracle_lib):
    D, bits = 128, 3
    cd = O.Codec(D, bits, O.PROD, 9)
    rng = np.random.default_rng(2)
    x = rng.standard_normal((200, D)).astype(np.float32)
    rec = cd.encode(x)
    R, S, c = (a.astype(np.float64) for a in (cd.R, cd.S, cd.c))
    for v in range(len(x)):
        xv = x[v].astype(np.float64)
        n = np.linalg.norm(xv)
        codes = O.unpack(rec["idx"][v], D, 2).astype(int)
        r = R @ xv / n - c[codes]
        assert abs(rec["rnorm"][v] - np.linalg.norm(r)) < 1e-5 * np.linalg.norm(r) + 1e-6
        z = S @ r
        sg = np.unpackbits(rec["sgn"][v].view(np.uint8), bitorder="little").astype(bool)
        clear = np.abs(z) > 1e-4 * np.abs(S) @ np.abs(r)
        assert np.array_equal(sg[clear], (z >= 0)[clear])


@pytest.mark.parametrize("bits,g", [(2, 32), (4, 64), (4, 32), (3, 16)])
def test_group_encode_bounds(oracle_lib, bits, g):
    D = 128
    cd = O.Codec(D, bits, O.GROUP, group=g)
    rng = np.random.default_rng(bits)
    x = (rng.standard_normal((300, D)) * 0.7 + rng.uniform(-3, 3, (300, 1))).astype(np.float32)
    x[1, :g] = 0.25            # a constant group: zero scale, all codes 0
    rec = cd.encode(x)
    qmax = (1 << bits) - 1
    for v in range(len(x)):
        codes = O.unpack(rec["idx"][v], D, bits).astype(np.float64)
        assert codes.max() <= qmax
        for gi in range(D // g):
            xs = x[v, gi * g:(gi + 1) * g]
            lo, hi = xs.min(), xs.max()
            s_want = np.float32((np.float32(hi) - np.float32(lo)) / np.float32(qmax)).astype(np.float16)
            m_want = np.float32(lo).astype(np.float16)
            assert rec["scale"][v, gi] == s_want.view(np.uint16)
            assert rec["min"][v, gi] == m_want.view(np.uint16)
            s, m0 = float(s_want), float(m_want)
            rec_x = codes[gi * g:(gi + 1) * g] * s + m0
            if s == 0:
                assert np.all(codes[gi * g:(gi + 1) * g] == 0)
                continue
            # within half a step (plus fp16 rounding of min and scale) of the input
            err = np.abs(rec_x - xs.astype(np.float64))
            slack = 0.5 * s + abs(m0 - lo) + qmax * abs(s - (hi - lo) / qmax) + 1e-6
            assert err.max() <= slack


@pytest.mark.parametrize("D,b", [(128, 2), (128, 4), (256, 3)])
def test_mse_distortion_matches_lloyd_max(oracle_lib, D, b):
    # relative squared error of n * (c @ R) equals the per-coordinate Lloyd-Max
    # distortion times D (the rotation is an isometry), averaged over inputs.
    cd = O.Codec(D, b, O.MSE, 4)
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3000, D)).astype(np.float32)
    xh = cd.dequant(cd.encode(x))
    rel = ((xh - x) ** 2).sum(1) / (x.astype(np.float64) ** 2).sum(1)
    c, m, _ = O.lloyd_max(D, b)
    f = lambda t: (1 - t * t) ** ((D - 3) / 2)
    e = np.concatenate([[-1.0], m, [1.0]])
    Z = integrate.quad(f, -1, 1, epsrel=1e-12)[0]
    dist = sum(integrate.quad(lambda t, cj=cj: (t - cj) ** 2 * f(t), e[j], e[j + 1])[0]
               for j, cj in enumerate(c)) / Z
    assert abs(rel.mean() / (D * dist) - 1) < 0.03


def test_qjl_estimator_unbiased_with_exact_variance(oracle_lib):
    # Over codec seeds, <q, x_prod> - <q, x> is zero-mean, with variance
    # E[((pi/2)|q|^2 |r|^2 - <Rq, r>^2) / D] per unit norm (QJL estimator).
    D, bits, M = 64, 2, 3000
    rng = np.random.default_rng(5)
    x = rng.standard_normal(D).astype(np.float32)
    q = (x + 0.5 * rng.standard_normal(D)).astype(np.float64)
    err, pred = [], []
    for s in range(M):
        cd = O.Codec(D, bits, O.PROD, 20000 + s)
        rec = cd.encode(x[None])
        n = float(rec["norm"][0])
        full = cd.dequant(rec)[0]
        rec0 = dict(rec, rnorm=np.zeros(1, np.float32))
        mse_part = cd.dequant(rec0)[0]
        qx = q @ x.astype(np.float64)
        qr = (qx - q @ mse_part) / n            # <R q, r>
        err.append((q @ full - qx) / n)
        g = float(rec["rnorm"][0])
        pred.append(((math.pi / 2) * (q @ q) * g * g - qr * qr) / D)
    err, pred = np.array(err), np.array(pred)
    assert abs(err.mean()) < 4 * err.std() / math.sqrt(M)
    assert abs((err ** 2).mean() / pred.mean() - 1) < 0.1

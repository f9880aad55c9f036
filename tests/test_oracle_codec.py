"""Pins of the oracle's codec builder against what the pages and the
mathematics fix: published generator outputs, orthogonality, the QR
definition, the Lloyd-Max centroid/midpoint conditions, closed forms and the
Gaussian limit, and an independent Monte-Carlo check of the coordinate density.
"""
import math

import numpy as np
import pytest
from scipy import integrate, special, stats

from conftest import read_golden

import oracle as O


def test_splitmix64_published_outputs(oracle_lib):
    for seed, i, val in read_golden("splitmix64.txt"):
        assert O.lib().tqo_splitmix64_at(int(seed), int(i)) == int(val)


def test_normals_are_standard_normal(oracle_lib):
    x = O.normals(7, 0, 400_000)
    assert abs(x.mean()) < 4 / math.sqrt(len(x))
    assert abs(x.var() - 1) < 0.01
    assert stats.kstest(x, "norm").pvalue > 1e-3
    # independent streams of one seed and of adjacent seeds differ
    assert not np.array_equal(O.normals(7, 1, 100), O.normals(7, 0, 100))
    assert not np.array_equal(O.normals(8, 0, 100), O.normals(7, 0, 100))
    assert np.array_equal(O.normals(7, 0, 101)[:100], O.normals(7, 0, 100))


@pytest.mark.parametrize("D", [64, 128, 256])
def test_rotation_is_orthogonal_qr_factor(oracle_lib, D):
    R = O.rotation_f64(D, 11)
    assert np.abs(R.T @ R - np.eye(D)).max() < 1e-12
    # R is the Q factor with positive diagonal of the seeded Gaussian matrix:
    # U = R^T G must be upper triangular with a positive diagonal.
    G = O.normals(11, 0, D * D).reshape(D, D)
    U = R.T @ G
    assert np.abs(np.tril(U, -1)).max() < 1e-10 * np.abs(U).max()
    assert (np.diag(U) > 0).all()
    # the stored fp32 table stays orthogonal to the benchmark spec's bound
    c = O.Codec(D, 4, O.MSE, 11)
    R32 = c.R.astype(np.float64)
    assert np.abs(R32.T @ R32 - np.eye(D)).max() < 1e-5


def test_rotation_haar_second_moment(oracle_lib):
    # For a Haar R, (R q)_i^2 has mean |q|^2 / D for every i.
    D, M = 64, 400
    q = np.random.default_rng(0).standard_normal(D)
    acc = np.zeros(D)
    for s in range(M):
        acc += (O.rotation_f64(D, 1000 + s) @ q) ** 2
    mean = acc / M
    target = q @ q / D
    # each entry is an average of M Beta-like variables with variance ~ 2 target^2
    assert np.abs(mean / target - 1).max() < 6 * math.sqrt(2 / M)


def _density(D):
    a = (D - 3) / 2
    return lambda t: (1 - t * t) ** a


@pytest.mark.parametrize("D", [64, 128, 256])
@pytest.mark.parametrize("b", [1, 2, 3, 4])
def test_lloyd_max_conditions(oracle_lib, D, b):
    c, m, _ = O.lloyd_max(D, b)
    L = 1 << b
    f = _density(D)
    # midpoint condition and ordering
    assert np.all(np.diff(c) > 0)
    assert np.allclose(m, (c[:-1] + c[1:]) / 2, rtol=0, atol=1e-17)
    # exact antisymmetry
    assert np.array_equal(c[::-1], -c)
    # centroid condition, by independent adaptive quadrature
    edges = np.concatenate([[-1.0], m, [1.0]])
    for j in range(L):
        lo, hi = edges[j], edges[j + 1]
        num = integrate.quad(lambda t: t * f(t), lo, hi, epsabs=0, epsrel=1e-13, limit=200)[0]
        den = integrate.quad(f, lo, hi, epsabs=0, epsrel=1e-13, limit=200)[0]
        assert abs(num / den - c[j]) < 1e-10 * max(1.0, abs(c[j]))


@pytest.mark.parametrize("D", [64, 128, 256, 1001])
def test_lloyd_max_one_bit_closed_form(oracle_lib, D):
    c, m, _ = O.lloyd_max(D, 1)
    exact = math.exp(math.lgamma(D / 2) - math.lgamma((D + 1) / 2)) / math.sqrt(math.pi)
    assert abs(c[1] - exact) < 1e-14 and c[0] == -c[1] and m[0] == 0.0


def test_lloyd_max_gaussian_limit(oracle_lib):
    # sqrt(D) * levels tend to the Gaussian Lloyd-Max levels with an O(1/D) gap.
    for row in read_golden("gaussian_lloyd_max.txt"):
        b, dist = int(row[0]), float(row[1])
        levels = np.array([float(v) for v in row[2:]])
        gaps = []
        for D in (128, 256, 512):
            c, m, _ = O.lloyd_max(D, b)
            half = c[len(c) // 2:] * math.sqrt(D)
            gaps.append(np.abs(half - levels).max() / levels.max())
        assert gaps[-1] < 0.006
        # gap roughly halves as D doubles (table rounding floor ~1e-3 relative)
        assert gaps[1] < 0.65 * gaps[0] + 1e-3 and gaps[2] < 0.65 * gaps[1] + 1e-3
        # per-coordinate distortion * D approaches the Gaussian distortion
        D = 512
        c, m, _ = O.lloyd_max(D, b)
        f = _density(D)
        edges = np.concatenate([[-1.0], m, [1.0]])
        Z = integrate.quad(f, -1, 1, epsrel=1e-12)[0]
        mse = sum(integrate.quad(lambda t, cj=cj: (t - cj) ** 2 * f(t), edges[j], edges[j + 1],
                                 epsrel=1e-12)[0] for j, cj in enumerate(c)) / Z
        assert abs(mse * D / dist - 1) < 0.02


@pytest.mark.parametrize("D,b", [(128, 2), (128, 3), (64, 4)])
def test_lloyd_max_density_is_unit_sphere_coordinate(oracle_lib, D, b):
    # Independent of the density formula: a coordinate of a uniform unit vector
    # in R^D has t^2 ~ Beta(1/2, (D-1)/2). Empirical cell means must match the
    # centroids to Monte-Carlo accuracy.
    rng = np.random.default_rng(123)
    n = 4_000_000
    t = np.sqrt(rng.beta(0.5, (D - 1) / 2, n)) * rng.choice([-1.0, 1.0], n)
    c, m, _ = O.lloyd_max(D, b)
    cell = np.searchsorted(m, t, side="left")
    for j in range(len(c)):
        tj = t[cell == j]
        se = tj.std() / math.sqrt(len(tj))
        assert abs(tj.mean() - c[j]) < 5 * se + 1e-12


def test_codec_determinism_and_seed_separation(oracle_lib):
    a = O.Codec(128, 3, O.PROD, 5)
    b = O.Codec(128, 3, O.PROD, 5)
    v = O.Codec(128, 3, O.PROD, 6)
    assert np.array_equal(a.R, b.R) and np.array_equal(a.S, b.S)
    assert not np.array_equal(a.R, v.R)
    # the QJL matrix is a different stream from the rotation of the same seed
    assert not np.allclose(a.S[:4], O.normals(5, 0, 4 * 128).reshape(4, 128))
    assert np.array_equal(a.S, O.normals(5, 1, 128 * 128).reshape(128, 128).astype(np.float32))
    # prod uses bits-1 index bits; its codebook is the (bits-1)-bit MSE codebook
    mse2 = O.Codec(128, 2, O.MSE, 5)
    assert a.ib == 2 and np.array_equal(a.c, mse2.c) and np.array_equal(a.R, mse2.R)


@pytest.mark.parametrize("D,bits,mode", [(128, 3, O.PROD), (128, 4, O.MSE), (256, 3, O.MSE), (64, 1, O.MSE),
                                         (128, 2, O.MSE), (256, 5, O.PROD)])
def test_stored_fp32_levels_meet_lloyd_max_conditions(oracle_lib, D, bits, mode):
    # The codec's stored fp32 tables, checked directly against the Lloyd-Max
    # conditions by independent adaptive quadrature: each stored level is the
    # centroid of the cell that the stored thresholds bound, and each stored
    # threshold is the midpoint of its two stored levels, both to fp32
    # precision (a few units in the last place).
    cd = O.Codec(D, bits, mode, 1)
    c = cd.c.astype(np.float64)
    m = cd.m.astype(np.float64)
    ulp = lambda x: np.spacing(np.float32(abs(x))).astype(np.float64)
    f = _density(D)
    edges = np.concatenate([[-1.0], m, [1.0]])
    for j in range(len(c)):
        lo, hi = edges[j], edges[j + 1]
        num = integrate.quad(lambda t: t * f(t), lo, hi, epsabs=0, epsrel=1e-13, limit=200)[0]
        den = integrate.quad(f, lo, hi, epsabs=0, epsrel=1e-13, limit=200)[0]
        assert abs(num / den - c[j]) <= 2 * ulp(c[j]), (j, num / den, c[j])
    for j in range(len(m)):
        assert abs((c[j] + c[j + 1]) / 2 - m[j]) <= ulp(m[j]) + 1e-300, (j, m[j])
    assert np.array_equal(cd.c[::-1], -cd.c)
    # levels are not rounded to a coarser grid: at least one level needs more
    # than the 11 significant bits of a half-precision number
    assert not np.array_equal(c, c.astype(np.float16).astype(np.float64))


def test_fractional_bits_split(oracle_lib):
    # the codec rebuild of "omlx/turboquant_kv.py" (_rebuild_codecs): a width
    # more than 1e-6 from an integer gives keys floor(b) and values ceil(b);
    # otherwise both get int(b), which truncates
    cases = {
        3.5: (3, 4), 2.5: (2, 3), 1.5: (1, 2), 2.25: (2, 3), 3.75: (3, 4),
        1.0: (1, 1), 2.0: (2, 2), 3.0: (3, 3), 4.0: (4, 4),
        3.0000005: (3, 3),      # inside the tolerance above 3
        2.9999995: (2, 2),      # inside the tolerance below 3: int() truncates
        3.00001: (3, 4),        # outside the tolerance: fractional
        2.99999: (2, 3),
    }
    for b, want in cases.items():
        assert O.bits_split(b) == want, b
    # a half-integer width averages exactly over one key and one value
    for b in (1.5, 2.5, 3.5):
        kb, vb = O.bits_split(b)
        assert (kb + vb) / 2 == b

// Host-side codec construction for libtq: seeded rotation, QJL matrix and
// Lloyd-Max codebook. Runs once per tq_codec_create, never on the decode path.
//
// Follows "omlx/turboquant_kv.py" (_rebuild_codecs: a codec is a pure function
// of head_dim, bits and seed) and "lightning-mlx/plan.md" (random orthogonal
// rotation + Lloyd-Max codebook). The construction below is fixed exactly so
// that the fp32 tables are reproducible on any machine:
//   normals: SplitMix64 stream seeded with 2*seed + stream, uniforms
//            ((z >> 12) + 1/2) / 2^52, Box-Muller pairs;
//   rotation: Householder QR of the Gaussian matrix (row-major fill), every
//            sum in ascending index order without fused multiply-add, then
//            the columns signed so that R's diagonal is positive;
//   codebook: Lloyd iteration on (1-t^2)^((D-3)/2) over [-1, 1]; levels and
//            midpoints stored as the nearest fp32 numbers.
// This file must be compiled without floating-point contraction.
#include "tq_internal.h"

#include <cmath>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

namespace tq {
namespace {

struct SplitMix64 {
    uint64_t state;
    uint64_t next() {
        state += 0x9E3779B97F4A7C15ULL;
        uint64_t z = state;
        z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
        z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
        return z ^ (z >> 31);
    }
    double uniform() { return (static_cast<double>(next() >> 12) + 0.5) * 0x1.0p-52; }
};

std::vector<double> gaussian_matrix(int D, uint64_t seed, int stream) {
    SplitMix64 g{seed * 2u + static_cast<uint64_t>(stream)};
    const size_t n = static_cast<size_t>(D) * D;
    std::vector<double> out(n);
    const double two_pi = 6.283185307179586;
    for (size_t k = 0; k < n; k += 2) {
        const double u1 = g.uniform();
        const double u2 = g.uniform();
        const double rad = std::sqrt(-2.0 * std::log(u1));
        const double ang = two_pi * u2;
        out[k] = rad * std::cos(ang);
        if (k + 1 < n) out[k + 1] = rad * std::sin(ang);
    }
    return out;
}

// Householder QR; returns Q * diag(sign(R_kk)) row-major.
std::vector<double> haar_rotation(int D, uint64_t seed) {
    // Work column-major: col[j][i] = A(i, j).
    std::vector<double> g = gaussian_matrix(D, seed, 0);
    std::vector<std::vector<double>> col(D, std::vector<double>(D));
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) col[j][i] = g[static_cast<size_t>(i) * D + j];

    std::vector<std::vector<double>> refl(D);  // reflector k, entries k..D-1
    std::vector<double> refl_sq(D, 0.0);
    std::vector<double> sgn(D, 1.0);
    for (int k = 0; k < D; ++k) {
        const std::vector<double>& x = col[k];
        double ss = 0.0;
        for (int i = k; i < D; ++i) ss = ss + x[i] * x[i];
        const double norm = std::sqrt(ss);
        const double alpha = (x[k] > 0.0) ? -norm : norm;
        sgn[k] = (alpha < 0.0) ? -1.0 : 1.0;
        std::vector<double> v(D, 0.0);
        v[k] = x[k] - alpha;
        for (int i = k + 1; i < D; ++i) v[i] = x[i];
        double vv = 0.0;
        for (int i = k; i < D; ++i) vv = vv + v[i] * v[i];
        refl[k] = v;
        refl_sq[k] = vv;
        if (vv == 0.0) continue;
        for (int j = k + 1; j < D; ++j) {
            std::vector<double>& a = col[j];
            double dot = 0.0;
            for (int i = k; i < D; ++i) dot = dot + v[i] * a[i];
            const double f = (2.0 * dot) / vv;
            for (int i = k; i < D; ++i) a[i] = a[i] - f * v[i];
        }
    }
    // Accumulate Q = H_0 ... H_{D-1} applied to the identity, last reflector first.
    std::vector<std::vector<double>> qcol(D, std::vector<double>(D, 0.0));
    for (int j = 0; j < D; ++j) qcol[j][j] = 1.0;
    for (int k = D - 1; k >= 0; --k) {
        if (refl_sq[k] == 0.0) continue;
        const std::vector<double>& v = refl[k];
        for (int j = 0; j < D; ++j) {
            std::vector<double>& a = qcol[j];
            double dot = 0.0;
            for (int i = k; i < D; ++i) dot = dot + v[i] * a[i];
            const double f = (2.0 * dot) / refl_sq[k];
            for (int i = k; i < D; ++i) a[i] = a[i] - f * v[i];
        }
    }
    std::vector<double> R(static_cast<size_t>(D) * D);
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) R[static_cast<size_t>(i) * D + j] = qcol[j][i] * sgn[j];
    return R;
}

// Gauss-Legendre nodes and weights on [-1, 1] (Newton on P_n).
void gauss_legendre(int n, std::vector<double>& x, std::vector<double>& w) {
    x.assign(n, 0.0);
    w.assign(n, 0.0);
    const double pi = 3.141592653589793;
    for (int i = 0; i < (n + 1) / 2; ++i) {
        double z = std::cos(pi * (i + 0.75) / (n + 0.5));
        double dp = 0.0;
        for (int it = 0; it < 100; ++it) {
            double p0 = 1.0, p1 = z;
            for (int k = 2; k <= n; ++k) {
                double p2 = ((2.0 * k - 1.0) * z * p1 - (k - 1.0) * p0) / k;
                p0 = p1;
                p1 = p2;
            }
            dp = n * (z * p1 - p0) / (z * z - 1.0);
            const double dz = p1 / dp;
            z -= dz;
            if (std::fabs(dz) < 1e-16) break;
        }
        x[i] = -z;
        x[n - 1 - i] = z;
        w[i] = w[n - 1 - i] = 2.0 / ((1.0 - z * z) * dp * dp);
    }
}

// Lloyd-Max levels for f(t) = (1 - t^2)^a on [-1, 1], a = (D-3)/2.
// Cell mass: composite Gauss-Legendre of f over [0, |e|] (odd extension);
// cell first moment: antiderivative -(1-t^2)^(a+1) / (2(a+1)).
void lloyd_max_levels(int D, int b, std::vector<double>& c, std::vector<double>& m) {
    const int L = 1 << b;
    const double a = 0.5 * (D - 3);
    std::vector<double> gx, gw;
    gauss_legendre(16, gx, gw);
    const int panels = 24;
    auto mass = [&](double e) {
        const double s = e < 0 ? -1.0 : 1.0;
        const double hi = std::fabs(e);
        if (hi == 0.0) return 0.0;
        const double h = hi / panels;
        double acc = 0.0;
        for (int p = 0; p < panels; ++p) {
            const double mid = (p + 0.5) * h;
            double part = 0.0;
            for (size_t i = 0; i < gx.size(); ++i) {
                const double t = mid + 0.5 * h * gx[i];
                const double u = 1.0 - t * t;
                part += gw[i] * (u > 0.0 ? std::pow(u, a) : 0.0);
            }
            acc += 0.5 * h * part;
        }
        return s * acc;
    };
    auto moment = [&](double e) {
        double u = 1.0 - e * e;
        if (u < 0.0) u = 0.0;
        return -std::pow(u, a + 1.0) / (2.0 * (a + 1.0));
    };
    c.assign(L, 0.0);
    const double spread = std::fmin(0.9, 3.0 / std::sqrt(static_cast<double>(D)));
    for (int j = 0; j < L; ++j) c[j] = spread * (2.0 * j + 1 - L) / L;
    std::vector<double> edge(L + 1), fe(L + 1), ge(L + 1);
    double best = 1e300;
    int stall = 0;
    for (int it = 0; it < 100000; ++it) {
        edge[0] = -1.0;
        edge[L] = 1.0;
        for (int j = 1; j < L; ++j) edge[j] = 0.5 * (c[j - 1] + c[j]);
        for (int j = 0; j <= L; ++j) {
            fe[j] = mass(edge[j]);
            ge[j] = moment(edge[j]);
        }
        double step = 0.0;
        for (int j = 0; j < L; ++j) {
            const double w = fe[j + 1] - fe[j];
            const double nc = w > 0.0 ? (ge[j + 1] - ge[j]) / w : 0.5 * (edge[j] + edge[j + 1]);
            step = std::fmax(step, std::fabs(nc - c[j]));
            c[j] = nc;
        }
        if (step <= 1e-17) break;
        if (step < best) {
            best = step;
            stall = 0;
        } else if (++stall >= 200) {
            break;
        }
    }
    for (int j = 0; j < L / 2; ++j) {
        const double h = 0.5 * (c[L - 1 - j] - c[j]);
        c[j] = -h;
        c[L - 1 - j] = h;
    }
    m.assign(L - 1, 0.0);
    for (int j = 0; j + 1 < L; ++j) m[j] = 0.5 * (c[j] + c[j + 1]);
}

// Nearest binary16 number to x, ties to even: spacing 2^(ilogb(x) - 10) in
// the normal half range and 2^-24 below it.
double nearest_half(double x) {
    if (x == 0.0) return x;
    int q = std::ilogb(x) - 10;
    if (q < -24) q = -24;
    return std::scalbn(std::nearbyint(std::scalbn(x, -q)), q);
}

// IEEE half bits of a value already on the fp16 grid (|h| < 65520).
uint16_t half_bits_of(double h) {
    const uint16_t sign = std::signbit(h) ? 0x8000u : 0u;
    const double a = std::fabs(h);
    if (a == 0.0) return sign;
    const int e = std::ilogb(a);
    if (e < -14) return static_cast<uint16_t>(sign | std::lround(std::scalbn(a, 24)));  // subnormal
    const long mant = std::lround(std::scalbn(a, 10 - e));                              // 1024..2047
    return static_cast<uint16_t>(sign | ((e + 15) << 10) | (mant - 1024));
}

}  // namespace

void build_tc_operand(const std::vector<float>& M, int D, double scale, std::vector<uint16_t>& out) {
    out.assign(static_cast<size_t>(2) * D * D, 0);
    const size_t lo_base = static_cast<size_t>(D) * D;
    for (int row = 0; row < D; ++row)
        for (int k = 0; k < D; ++k) {
            const double v = scale * static_cast<double>(M[static_cast<size_t>(row) * D + k]);
            const double hi = nearest_half(v);
            const double lo = nearest_half(v - hi);
            const size_t at = (static_cast<size_t>(row / 8) * (D / 8) + k / 8) * 64 + (row % 8) * 8 + (k % 8);
            out[at] = half_bits_of(hi);
            out[lo_base + at] = half_bits_of(lo);
        }
}

// Scale of the half-precision operand levels: the alpha in [1, 2) (on a grid
// of 2^-21) minimising the largest relative error of rounding alpha * |c_j|
// to fp16 over the distinct magnitudes; ties keep the smaller alpha. The
// decode multiplies fp16 levels with fp16 query or weight operands on the
// tensor cores; a well-chosen common scale leaves one or two magnitudes
// (1- and 2-bit codebooks) almost exact and cuts the error of the larger
// codebooks several-fold compared with rounding the levels themselves.
static double operand_scale(const std::vector<float>& levels) {
    std::vector<double> mags;
    for (float v : levels)
        if (v > 0.0f) mags.push_back(static_cast<double>(v));
    if (mags.empty()) return 1.0;
    double best_err = INFINITY, best = 1.0;
    constexpr int kSteps = 1 << 21;
    for (int i = 0; i < kSteps; ++i) {
        const double a = 1.0 + std::ldexp(static_cast<double>(i), -21);
        double worst = 0.0;
        for (double m : mags) {
            const double v = a * m;
            const double e = std::fabs(nearest_half(v) - v) / v;
            if (e > worst) {
                worst = e;
                if (worst >= best_err) break;
            }
        }
        if (worst < best_err) {
            best_err = worst;
            best = a;
        }
    }
    return best;
}

void build_codec_tables(int D, int index_bits, bool with_qjl, uint64_t seed, HostTables& out) {
    static std::mutex mu;
    struct Levels {
        std::vector<double> c, m;
        double scale;
    };
    static std::map<std::pair<int, int>, Levels> cache;
    std::vector<double> c, m;
    double scale = 1.0;
    {
        std::lock_guard<std::mutex> lk(mu);
        auto key = std::make_pair(D, index_bits);
        auto it = cache.find(key);
        if (it == cache.end()) {
            lloyd_max_levels(D, index_bits, c, m);
            std::vector<float> cf(c.size());
            for (size_t i = 0; i < c.size(); ++i) cf[i] = static_cast<float>(c[i]);
            scale = operand_scale(cf);
            cache[key] = {c, m, scale};
        } else {
            c = it->second.c;
            m = it->second.m;
            scale = it->second.scale;
        }
    }
    const std::vector<double> R = haar_rotation(D, seed);
    out.rotation.resize(R.size());
    for (size_t i = 0; i < R.size(); ++i) out.rotation[i] = static_cast<float>(R[i]);
    out.qjl.clear();
    if (with_qjl) {
        const std::vector<double> S = gaussian_matrix(D, seed, 1);
        out.qjl.resize(S.size());
        for (size_t i = 0; i < S.size(); ++i) out.qjl[i] = static_cast<float>(S[i]);
    }
    // Stored levels and thresholds: the fp32 numbers nearest to the fp64
    // levels and to the fp64 midpoints between adjacent levels.
    out.centroids.resize(c.size());
    for (size_t i = 0; i < c.size(); ++i) out.centroids[i] = static_cast<float>(c[i]);
    out.midpoints.resize(m.size());
    for (size_t i = 0; i < m.size(); ++i) out.midpoints[i] = static_cast<float>(m[i]);
    out.op_scale = static_cast<float>(scale);
    out.op_levels.resize(c.size());
    for (size_t i = 0; i < c.size(); ++i)
        out.op_levels[i] = static_cast<float>(nearest_half(scale * static_cast<double>(out.centroids[i])));
}

}  // namespace tq

/*
 * tq_oracle.c -- plain, slow, CPU oracle for TurboQuant KV-cache compression
 * and decode attention over the compressed cache.
 *
 * TEST INFRASTRUCTURE. Only the tests, the smoke check and the benchmark's
 * CPU-baseline / reference arm may load or call this library. It shares no
 * code, header, table or constant generator with the GPU library.
 *
 * Sources, by page title:
 *  - "lightning-mlx/plan.md", section "Estado atual do código": the codec is a
 *    random orthogonal rotation followed by a Lloyd-Max scalar codebook, with
 *    the norm stored apart; reconstruction unpacks the indices, looks up the
 *    codebook, denormalises groups (x scale + offset) and applies the inverse
 *    rotation as `rotated @ Q` in fp32.
 *  - "omlx/turboquant_kv.py", `_infer_head_dim` and `_rebuild_codecs`: indices
 *    are packed into uint32 words, packed_width = ceil(head_dim*bits/32); a prod
 *    state packs its MSE indices with bits-1; codecs are fully determined by
 *    (head_dim, bits, seed) and the value codec uses seed+1; state fields
 *    (norms, indices) and (norms, mse_indices, residual_norms, qjl_signs).
 *  - "turboquant/validate_moe_phase2.py", TEST 1 and TEST 2: TurboQuantProd =
 *    MSE indices + QJL signs + residual norm + norm, norms stored as float32;
 *    the rotation Pi and the QJL matrix S are head_dim x head_dim fp32; values
 *    use group quantisation with per-group scales and zeros; attention scale is
 *    1/sqrt(head_dim).
 *
 * Readings taken where the pages are silent (all listed in the design notes):
 *  [R1] random numbers: SplitMix64 streams, Box-Muller normals;
 *  [R2] rotation: Householder QR of a Gaussian matrix with the sign of R's
 *       diagonal folded into Q (Haar); forward y = R x, inverse x = R^T y;
 *  [R3] Lloyd-Max density: exact marginal of one coordinate of a uniform unit
 *       vector in R^D, f(t) ~ (1 - t^2)^((D-3)/2) on [-1, 1];
 *  [R4] encode arithmetic in fp32 with sequential fused multiply-adds (the
 *       pages rotate in fp32); index = number of midpoints strictly below y;
 *  [R5] prod residual taken in the rotated unit domain; sign bit set for
 *       (S r)_j >= 0; QJL estimator constant sqrt(pi/2)/D;
 *  [R6] group quantisation: fp16 scale = (max-min)/(2^b-1), fp16 min,
 *       code = clamp(rint((x - min)/scale)), values are not rotated;
 *  [R7] decode: contiguous GQA grouping, query l of Lq sees keys
 *       t <= N - Lq + l;
 *  [R10] stored codebook: the fp32 roundings of the fp64 Lloyd-Max levels and
 *       of the fp64 midpoints between adjacent levels.
 */
#include "tq_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

#define TQO_MSE 0
#define TQO_PROD 1
#define TQO_GROUP 2

int tqo_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops that follow (timing on one core and on all). */
void tqo_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------ */
/* [R1] SplitMix64 (Vigna): state += golden gamma, then the mix.       */
/* ------------------------------------------------------------------ */
static uint64_t sm64_mix(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

uint64_t tqo_splitmix64_at(uint64_t s, uint64_t i) {
    return sm64_mix(s + (i + 1) * 0x9E3779B97F4A7C15ULL);
}

/* Uniform in (0,1): ((z >> 12) + 1/2) / 2^52, exact in double. */
static double u01(uint64_t z) { return ((double)(z >> 12) + 0.5) * 0x1.0p-52; }

/* Stream (seed, j) is SplitMix64 seeded with 2*seed + j; normals come in
 * Box-Muller pairs from consecutive uniforms (u1, u2):
 *   g0 = sqrt(-2 ln u1) cos(2 pi u2),  g1 = sqrt(-2 ln u1) sin(2 pi u2). */
void tqo_normals(uint64_t seed, int stream, int64_t n, double *out) {
    const uint64_t s0 = seed * 2u + (uint64_t)stream;
    const double two_pi = 6.283185307179586;
    for (int64_t k = 0; 2 * k < n; ++k) {
        double u1 = u01(tqo_splitmix64_at(s0, (uint64_t)(2 * k)));
        double u2 = u01(tqo_splitmix64_at(s0, (uint64_t)(2 * k + 1)));
        double r = sqrt(-2.0 * log(u1));
        double th = two_pi * u2;
        out[2 * k] = r * cos(th);
        if (2 * k + 1 < n) out[2 * k + 1] = r * sin(th);
    }
}

/* ------------------------------------------------------------------ */
/* [R2] Rotation: Householder QR of G (row-major, G[i][j] = normal     */
/* number i*D+j of stream 0), then R = Q diag(d), d_k = sign(R_kk).    */
/* Every sum runs in ascending index order with separate multiply and  */
/* add, so the result is a fixed function of G.                        */
/* ------------------------------------------------------------------ */
int tqo_rotation_f64(int D, uint64_t seed, double *Rout) {
    if (D < 2) return -1;
    double *A = (double *)malloc(sizeof(double) * D * D);
    double *V = (double *)malloc(sizeof(double) * D * D); /* v_k in row k, entries k..D-1 */
    double *vv = (double *)malloc(sizeof(double) * D);
    double *d = (double *)malloc(sizeof(double) * D);
    tqo_normals(seed, 0, (int64_t)D * D, A);
    for (int k = 0; k < D; ++k) {
        double s = 0.0;
        for (int i = k; i < D; ++i) s = s + A[i * D + k] * A[i * D + k];
        double nrm = sqrt(s);
        double alpha = (A[k * D + k] > 0.0) ? -nrm : nrm;
        d[k] = (alpha < 0.0) ? -1.0 : 1.0;
        double *v = V + (size_t)k * D;
        v[k] = A[k * D + k] - alpha;
        for (int i = k + 1; i < D; ++i) v[i] = A[i * D + k];
        double w2 = 0.0;
        for (int i = k; i < D; ++i) w2 = w2 + v[i] * v[i];
        vv[k] = w2;
        if (w2 == 0.0) continue;
        for (int j = k + 1; j < D; ++j) {
            double w = 0.0;
            for (int i = k; i < D; ++i) w = w + v[i] * A[i * D + j];
            double f = (2.0 * w) / w2;
            for (int i = k; i < D; ++i) A[i * D + j] = A[i * D + j] - f * v[i];
        }
    }
    /* Q = H_0 H_1 ... H_{D-1} I, applied from the last reflector. */
    double *Q = A; /* reuse */
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) Q[i * D + j] = (i == j) ? 1.0 : 0.0;
    for (int k = D - 1; k >= 0; --k) {
        if (vv[k] == 0.0) continue;
        const double *v = V + (size_t)k * D;
        for (int j = 0; j < D; ++j) {
            double w = 0.0;
            for (int i = k; i < D; ++i) w = w + v[i] * Q[i * D + j];
            double f = (2.0 * w) / vv[k];
            for (int i = k; i < D; ++i) Q[i * D + j] = Q[i * D + j] - f * v[i];
        }
    }
    for (int i = 0; i < D; ++i)
        for (int j = 0; j < D; ++j) Rout[i * D + j] = Q[i * D + j] * d[j];
    free(A); free(V); free(vv); free(d);
    return 0;
}

int tqo_qjl_f64(int D, uint64_t seed, double *S) {
    tqo_normals(seed, 1, (int64_t)D * D, S);
    return 0;
}

/* ------------------------------------------------------------------ */
/* [R3] Lloyd-Max for f(t) = (1-t^2)^a, a = (D-3)/2, on [-1,1].        */
/* Cell mass uses the exact antiderivative of (1-t^2)^a built by the   */
/* recurrence I_a = (t(1-t^2)^a + 2a I_{a-1}) / (2a+1); the cell's     */
/* first moment uses the closed form -(1-t^2)^(a+1) / (2(a+1)).        */
/* ------------------------------------------------------------------ */
static double mass_F(double t, int D) {
    /* integral_0^t (1-s^2)^((D-3)/2) ds */
    double u = 1.0 - t * t;
    if (u < 0.0) u = 0.0;
    double I, p; /* p = u^a_j for the current a_j */
    double a;
    if (D % 2 == 1) { /* integer exponents from 0 */
        I = t; p = 1.0; a = 0.0;
    } else {          /* half-integer exponents from 1/2 */
        p = sqrt(u);
        I = 0.5 * (t * p + asin(t));
        a = 0.5;
    }
    const double target = 0.5 * (double)(D - 3);
    while (a < target - 0.25) {
        a = a + 1.0;
        p = p * u;
        I = (t * p + 2.0 * a * I) / (2.0 * a + 1.0);
    }
    return I;
}

static double moment_G(double t, int D) {
    double a = 0.5 * (double)(D - 3);
    double u = 1.0 - t * t;
    if (u < 0.0) u = 0.0;
    return -pow(u, a + 1.0) / (2.0 * (a + 1.0));
}

int tqo_lloyd_max(int D, int b, double *c, double *m) {
    if (D < 3 || b < 1 || b > 8) return -1;
    const int L = 1 << b;
    double *e = (double *)malloc(sizeof(double) * (L + 1));
    double *Fe = (double *)malloc(sizeof(double) * (L + 1));
    double *Ge = (double *)malloc(sizeof(double) * (L + 1));
    double spread = 3.0 / sqrt((double)D);
    if (spread > 0.9) spread = 0.9;
    for (int j = 0; j < L; ++j) c[j] = spread * (double)(2 * j + 1 - L) / (double)L;
    /* Lloyd iterations converge linearly; stop at a step of at most 1e-17 or
     * once the smallest step seen has not shrunk for 200 iterations (the
     * floating-point noise floor). */
    int it, stall = 0;
    double best = INFINITY;
    for (it = 0; it < 100000; ++it) {
        e[0] = -1.0;
        e[L] = 1.0;
        for (int j = 1; j < L; ++j) e[j] = 0.5 * (c[j - 1] + c[j]);
        for (int j = 0; j <= L; ++j) { Fe[j] = mass_F(e[j], D); Ge[j] = moment_G(e[j], D); }
        double delta = 0.0;
        for (int j = 0; j < L; ++j) {
            double mass = Fe[j + 1] - Fe[j];
            double mom = Ge[j + 1] - Ge[j];
            double cn = (mass > 0.0) ? mom / mass : 0.5 * (e[j] + e[j + 1]);
            double dd = fabs(cn - c[j]);
            if (dd > delta) delta = dd;
            c[j] = cn;
        }
        if (delta <= 1e-17) break;
        if (delta < best) { best = delta; stall = 0; }
        else if (++stall >= 200) break;
    }
    /* exact antisymmetry c[L-1-j] = -c[j] */
    for (int j = 0; j < L / 2; ++j) {
        double s = 0.5 * (c[L - 1 - j] - c[j]);
        c[j] = -s;
        c[L - 1 - j] = s;
    }
    for (int j = 0; j + 1 < L; ++j) m[j] = 0.5 * (c[j] + c[j + 1]);
    free(e); free(Fe); free(Ge);
    return it;
}

int tqo_index_bits(int bits, int mode) { return mode == TQO_PROD ? bits - 1 : bits; }

int tqo_packed_words(int D, int ib) { return (D * ib + 31) / 32; }

int tqo_record_bytes(int D, int bits, int mode, int group) {
    int ib = tqo_index_bits(bits, mode);
    int w = tqo_packed_words(D, ib);
    if (mode == TQO_MSE) return 4 * w + 4;
    if (mode == TQO_PROD) return 4 * w + 4 * (D / 32) + 8;
    return 4 * w + 4 * (D / group); /* fp16 scale + fp16 min per group */
}

/* Key and value widths of a possibly fractional width b, as the codec rebuild
 * of "omlx/turboquant_kv.py" (_rebuild_codecs) computes them: b is
 * fractional unless it lies within 1e-6 of round(b); a fractional b gives keys
 * floor(b) and values ceil(b), any other b gives int(b) (truncation) to both. */
void tqo_bits_split(double b, int *key_bits, int *value_bits) {
    int fractional = fabs(b - nearbyint(b)) > 1e-6;
    *key_bits = fractional ? (int)floor(b) : (int)b;
    *value_bits = fractional ? (int)ceil(b) : (int)b;
}

int tqo_codec_tables(int D, int bits, int mode, uint64_t seed,
                     float *R, float *S, float *c, float *m) {
    if (mode == TQO_GROUP) return 0;
    int ib = tqo_index_bits(bits, mode);
    if (ib < 1 || ib > 8) return -1;
    double *R64 = (double *)malloc(sizeof(double) * D * D);
    if (tqo_rotation_f64(D, seed, R64) != 0) { free(R64); return -1; }
    for (int i = 0; i < D * D; ++i) R[i] = (float)R64[i];
    if (mode == TQO_PROD && S) {
        tqo_qjl_f64(D, seed, R64);
        for (int i = 0; i < D * D; ++i) S[i] = (float)R64[i];
    }
    free(R64);
    int L = 1 << ib;
    double c64[256], m64[255];
    tqo_lloyd_max(D, ib, c64, m64);
    /* The stored levels and decision thresholds are the fp32 numbers nearest
     * to the fp64 Lloyd-Max levels and to the fp64 midpoints between them. */
    for (int j = 0; j < L; ++j) c[j] = (float)c64[j];
    for (int j = 0; j + 1 < L; ++j) m[j] = (float)m64[j];
    return 0;
}

/* ------------------------------------------------------------------ */
/* Bit packing: code i occupies bits [i*b, i*b+b) of the word stream,   */
/* least significant bit first; a code may straddle two words.          */
/* ------------------------------------------------------------------ */
void tqo_pack(const uint8_t *codes, int D, int b, uint32_t *words) {
    int W = tqo_packed_words(D, b);
    for (int w = 0; w < W; ++w) words[w] = 0;
    for (int i = 0; i < D; ++i) {
        int p = i * b;
        uint64_t v = (uint64_t)codes[i] << (p & 31);
        words[p >> 5] |= (uint32_t)v;
        if ((p & 31) + b > 32) words[(p >> 5) + 1] |= (uint32_t)(v >> 32);
    }
}

void tqo_unpack(const uint32_t *words, int D, int b, uint8_t *codes) {
    for (int i = 0; i < D; ++i) {
        int p = i * b;
        uint64_t v = words[p >> 5] >> (p & 31);
        if ((p & 31) + b > 32) v |= (uint64_t)words[(p >> 5) + 1] << (32 - (p & 31));
        codes[i] = (uint8_t)(v & ((1u << b) - 1));
    }
}

/* ------------------------------------------------------------------ */
/* IEEE binary16, round to nearest even.                                */
/* ------------------------------------------------------------------ */
uint16_t tqo_f32_to_f16(float f) {
    uint32_t x;
    memcpy(&x, &f, 4);
    uint32_t sign = (x >> 16) & 0x8000u;
    uint32_t ax = x & 0x7FFFFFFFu;
    if (ax >= 0x7F800000u) {
        if (ax == 0x7F800000u) return (uint16_t)(sign | 0x7C00u);
        return (uint16_t)(sign | 0x7E00u | ((ax >> 13) & 0x3FFu));
    }
    if (ax >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u); /* >= 65520 */
    int E = (int)(ax >> 23) - 127;
    uint32_t M = (ax & 0x7FFFFFu) | 0x800000u;
    if (E >= -14) { /* normal result */
        uint32_t h = ((uint32_t)(E + 15) << 10) | ((ax & 0x7FFFFFu) >> 13);
        uint32_t rem = ax & 0x1FFFu;
        if (rem > 0x1000u || (rem == 0x1000u && (h & 1u))) h += 1u;
        return (uint16_t)(sign | h);
    }
    if (E < -25) return (uint16_t)sign; /* below half the smallest subnormal */
    int s = -E - 1; /* 14..24: value / 2^-24 = M >> s */
    uint32_t k = M >> s;
    uint32_t rem = M & ((1u << s) - 1u);
    uint32_t half = 1u << (s - 1);
    if (rem > half || (rem == half && (k & 1u))) k += 1u;
    return (uint16_t)(sign | k);
}

float tqo_f16_to_f32(uint16_t h) {
    uint32_t sign = ((uint32_t)h & 0x8000u) << 16;
    uint32_t e = (h >> 10) & 0x1Fu, mant = h & 0x3FFu;
    float r;
    if (e == 0) {
        r = ldexpf((float)mant, -24);
        uint32_t bits;
        memcpy(&bits, &r, 4);
        bits |= sign;
        memcpy(&r, &bits, 4);
        return r;
    }
    uint32_t bits;
    if (e == 31) bits = sign | 0x7F800000u | (mant << 13);
    else bits = sign | ((e - 15 + 127) << 23) | (mant << 13);
    memcpy(&r, &bits, 4);
    return r;
}

/* ------------------------------------------------------------------ */
/* [R4] MSE encode of one vector, fp32 with sequential fmaf:            */
/*   n = sqrt(sum_k x_k^2); y_i = (sum_k R_ik x_k) / n (0 if n == 0);   */
/*   code_i = #{j : y_i > m_j}.                                         */
/* ------------------------------------------------------------------ */
static void mse_one(int D, const float *x, const float *R, const float *m, int b,
                    uint8_t *codes, float *y, float *norm) {
    float n2 = 0.0f;
    for (int k = 0; k < D; ++k) n2 = fmaf(x[k], x[k], n2);
    float n = sqrtf(n2);
    const int nm = (1 << b) - 1;
    for (int i = 0; i < D; ++i) {
        float t = 0.0f;
        for (int k = 0; k < D; ++k) t = fmaf(R[(size_t)i * D + k], x[k], t);
        float yi = (n > 0.0f) ? t / n : 0.0f;
        int code = 0;
        for (int j = 0; j < nm; ++j) code += (yi > m[j]) ? 1 : 0;
        codes[i] = (uint8_t)code;
        y[i] = yi;
    }
    *norm = n;
}

void tqo_encode_mse(int64_t n, int D, const float *x, const float *R, const float *m,
                    int b, uint32_t *idx, float *norm) {
    const int W = tqo_packed_words(D, b);
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < n; ++v) {
        uint8_t codes[512];
        float y[512];
        mse_one(D, x + v * D, R, m, b, codes, y, norm + v);
        tqo_pack(codes, D, b, idx + v * W);
    }
}

/* [R5] prod: (bits-1)-bit MSE, residual r = y - c[code] in the rotated unit
 * domain, rnorm = sqrt(sum r_i^2), sign bit j = ((S r)_j >= 0). */
void tqo_encode_prod(int64_t n, int D, const float *x, const float *R, const float *S,
                     const float *c, const float *m, int bits, uint32_t *idx,
                     uint32_t *sgn, float *norm, float *rnorm) {
    const int b = bits - 1;
    const int W = tqo_packed_words(D, b);
    const int Ws = D / 32;
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < n; ++v) {
        uint8_t codes[512];
        float y[512], r[512];
        mse_one(D, x + v * D, R, m, b, codes, y, norm + v);
        tqo_pack(codes, D, b, idx + v * W);
        float g2 = 0.0f;
        for (int i = 0; i < D; ++i) {
            r[i] = y[i] - c[codes[i]];
            g2 = fmaf(r[i], r[i], g2);
        }
        rnorm[v] = sqrtf(g2);
        uint32_t *sw = sgn + v * Ws;
        for (int w = 0; w < Ws; ++w) sw[w] = 0;
        for (int j = 0; j < D; ++j) {
            float z = 0.0f;
            for (int i = 0; i < D; ++i) z = fmaf(S[(size_t)j * D + i], r[i], z);
            if (z >= 0.0f) sw[j >> 5] |= 1u << (j & 31);
        }
    }
}

/* [R6] group quantisation of one vector, groups of g consecutive coords. */
void tqo_encode_group(int64_t n, int D, const float *x, int bits, int g,
                      uint32_t *data, uint16_t *scale, uint16_t *mn) {
    const int W = tqo_packed_words(D, bits);
    const int ng = D / g;
    const int qmax = (1 << bits) - 1;
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < n; ++v) {
        const float *xv = x + v * D;
        uint8_t codes[512];
        for (int gi = 0; gi < ng; ++gi) {
            float lo = xv[gi * g], hi = xv[gi * g];
            for (int k = 1; k < g; ++k) {
                float t = xv[gi * g + k];
                lo = (t < lo) ? t : lo;
                hi = (t > hi) ? t : hi;
            }
            float s32 = (hi - lo) / (float)qmax;
            uint16_t sh = tqo_f32_to_f16(s32), mh = tqo_f32_to_f16(lo);
            scale[v * ng + gi] = sh;
            mn[v * ng + gi] = mh;
            float sf = tqo_f16_to_f32(sh), mf = tqo_f16_to_f32(mh);
            for (int k = 0; k < g; ++k) {
                int q = 0;
                if (sf != 0.0f) {
                    float r = rintf((xv[gi * g + k] - mf) / sf);
                    if (!(r > 0.0f)) q = 0;
                    else if (r > (float)qmax) q = qmax;
                    else q = (int)r;
                }
                codes[gi * g + k] = (uint8_t)q;
            }
        }
        tqo_pack(codes, D, bits, data + v * W);
    }
}

/* ------------------------------------------------------------------ */
/* Dequantisation to fp64 (plain definitions).                          */
/*  MSE : x = n * (c[code] @ R)                                          */
/*  prod: x = n * ((c[code] + sqrt(pi/2)/D * rnorm * S^T sigma) @ R)     */
/*  group: x = code * scale + min                                        */
/* ------------------------------------------------------------------ */
void tqo_dequant_mse(int64_t n, int D, const uint32_t *idx, const float *norm,
                     const float *R, const float *c, int b, double *out) {
    const int W = tqo_packed_words(D, b);
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < n; ++v) {
        uint8_t codes[512];
        tqo_unpack(idx + v * W, D, b, codes);
        for (int d = 0; d < D; ++d) {
            double s = 0.0;
            for (int i = 0; i < D; ++i) s += (double)c[codes[i]] * (double)R[(size_t)i * D + d];
            out[v * D + d] = (double)norm[v] * s;
        }
    }
}

void tqo_dequant_prod(int64_t n, int D, const uint32_t *idx, const uint32_t *sgn,
                      const float *norm, const float *rnorm, const float *R,
                      const float *S, const float *c, int bits, double *out) {
    const int b = bits - 1;
    const int W = tqo_packed_words(D, b);
    const int Ws = D / 32;
    const double kappa = sqrt(M_PI / 2.0) / (double)D;
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < n; ++v) {
        uint8_t codes[512];
        double yh[512];
        tqo_unpack(idx + v * W, D, b, codes);
        const uint32_t *sw = sgn + v * Ws;
        for (int i = 0; i < D; ++i) {
            double st = 0.0;
            for (int j = 0; j < D; ++j) {
                double sg = ((sw[j >> 5] >> (j & 31)) & 1u) ? 1.0 : -1.0;
                st += (double)S[(size_t)j * D + i] * sg;
            }
            yh[i] = (double)c[codes[i]] + kappa * (double)rnorm[v] * st;
        }
        for (int d = 0; d < D; ++d) {
            double s = 0.0;
            for (int i = 0; i < D; ++i) s += yh[i] * (double)R[(size_t)i * D + d];
            out[v * D + d] = (double)norm[v] * s;
        }
    }
}

void tqo_dequant_group(int64_t n, int D, const uint32_t *data, const uint16_t *scale,
                       const uint16_t *mn, int bits, int g, double *out) {
    const int W = tqo_packed_words(D, bits);
    const int ng = D / g;
#pragma omp parallel for schedule(static)
    for (int64_t v = 0; v < n; ++v) {
        uint8_t codes[512];
        tqo_unpack(data + v * W, D, bits, codes);
        for (int d = 0; d < D; ++d) {
            double s = tqo_f16_to_f32(scale[v * ng + d / g]);
            double m0 = tqo_f16_to_f32(mn[v * ng + d / g]);
            out[v * D + d] = (double)codes[d] * s + m0;
        }
    }
}

/* ------------------------------------------------------------------ */
/* [R7] plain softmax(q K^T * scale) V in fp64.                          */
/* ------------------------------------------------------------------ */
void tqo_attention_f64(int D, int64_t N, int G, int Lq, const double *q,
                       const double *K, const double *V, double scale, double *out) {
#pragma omp parallel for schedule(static)
    for (int r = 0; r < G * Lq; ++r) {
        const int l = r % Lq;
        const int64_t nv = N - Lq + l + 1;
        const double *qr = q + (size_t)r * D;
        double *o = out + (size_t)r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (nv <= 0) continue;
        double *s = (double *)malloc(sizeof(double) * nv);
        double mx = -INFINITY;
        for (int64_t t = 0; t < nv; ++t) {
            double a = 0.0;
            for (int d = 0; d < D; ++d) a += qr[d] * K[t * D + d];
            s[t] = a * scale;
            if (s[t] > mx) mx = s[t];
        }
        double den = 0.0;
        for (int64_t t = 0; t < nv; ++t) {
            double p = exp(s[t] - mx);
            den += p;
            for (int d = 0; d < D; ++d) o[d] += p * V[t * D + d];
        }
        for (int d = 0; d < D; ++d) o[d] /= den;
        free(s);
    }
}

/* Rotated-domain decode: with q' = R_k q and q'' = S q',
 *   score_t = scale * n_t * (<q', c[code_t]> + sqrt(pi/2)/D * rnorm_t <q'', sigma_t>)
 * and for MSE values out = (sum_t p_t n_t c_v[code_t]) @ R_v / sum_t p_t;
 * group values are summed in the original domain. */
void tqo_decode_rotated(int D, int64_t N, int G, int Lq, const double *q,
                        int kmode, int kbits, const uint32_t *kidx, const uint32_t *ksgn,
                        const float *knorm, const float *krn, const float *kR,
                        const float *kS, const float *kc,
                        int vmode, int vbits, int vgroup, const uint32_t *vidx,
                        const float *vnorm, const uint16_t *vscale, const uint16_t *vmin,
                        const float *vR, const float *vc, double scale, double *out) {
    const int kb = tqo_index_bits(kbits, kmode);
    const int Wk = tqo_packed_words(D, kb);
    const int Ws = D / 32;
    const int Wv = tqo_packed_words(D, vbits);
    const double kappa = sqrt(M_PI / 2.0) / (double)D;
    const int ng = (vmode == TQO_GROUP) ? D / vgroup : 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < G * Lq; ++r) {
        const int l = r % Lq;
        const int64_t nv = N - Lq + l + 1;
        const double *qr = q + (size_t)r * D;
        double *o = out + (size_t)r * D;
        double q1[512], q2[512], acc[512];
        uint8_t codes[512];
        for (int i = 0; i < D; ++i) {
            double s = 0.0;
            for (int k = 0; k < D; ++k) s += (double)kR[(size_t)i * D + k] * qr[k];
            q1[i] = s;
        }
        if (kmode == TQO_PROD) {
            for (int j = 0; j < D; ++j) {
                double s = 0.0;
                for (int i = 0; i < D; ++i) s += (double)kS[(size_t)j * D + i] * q1[i];
                q2[j] = s;
            }
        }
        for (int d = 0; d < D; ++d) { acc[d] = 0.0; o[d] = 0.0; }
        if (nv <= 0) continue;
        double mx = -INFINITY, den = 0.0;
        for (int64_t t = 0; t < nv; ++t) {
            tqo_unpack(kidx + t * Wk, D, kb, codes);
            double a = 0.0;
            for (int i = 0; i < D; ++i) a += q1[i] * (double)kc[codes[i]];
            if (kmode == TQO_PROD) {
                double z = 0.0;
                const uint32_t *sw = ksgn + t * Ws;
                for (int j = 0; j < D; ++j)
                    z += ((sw[j >> 5] >> (j & 31)) & 1u) ? q2[j] : -q2[j];
                a += kappa * (double)krn[t] * z;
            }
            double s = scale * (double)knorm[t] * a;
            /* online softmax in fp64 */
            double mnew = s > mx ? s : mx;
            double corr = exp(mx - mnew);
            double p = exp(s - mnew);
            den = den * corr + p;
            for (int d = 0; d < D; ++d) acc[d] *= corr;
            mx = mnew;
            tqo_unpack(vidx + t * Wv, D, vbits, codes);
            if (vmode == TQO_MSE) {
                double w = p * (double)vnorm[t];
                for (int d = 0; d < D; ++d) acc[d] += w * (double)vc[codes[d]];
            } else {
                for (int d = 0; d < D; ++d) {
                    double sc = tqo_f16_to_f32(vscale[t * ng + d / vgroup]);
                    double m0 = tqo_f16_to_f32(vmin[t * ng + d / vgroup]);
                    acc[d] += p * ((double)codes[d] * sc + m0);
                }
            }
        }
        if (vmode == TQO_MSE) {
            for (int d = 0; d < D; ++d) {
                double s = 0.0;
                for (int i = 0; i < D; ++i) s += acc[i] * (double)vR[(size_t)i * D + d];
                o[d] = s / den;
            }
        } else {
            for (int d = 0; d < D; ++d) o[d] = acc[d] / den;
        }
    }
}

/* ------------------------------------------------------------------ */
/* Sequence-sharded decode. A shard holds tokens [offset, offset + N) of  */
/* each sequence; its rows keep the unnormalised softmax state over them: */
/*   m = max_t s_t, l = sum_t exp(s_t - m), acc = sum_t exp(s_t - m) v_t  */
/* with v_t the value in the rotated domain (MSE) or the dequantised      */
/* value (group). A key at local index t is visible to query l of Lq when */
/* t <= E - Lq + l, where E = (global sequence length) - offset is the    */
/* shard's causal end. Parts merge by the log-sum-exp rule:               */
/*   M = max_p m_p, L = sum_p exp(m_p - M) l_p,                           */
/*   acc = sum_p exp(m_p - M) acc_p, out = (acc / L) (@ R_v for MSE).     */
/* A part with no visible key has m = -inf, l = 0, acc = 0 and adds       */
/* nothing. The plain decode is the merge of one part with E = N.         */
/* ------------------------------------------------------------------ */
void tqo_decode_partial(int D, int64_t N, int64_t E, int G, int Lq, const double *q,
                        int kmode, int kbits, const uint32_t *kidx, const uint32_t *ksgn,
                        const float *knorm, const float *krn, const float *kR,
                        const float *kS, const float *kc,
                        int vmode, int vbits, int vgroup, const uint32_t *vidx,
                        const float *vnorm, const uint16_t *vscale, const uint16_t *vmin,
                        const float *vc, double scale, double *m_out, double *l_out,
                        double *acc_out) {
    const int kb = tqo_index_bits(kbits, kmode);
    const int Wk = tqo_packed_words(D, kb);
    const int Ws = D / 32;
    const int Wv = tqo_packed_words(D, vbits);
    const double kappa = sqrt(M_PI / 2.0) / (double)D;
    const int ng = (vmode == TQO_GROUP) ? D / vgroup : 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < G * Lq; ++r) {
        const int l = r % Lq;
        int64_t nv = E - Lq + l + 1; /* visible local keys t < nv */
        if (nv > N) nv = N;
        const double *qr = q + (size_t)r * D;
        double *acc = acc_out + (size_t)r * D;
        double q1[512], q2[512];
        uint8_t codes[512];
        for (int i = 0; i < D; ++i) {
            double s = 0.0;
            for (int k = 0; k < D; ++k) s += (double)kR[(size_t)i * D + k] * qr[k];
            q1[i] = s;
        }
        if (kmode == TQO_PROD) {
            for (int j = 0; j < D; ++j) {
                double s = 0.0;
                for (int i = 0; i < D; ++i) s += (double)kS[(size_t)j * D + i] * q1[i];
                q2[j] = s;
            }
        }
        for (int d = 0; d < D; ++d) acc[d] = 0.0;
        double mx = -INFINITY, den = 0.0;
        for (int64_t t = 0; t < nv; ++t) {
            tqo_unpack(kidx + t * Wk, D, kb, codes);
            double a = 0.0;
            for (int i = 0; i < D; ++i) a += q1[i] * (double)kc[codes[i]];
            if (kmode == TQO_PROD) {
                double z = 0.0;
                const uint32_t *sw = ksgn + t * Ws;
                for (int j = 0; j < D; ++j)
                    z += ((sw[j >> 5] >> (j & 31)) & 1u) ? q2[j] : -q2[j];
                a += kappa * (double)krn[t] * z;
            }
            double s = scale * (double)knorm[t] * a;
            double mnew = s > mx ? s : mx;
            double corr = exp(mx - mnew);
            double p = exp(s - mnew);
            den = den * corr + p;
            for (int d = 0; d < D; ++d) acc[d] *= corr;
            mx = mnew;
            tqo_unpack(vidx + t * Wv, D, vbits, codes);
            if (vmode == TQO_MSE) {
                double w = p * (double)vnorm[t];
                for (int d = 0; d < D; ++d) acc[d] += w * (double)vc[codes[d]];
            } else {
                for (int d = 0; d < D; ++d) {
                    double sc = tqo_f16_to_f32(vscale[t * ng + d / vgroup]);
                    double m0 = tqo_f16_to_f32(vmin[t * ng + d / vgroup]);
                    acc[d] += p * ((double)codes[d] * sc + m0);
                }
            }
        }
        m_out[r] = mx;
        l_out[r] = den;
    }
}

void tqo_merge_partials(int D, int P, int64_t rows, const double *m, const double *l,
                        const double *acc, int vmode, const float *vR, double *out) {
    for (int64_t r = 0; r < rows; ++r) {
        double M = -INFINITY;
        for (int p = 0; p < P; ++p)
            if (m[(size_t)p * rows + r] > M) M = m[(size_t)p * rows + r];
        double L = 0.0, a[512];
        for (int d = 0; d < D; ++d) a[d] = 0.0;
        if (M != -INFINITY) {
            for (int p = 0; p < P; ++p) {
                const double mp = m[(size_t)p * rows + r];
                if (mp == -INFINITY) continue;
                const double w = exp(mp - M);
                L += w * l[(size_t)p * rows + r];
                const double *ap = acc + ((size_t)p * rows + r) * D;
                for (int d = 0; d < D; ++d) a[d] += w * ap[d];
            }
        }
        double *o = out + (size_t)r * D;
        for (int d = 0; d < D; ++d) {
            if (!(L > 0.0)) { o[d] = 0.0; continue; }
            if (vmode == TQO_MSE) {
                double s = 0.0;
                for (int i = 0; i < D; ++i) s += a[i] * (double)vR[(size_t)i * D + d];
                o[d] = s / L;
            } else {
                o[d] = a[d] / L;
            }
        }
    }
}

/* ------------------------------------------------------------------ */
/* Paged pool layout. A layer pool is an array of blocks; block p holds  */
/* BT tokens of every kv head; the (p, h) sub-block starts at byte       */
/* (p*Hkv + h) * BT * record_bytes and stores its streams one after      */
/* another, each token-major: key indices, key signs (prod), key norms,  */
/* key residual norms (prod), value indices/data, then value norms (MSE) */
/* or value scales and mins (group).                                     */
/* ------------------------------------------------------------------ */
int64_t tqo_subblock_layout(int D, int kmode, int kbits, int vmode, int vbits, int vgroup,
                            int BT, int64_t off[7]) {
    int64_t o = 0;
    for (int i = 0; i < 7; ++i) off[i] = -1;
    int kb = tqo_index_bits(kbits, kmode);
    off[0] = o; o += (int64_t)BT * 4 * tqo_packed_words(D, kb);
    if (kmode == TQO_PROD) { off[1] = o; o += (int64_t)BT * 4 * (D / 32); }
    off[2] = o; o += (int64_t)BT * 4;
    if (kmode == TQO_PROD) { off[3] = o; o += (int64_t)BT * 4; }
    off[4] = o; o += (int64_t)BT * 4 * tqo_packed_words(D, vbits);
    if (vmode == TQO_MSE) { off[5] = o; o += (int64_t)BT * 4; }
    else {
        off[5] = o; o += (int64_t)BT * 2 * (D / vgroup);
        off[6] = o; o += (int64_t)BT * 2 * (D / vgroup);
    }
    return o;
}

void tqo_pool_write(uint8_t *pool, int D, int Hkv, int BT, const int32_t *table,
                    int max_blocks, int seq, int h, int64_t t0, int64_t n,
                    int kmode, int kbits, int vmode, int vbits, int vgroup,
                    const uint32_t *kidx, const uint32_t *ksgn, const float *knorm,
                    const float *krn, const uint32_t *vidx, const float *vnorm,
                    const uint16_t *vscale, const uint16_t *vmin) {
    int64_t off[7];
    int64_t sub = tqo_subblock_layout(D, kmode, kbits, vmode, vbits, vgroup, BT, off);
    int kb = tqo_index_bits(kbits, kmode);
    int Wk = tqo_packed_words(D, kb), Ws = D / 32, Wv = tqo_packed_words(D, vbits);
    int ng = (vmode == TQO_GROUP) ? D / vgroup : 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t t = t0 + i;
        int64_t lb = t / BT, slot = t % BT;
        int64_t p = table ? table[(int64_t)seq * max_blocks + lb] : (int64_t)seq * max_blocks + lb;
        uint8_t *base = pool + (p * Hkv + h) * sub;
        memcpy(base + off[0] + slot * 4 * Wk, kidx + i * Wk, 4 * Wk);
        if (kmode == TQO_PROD) memcpy(base + off[1] + slot * 4 * Ws, ksgn + i * Ws, 4 * Ws);
        memcpy(base + off[2] + slot * 4, knorm + i, 4);
        if (kmode == TQO_PROD) memcpy(base + off[3] + slot * 4, krn + i, 4);
        memcpy(base + off[4] + slot * 4 * Wv, vidx + i * Wv, 4 * Wv);
        if (vmode == TQO_MSE) memcpy(base + off[5] + slot * 4, vnorm + i, 4);
        else {
            memcpy(base + off[5] + slot * 2 * ng, vscale + i * ng, 2 * ng);
            memcpy(base + off[6] + slot * 2 * ng, vmin + i * ng, 2 * ng);
        }
    }
}

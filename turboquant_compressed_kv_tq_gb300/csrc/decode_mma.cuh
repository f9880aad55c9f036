// Tensor-core split-K decode attention over the TurboQuant cache, head_dim 128.
//
// Per (token split, kv head, row group of 16 query rows, sequence) one CTA of
// kWarps warps. Every warp streams its own tiles of compressed records from
// HBM into a private ring of shared-memory stages with 1-D bulk copies
// (cp.async.bulk, completion on an mbarrier), and runs, 16 tokens at a time:
//   scores  S = Q' K_hat^T (+ Q'' sigma^T for prod keys) on mma.sync
//           m16n8k16 (fp16 operands, fp32 accumulate); the key operand is
//           decoded from the packed indices straight into MMA fragments with
//           byte-permute table lookups (no shared-memory round trip);
//   softmax online, in log2 units (scale * log2(e) folded into the query);
//   values  O += P' V_hat on mma.sync, P' = p * value norm, V_hat decoded per
//           token into registers and transposed to the MMA operand layout with
//           movmatrix.
// Warps merge in shared memory; the CTA writes (max, sum, acc) partials and
// the last CTA of each (sequence, head, row group) merges the splits, applies
// the inverse value rotation and writes the output.
//
// Query fragments are prepared by a separate kernel in the coordinate order the
// decoders produce (the contraction over head_dim is invariant under a common
// permutation of both operands).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cstdint>

#include "tq_internal.h"

namespace tq {
namespace mmadec {

constexpr int kD = 128;
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kStages = 2;
constexpr int kRows = 16;
constexpr int kMaxTile = 64;
constexpr int kQFragBytes = 2 * 8 * 32 * 16;  // query fragments of one unit
constexpr unsigned kSpinLimit = 1u << 22;

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;\n" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// prmt.b32 in its default mode: each selector nibble picks a byte of {b, a};
// a set msb in the nibble replicates that byte's sign bit instead.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;\n" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_inval(uint64_t* bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Bounded wait on a phase; returns false if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, unsigned phase) {
    const uint32_t a = smem_u32(bar);
    for (unsigned it = 0; it < kSpinLimit; ++it) {
        uint32_t done;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(done)
            : "r"(a), "r"(phase)
            : "memory");
        if (done) return true;
    }
    return false;
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// L2 policy for data read exactly once (the compressed records): evicted
// first, so codec tables and workspaces shared between launches stay cached.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_g2s_once(void* dst, const void* src, unsigned bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// ------------------------------------------------------------------ codebooks in registers

// Byte tables for __byte_perm lookups: for a 4-entry fp16 table T,
// lo holds the low bytes of T[0..3] and hi the high bytes, so
// prmt(lo, hi, sel) with selector nibbles (c, c+4) returns T[c].
struct Tab4 {
    uint32_t lo, hi;
};
// 8-entry table: lo bytes in lo0 (entries 0..3) and lo1 (4..7), same for hi.
struct Tab8 {
    uint32_t lo0, lo1, hi0, hi1;
};

__device__ __forceinline__ uint32_t h_bits(float x) { return __half_as_ushort(__float2half_rn(x)); }

__device__ inline Tab4 make_tab4(const float* c) {
    Tab4 t{0, 0};
    for (int i = 0; i < 4; ++i) {
        const uint32_t h = h_bits(c[i]);
        t.lo |= (h & 0xFFu) << (8 * i);
        t.hi |= (h >> 8) << (8 * i);
    }
    return t;
}

__device__ inline Tab8 make_tab8(const float* c) {
    Tab8 t{0, 0, 0, 0};
    for (int i = 0; i < 8; ++i) {
        const uint32_t h = h_bits(c[i]);
        if (i < 4) {
            t.lo0 |= (h & 0xFFu) << (8 * i);
            t.hi0 |= (h >> 8) << (8 * i);
        } else {
            t.lo1 |= (h & 0xFFu) << (8 * (i - 4));
            t.hi1 |= (h >> 8) << (8 * (i - 4));
        }
    }
    return t;
}

// ------------------------------------------------------------------ decoders
//
// A thread decodes one 32-coordinate chunk of one token into 16 half2 values.
// Pair p of the chunk holds coordinates (pair_a(p), pair_b(p)); the score MMA
// uses pairs (2ks, 2ks+1) as the (b0b1, b2b3) registers of k-step ks.

// 2-bit codes, 16 per word: the codes s, s+4, s+8, s+12 of a word sit in the
// bytes of (w >> 2s) & 0x03030303.
__device__ __forceinline__ void dec2_pair(uint32_t w, int s, const Tab4& t, uint32_t& h0, uint32_t& h1) {
    const uint32_t x = (w >> (2 * s)) & 0x03030303u;
    const uint32_t sel = x * 0x11u + 0x40404040u;
    h0 = prmt(t.lo, t.hi, sel);          // codes s, s+4
    h1 = prmt(t.lo, t.hi, sel >> 16);    // codes s+8, s+12
}

// Sign-magnitude 4-bit decode of 8 codes (one word) with a symmetric codebook:
// value = +mu[k-8] for k >= 8 and -mu[7-k] below. Produces pairs (0,1),(2,3),
// (4,5),(6,7).
__device__ __forceinline__ void dec4_word(uint32_t w, const Tab8& mu, uint32_t (&h)[4]) {
    const uint32_t f = (~(w >> 3)) & 0x11111111u;         // 1 where the code is negative
    const uint32_t u = (w ^ (f * 7u)) & 0x77777777u;      // magnitude index per nibble
    const uint32_t ws = w << 4;
    {
        const uint32_t lo4 = prmt(mu.lo0, mu.lo1, u);
        uint32_t hi4 = prmt(mu.hi0, mu.hi1, u);
        const uint32_t s4 = prmt(ws, w, 0xD9C8);   // 0xFF where positive (codes 0..3)
        hi4 ^= ~s4 & 0x80808080u;
        h[0] = prmt(lo4, hi4, 0x5140);
        h[1] = prmt(lo4, hi4, 0x7362);
    }
    {
        const uint32_t u2 = u >> 16;
        const uint32_t lo4 = prmt(mu.lo0, mu.lo1, u2);
        uint32_t hi4 = prmt(mu.hi0, mu.hi1, u2);
        const uint32_t s4 = prmt(ws, w, 0xFBEA);   // codes 4..7
        hi4 ^= ~s4 & 0x80808080u;
        h[2] = prmt(lo4, hi4, 0x5140);
        h[3] = prmt(lo4, hi4, 0x7362);
    }
}

// 3-bit: 8 codes (24 bits) spread into nibbles, then an 8-entry lookup.
__device__ __forceinline__ void dec3_group(uint32_t v, const Tab8& t, uint32_t (&h)[4]) {
    uint32_t x = (v & 0x00000FFFu) | ((v << 4) & 0x0FFF0000u);
    x = (x & 0x003F003Fu) | ((x << 2) & 0x3F003F00u);
    x = (x & 0x07070707u) | ((x << 1) & 0x70707070u);
    {
        const uint32_t lo4 = prmt(t.lo0, t.lo1, x);
        const uint32_t hi4 = prmt(t.hi0, t.hi1, x);
        h[0] = prmt(lo4, hi4, 0x5140);
        h[1] = prmt(lo4, hi4, 0x7362);
    }
    {
        const uint32_t x2 = x >> 16;
        const uint32_t lo4 = prmt(t.lo0, t.lo1, x2);
        const uint32_t hi4 = prmt(t.hi0, t.hi1, x2);
        h[2] = prmt(lo4, hi4, 0x5140);
        h[3] = prmt(lo4, hi4, 0x7362);
    }
}

// One-bit codes / QJL signs: bit i of the word for coordinate i; pair (s, s+16)
// and (s+8, s+24); `neg2` holds (-v, -v) so that a set bit yields +v.
__device__ __forceinline__ uint32_t dec1(uint32_t w, int sh, uint32_t neg2) {
    return ((w << sh) & 0x80008000u) ^ neg2;
}

// Decode a whole 32-coordinate chunk into 16 pairs (MSE codebooks).
template <int B>
struct MseChunk;

template <>
struct MseChunk<1> {
    static constexpr int kWords = 1;
    __device__ __forceinline__ static void run(const uint32_t* w, const Tab4& t, uint32_t (&h)[16]) {
        const uint32_t neg2 = t.lo;  // (-c, -c) packed (see table setup)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            h[2 * ks] = dec1(w[0], 15 - ks, neg2);
            h[2 * ks + 1] = dec1(w[0], 7 - ks, neg2);
        }
    }
};

template <>
struct MseChunk<2> {
    static constexpr int kWords = 2;
    __device__ __forceinline__ static void run(const uint32_t* w, const Tab4& t, uint32_t (&h)[16]) {
#pragma unroll
        for (int s = 0; s < 4; ++s) {
#pragma unroll
            for (int hw = 0; hw < 2; ++hw) {
                const int ks = 2 * s + hw;
                dec2_pair(w[hw], s, t, h[2 * ks], h[2 * ks + 1]);
            }
        }
    }
};

template <>
struct MseChunk<3> {
    static constexpr int kWords = 3;
    __device__ __forceinline__ static void run(const uint32_t* w, const Tab8& t, uint32_t (&h)[16]) {
        const uint32_t v0 = w[0] & 0xFFFFFFu;
        const uint32_t v1 = __funnelshift_r(w[0], w[1], 24) & 0xFFFFFFu;
        const uint32_t v2 = __funnelshift_r(w[1], w[2], 16) & 0xFFFFFFu;
        const uint32_t v3 = w[2] >> 8;
        uint32_t g[4];
        dec3_group(v0, t, g);
        h[0] = g[0]; h[1] = g[1]; h[2] = g[2]; h[3] = g[3];
        dec3_group(v1, t, g);
        h[4] = g[0]; h[5] = g[1]; h[6] = g[2]; h[7] = g[3];
        dec3_group(v2, t, g);
        h[8] = g[0]; h[9] = g[1]; h[10] = g[2]; h[11] = g[3];
        dec3_group(v3, t, g);
        h[12] = g[0]; h[13] = g[1]; h[14] = g[2]; h[15] = g[3];
    }
};

template <>
struct MseChunk<4> {
    static constexpr int kWords = 4;
    __device__ __forceinline__ static void run(const uint32_t* w, const Tab8& t, uint32_t (&h)[16]) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint32_t g[4];
            dec4_word(w[i], t, g);
            h[4 * i] = g[0]; h[4 * i + 1] = g[1]; h[4 * i + 2] = g[2]; h[4 * i + 3] = g[3];
        }
    }
};

// Coordinates (within the 32-coordinate chunk) of pair p for an MSE decoder.
__host__ __device__ inline void mse_pair(int bits, int p, int& a, int& b) {
    const int ks = p >> 1, e = p & 1;
    if (bits == 1) {
        a = ks + 8 * e;
        b = a + 16;
    } else if (bits == 2) {
        const int s = ks >> 1, hw = ks & 1;
        a = 16 * hw + 8 * e + s;
        b = a + 4;
    } else {
        a = 2 * p;
        b = a + 1;
    }
}

// Group-quantised values: q*scale + min with one rounding. The code is placed
// in the mantissa of 1.0 (exact 1 + q/16 for 4 bits, 1 + q/4 for 2 bits), 1.0 is
// subtracted exactly, and one fused multiply-add gives (q/16)*(16*scale) + min.
// 4-bit: pair (i, i+4) of word wi -> p = 4*wi + i; 2-bit: pair (i, i+8) of
// word w -> p = 8*w + i.
__host__ __device__ inline void group_pair(int bits, int p, int& a, int& b) {
    if (bits == 4) {
        a = 8 * (p >> 2) + (p & 3);
        b = a + 4;
    } else {
        a = 16 * (p >> 3) + (p & 7);
        b = a + 8;
    }
}

template <int B>
struct GroupChunk;

template <>
struct GroupChunk<4> {
    static constexpr int kWords = 4;
    __device__ __forceinline__ static void run(const uint32_t* w, uint32_t mul2, uint32_t add2, uint32_t (&h)[16]) {
        const __half2 m = *reinterpret_cast<const __half2*>(&mul2);
        const __half2 c = *reinterpret_cast<const __half2*>(&add2);
#pragma unroll
        for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int sh = 6 - 4 * i;
                const uint32_t x = sh >= 0 ? (w[wi] << sh) : (w[wi] >> (-sh));
                const uint32_t v = (x & 0x03C003C0u) | 0x3C003C00u;  // 1 + q/16 in each half
                const __half2 f = __hsub2(*reinterpret_cast<const __half2*>(&v), __float2half2_rn(1.0f));
                const __half2 r = __hfma2(f, m, c);
                h[4 * wi + i] = *reinterpret_cast<const uint32_t*>(&r);
            }
        }
    }
};

template <>
struct GroupChunk<2> {
    static constexpr int kWords = 2;
    __device__ __forceinline__ static void run(const uint32_t* w, uint32_t mul2, uint32_t add2, uint32_t (&h)[16]) {
        const __half2 m = *reinterpret_cast<const __half2*>(&mul2);
        const __half2 c = *reinterpret_cast<const __half2*>(&add2);
#pragma unroll
        for (int wi = 0; wi < 2; ++wi) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int sh = 8 - 2 * i;
                const uint32_t x = sh >= 0 ? (w[wi] << sh) : (w[wi] >> (-sh));
                const uint32_t v = (x & 0x03000300u) | 0x3C003C00u;  // 1 + q/4 in each half
                const __half2 f = __hsub2(*reinterpret_cast<const __half2*>(&v), __float2half2_rn(1.0f));
                const __half2 r = __hfma2(f, m, c);
                h[8 * wi + i] = *reinterpret_cast<const uint32_t*>(&r);
            }
        }
    }
};

}  // namespace mmadec
}  // namespace tq

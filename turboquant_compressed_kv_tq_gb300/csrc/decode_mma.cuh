// Tensor-core split-K decode attention over the TurboQuant cache (head_dims
// 64, 128 and 256; 64 runs in the 128 layout, 256 as two CTAs per unit, one
// per 128-column half of the values).
//
// Per (token split, kv head, row group of 16 query rows, sequence) one CTA of
// kWarps warps. Every warp streams its own tiles of compressed records from
// HBM into a private ring of shared-memory stages with 1-D bulk copies
// (cp.async.bulk, completion on an mbarrier), and runs, 32 tokens at a time:
//   scores  S = Q' K_hat^T (+ Q'' sigma^T for prod keys) on mma.sync
//           m16n8k16 (fp16 operands, fp32 accumulate); the key operand is
//           decoded from the packed indices straight into MMA fragments:
//           2-bit indices through a shared table of code quads (one 64-bit
//           load per four levels), 4-bit MSE indices through a shared table
//           of code pairs, other widths with byte-permute lookups in
//           registers; QJL signs as exact +-1 operands (with 3-bit MSE values
//           through a shared table of sign nibbles), their products weighted
//           by the residual norm in fp32; codebook operands are the fp16
//           numbers nearest to op_scale * level (a per-codebook scale that
//           keeps the rounding error small), op_scale divided out in the
//           query (keys) and in the merge (values);
//   softmax online, in log2 units (scale * log2(e) folded into the query),
//           with a lagging row maximum;
//   values  O += P' V_hat on mma.sync, P' = p * value norm, V_hat decoded per
//           token into registers (3- and 4-bit MSE indices through shared
//           tables of code pairs; group codes or-ed into the mantissa of an
//           fp16 1.0, then one subtraction and one multiply-add by the
//           group's scale and minimum) and transposed to the MMA operand
//           layout with movmatrix.
// With at most 8 query rows per KV head a transposed form puts 16 tokens on
// the MMA's M and the rows on N (S^T = K Q^T, O^T = V^T P^T). Warps merge in
// shared memory; each CTA writes its split's (max, sum, acc) rows, and a
// separate merge kernel (one CTA per output row) combines the splits, applies
// the inverse value rotation and writes the output.
//
// Query fragments are prepared by a separate kernel (or inside the fused
// decode-step launch) in the coordinate order the decoders produce (the
// contraction over head_dim is invariant under a common permutation of both
// operands).
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
// Dynamic shared memory the split kernel may use: the 227 KB per-block opt-in
// of the GPU less a margin for its static shared memory.
constexpr size_t kSmemBudget = 227 * 1024 - 1024;
constexpr int kQFragBytes = 2 * 8 * 32 * 16;  // query fragments of one unit
// End of the split kernel: the warps merge their (max, sum, accumulator) rows
// in shared memory from offset 0 (rows of kCoStride floats, a column d at
// d + d / 32 so that the fragment layout stores without bank conflicts).
constexpr int kCoStride = kD + 4;
constexpr int kWarpMergeBytes = (2 * kWarps * kRows + kWarps * kRows * kCoStride) * 4;
constexpr unsigned kSpinLimit = 1u << 22;
// Pair table of 3-bit value codes: 64 entries x 32 bank copies x 4 bytes,
// placed at an 8 KB-aligned shared address inside a 16 KB region.
constexpr int kVPairBytes = 64 * 32 * 4;
constexpr int kVPairRegion = 2 * kVPairBytes;
// Quad table of 2-bit key codes: 256 entries x 16 bank copies x 8 bytes. Used
// for 2-bit key indices except with prod keys and group values, whose records
// leave no room for it next to the 64-token stages.
constexpr int kKQuadBytes = 256 * 16 * 8;
__host__ __device__ constexpr bool quad_keys(int kb, bool kprod, bool vgroup) { return kb == 2 && !(kprod && vgroup); }
// Pair table of 4-bit MSE codes: 256 entries (a byte: two codes) x 32 bank
// copies x 4 bytes. Used with MSE keys at head_dims up to 128: for 4-bit keys,
// and for 4-bit values (with prod keys, or at head_dim 256, the stages would
// have to shrink to make room).
constexpr int kPair4Bytes = 256 * 32 * 4;
__host__ __device__ constexpr bool pair4_keys(int d, int kb, bool kprod) { return d <= kD && !kprod && kb == 4; }
__host__ __device__ constexpr bool pair4_values(int d, bool kprod, bool vgroup, int vb) {
    return d <= kD && !kprod && !vgroup && vb == 4;
}
// With 4-bit MSE keys and values both: one table of 256-byte entries at
// shared offset 0 (256 entries x two sets of 32 bank copies x 4 bytes; keys
// read set 0, values set 1), the lane's address one byte permute of the code
// word (the byte of codes x 256 + the lane's copy) with the table's base
// folded into the load.
constexpr int kPair4WBytes = 256 * 64 * 4;
__host__ __device__ constexpr bool pair4_wide(int d, int kb, bool kprod, bool vgroup, int vb) {
    return pair4_keys(d, kb, kprod) && pair4_values(d, kprod, vgroup, vb);
}
// QJL sign operands through a shared table of sign nibbles (16 entries x 16
// bank copies x 8 bytes) at a 2 KB-aligned shared address: prod keys with
// 3-bit MSE values (in the slack of the value pair table's region) or with
// group values (in a 4 KB region of its own).
constexpr int kQNibBytes = 16 * 16 * 8;
constexpr int kQNibRegion = 4096;
__host__ __device__ constexpr bool nibble_qjl(bool kprod, bool vgroup, int vb) {
    return kprod && (vgroup || vb == 3);
}
// Coordinate order of the query fragments: bit 0 natural pair order of the
// codebook part (quad-table keys), bit 1 natural pair order of the QJL part
// (nibble-table signs); otherwise the byte-permute decoders' orders.
__host__ __device__ constexpr int frag_order(int kb, bool kprod, bool vgroup, int vb) {
    return (quad_keys(kb, kprod, vgroup) ? 1 : 0) | (nibble_qjl(kprod, vgroup, vb) ? 2 : 0);
}

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

__device__ __forceinline__ float rcp_approx(float x) {
    float y;
    asm("rcp.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
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

// The 32 bits of an fp16 pair.
__device__ __forceinline__ uint32_t h2_bits(__half2 x) {
    uint32_t r;
    memcpy(&r, &x, sizeof(r));
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

// ------------------------------------------------------------------ integer work on the FMA pipe
//
// The decoders are bound by the ALU pipe (logic, shifts, byte permutes, integer
// adds). Left shifts and the shift-and-add steps of the bit spreading are
// written as integer multiply-adds instead, which issue to the FMA pipe:
// x << k is x * 2^k, and moving a masked field m of v up by k bits is
// v + (2^k - 1) m. The multipliers sit in constant memory so that the compiler
// keeps them as multiplies rather than folding them back into shifts and adds.
// (Right shifts stay shifts: as the high word of a product they take two
// issue cycles of the FMA pipe, measured slower than the shift.)
struct DecConst {
    uint32_t pow2[32];  // 2^k
    uint32_t m3, m15, m11, m10001;
};
static __constant__ DecConst kDc = {
    {1u << 0,  1u << 1,  1u << 2,  1u << 3,  1u << 4,  1u << 5,  1u << 6,  1u << 7,
     1u << 8,  1u << 9,  1u << 10, 1u << 11, 1u << 12, 1u << 13, 1u << 14, 1u << 15,
     1u << 16, 1u << 17, 1u << 18, 1u << 19, 1u << 20, 1u << 21, 1u << 22, 1u << 23,
     1u << 24, 1u << 25, 1u << 26, 1u << 27, 1u << 28, 1u << 29, 1u << 30, 1u << 31},
    3u, 15u, 0x11u, 0x10001u};

__device__ __forceinline__ uint32_t mad_lo(uint32_t a, uint32_t b, uint32_t c) {
    uint32_t d;
    asm("mad.lo.u32 %0, %1, %2, %3;\n" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// x << k (k a compile-time constant after unrolling, 0..31).
__device__ __forceinline__ uint32_t shl_f(uint32_t x, int k) { return k == 0 ? x : mad_lo(x, kDc.pow2[k], 0u); }

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
// Selector nibbles (c, c + 4) per byte: x * 0x11 + 0x40404040.
__device__ __forceinline__ void dec2_pair(uint32_t w, int s, const Tab4& t, uint32_t& h0, uint32_t& h1) {
    const uint32_t x = (w >> (2 * s)) & 0x03030303u;
    const uint32_t sel = mad_lo(x, kDc.m11, 0x40404040u);
    h0 = prmt(t.lo, t.hi, sel);          // codes s, s+4
    h1 = prmt(t.lo, t.hi, sel >> 16);    // codes s+8, s+12
}

// Sign-magnitude 4-bit decode of 8 codes (one word) with a symmetric codebook:
// value = +mu[k-8] for k >= 8 and -mu[7-k] below. Produces pairs (0,1),(2,3),
// (4,5),(6,7).
__device__ __forceinline__ void dec4_word(uint32_t w, const Tab8& mu, uint32_t (&h)[4]) {
    const uint32_t f = (~(w >> 3)) & 0x11111111u;     // 1 where the code is negative
    const uint32_t u = (w ^ (f * 7u)) & 0x77777777u;      // magnitude index per nibble
    const uint32_t ws = shl_f(w, 4);
    {
        const uint32_t lo4 = prmt(mu.lo0, mu.lo1, u);
        uint32_t hi4 = prmt(mu.hi0, mu.hi1, u);
        const uint32_t s4 = prmt(ws, w, 0xD9C8);   // 0xFF where positive (codes 0..3)
        hi4 ^= ~s4 & 0x80808080u;
        h[0] = prmt(lo4, hi4, 0x5140);
        h[1] = prmt(lo4, hi4, 0x7362);
    }
    {
        const uint32_t u2 = (u >> 16);
        const uint32_t lo4 = prmt(mu.lo0, mu.lo1, u2);
        uint32_t hi4 = prmt(mu.hi0, mu.hi1, u2);
        const uint32_t s4 = prmt(ws, w, 0xFBEA);   // codes 4..7
        hi4 ^= ~s4 & 0x80808080u;
        h[2] = prmt(lo4, hi4, 0x5140);
        h[3] = prmt(lo4, hi4, 0x7362);
    }
}

// 3-bit: 8 codes (v < 2^24) spread into nibbles, then an 8-entry lookup.
// Each spread step moves a masked field up by k bits as v + (2^k - 1)(v & m).
__device__ __forceinline__ void dec3_group(uint32_t v, const Tab8& t, uint32_t (&h)[4]) {
    uint32_t x = mad_lo(v & 0x00FFF000u, kDc.m15, v);     // codes 4..7 up by 4
    x = mad_lo(x & 0x0FC00FC0u, kDc.m3, x);                // codes 2, 3, 6, 7 up by 2
    x = mad_lo(x & 0x38383838u, kDc.pow2[0], x);           // odd codes up by 1
    {
        const uint32_t lo4 = prmt(t.lo0, t.lo1, x);
        const uint32_t hi4 = prmt(t.hi0, t.hi1, x);
        h[0] = prmt(lo4, hi4, 0x5140);
        h[1] = prmt(lo4, hi4, 0x7362);
    }
    {
        const uint32_t x2 = (x >> 16);
        const uint32_t lo4 = prmt(t.lo0, t.lo1, x2);
        const uint32_t hi4 = prmt(t.hi0, t.hi1, x2);
        h[2] = prmt(lo4, hi4, 0x5140);
        h[3] = prmt(lo4, hi4, 0x7362);
    }
}

// One-bit codes / QJL signs: bit i of the word for coordinate i; pair (s, s+16)
// and (s+8, s+24); `neg2` holds (-v, -v) so that a set bit yields +v.
__device__ __forceinline__ uint32_t dec1(uint32_t w, int sh, uint32_t neg2) {
    return (shl_f(w, sh) & 0x80008000u) ^ neg2;
}

// (h, h) from the fp16 bits h.
__device__ __forceinline__ uint32_t dup_half(uint32_t h) { return mad_lo(h, kDc.m10001, 0u); }

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
        // the four 24-bit groups of the 96-bit chunk
        const uint32_t v0 = w[0] & 0xFFFFFFu;
        const uint32_t v1 = mad_lo(w[1] & 0xFFFFu, kDc.pow2[8], (w[0] >> 24));
        const uint32_t v2 = mad_lo(w[2] & 0xFFu, kDc.pow2[16], (w[1] >> 16));
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

// 3-bit codes through a shared-memory table of code pairs, moving the lookups
// from the ALU pipe (byte permutes) to the load pipe. Entry e holds the fp16
// pair (c[e & 7], c[e >> 3]); the copy for lane L of entry e sits at byte
// 128 e + 4 L of an 8 KB-aligned table, so the 32 lanes of a warp always read
// 32 different banks. `lane_addr` is the table's shared address + 4 L. Field p
// of the 96-bit chunk (codes 2p, 2p + 1, bits 6p..6p+5) is shifted to bit 7,
// masked and or-ed onto the lane address: one shift, one logic op and one
// load per pair, in the same pair order as MseChunk<3>.
// Plain shared loads of the lookup tables. The tables are written once before a
// CTA barrier; every lookup address depends on record words loaded after that
// barrier, so the loads (not volatile, free to be scheduled) cannot move above it.
__device__ __forceinline__ uint32_t lds_u32(uint32_t addr) {
    uint32_t v;
    asm("ld.shared.u32 %0, [%1];\n" : "=r"(v) : "r"(addr));
    return v;
}

__device__ __forceinline__ void pair3_chunk(const uint32_t* w, uint32_t lane_addr, uint32_t (&h)[16]) {
#pragma unroll
    for (int p = 0; p < 16; ++p) {
        const int b = 6 * p, wi = b >> 5, off = b & 31;
        uint32_t f;
        if (off + 6 > 32) f = __funnelshift_r(w[wi], w[wi + 1], off - 7);
        else if (off >= 7) f = w[wi] >> (off - 7);
        else f = shl_f(w[wi], 7 - off);
        h[p] = lds_u32((f & 0x1F80u) | lane_addr);
    }
}

// 2-bit codes through a shared-memory table of code quads: entry e (one byte
// of codes, four coordinates) holds the fp16 pairs (c[e & 3], c[(e >> 2) & 3])
// and (c[(e >> 4) & 3], c[e >> 6]); the copy for lane L of entry e sits at byte
// 128 e + 8 (L % 16), so each half-warp's 64-bit loads hit 16 different bank
// pairs. `lane_addr` is the table's shared address + 8 (L % 16). Byte k of word
// hw of the chunk gives pairs 8 hw + 2k and 8 hw + 2k + 1, i.e. coordinates in
// natural order (pair p = coordinates 2p, 2p + 1).
__device__ __forceinline__ uint2 lds_u64(uint32_t addr) {
    uint2 v;
    asm("ld.shared.v2.u32 {%0, %1}, [%2];\n" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ void quad2_chunk(const uint32_t* w, uint32_t lane_addr, uint32_t (&h)[16]) {
#pragma unroll
    for (int hw = 0; hw < 2; ++hw) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t f = k == 0 ? shl_f(w[hw], 7) : (w[hw] >> (8 * k - 7));
            const uint2 v = lds_u64(mad_lo(f & 0x7F80u, kDc.pow2[0], lane_addr));
            h[8 * hw + 2 * k] = v.x;
            h[8 * hw + 2 * k + 1] = v.y;
        }
    }
}

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
                const uint32_t x = sh >= 0 ? shl_f(w[wi], sh) : (w[wi] >> (-sh));
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
                const uint32_t x = sh >= 0 ? shl_f(w[wi], sh) : (w[wi] >> (-sh));
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

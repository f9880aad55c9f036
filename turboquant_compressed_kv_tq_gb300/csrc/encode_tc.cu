// Tensor-core encode for long appends (chunked prefill): MSE and prod codecs,
// head_dim 64 or 128, bf16 or f16 inputs.
//
// The D x D rotation (and, for prod keys, the QJL projection of the residual)
// runs on the 5th-generation tensor cores: one persistent CTA per SM keeps the
// codec's operand tables in shared memory and, per 128-token tile,
//   GEMM 1  Y = X~ (R_hi + R_lo)^T      (tcgen05.mma kind::f16, fp32 in TMEM)
//   epilogue: y = Y * 2^e / (16 n), the Lloyd-Max index #{midpoints < y}, the
//            packed indices, and for prod keys the residual r = y - c[index],
//            its norm, and r~ = 256 r split into fp16 hi/lo operand tiles
//   GEMM 2  Z = (r~_hi + r~_lo)(S_hi + S_lo)^T, minus the lo*lo term (prod)
//   epilogue: sign bits (Z >= 0), residual norm and norm stored.
// The work is split across warps and pipelined over tiles:
//   producer warps (4, one thread per token) load a token, compute its norm
//            in the specification's sequential fused multiply-add order
//            (bit-exact) and write X~ = x * 2^-e into the operand tile;
//   MMA warp issues GEMM 1 of tile i + 1 while tile i's epilogue runs (two
//            TMEM accumulators), then GEMM 2 of tile i;
//   epilogue warps (8, two threads per token, column halves of its TMEM row)
//            quantise, pack and store, and form the residual operands.
// Hand-offs are mbarriers (per buffer: a producer arrives for a buffer's next
// use only after the consumer of its previous use has signalled it free).
// Operands: X~ is exact in fp16 for bf16 or f16 inputs down to 2^-14 of the
// norm; 16 R and S are split into fp16 hi + lo (about 22 significant bits).
// Products are exact and sums are fp32, so y and S r carry errors far below
// the fp32 dot-product bound of the sequential specification: an index or
// sign can differ from it only where the exact value lies within rounding
// distance of a decision threshold (a midpoint, or 0).
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_ptx.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kTileRows = 128;   // tokens per tile = MMA M = TMEM lanes used
constexpr int kProdWarps = 4;    // warps 0..3: one thread per token
constexpr int kEpiWarps = 8;     // warps 4..11: lane quarter warp % 4, column half (warp - 4) / 4
constexpr int kMmaWarp = kProdWarps + kEpiWarps;
constexpr int kEncThreads = 32 * (kMmaWarp + 1);
constexpr int kEpiBar = 1;       // named barrier of the epilogue warps

// mbarriers
enum : int {
    kBarTab = 0,        // codec tables copied
    kBarAFull = 1,      // X~ tile written (4 producer warps)
    kBarAEmpty = 2,     // GEMM 1 read it (commit)
    kBarYFull = 3,      // [2] GEMM 1 done (commit)
    kBarYEmpty = 5,     // [2] accumulator free again: the epilogue read it (8 warps), or
                        //     for prod keys GEMM 2 read the residual stored over it (commit)
    kBarRFull = 7,      // [2] prod keys: the residual stored over accumulator b (8 epilogue warps)
    kBarZFull = 9,      // GEMM 2 done (commit)
    kBarZEmpty = 10,    // epilogue read Z (8 epilogue warps)
    kBarNorm = 11,      // [3] a tile's norms written (4 producer warps)
    kNumBars = 14
};

template <int D, bool PROD>
struct TcLayout {
    static constexpr int kTab = 2 * D * D * 2;           // hi + lo fp16 tables
    static constexpr int kTile = kTileRows * D * 2;      // one fp16 operand tile
    static constexpr int oR = 0;
    static constexpr int oS = oR + kTab;
    static constexpr int oA = oS + (PROD ? kTab : 0);    // X~
    static constexpr int oNorm = oA + kTile;                  // [3][128] norms
    static constexpr int oG2 = oNorm + 3 * kTileRows * 4;     // [3][128] residual sums of half 1 (prod)
    static constexpr int oCb = oG2 + 3 * kTileRows * 4;       // centroids [16], midpoints [16]
    static constexpr int oBar = oCb + 128;
    static constexpr int kBytes = oBar + 128;
    static constexpr uint32_t kLbo = 128;                // next 8 columns (K)
    static constexpr uint32_t kSbo = 16 * D;             // next 8 rows (M/N)
    // TMEM: accumulators Y[2] (D columns each) and Z (prod)
    static constexpr uint32_t kCols = PROD ? (D == 128 ? 512 : 256) : (D == 128 ? 256 : 128);
};

// Byte offset of element (row, k) of a [rows][D] fp16 operand tile in the
// no-swizzle K-major core-matrix layout.
template <int D>
__device__ __forceinline__ int core_off(int row, int k) {
    return ((row >> 3) * (D / 8) + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

__device__ __forceinline__ float elem_f32(const uint4& v, int e, int dtype) {
    const uint32_t w = (&v.x)[e >> 1];
    const uint32_t h = (e & 1) ? (w >> 16) : (w & 0xFFFFu);
    if (dtype == TQ_BF16) return __uint_as_float(h << 16);
    return __half2float(__ushort_as_half(static_cast<unsigned short>(h)));
}

__device__ __forceinline__ uint32_t half2_bits(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Store 8 consecutive columns (k0 multiple of 8) of this thread's row as the
// fp16 hi part in tile a0 and, if a1, the lo remainder in tile a1.
template <int D>
__device__ __forceinline__ void store8(unsigned char* a0, unsigned char* a1, int row, int k0, const float (&f)[8]) {
    uint32_t hi[4], lo[4];
#pragma unroll
    for (int p = 0; p < 4; ++p) {
        hi[p] = half2_bits(f[2 * p], f[2 * p + 1]);
        if (a1) {
            const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&hi[p]));
            lo[p] = half2_bits(f[2 * p] - back.x, f[2 * p + 1] - back.y);
        }
    }
    const int off = core_off<D>(row, k0);
    *reinterpret_cast<uint4*>(a0 + off) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    if (a1) *reinterpret_cast<uint4*>(a1 + off) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
}

// N words at dst (dst aligned to the widest access that divides N words).
template <int N>
__device__ __forceinline__ void store_words(uint32_t* dst, const uint32_t (&w)[N]) {
    if constexpr (N % 4 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 4) reinterpret_cast<uint4*>(dst)[i / 4] = make_uint4(w[i], w[i + 1], w[i + 2], w[i + 3]);
    } else if constexpr (N % 2 == 0) {
#pragma unroll
        for (int i = 0; i < N; i += 2) reinterpret_cast<uint2*>(dst)[i / 2] = make_uint2(w[i], w[i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < N; ++i) dst[i] = w[i];
    }
}

// Lloyd-Max index #{j : y > m_j} over the 2^KB - 1 sorted midpoints, as a
// binary search with register selects (KB compares instead of 2^KB - 1).
template <int KB>
__device__ __forceinline__ int lm_index(float y, const float (&m)[(1 << KB) - 1]) {
    if constexpr (KB == 1) {
        return y > m[0] ? 1 : 0;
    } else if constexpr (KB == 2) {
        const int b1 = y > m[1];
        const int b0 = y > (b1 ? m[2] : m[0]);
        return 2 * b1 + b0;
    } else if constexpr (KB == 3) {
        const int b2 = y > m[3];
        const int b1 = y > (b2 ? m[5] : m[1]);
        const float t0 = b2 ? (b1 ? m[6] : m[4]) : (b1 ? m[2] : m[0]);
        const int b0 = y > t0;
        return 4 * b2 + 2 * b1 + b0;
    } else {
        const int b3 = y > m[7];
        const int b2 = y > (b3 ? m[11] : m[3]);
        const float t1 = b3 ? (b2 ? m[13] : m[9]) : (b2 ? m[5] : m[1]);
        const int b1 = y > t1;
        const int hi = 4 * b3 + 2 * b2 + b1;   // which pair of midpoints is left: m[2 hi], m[2 hi + ...]
        float t0 = m[0];
#pragma unroll
        for (int k = 1; k < 8; ++k) t0 = hi == k ? m[2 * k] : t0;
        const int b0 = y > t0;
        return 2 * hi + b0;
    }
}

// One tensor's tiles t0, t0 + stride, ... (n_it of them) through the pipeline
// below, with the shared memory laid out by TcLayout<D, PROD> and the TMEM
// columns from tmem; returns whether a wait ran out. Every thread of the CTA
// calls it; its barriers are initialised here and invalidated at the end, so
// that a CTA can run one phase per tensor.
template <int D, int KB, bool PROD>
__device__ __forceinline__ bool tc_phase(const EncodeAppendArgs& a, int is_v, int tiles_per_seq, int64_t t0,
                                         int64_t stride, int n_it, unsigned char* smem, uint32_t tmem) {
    using L = TcLayout<D, PROD>;
    constexpr int NM = (1 << KB) - 1;   // midpoints
    constexpr int W = D * KB / 32;      // index words
    constexpr int WS = D / 32;          // sign words
    constexpr int DH = D / 2;           // columns per epilogue thread
    constexpr int CH = DH / 32;         // 32-column chunks per epilogue thread
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::oBar);
    float* s_norm = reinterpret_cast<float*>(smem + L::oNorm);
    float* s_g2 = reinterpret_cast<float*>(smem + L::oG2);
    float* s_c = reinterpret_cast<float*>(smem + L::oCb);
    float* s_m = s_c + 16;

    const CodecDev& cd = is_v ? a.vc : a.kc;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t sbase = tc::smem_addr(smem);
    const int Hkv = a.pool.Hkv;
    auto tile_of = [&](int it) { return t0 + static_cast<int64_t>(it) * stride; };
    // The input rows of a tile are contiguous: thread 0 prefetches a tile's
    // rows into L2 one tile ahead of the producers (the first at launch, while
    // the prologue and the previous kernel's tail run).
    const char* src = static_cast<const char*>(is_v ? a.v : a.k);
    auto prefetch_tile = [&](int it) {
        if (tid != 0 || it >= n_it) return;
        const int64_t tile = tile_of(it);
        const int ts = static_cast<int>(tile % tiles_per_seq);
        const int bh = static_cast<int>(tile / tiles_per_seq);
        const int t0 = ts * kTileRows;
        const int rows = a.n_new - t0 < kTileRows ? a.n_new - t0 : kTileRows;
        tc::bulk_prefetch_l2(src + (static_cast<int64_t>(bh) * a.n_new + t0) * D * 2,
                             static_cast<unsigned>(rows) * D * 2);
    };
    prefetch_tile(0);
    if (tid == 0) {
        tc::mbar_init(&bars[kBarTab], 1);
        tc::mbar_init(&bars[kBarAFull], kProdWarps);
        tc::mbar_init(&bars[kBarAEmpty], 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&bars[kBarYFull + i], 1);
            tc::mbar_init(&bars[kBarYEmpty + i], PROD ? 1 : kEpiWarps);
            tc::mbar_init(&bars[kBarRFull + i], kEpiWarps);
        }
        tc::mbar_init(&bars[kBarZFull], 1);
        tc::mbar_init(&bars[kBarZEmpty], kEpiWarps);
        for (int i = 0; i < 3; ++i) tc::mbar_init(&bars[kBarNorm + i], kProdWarps);
        tc::mbar_fence_init();
        tc::mbar_expect_tx(&bars[kBarTab], (PROD ? 2 : 1) * L::kTab);
        tc::bulk_g2s(smem + L::oR, cd.Rtc, L::kTab, &bars[kBarTab]);
        if constexpr (PROD) tc::bulk_g2s(smem + L::oS, cd.Stc, L::kTab, &bars[kBarTab]);
    }
    if (tid < 16) {
        s_c[tid] = tid <= NM ? cd.c[tid] : 0.0f;
        s_m[tid] = tid < NM ? cd.m[tid] : 0.0f;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const bool tables_failed = __syncthreads_or(!tc::mbar_wait(&bars[kBarTab], 0));

    bool failed = tables_failed;

    if (warp < kProdWarps) {
        // ---------------- producers: norm (sequential order) and X~ of one token
        const int row = tid;
        for (int it = 0; it < n_it && !failed; ++it) {
            prefetch_tile(it + 1);
            const int64_t tile = tile_of(it);
            const int ts = static_cast<int>(tile % tiles_per_seq);
            const int bh = static_cast<int>(tile / tiles_per_seq);
            const int t = ts * kTileRows + row;
            const bool valid = t < a.n_new;
            const uint4* p = reinterpret_cast<const uint4*>(src + (static_cast<int64_t>(bh) * a.n_new + t) * D * 2);
            uint4 raw[D / 8];
#pragma unroll
            for (int c8 = 0; c8 < D / 8; ++c8) raw[c8] = valid ? __ldg(p + c8) : make_uint4(0, 0, 0, 0);
            float n2 = 0.0f;
#pragma unroll
            for (int c8 = 0; c8 < D / 8; ++c8)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float f = elem_f32(raw[c8], e, a.dtype);
                    n2 = __fmaf_rn(f, f, n2);
                }
            const float n = __fsqrt_rn(n2);
            const float down = scalbnf(1.0f, n > 0.0f ? -ilogbf(n) : 0);
            // the operand tile and this stash slot are free once GEMM 1 of the
            // previous tile has read the tile (which also means the epilogue of
            // the tile three back, the slot's previous user, has finished)
            if (!tc::mbar_wait(&bars[kBarAEmpty], (it & 1) ^ 1)) {
                failed = true;
                break;
            }
            s_norm[(it % 3) * kTileRows + row] = n;
#pragma unroll
            for (int c8 = 0; c8 < D / 8; ++c8) {
                float f[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) f[e] = elem_f32(raw[c8], e, a.dtype) * down;
                store8<D>(smem + L::oA, nullptr, row, 8 * c8, f);
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
                tc::mbar_arrive(&bars[kBarAFull]);
                tc::mbar_arrive(&bars[kBarNorm + it % 3]);
            }
        }
    } else if (warp == kMmaWarp) {
        // ---------------- MMAs: GEMM 1 of tile it + 1 before GEMM 2 of tile it
        if (lane == 0 && !failed) {
            constexpr uint32_t idesc = tc::idesc_f16_f32(kTileRows, D);
            auto lo_of = [&](int off) { return static_cast<uint32_t>(tc::smem_desc(sbase + off, L::kLbo, 0) & 0xFFFFFFFFu); };
            const uint32_t hi = static_cast<uint32_t>(tc::smem_desc(0, 0, L::kSbo) >> 32);
            const uint64_t hi64 = static_cast<uint64_t>(hi) << 32;
            const uint32_t la = lo_of(L::oA), lrh = lo_of(L::oR), lrl = lo_of(L::oR + L::kTab / 2);
            bool ok = true;
            int g1 = 0, g2n = 0;
            auto gemm1 = [&](int it) {
                const int bb = it & 1;
                ok = tc::mbar_wait(&bars[kBarAFull], it & 1) &&
                     tc::mbar_wait(&bars[kBarYEmpty + bb], ((it >> 1) & 1) ^ 1);
                if (!ok) return;
                tc::tc_fence_after();
                const uint32_t d = tmem + bb * D;
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    tc::mma_f16(d, hi64 | (la + 16 * s), hi64 | (lrh + 16 * s), idesc, s > 0);
                    tc::mma_f16(d, hi64 | (la + 16 * s), hi64 | (lrl + 16 * s), idesc, 1);
                }
                tc::mma_commit(&bars[kBarYFull + bb]);
                tc::mma_commit(&bars[kBarAEmpty]);
                ++g1;
            };
            if (n_it > 0) gemm1(0);
            for (int it = 0; it < n_it && ok; ++it) {
                if (it + 1 < n_it) gemm1(it + 1);
                if (!ok) break;
                if constexpr (PROD) {
                    // GEMM 2 of tile it: its A operand, the residual r~ as fp16 hi / lo
                    // pairs, lies over accumulator bb: 32-coordinate chunk q in
                    // columns 32 q .. 32 q + 15 (hi) and 32 q + 16 .. 32 q + 31 (lo)
                    const int bb = it & 1;
                    ok = tc::mbar_wait(&bars[kBarRFull + bb], (it >> 1) & 1) &&
                         tc::mbar_wait(&bars[kBarZEmpty], (it & 1) ^ 1);
                    if (!ok) break;
                    tc::tc_fence_after();
                    const uint32_t d = tmem + 2 * D;
                    const uint32_t yb = tmem + bb * D;
                    const uint32_t lsh = lo_of(L::oS), lsl = lo_of(L::oS + L::kTab / 2);
#pragma unroll
                    for (int s = 0; s < D / 16; ++s) {
                        const uint32_t ah = yb + 32 * (s >> 1) + 8 * (s & 1), al = ah + 16;
                        tc::mma_f16_ta(d, ah, hi64 | (lsh + 16 * s), idesc, s > 0);
                        tc::mma_f16_ta(d, al, hi64 | (lsh + 16 * s), idesc, 1);
                        tc::mma_f16_ta(d, ah, hi64 | (lsl + 16 * s), idesc, 1);
                    }
                    tc::mma_commit(&bars[kBarZFull]);
                    tc::mma_commit(&bars[kBarYEmpty + bb]);   // the accumulator takes tile it + 2
                    ++g2n;
                }
            }
            if (!ok) {
                failed = true;
                atomicOr(a.err, TQ_DEVERR_TIMEOUT);
            }
            // drain (after a timeout elsewhere): the last commits of each kind
            if (g1) (void)tc::mbar_wait(&bars[kBarAEmpty], (g1 - 1) & 1);
            if (g2n) (void)tc::mbar_wait(&bars[kBarZFull], (g2n - 1) & 1);
        }
        __syncwarp();
    } else {
        // ---------------- epilogue: two threads per token (column halves)
        const int ew = warp - kProdWarps;
        const int lq = warp & 3, half = ew >> 2;
        const int row = 32 * lq + lane;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(32 * lq) << 16) + DH * half;
        float mreg[NM];
#pragma unroll
        for (int j = 0; j < NM; ++j) mreg[j] = s_m[j];
        // 2-bit codebooks: levels from registers, as -256 c (the residual is
        // formed directly as r~ = 256 y - 256 c, see below)
        const float creg[4] = {-256.0f * s_c[0], -256.0f * s_c[1], -256.0f * s_c[2], -256.0f * s_c[3]};
        const int64_t o_idx = is_v ? a.pool.off[4] : a.pool.off[0];
        const int64_t o_norm = is_v ? a.pool.off[5] : a.pool.off[2];
        // destination of this thread's token of tile it in the pool (null: out of
        // range, flagged); computed one tile ahead, so that its loads (sequence
        // length, block table) are in flight while the current tile is processed
        auto dest_of = [&](int it, char*& sub, int& slot) {
            const int64_t tile = tile_of(it);
            const int ts = static_cast<int>(tile % tiles_per_seq);
            const int bh = static_cast<int>(tile / tiles_per_seq);
            const int h = bh % Hkv, b = bh / Hkv;
            const int t = ts * kTileRows + row;
            sub = nullptr;
            slot = 0;
            if (t >= a.n_new) return;
            const int pos = a.seq_lens[b] + t;
            const int BT = a.pool.BT;
            const int lb = pos / BT;
            slot = pos - lb * BT;
            if (pos < 0 || lb >= a.max_blocks) {
                atomicOr(a.err, TQ_DEVERR_CAPACITY);
                return;
            }
            const int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(b) * a.max_blocks + lb])
                                       : static_cast<int64_t>(b) * a.max_blocks + lb;
            if (pb < 0 || pb >= a.pool.num_blocks) atomicOr(a.err, TQ_DEVERR_BLOCK);
            else sub = a.pool.base + (pb * Hkv + h) * a.pool.sub_bytes;
        };
        // Index pass of tile j: Lloyd-Max indices packed and stored, the norm
        // stored; for prod keys also the residual r~ = 256 (y - c), stored as fp16
        // hi / lo pairs over the 32-column accumulator chunk the thread has just
        // read (the A operand of GEMM 2), and this half's residual sum.
        auto index_pass = [&](int j, char*& sub, int& slot, float& g2) -> bool {
            const int bj = j & 1;
            const bool okw = tc::mbar_wait(&bars[kBarYFull + bj], (j >> 1) & 1) &&
                             tc::mbar_wait(&bars[kBarNorm + j % 3], (j / 3) & 1);
            tc::tc_fence_after();
            dest_of(j, sub, slot);
            const float n = s_norm[(j % 3) * kTileRows + row];
            const int ex = n > 0.0f ? ilogbf(n) : 0;
            const float inv = n > 0.0f ? __fdiv_rn(scalbnf(1.0f, ex - 4), n) : 0.0f;
            uint32_t* widx = sub ? reinterpret_cast<uint32_t*>(sub + o_idx) + static_cast<int64_t>(slot) * W : nullptr;
            float g2p[4] = {0.0f, 0.0f, 0.0f, 0.0f};   // 2^16 x the residual sum of squares, four chains
#pragma unroll 1
            for (int ch = 0; ch < CH; ++ch) {
                float v[32];
                const uint32_t tcol = t_lane + bj * D + 32 * ch;
                tc::tmem_ld32(tcol, v);
                uint32_t cw[KB];
#pragma unroll
                for (int q = 0; q < KB; ++q) cw[q] = 0u;
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const float y = v[i] * inv;
                    int code;
                    float cc = 0.0f;   // -256 x the index's level (prod keys)
                    if constexpr (PROD && KB == 2) {
                        // the index and its level from the same two comparisons
                        const bool p1 = y > mreg[1];
                        const bool p0 = y > (p1 ? mreg[2] : mreg[0]);
                        code = (p1 ? 2 : 0) + (p0 ? 1 : 0);
                        cc = p1 ? (p0 ? creg[3] : creg[2]) : (p0 ? creg[1] : creg[0]);
                    } else {
                        code = lm_index<KB>(y, mreg);
                    }
                    const int bit = i * KB;
                    cw[bit >> 5] += static_cast<uint32_t>(code) << (bit & 31);   // disjoint bits: a shift-add
                    if ((bit & 31) + KB > 32) cw[(bit >> 5) + 1] |= static_cast<uint32_t>(code) >> (32 - (bit & 31));
                    if constexpr (PROD) {
                        if constexpr (KB == 1) cc = (code & 1) ? creg[1] : creg[0];
                        else if constexpr (KB > 2) cc = -256.0f * s_c[code];
                        // r~ = 256 (y - c) in one rounding: scaling by a power of two
                        // commutes with rounding (y - c is 0 or a normal number), so
                        // r~ is bit for bit 256 x fp32(y - c); the sums of r~^2 are
                        // then exactly 2^16 x the sums of r^2
                        const float rs = __fmaf_rn(y, 256.0f, cc);
                        g2p[i & 3] = __fmaf_rn(rs, rs, g2p[i & 3]);
                        v[i] = rs;
                    }
                }
                if (widx) store_words<KB>(widx + KB * (CH * half + ch), cw);
                if constexpr (PROD) {
                    uint32_t hi[16], lo[16];
#pragma unroll
                    for (int p = 0; p < 16; ++p) {
                        hi[p] = half2_bits(v[2 * p], v[2 * p + 1]);
                        const float2 back = __half22float2(*reinterpret_cast<const __half2*>(&hi[p]));
                        lo[p] = half2_bits(v[2 * p] - back.x, v[2 * p + 1] - back.y);
                    }
                    tc::tmem_st16u(tcol, hi);
                    tc::tmem_st16u(tcol + 16, lo);
                }
            }
            if (sub && half == 0) reinterpret_cast<float*>(sub + o_norm)[slot] = n;
            g2 = (g2p[0] + g2p[1]) + (g2p[2] + g2p[3]);
            tc::tc_fence_before();
            __syncwarp();
            if constexpr (PROD) {
                if (half == 1) s_g2[(j % 3) * kTileRows + row] = g2;
                if (lane == 0) tc::mbar_arrive(&bars[kBarRFull + bj]);   // GEMM 2 may read the residual
            } else {
                if (lane == 0) tc::mbar_arrive(&bars[kBarYEmpty + bj]);  // the accumulator may take the tile after next
            }
            return okw;
        };
        if constexpr (PROD) {
            // Sign pass of tile j: the signs of S r and the residual norm (the
            // other half's residual sum from shared memory, after the barrier).
            auto sign_pass = [&](int j, char* sub, int slot, float g2, bool ok) -> bool {
                ok = ok && tc::mbar_wait(&bars[kBarZFull], j & 1);
                tc::tc_fence_after();
                uint32_t sw[CH];
#pragma unroll
                for (int ch = 0; ch < CH; ++ch) {
                    float v[32];
                    tc::tmem_ld32(t_lane + 2 * D + 32 * ch, v);
                    uint32_t w = 0u;
#pragma unroll
                    for (int i = 0; i < 32; ++i) w |= (v[i] >= 0.0f ? 1u : 0u) << i;
                    sw[ch] = w;
                }
                tc::tc_fence_before();
                __syncwarp();
                if (lane == 0) tc::mbar_arrive(&bars[kBarZEmpty]);
                if (tc::bar_or(kEpiBar, 32 * kEpiWarps, !ok)) return false;   // uniform failure exit
                if (sub) {
                    store_words<CH>(reinterpret_cast<uint32_t*>(sub + a.pool.off[1]) + static_cast<int64_t>(slot) * WS +
                                        CH * half,
                                    sw);
                    if (half == 0)
                        reinterpret_cast<float*>(sub + a.pool.off[3])[slot] =
                            __fsqrt_rn(g2 + s_g2[(j % 3) * kTileRows + row]) * 0.00390625f;   // sqrt(2^16 x) / 256, exact
                }
                return true;
            };
            // the index pass runs one tile ahead: GEMM 2 of tile it overlaps the
            // index pass of tile it + 1 (the residual of tile it + 1 lies over the
            // other accumulator; the residual sums rotate through three slots)
            char* sub_c = nullptr;
            char* sub_n = nullptr;
            int slot_c = 0, slot_n = 0;
            float g2_c = 0.0f, g2_n = 0.0f;
            bool ok = n_it > 0 ? index_pass(0, sub_c, slot_c, g2_c) : true;
            for (int it = 0; it < n_it && !failed; ++it) {
                if (it + 1 < n_it) ok = index_pass(it + 1, sub_n, slot_n, g2_n) && ok;
                if (!sign_pass(it, sub_c, slot_c, g2_c, ok)) {
                    failed = true;
                    break;
                }
                sub_c = sub_n;
                slot_c = slot_n;
                g2_c = g2_n;
            }
        } else {
            for (int it = 0; it < n_it && !failed; ++it) {
                char* sub = nullptr;
                int slot = 0;
                float g2 = 0.0f;
                const bool ok = index_pass(it, sub, slot, g2);
                if (tc::bar_or(kEpiBar, 32 * kEpiWarps, !ok)) {
                    failed = true;
                    break;
                }
            }
        }
    }

    failed = __syncthreads_or(failed);
    if (failed && tid == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (tid == 0)
        for (int i = 0; i < kNumBars; ++i) tc::mbar_inval(&bars[i]);
    __syncthreads();  // the next phase may reuse this shared memory and these TMEM columns
    return failed;
}

// The CTA's TMEM columns for its phases (the widest layout's), allocated by
// warp 0; the next kernel may take SMs as they free up at this launch's tail
// (it shares no data with this one); this kernel completes only after its
// predecessor (the wait at exit).
template <int COLS>
__device__ __forceinline__ uint32_t tc_begin(uint32_t* slot) {
    tc::grid_release_dependents();
    if (threadIdx.x < 32) {
        tc::tmem_alloc(slot, COLS);
        tc::tmem_relinquish();
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    return *slot;
}

template <int COLS>
__device__ __forceinline__ void tc_end(uint32_t tmem) {
    if (threadIdx.x < 32) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, COLS);
    }
    tc::grid_wait_prior();
}

// One tensor (keys: is_v = 0, values: is_v = 1), persistent CTAs over its tiles.
template <int D, int KB, bool PROD>
__global__ void __launch_bounds__(kEncThreads, 1)
    encode_tc_kernel(EncodeAppendArgs a, int is_v, int tiles_per_seq) {
    using L = TcLayout<D, PROD>;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint32_t s_tmem;
    const uint32_t tmem = tc_begin<L::kCols>(&s_tmem);
    const int64_t ntiles = static_cast<int64_t>(a.batch) * a.pool.Hkv * tiles_per_seq;
    const int n_it = blockIdx.x < ntiles ? static_cast<int>((ntiles - 1 - blockIdx.x) / gridDim.x + 1) : 0;
    (void)tc_phase<D, KB, PROD>(a, is_v, tiles_per_seq, blockIdx.x, gridDim.x, n_it, smem, tmem);
    tc_end<L::kCols>(tmem);
}

// Keys and values of one append in one launch: the first GK CTAs run the
// keys' tiles (CTA c takes c, c + GK, ...), the others the values' tiles, both
// tensors side by side on disjoint SMs. GK splits the grid by the tensors'
// relative tile cost (a prod tile, with its QJL GEMM and sign pass, costs about
// 1.2 MSE tiles), so that both halves finish together; each CTA runs one
// phase, with no switch of tables or barriers inside a CTA.
template <int D, int KBK, bool PRODK, int KBV, bool PRODV>
__global__ void __launch_bounds__(kEncThreads, 1)
    encode_tc_pair_kernel(EncodeAppendArgs a, int tiles_per_seq, int gk) {
    using LK = TcLayout<D, PRODK>;
    using LV = TcLayout<D, PRODV>;
    constexpr int kCols = LK::kCols > LV::kCols ? LK::kCols : LV::kCols;
    extern __shared__ __align__(1024) unsigned char smem[];
    __shared__ uint32_t s_tmem;
    const uint32_t tmem = tc_begin<kCols>(&s_tmem);
    const int64_t nt = static_cast<int64_t>(a.batch) * a.pool.Hkv * tiles_per_seq;   // per tensor
    const int64_t c = blockIdx.x;
    if (c < gk) {
        const int n = c < nt ? static_cast<int>((nt - 1 - c) / gk + 1) : 0;
        (void)tc_phase<D, KBK, PRODK>(a, 0, tiles_per_seq, c, gk, n, smem, tmem);
    } else {
        const int64_t cv = c - gk, gv = gridDim.x - gk;
        const int n = cv < nt ? static_cast<int>((nt - 1 - cv) / gv + 1) : 0;
        (void)tc_phase<D, KBV, PRODV>(a, 1, tiles_per_seq, cv, gv, n, smem, tmem);
    }
    tc_end<kCols>(tmem);
}

int sm_count() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int v = cache[dev & 63].load();
    if (v == 0) {
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev & 63].store(v);
    }
    return v;
}

template <int D, int KB, bool PROD>
cudaError_t launch_tc(const EncodeAppendArgs& a, int is_v, cudaStream_t s) {
    using L = TcLayout<D, PROD>;
    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(encode_tc_kernel<D, KB, PROD>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, L::kBytes);
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        attr_set.fetch_or(bit);
    }
    const int tiles_per_seq = (a.n_new + kTileRows - 1) / kTileRows;
    const int64_t ntiles = static_cast<int64_t>(a.batch) * a.pool.Hkv * tiles_per_seq;
    int64_t grid = static_cast<int64_t>(sm_count());
    if (grid <= 0) return cudaErrorInvalidDevice;
    if (grid > ntiles) grid = ntiles;
    const cudaError_t e = launch_overlapped(encode_tc_kernel<D, KB, PROD>, dim3(static_cast<unsigned>(grid)),
                                            dim3(kEncThreads), L::kBytes, s, a, is_v, tiles_per_seq);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e;
}

template <int D, int KBK, bool PRODK, int KBV, bool PRODV>
cudaError_t launch_tc_pair(const EncodeAppendArgs& a, cudaStream_t s) {
    constexpr size_t kBytes = TcLayout<D, PRODK>::kBytes > TcLayout<D, PRODV>::kBytes ? TcLayout<D, PRODK>::kBytes
                                                                                       : TcLayout<D, PRODV>::kBytes;
    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(encode_tc_pair_kernel<D, KBK, PRODK, KBV, PRODV>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kBytes));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        attr_set.fetch_or(bit);
    }
    const int tiles_per_seq = (a.n_new + kTileRows - 1) / kTileRows;
    const int64_t nt = static_cast<int64_t>(a.batch) * a.pool.Hkv * tiles_per_seq;   // per tensor
    int64_t grid = static_cast<int64_t>(sm_count());
    if (grid <= 0) return cudaErrorInvalidDevice;
    if (grid > 2 * nt) grid = 2 * nt;
    if (grid < 2) grid = 2;
    // CTAs for the keys: the split that minimises the later of the two halves'
    // ends, each half's time its most tiles per CTA x its tiles' relative cost
    // (a prod tile costs about 1.2 MSE tiles)
    constexpr double wk = PRODK ? 1.2 : 1.0, wv = PRODV ? 1.2 : 1.0;
    int64_t gk = 1;
    double best = 1e300;
    for (int64_t g = 1; g < grid; ++g) {
        const double t = std::max(static_cast<double>((nt + g - 1) / g) * wk,
                                  static_cast<double>((nt + grid - g - 1) / (grid - g)) * wv);
        if (t < best) {
            best = t;
            gk = g;
        }
    }
    const cudaError_t e = launch_overlapped(encode_tc_pair_kernel<D, KBK, PRODK, KBV, PRODV>,
                                            dim3(static_cast<unsigned>(grid)), dim3(kEncThreads), kBytes, s, a,
                                            tiles_per_seq, static_cast<int>(gk));
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e;
}

template <int D>
cudaError_t dispatch_kb(const EncodeAppendArgs& a, int is_v, const CodecDev& cd, cudaStream_t s) {
    const bool prod = cd.mode == TQ_MODE_PROD;
    switch (cd.ib) {
        case 1: return prod ? launch_tc<D, 1, true>(a, is_v, s) : launch_tc<D, 1, false>(a, is_v, s);
        case 2: return prod ? launch_tc<D, 2, true>(a, is_v, s) : launch_tc<D, 2, false>(a, is_v, s);
        case 3: return prod ? launch_tc<D, 3, true>(a, is_v, s) : launch_tc<D, 3, false>(a, is_v, s);
        case 4: return prod ? launch_tc<D, 4, true>(a, is_v, s) : launch_tc<D, 4, false>(a, is_v, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace

bool encode_tc_supported(const EncodeAppendArgs& a, int is_v) {
    const CodecDev& cd = is_v ? a.vc : a.kc;
    if (cd.mode != TQ_MODE_MSE && cd.mode != TQ_MODE_PROD) return false;
    if (cd.D != 64 && cd.D != 128) return false;
    if (!cd.Rtc || (cd.mode == TQ_MODE_PROD && !cd.Stc)) return false;
    return a.dtype == TQ_BF16 || a.dtype == TQ_F16;
}

// Keys and values in one tensor-core launch, for the codec pairs built as
// one kernel (head_dim 128: prod keys of 3 bits with 3- or 4-bit MSE values,
// 4-bit MSE keys and values); false for the others (two launches instead).
bool launch_encode_tc_pair(const EncodeAppendArgs& a, cudaStream_t s, cudaError_t* err) {
    if (a.kc.D != 128 || a.vc.D != 128) return false;
    const bool kp = a.kc.mode == TQ_MODE_PROD, vp = a.vc.mode == TQ_MODE_PROD;
    if (kp && a.kc.ib == 2 && !vp && a.vc.ib == 3) *err = launch_tc_pair<128, 2, true, 3, false>(a, s);
    else if (kp && a.kc.ib == 2 && !vp && a.vc.ib == 4) *err = launch_tc_pair<128, 2, true, 4, false>(a, s);
    else if (!kp && a.kc.ib == 4 && !vp && a.vc.ib == 4) *err = launch_tc_pair<128, 4, false, 4, false>(a, s);
    else return false;
    return true;
}

// Tensor-core encode of one tensor (keys: is_v = 0, values: is_v = 1).
cudaError_t launch_encode_tc(const EncodeAppendArgs& a, int is_v, cudaStream_t s) {
    const CodecDev& cd = is_v ? a.vc : a.kc;
    if (cd.D == 64) return dispatch_kb<64>(a, is_v, cd, s);
    if (cd.D == 128) return dispatch_kb<128>(a, is_v, cd, s);
    return cudaErrorInvalidValue;
}

}  // namespace tq

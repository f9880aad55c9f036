// Tensor-core encode for long appends (chunked prefill): MSE and prod codecs,
// head_dim 64 or 128, bf16 or f16 inputs.
//
// The D x D rotation (and, for prod keys, the QJL projection of the residual)
// runs on the 5th-generation tensor cores: one persistent CTA per SM keeps the
// codec's operand tables in shared memory and, per 128-token tile,
//   GEMM 1  Y = X~ (R_hi + R_lo)^T      (tcgen05.mma kind::f16, fp32 in TMEM)
//   epilogue: one thread per token reads its row of Y from TMEM, forms
//            y = Y * 2^e / (16 n), the Lloyd-Max index #{midpoints < y}, packs
//            the indices, and for prod keys the residual r = y - c[index],
//            its norm, and r~ = 256 r split into fp16 hi/lo operand tiles
//   GEMM 2  Z = (r~_hi + r~_lo)(S_hi + S_lo)^T, minus the lo*lo term (prod)
//   epilogue: sign bits (Z >= 0), residual norm and norm stored.
// Operands: X~ = x * 2^-e (e = exponent of the norm) is exact in fp16 for bf16
// or f16 inputs down to 2^-14 of the norm; 16 R and S are split into fp16
// hi + lo (about 22 significant bits). Products are exact and sums are fp32,
// so y and S r carry errors far below the fp32 dot-product bound of the
// sequential specification: an index or sign can differ from it only where the
// exact value lies within rounding distance of a decision threshold (a
// midpoint, or 0). The norm keeps the specification's sequential fused
// multiply-add order and is bit-exact.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_ptx.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kTileRows = 128;  // tokens per tile = MMA M = TMEM lanes used

// Threads per token: prod keys (one CTA per SM: their operand tables fill
// shared memory) split each token's TMEM row between two threads; MSE codecs
// run two CTAs per SM with one thread per token.
template <bool PROD>
struct Split {
    static constexpr int kTPT = PROD ? 2 : 1;
    static constexpr int kThreads = kTileRows * kTPT;
};

template <int D, bool PROD>
struct TcLayout {
    static constexpr int kTab = 2 * D * D * 2;           // hi + lo fp16 tables
    static constexpr int kTile = kTileRows * D * 2;      // one fp16 operand tile
    static constexpr int oR = 0;
    static constexpr int oS = oR + kTab;
    static constexpr int oA0 = oS + (PROD ? kTab : 0);   // inputs, then residual hi
    static constexpr int oA1 = oA0 + kTile;              // residual lo (prod)
    static constexpr int oMisc = oA1 + (PROD ? kTile : 0);
    static constexpr int kBytes = oMisc + 2048;
    static constexpr uint32_t kLbo = 128;                // next 8 columns (K)
    static constexpr uint32_t kSbo = 16 * D;             // next 8 rows (M/N)
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

template <int D, int KB, bool PROD>
__global__ void __launch_bounds__(Split<PROD>::kThreads, 1)
    encode_tc_kernel(EncodeAppendArgs a, int is_v, int tiles_per_seq) {
    using L = TcLayout<D, PROD>;
    constexpr int TPT = Split<PROD>::kTPT;
    constexpr int NM = (1 << KB) - 1;   // midpoints
    constexpr int W = D * KB / 32;      // index words
    constexpr int WS = D / 32;          // sign words
    constexpr int DH = D / TPT;         // columns per thread
    constexpr int CH = DH / 32;         // 32-column chunks per thread
    extern __shared__ __align__(1024) unsigned char smem[];
    float* s_c = reinterpret_cast<float*>(smem + L::oMisc);
    float* s_m = s_c + 16;
    uint64_t* bar_tab = reinterpret_cast<uint64_t*>(smem + L::oMisc + 128);
    uint64_t* bar_mma = bar_tab + 1;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_tab + 2);
    float* s_n2 = reinterpret_cast<float*>(smem + L::oMisc + 256);    // [128] first-half norm sums
    float* s_nrm = s_n2 + kTileRows;                                  // [128] norms
    float* s_g2 = s_nrm + kTileRows;                                  // [128] second-half residual sums

    const CodecDev& cd = is_v ? a.vc : a.kc;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int row = tid & (kTileRows - 1), half = TPT == 2 ? (tid >> 7) : 0;
    const uint32_t sbase = tc::smem_addr(smem);

    if (warp == 0) {
        tc::tmem_alloc(s_tmem, D);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        tc::mbar_init(bar_tab, 1);
        tc::mbar_init(bar_mma, 1);
        tc::mbar_fence_init();
        tc::mbar_expect_tx(bar_tab, (PROD ? 2 : 1) * L::kTab);
        tc::bulk_g2s(smem + L::oR, cd.Rtc, L::kTab, bar_tab);
        if constexpr (PROD) tc::bulk_g2s(smem + L::oS, cd.Stc, L::kTab, bar_tab);
    }
    if (tid < 16) {
        s_c[tid] = tid <= NM ? cd.c[tid] : 0.0f;
        s_m[tid] = tid < NM ? cd.m[tid] : 0.0f;
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const uint32_t tmem = *s_tmem;
    const uint32_t tmem_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16) + DH * half;
    float mreg[NM];
#pragma unroll
    for (int j = 0; j < NM; ++j) mreg[j] = s_m[j];

    bool ok = tc::mbar_wait(bar_tab, 0);
    const bool tables_failed = __syncthreads_or(!ok);

    const int Hkv = a.pool.Hkv;
    const int64_t ntiles = static_cast<int64_t>(a.batch) * Hkv * tiles_per_seq;
    const char* src = static_cast<const char*>(is_v ? a.v : a.k);
    const int64_t o_idx = is_v ? a.pool.off[4] : a.pool.off[0];
    const int64_t o_norm = is_v ? a.pool.off[5] : a.pool.off[2];
    constexpr uint32_t idesc = tc::idesc_f16_f32(kTileRows, D);
    unsigned phase = 0;
    bool failed = tables_failed;
    unsigned char* A0 = smem + L::oA0;
    unsigned char* A1 = smem + L::oA1;

    // this thread's columns of its token in a tile, loaded one tile ahead
    uint4 nraw[DH / 8];
    auto load_row = [&](int64_t tl) {
        const int ts = static_cast<int>(tl % tiles_per_seq);
        const int bh = static_cast<int>(tl / tiles_per_seq);
        const int t = ts * kTileRows + row;
        const bool ok_row = tl < ntiles && t < a.n_new;
        const int64_t r = (static_cast<int64_t>(bh / Hkv) * Hkv + bh % Hkv) * a.n_new + t;
        const uint4* p = reinterpret_cast<const uint4*>(src + r * D * 2) + half * (DH / 8);
#pragma unroll
        for (int c8 = 0; c8 < DH / 8; ++c8) nraw[c8] = ok_row ? __ldg(p + c8) : make_uint4(0, 0, 0, 0);
    };
    load_row(blockIdx.x);

    for (int64_t tile = blockIdx.x; tile < ntiles && !failed; tile += gridDim.x) {
        const int ts = static_cast<int>(tile % tiles_per_seq);
        const int bh = static_cast<int>(tile / tiles_per_seq);
        const int h = bh % Hkv, b = bh / Hkv;
        const int t = ts * kTileRows + row;
        const bool valid = t < a.n_new;

        // ---------------- this thread's columns (loaded during the previous tile):
        // the norm's sequential fma chain runs over the first half, then
        // continues over the second half in the other thread of the token
        uint4 raw[DH / 8];
#pragma unroll
        for (int c8 = 0; c8 < DH / 8; ++c8) raw[c8] = nraw[c8];
        float n2 = 0.0f;
        if (TPT == 1 || half == 0) {
#pragma unroll
            for (int c8 = 0; c8 < DH / 8; ++c8)
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const float f = elem_f32(raw[c8], e, a.dtype);
                    n2 = __fmaf_rn(f, f, n2);
                }
        }
        float n;
        if constexpr (TPT == 2) {
            if (half == 0) s_n2[row] = n2;
            __syncthreads();
            if (half == 1) {
                n2 = s_n2[row];
#pragma unroll
                for (int c8 = 0; c8 < DH / 8; ++c8)
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const float f = elem_f32(raw[c8], e, a.dtype);
                        n2 = __fmaf_rn(f, f, n2);
                    }
                s_nrm[row] = __fsqrt_rn(n2);
            }
            __syncthreads();
            n = s_nrm[row];
        } else {
            n = __fsqrt_rn(n2);
        }
        const int ex = n > 0.0f ? ilogbf(n) : 0;
        const float down = scalbnf(1.0f, -ex);
#pragma unroll
        for (int c8 = 0; c8 < DH / 8; ++c8) {
            float f[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = elem_f32(raw[c8], e, a.dtype) * down;
            store8<D>(A0, nullptr, row, DH * half + 8 * c8, f);
        }
        tc::fence_proxy_async_smem();
        tc::tc_fence_before();
        __syncthreads();

        // ---------------- GEMM 1: Y = X~ (16 R)^T in two fp16 parts
        if (tid == 0) {
            tc::tc_fence_after();
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const uint64_t ad = tc::smem_desc(sbase + L::oA0 + 256 * s, L::kLbo, L::kSbo);
                tc::mma_f16(tmem, ad, tc::smem_desc(sbase + L::oR + 256 * s, L::kLbo, L::kSbo), idesc, s > 0);
                tc::mma_f16(tmem, ad, tc::smem_desc(sbase + L::oR + L::kTab / 2 + 256 * s, L::kLbo, L::kSbo),
                            idesc, 1);
            }
            tc::mma_commit(bar_mma);
        }
        load_row(tile + gridDim.x);  // next tile's row, in flight during this tile
        ok = tc::mbar_wait(bar_mma, phase);
        if (__syncthreads_or(!ok)) {
            failed = true;  // the commit of `phase` is still outstanding
            break;
        }
        phase ^= 1;
        tc::tc_fence_after();

        // ---------------- epilogue 1: indices (and residual operands for prod),
        // 32 columns at a time; their KB index words are stored directly
        const float inv = n > 0.0f ? __fdiv_rn(scalbnf(1.0f, ex - 4), n) : 0.0f;

        // destination of this token in the pool
        char* sub = nullptr;
        int slot = 0;
        if (valid) {
            const int pos = a.seq_lens[b] + t;
            const int BT = a.pool.BT;
            const int lb = pos / BT;
            slot = pos - lb * BT;
            if (pos < 0 || lb >= a.max_blocks) {
                atomicOr(a.err, TQ_DEVERR_CAPACITY);
            } else {
                const int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(b) * a.max_blocks + lb])
                                           : static_cast<int64_t>(b) * a.max_blocks + lb;
                if (pb < 0 || pb >= a.pool.num_blocks) atomicOr(a.err, TQ_DEVERR_BLOCK);
                else sub = a.pool.base + (pb * Hkv + h) * a.pool.sub_bytes;
            }
        }
        uint32_t* widx = sub ? reinterpret_cast<uint32_t*>(sub + o_idx) + static_cast<int64_t>(slot) * W : nullptr;

        float g2 = 0.0f;
#pragma unroll 1
        for (int ch = 0; ch < CH; ++ch) {
            float v[32];
            tc::tmem_ld32(tmem_row + 32 * ch, v);
            uint32_t cw[KB];
#pragma unroll
            for (int q = 0; q < KB; ++q) cw[q] = 0u;
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const float y = v[i] * inv;
                int code = 0;
#pragma unroll
                for (int j = 0; j < NM; ++j) code += y > mreg[j] ? 1 : 0;
                const int bit = i * KB;
                cw[bit >> 5] |= static_cast<uint32_t>(code) << (bit & 31);
                if ((bit & 31) + KB > 32) cw[(bit >> 5) + 1] |= static_cast<uint32_t>(code) >> (32 - (bit & 31));
                if constexpr (PROD) {
                    const float r = __fsub_rn(y, s_c[code]);
                    g2 = __fmaf_rn(r, r, g2);
                    v[i] = r * 256.0f;
                }
            }
            if (widx) store_words<KB>(widx + KB * (CH * half + ch), cw);
            if constexpr (PROD) {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float f[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) f[e] = v[8 * q + e];
                    store8<D>(A0, A1, row, DH * half + 32 * ch + 8 * q, f);
                }
            }
        }
        if (sub && half == 0) reinterpret_cast<float*>(sub + o_norm)[slot] = n;

        if constexpr (PROD) {
            // ---------------- GEMM 2: Z = r~ S^T in three fp16 parts
            if (TPT == 2 && half == 1) s_g2[row] = g2;
            tc::fence_proxy_async_smem();
            tc::tc_fence_before();
            __syncthreads();
            if (tid == 0) {
                tc::tc_fence_after();
#pragma unroll
                for (int s = 0; s < D / 16; ++s) {
                    const uint64_t ah = tc::smem_desc(sbase + L::oA0 + 256 * s, L::kLbo, L::kSbo);
                    const uint64_t al = tc::smem_desc(sbase + L::oA1 + 256 * s, L::kLbo, L::kSbo);
                    const uint64_t bh_ = tc::smem_desc(sbase + L::oS + 256 * s, L::kLbo, L::kSbo);
                    const uint64_t bl = tc::smem_desc(sbase + L::oS + L::kTab / 2 + 256 * s, L::kLbo, L::kSbo);
                    tc::mma_f16(tmem, ah, bh_, idesc, s > 0);
                    tc::mma_f16(tmem, al, bh_, idesc, 1);
                    tc::mma_f16(tmem, ah, bl, idesc, 1);
                }
                tc::mma_commit(bar_mma);
            }
            ok = tc::mbar_wait(bar_mma, phase);
            if (__syncthreads_or(!ok)) {
                failed = true;
                break;
            }
            phase ^= 1;
            tc::tc_fence_after();
            uint32_t sw[CH];
#pragma unroll
            for (int ch = 0; ch < CH; ++ch) {
                float v[32];
                tc::tmem_ld32(tmem_row + 32 * ch, v);
                uint32_t w = 0u;
#pragma unroll
                for (int i = 0; i < 32; ++i) w |= (v[i] >= 0.0f ? 1u : 0u) << i;
                sw[ch] = w;
            }
            if (sub) {
                store_words<CH>(reinterpret_cast<uint32_t*>(sub + a.pool.off[1]) + static_cast<int64_t>(slot) * WS + CH * half,
                                sw);
                if (half == 0)
                    reinterpret_cast<float*>(sub + a.pool.off[3])[slot] = __fsqrt_rn(TPT == 2 ? g2 + s_g2[row] : g2);
            }
        }
        // TMEM reads of this tile are complete before the next tile's MMAs
        tc::tc_fence_before();
    }

    if (failed) {
        if (tid == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
        // let the table copies and an MMA group already committed finish
        // (bounded) before the shared and tensor memory go away
        (void)tc::mbar_wait(bar_tab, 0);
        if (!tables_failed) (void)tc::mbar_wait(bar_mma, phase);
    }
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, D);
    }
    if (tid == 0) {
        tc::mbar_inval(bar_tab);
        tc::mbar_inval(bar_mma);
    }
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
    const int per_sm = PROD ? 1 : 2;
    int64_t grid = static_cast<int64_t>(sm_count()) * per_sm;
    if (grid <= 0) return cudaErrorInvalidDevice;
    if (grid > ntiles) grid = ntiles;
    encode_tc_kernel<D, KB, PROD><<<static_cast<unsigned>(grid), Split<PROD>::kThreads, L::kBytes, s>>>(a, is_v,
                                                                                                   tiles_per_seq);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
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

// Tensor-core encode of one tensor (keys: is_v = 0, values: is_v = 1).
cudaError_t launch_encode_tc(const EncodeAppendArgs& a, int is_v, cudaStream_t s) {
    const CodecDev& cd = is_v ? a.vc : a.kc;
    if (cd.D == 64) return dispatch_kb<64>(a, is_v, cd, s);
    if (cd.D == 128) return dispatch_kb<128>(a, is_v, cd, s);
    return cudaErrorInvalidValue;
}

}  // namespace tq

// Kernel templates of the tensor-core decode path (see decode_mma.cuh).
#pragma once

#include <type_traits>

#include "decode_mma.cuh"
#include "tc_ptx.cuh"

namespace tq {
namespace mmadec {

constexpr float kLog2e = 1.4426950408889634f;
// Running row maximum before any score: finite, so that ex2(score - max) and
// ex2(old - new max) need no guard (a masked score is -inf and gives 0).
constexpr float kNoMax = -3.402823466e38f;
// Lagging row maximum: the reference maximum m of p = 2^(x - m) moves only
// when a score passes it by more than kLag (log2 units), so p <= 2^kLag and
// most 16-token steps skip the rescale of the accumulators. P' = fp16(p * value
// norm) stays finite while norms are at most kLagNorm (2^8 * 2^7 < 65504); in
// a tile holding a larger norm, m follows the exact maximum instead.
constexpr float kLag = 8.0f;
constexpr float kLagNorm = 128.0f;
constexpr float kSqrtHalfPi = 1.2533141373155003f;  // sqrt(pi/2)

// Per-launch layout of one shared-memory stage (TT tokens of every stream).
struct StageLayout {
    int tt;                 // tokens per stage (= tile), 16..64, divides block_tokens
    int bytes;              // stage bytes rounded up to 128
    int off[7];             // stream offsets inside a stage (-1 = absent)
    int field[7];           // bytes per token of each stream
    int bar_off;            // byte offset of the mbarriers (past ring and merge areas)
    int qs_off;             // byte offset of the query fragments (past the ring)
    int vt_off;             // byte offset of the value pair table region (-1: none)
    int kt_off;             // byte offset of the key quad table (-1: none)
    int ring_off;           // byte offset of the stage rings
};

struct MmaArgs {
    DecodeArgs a;
    StageLayout st;
    const uint4* qfrag;     // [unit][2][8][32] uint4
    float* part;            // [unit][splits][16][128]
    float* ml;              // [unit][splits][16][2]
};

// ------------------------------------------------------------------ query fragments

// q' = R_k q * scale * log2(e) and q'' = S_k q' * sqrt(pi/2)/D (same scale),
// written as fp16 A fragments of mma.m16n8k16 in the decoders' coordinate order.
// Slot 0 holds fp16(q'); slot 1 holds q'' for prod keys, and for MSE keys the
// rounding remainder fp16(q' - fp16(q')), so that two MMAs against the exact
// fp16 codebook operand carry q' to about 22 bits.
constexpr int kQThreads = 256;
constexpr int kQStride = kD + 8;  // fp16 row stride of the query operand tiles (conflict-free fragments)

struct QSmem {
    uint16_t R[2][kD * kD];         // 16 R_k, fp16 hi / lo, core-matrix layout
    uint16_t S[2][kD * kD];         // S_k, fp16 hi / lo (prod keys)
    uint16_t A[2][kRows * kQStride];  // scaled operand rows, fp16 hi / lo
    float q1[kRows][kD];            // q' (fp32)
    float q2[kRows][kD];            // q'' (fp32, prod keys)
    float ex[kRows];                // per-row power-of-two scale exponents
    uint64_t bar;
};

// Rows of the A tiles from fp32 values v[16][kD] scaled by 2^-ex[row]: hi and lo fp16.
__device__ __forceinline__ void q_split_rows(QSmem& sm, const float* v, int tid) {
    for (int e = tid; e < kRows * kD / 2; e += kQThreads) {
        const int r = e / (kD / 2), k = 2 * (e % (kD / 2));
        const float sc = scalbnf(1.0f, -static_cast<int>(sm.ex[r]));
        const float a = v[r * kD + k] * sc, b = v[r * kD + k + 1] * sc;
        const __half2 hi = __floats2half2_rn(a, b);
        const float2 back = __half22float2(hi);
        const __half2 lo = __floats2half2_rn(a - back.x, b - back.y);
        *reinterpret_cast<__half2*>(&sm.A[0][r * kQStride + k]) = hi;
        *reinterpret_cast<__half2*>(&sm.A[1][r * kQStride + k]) = lo;
    }
}

// out[16][kD] = (A_hi + A_lo) (T_hi + T_lo)^T without the lo*lo term, times
// 2^ex[row] / tscale: warp w computes output columns 16w .. 16w+15.
__device__ __forceinline__ void q_gemm(QSmem& sm, const uint16_t (*T)[kD * kD], float tscale, float* out, int warp,
                                       int lane) {
    const int g = lane >> 2, j = lane & 3;
    float acc[2][4] = {};
#pragma unroll
    for (int ks = 0; ks < kD / 16; ++ks) {
        uint32_t ah[4], al[4];
        const int k0 = 16 * ks + 2 * j;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint16_t* A = sm.A[h];
            uint32_t* dst = h ? al : ah;
            dst[0] = *reinterpret_cast<const uint32_t*>(A + g * kQStride + k0);
            dst[1] = *reinterpret_cast<const uint32_t*>(A + (g + 8) * kQStride + k0);
            dst[2] = *reinterpret_cast<const uint32_t*>(A + g * kQStride + k0 + 8);
            dst[3] = *reinterpret_cast<const uint32_t*>(A + (g + 8) * kQStride + k0 + 8);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            const int n8 = 2 * warp + nt;  // core-matrix row group of the output columns
            const int o0 = (n8 * (kD / 8) + 2 * ks) * 64 + g * 8 + 2 * j;
            const uint32_t bh0 = *reinterpret_cast<const uint32_t*>(T[0] + o0);
            const uint32_t bh1 = *reinterpret_cast<const uint32_t*>(T[0] + o0 + 64);
            const uint32_t bl0 = *reinterpret_cast<const uint32_t*>(T[1] + o0);
            const uint32_t bl1 = *reinterpret_cast<const uint32_t*>(T[1] + o0 + 64);
            mma16816(acc[nt], ah, bh0, bh1);
            mma16816(acc[nt], ah, bl0, bl1);
            mma16816(acc[nt], al, bh0, bh1);
        }
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
        const int c = 16 * warp + 8 * nt + 2 * j;
        const float s0 = scalbnf(1.0f, static_cast<int>(sm.ex[g])) / tscale;
        const float s1 = scalbnf(1.0f, static_cast<int>(sm.ex[g + 8])) / tscale;
        out[g * kD + c] = acc[nt][0] * s0;
        out[g * kD + c + 1] = acc[nt][1] * s0;
        out[(g + 8) * kD + c] = acc[nt][2] * s1;
        out[(g + 8) * kD + c + 1] = acc[nt][3] * s1;
    }
}

// Persistent query prep over the units (sequence x kv head, row group): CTA
// `cta` of `ncta` takes units cta, cta + ncta, ...; the tables are staged once
// per CTA by one bulk copy; per unit q' = Q R^T and q'' = q' S^T for the 16
// rows on the tensor cores, both operands split into fp16 hi + lo (about 22
// significant bits). Runs in a block of kQThreads threads.
// ORD (frag_order): bit 0 puts the codebook part in natural pair order (the
// split kernel's quad-table key decoder), bit 1 the QJL part (its nibble-table
// sign decoder); otherwise the byte-permute decoders' orders.
template <int KB, int ORD = 0>
__device__ __forceinline__ void qfrag_body(const MmaArgs& m, unsigned char* qsm_raw, int cta, int ncta) {
    QSmem& sm = *reinterpret_cast<QSmem*>(qsm_raw);
    const DecodeArgs& a = m.a;
    const bool prod = a.kc.mode == TQ_MODE_PROD;
    const int Hkv = a.pool.Hkv;
    const int RG = a.plan.row_groups;
    const int units = a.batch * Hkv * RG;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(&sm.bar, 1);
        mbar_fence_init();
        mbar_expect_tx(&sm.bar, (prod ? 2u : 1u) * 2u * kD * kD * 2u);
        bulk_g2s(sm.R, a.kc.Rtc, 2 * kD * kD * 2, &sm.bar);
        if (prod) bulk_g2s(sm.S, a.kc.Stc, 2 * kD * kD * 2, &sm.bar);
    }
    bool first = true;
    for (int unit = cta; unit < units; unit += ncta) {
        const int bh = unit / RG, rg = unit % RG;
        const int b = bh / Hkv, h = bh % Hkv;
        // query rows (fp32) into q2 as scratch, and each row's scale exponent
        for (int e = tid; e < kRows * kD; e += kQThreads) {
            const int rr = e / kD, k = e % kD;
            const int r = rg * kRows + rr;
            float v = 0.0f;
            if (r < a.plan.rows) {
                const int gq = r / a.Lq, l = r % a.Lq;
                const int64_t src = ((static_cast<int64_t>(b) * a.Hq + h * a.G + gq) * a.Lq + l) * kD + k;
                if (a.q_dtype == TQ_F32) v = static_cast<const float*>(a.q)[src];
                else if (a.q_dtype == TQ_BF16) v = __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[src]);
                else v = __half2float(static_cast<const __half*>(a.q)[src]);
            }
            sm.q2[rr][k] = v;
        }
        __syncthreads();
        if (tid < kRows) {
            float mx = 0.0f;
            for (int k = 0; k < kD; ++k) mx = fmaxf(mx, fabsf(sm.q2[tid][k]));
            sm.ex[tid] = mx > 0.0f ? static_cast<float>(ilogbf(mx)) : 0.0f;  // |q| * 2^-ex < 2
        }
        __syncthreads();
        q_split_rows(sm, &sm.q2[0][0], tid);
        if (first) {
            const bool ok = mbar_wait(&sm.bar, 0);
            if (__syncthreads_or(!ok)) {
                if (tid == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
                (void)mbar_wait(&sm.bar, 0);
                tc::grid_wait_prior();
                tc::grid_release_dependents();
                return;
            }
        }
        q_gemm(sm, sm.R, 16.0f, &sm.q1[0][0], warp, lane);  // the table holds 16 R
        __syncthreads();
        if (prod) {
            // |q'| <= |q|_2 <= sqrt(128) * 2^(ex+1): scale q' by 2^-(ex+4)
            if (tid < kRows) sm.ex[tid] += 4.0f;
            __syncthreads();
            q_split_rows(sm, &sm.q1[0][0], tid);
            __syncthreads();
            q_gemm(sm, sm.S, 1.0f, &sm.q2[0][0], warp, lane);
            __syncthreads();
        }
        if (first) {
            first = false;
            // the workspace is written below: wait until the kernels before this
            // one are done (the queries and tables it has read so far are no
            // kernel's output in this chain; the append before it waits for the
            // decode before that); the split kernel may then start fetching
            // records, which are all written by now
            tc::grid_wait_prior();
            tc::grid_release_dependents();
        }
        // entry (row rr, which, ks, j, e): lane 4*(rr%8)+j, register 2e + (rr >= 8)
        // the key codebook operand is fp16(op_scale * level): the q' operand
        // carries 1 / op_scale so that their product is q' * level
        const float s1 = a.scale * kLog2e / a.kc.cq_scale;
        const float s2 = a.scale * kLog2e * kSqrtHalfPi / static_cast<float>(kD);
        uint32_t* dst = reinterpret_cast<uint32_t*>(const_cast<uint4*>(m.qfrag)) + static_cast<int64_t>(unit) * 2 * 8 * 32 * 4;
        for (int e = tid; e < kRows * 128; e += kQThreads) {
            const int rr = e >> 7, x = e & 127;
            const int which = x >> 6, ks = (x >> 3) & 7, j = (x >> 1) & 3, ee = x & 1;
            const int ln = 4 * (rr & 7) + j;
            const int reg = 2 * ee + (rr >= 8 ? 1 : 0);
            int pa, pb;
            const bool qjl = which && prod;
            if (qjl ? (ORD & 2) != 0 : (ORD & 1) != 0) {
                pa = 2 * (2 * ks + ee);
                pb = pa + 1;
            } else {
                mse_pair(qjl ? 1 : KB, 2 * ks + ee, pa, pb);
            }
            const float* q = qjl ? sm.q2[rr] : sm.q1[rr];
            const float sc = qjl ? s2 : s1;
            float va = q[32 * j + pa] * sc, vb = q[32 * j + pb] * sc;
            if (which && !qjl) {
                va -= __half2float(__float2half_rn(va));
                vb -= __half2float(__float2half_rn(vb));
            }
            dst[((which * 8 + ks) * 32 + ln) * 4 + reg] = pack_half2(va, vb);
        }
        __syncthreads();   // q1 / q2 / A are rewritten by the next unit
    }
    if (first && tid == 0) {   // no unit for this CTA: release the tables' copy
        (void)mbar_wait(&sm.bar, 0);
    }
    if (tid == 0) mbar_inval(&sm.bar);
}

template <int KB, int ORD = 0>
__global__ void __launch_bounds__(kQThreads) qfrag_kernel(MmaArgs m) {
    extern __shared__ __align__(16) unsigned char qsm_raw[];
    qfrag_body<KB, ORD>(m, qsm_raw, blockIdx.x, gridDim.x);
}

// CTAs of the query-prep kernel: one per unit up to one per SM.
inline int qfrag_grid(int units) {
    static std::atomic<int> sms[64];
    int dev = 0;
    cudaGetDevice(&dev);
    int n = sms[dev & 63].load();
    if (n == 0) {
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
        sms[dev & 63].store(n);
    }
    return units < n ? units : n;
}

// ------------------------------------------------------------------ split kernel

// Key operands of k-steps 2 q2 and 2 q2 + 1 (four half2: (b0, b1) of each)
// from one token's index words, in the pair order the query fragments use.
template <int KB, bool QUAD, typename Tab>
__device__ __forceinline__ void key_ks2(const uint32_t (&w)[KB], const Tab& t, uint32_t lane_addr, int q2,
                                        uint32_t (&h)[4]) {
    if constexpr (QUAD) {
        // 2-bit codes, natural pair order: byte k of word hw is k-step 4 hw + k
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int ks = 2 * q2 + e, hw = ks >> 2, k = ks & 3;
            const uint32_t f = k == 0 ? shl_f(w[hw], 7) : (w[hw] >> (8 * k - 7));
            const uint2 v = lds_u64(mad_lo(f & 0x7F80u, kDc.pow2[0], lane_addr));
            h[2 * e] = v.x;
            h[2 * e + 1] = v.y;
        }
    } else if constexpr (KB == 1) {
        const uint32_t neg2 = t.lo;
#pragma unroll
        for (int e = 0; e < 2; ++e) {
            const int ks = 2 * q2 + e;
            h[2 * e] = dec1(w[0], 15 - ks, neg2);
            h[2 * e + 1] = dec1(w[0], 7 - ks, neg2);
        }
    } else if constexpr (KB == 2) {
        // k-step 2 s + hw from word hw, code group s
        dec2_pair(w[0], q2, t, h[0], h[1]);
        dec2_pair(w[1], q2, t, h[2], h[3]);
    } else if constexpr (KB == 3) {
        uint32_t v;
        if (q2 == 0) v = w[0] & 0xFFFFFFu;
        else if (q2 == 1) v = mad_lo(w[1] & 0xFFFFu, kDc.pow2[8], (w[0] >> 24));
        else if (q2 == 2) v = mad_lo(w[2] & 0xFFu, kDc.pow2[16], (w[1] >> 16));
        else v = w[2] >> 8;
        dec3_group(v, t, h);
    } else {
        dec4_word(w[q2], t, h);
    }
}

template <int NW>
__device__ __forceinline__ void load_words(const uint32_t* p, uint32_t (&w)[NW]) {
    if constexpr (NW == 4) {
        const uint4 v = *reinterpret_cast<const uint4*>(p);
        w[0] = v.x; w[1] = v.y; w[2] = v.z; w[3] = v.w;
    } else if constexpr (NW == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(p);
        w[0] = v.x; w[1] = v.y;
    } else {
#pragma unroll
        for (int k = 0; k < NW; ++k) w[k] = p[k];
    }
}

// The fp16 pairs of one word's four bytes (codes 2k, 2k + 1 for byte k) from
// the 4-bit pair table: entry e (a byte) at 128 e + 4 L for lane L; byte k is
// shifted to bit 7, masked and added to the lane's address (one shift, one
// logic op, one add and one load per pair).
__device__ __forceinline__ void pair4_word(uint32_t w, uint32_t lane_addr, uint32_t (&h)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const uint32_t f = k == 0 ? shl_f(w, 7) : (w >> (8 * k - 7));
        h[k] = lds_u32(mad_lo(f & 0x7F80u, kDc.pow2[0], lane_addr));
    }
}

// The same from the table of 256-byte entries at the start of shared memory:
// the entry's offset is byte k of w times 256, the lane's copy lane_b (< 256),
// so one byte permute gives the offset (byte 0 = lane_b, byte 1 = byte k of w).
__device__ __forceinline__ void pair4w_word(const unsigned char* tab, uint32_t w, uint32_t lane_b, uint32_t (&h)[4]) {
#pragma unroll
    for (int k = 0; k < 4; ++k)
        h[k] = *reinterpret_cast<const uint32_t*>(tab + __byte_perm(w, lane_b, 0x5504u | (k << 4)));
}

template <int B>
struct MseTable {
    using type = Tab8;
};
template <>
struct MseTable<1> {
    using type = Tab4;
};
template <>
struct MseTable<2> {
    using type = Tab4;
};

// Register tables for an MSE codebook of 2^B centroids.
template <int B>
__device__ inline typename MseTable<B>::type mse_table(const float* cg) {
    float c[16];
    for (int k = 0; k < (1 << B); ++k) c[k] = __ldg(cg + k);
    if constexpr (B == 1) {
        const uint32_t h = h_bits(c[0]);
        return Tab4{h | (h << 16), 0u};
    } else if constexpr (B == 2) {
        return make_tab4(c);
    } else if constexpr (B == 3) {
        return make_tab8(c);
    } else {
        return make_tab8(c + 8);  // magnitudes of the positive half
    }
}

template <int B>
__device__ __forceinline__ void mse_chunk(const uint32_t* w, const typename MseTable<B>::type& t, uint32_t (&h)[16]) {
    MseChunk<B>::run(w, t, h);
}

// Merge of a unit's split partials, one CTA per (unit, row), launched after
// the split kernel with programmatic dependent launch: R_v is staged in shared
// memory before the CTA waits for the split kernel (head_dim 64 and 128; at
// 256 the rotation reads R_v's rows from L2); then the CTA takes the row's maximum
// over the splits, weights each split's (sum, accumulator) by 2^(m - max),
// divides by the merged sum and applies the inverse value rotation (or, for a
// shard's state, writes the merged (max, sum, accumulator) without the
// rotation). Thread d < D owns output column d; at head_dim 256 the split
// kernel's two 128-column halves are separate partial rows (the same max and
// sum in both), and with MSE values the CTA has 4 D threads: quarter k of
// them sums rows [D k / 4, D (k + 1) / 4) of the rotation (four L2 loads of
// R_v in flight per column instead of one), the quarters' sums added in a
// fixed order.
template <bool VGROUP, int D>
__host__ __device__ constexpr int merge_threads() { return D <= kD || VGROUP ? D : 4 * D; }

template <bool VGROUP, int D = kD>
__global__ void __launch_bounds__(merge_threads<VGROUP, D>()) merge_rows_kernel(MmaArgs m) {
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int NH = D > kD ? D / kD : 1, kW = D / 32;
    constexpr int kQ = merge_threads<VGROUP, D>() / D;   // rotation quarters (1: no split of the rotation)
    const DecodeArgs& a = m.a;
    tc::grid_release_dependents();  // the next kernel waits for this grid before the workspace
    const int unit = blockIdx.x, r = blockIdx.y;
    const int RG = a.plan.row_groups;
    const int rg = unit % RG, bh = unit / RG;
    const int b = bh / a.pool.Hkv, h = bh % a.pool.Hkv;
    const int row = rg * kRows + r;
    if (row >= a.plan.rows) return;  // padding row of the last group
    const int d = threadIdx.x % D, quarter = threadIdx.x / D, lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const bool col = quarter == 0;   // the threads of the split merge (one per column)
    const int h2 = d / kD, cc = d % kD;
    const bool rotate = !VGROUP && !a.part_acc;
    const bool stage_r = rotate && D <= kD;
    float* sR = reinterpret_cast<float*>(smem);      // [D][D], staged rotation only
    float* so = sR + (stage_r ? D * D : 0);          // [D] the merged row
    float* sw = so + D;                              // [D] weights of a chunk of splits
    float* sred = sw + D;                            // [kW] per-warp maxima / sums
    float* sq = sred + kW;                           // [kQ][D] the rotation quarters' sums
    __shared__ uint64_t bar;
    if (stage_r && threadIdx.x == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        mbar_expect_tx(&bar, D * D * 4);
        bulk_g2s(sR, a.vc.R, D * D * 4, &bar);
    }
    tc::grid_wait_prior();  // the split kernel's partials
    const int S = a.plan.splits;
    // (max, sum) rows of the unit's first half; accumulator column cc of half h2
    const float* mlr = m.ml + (static_cast<int64_t>(unit) * NH * S * kRows + r) * 2;     // split s at + s * 32
    const float* pr = m.part + ((static_cast<int64_t>(unit) * NH + h2) * S * kRows + r) * kD + cc;  // + s * 16 x 128
    // every load of the first kMPre splits issued at once (one L2 round trip):
    // thread d's column of each split's accumulator, and the (max, sum) of
    // split d
    constexpr int kMPre = 32;
    float pv[kMPre];
#pragma unroll
    for (int s = 0; s < kMPre; ++s) pv[s] = col && s < S ? __ldcg(pr + static_cast<int64_t>(s) * kRows * kD) : 0.0f;
    float2 myml = make_float2(-INFINITY, 0.0f);
    if (col && d < S) myml = __ldcg(reinterpret_cast<const float2*>(mlr + d * kRows * 2));
    // the row's maximum over the splits
    float mx = myml.x;
    if (col)
        for (int s = d + D; s < S; s += D) mx = fmaxf(mx, __ldcg(mlr + s * kRows * 2));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    if (col && lane == 0) sred[wid] = mx;
    __syncthreads();
    float M = sred[0];
#pragma unroll
    for (int w = 1; w < kW; ++w) M = fmaxf(M, sred[w]);
    // weights 2^(m - M) of the first D splits (a split that saw no score has
    // (-inf, 0) and a zero accumulator); thread d's share of the sum
    float lsum = 0.0f;
    if (col && d < S) {
        const float w = myml.x == -INFINITY ? 0.0f : ex2(myml.x - M);
        sw[d] = w;
        lsum = w * myml.y;
    }
    __syncthreads();
    float acc = 0.0f;
#pragma unroll
    for (int s = 0; s < kMPre; ++s)
        if (s < S) acc = fmaf(sw[s], pv[s], acc);
    // splits past the first kMPre (long sequences over few units)
    for (int s0 = 0; s0 < S; s0 += D) {
        const int n = S - s0 < D ? S - s0 : D;
        if (s0 > 0) {
            __syncthreads();
            if (col && d < n) {
                const float2 ml = __ldcg(reinterpret_cast<const float2*>(mlr + (s0 + d) * kRows * 2));
                const float w = ml.x == -INFINITY ? 0.0f : ex2(ml.x - M);
                sw[d] = w;
                lsum = fmaf(w, ml.y, lsum);
            }
            __syncthreads();
        }
        if (col) {
#pragma unroll 8
            for (int s = s0 > 0 ? 0 : kMPre; s < n; ++s)
                acc = fmaf(sw[s], __ldcg(pr + static_cast<int64_t>(s0 + s) * kRows * kD), acc);
        }
    }
    __syncthreads();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
    if (col && lane == 0) sred[wid] = lsum;
    __syncthreads();
    float L = sred[0];
#pragma unroll
    for (int w = 1; w < kW; ++w) L += sred[w];
    // MSE values were multiplied as fp16(op_scale * level): divide op_scale out
    const float vs = VGROUP ? 1.0f : a.vc.cq_scale;
    const int gq = row / a.Lq, l = row % a.Lq;
    const int64_t oo = (static_cast<int64_t>(b) * a.Hq + h * a.G + gq) * a.Lq + l;
    if (a.part_acc) {
        // a shard's state: max in natural-log units, sum, accumulator
        if (!col) return;
        a.part_acc[oo * D + d] = acc * (1.0f / vs);
        if (d == 0) {
            a.part_ml[2 * oo] = M == -INFINITY ? -INFINITY : M * 0.6931471805599453f;
            a.part_ml[2 * oo + 1] = L;
        }
        return;
    }
    const float x = L > 0.0f ? acc * (1.0f / (L * vs)) : 0.0f;
    if (!rotate) {
        if (col) a.out[oo * D + d] = x;
        return;
    }
    if (col) so[d] = x;
    __syncthreads();
    // out[d] = sum_i row[i] R_v[i][d]: R_v's row i is one contiguous load, the
    // merged row's values are broadcasts (four at a time)
    float y0 = 0.0f, y1 = 0.0f;
    const float4* so4 = reinterpret_cast<const float4*>(so);
    if (stage_r) {
        if (!mbar_wait(&bar, 0)) {
            if (d == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
            (void)mbar_wait(&bar, 0);
        }
#pragma unroll 4
        for (int i4 = 0; i4 < D / 4; ++i4) {
            const float4 v = so4[i4];
            y0 = fmaf(v.x, sR[(4 * i4) * D + d], y0);
            y1 = fmaf(v.y, sR[(4 * i4 + 1) * D + d], y1);
            y0 = fmaf(v.z, sR[(4 * i4 + 2) * D + d], y0);
            y1 = fmaf(v.w, sR[(4 * i4 + 3) * D + d], y1);
        }
    } else {
        // rows [D quarter / kQ, D (quarter + 1) / kQ) of R_v, from L2
        const float* R = a.vc.R + static_cast<int64_t>(quarter) * (D / kQ) * D;
        const float4* sq4 = so4 + quarter * (D / kQ / 4);
#pragma unroll 8
        for (int i4 = 0; i4 < D / kQ / 4; ++i4) {
            const float4 v = sq4[i4];
            y0 = fmaf(v.x, __ldg(R + (4 * i4) * D + d), y0);
            y1 = fmaf(v.y, __ldg(R + (4 * i4 + 1) * D + d), y1);
            y0 = fmaf(v.z, __ldg(R + (4 * i4 + 2) * D + d), y0);
            y1 = fmaf(v.w, __ldg(R + (4 * i4 + 3) * D + d), y1);
        }
        if constexpr (kQ > 1) {
            sq[quarter * D + d] = y0 + y1;
            __syncthreads();
            if (!col) return;
            y0 = sq[d];
            y1 = 0.0f;
#pragma unroll
            for (int k = 1; k < kQ; ++k) y0 += sq[k * D + d];
        }
    }
    a.out[oo * D + d] = y0 + y1;
    if (stage_r && threadIdx.x == 0) mbar_inval(&bar);
}

// Dynamic shared memory of merge_rows_kernel.
template <bool VGROUP, int D = kD>
inline size_t merge_rows_smem(bool rotate) {
    constexpr int nt = merge_threads<VGROUP, D>();
    return (rotate && D <= kD ? static_cast<size_t>(D) * D * 4 : 0) + (2 * D + D / 32 + (nt > D ? nt : 0)) * 4;
}

// Query fragments of one unit (16 rows) from its fp32 q' and q'' rows, in the
// layout and coordinate order qfrag_body writes for head_dim 128, over D / 16
// k-steps: entry (which, k-step 8 c + ks, lane 4 (row % 8) + j, register
// 2 e + (row >= 8)) holds the pair (pa, pb) of the lane's chunk j D / 128 + c.
// Slot 1 holds q'' for prod keys and fp16(q') 's rounding remainder otherwise.
// A block of NT threads: every thread issues all of its loads (L2) before it
// converts any, so the rows arrive in one round trip. Head_dim 64 takes the
// head_dim-128 layout with the coordinates past 64 zero (the lanes whose
// chunk lies past the vector's end then contribute nothing to a score).
template <int KB, int ORD, int D, int NT>
__device__ __forceinline__ void frag_from_rows(uint32_t* dst, const float* q1, const float* q2, bool prod, float s1,
                                               float s2, int tid) {
    constexpr int DV = D < kD ? kD : D;   // the layout's head_dim
    constexpr int KS = DV / 16, NC = DV / kD;
    constexpr int kPerRow = 2 * KS * 4 * 2;
    constexpr int kTotal = kRows * kPerRow, kIter = (kTotal + NT - 1) / NT;
    // entry e: (row, which, k-step, lane chunk j, e) and the source pair
    auto where = [&](int e, int& out, const float*& q, int& pa, int& pb, bool& qjl, bool& rem) {
        const int rr = e / kPerRow, x = e % kPerRow;
        const int which = x / (KS * 8), ksg = (x / 8) % KS, j = (x >> 1) & 3, ee = x & 1;
        const int c = ksg / 8, ks = ksg % 8;
        out = ((which * KS + ksg) * 32 + 4 * (rr & 7) + j) * 4 + 2 * ee + (rr >= 8 ? 1 : 0);
        qjl = which && prod;
        rem = which && !prod;
        if (qjl ? (ORD & 2) != 0 : (ORD & 1) != 0) {
            pa = 2 * (2 * ks + ee);
            pb = pa + 1;
        } else {
            mse_pair(qjl ? 1 : KB, 2 * ks + ee, pa, pb);
        }
        const int chunk = j * NC + c;
        q = chunk < D / 32 ? (qjl ? q2 : q1) + rr * D + 32 * chunk : nullptr;
    };
    float va[kIter], vb[kIter];
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const int e = tid + it * NT;
        va[it] = vb[it] = 0.0f;
        if (e < kTotal) {
            int out, pa, pb;
            const float* q;
            bool qjl, rem;
            where(e, out, q, pa, pb, qjl, rem);
            if (q) {
                va[it] = __ldcg(q + pa);
                vb[it] = __ldcg(q + pb);
            }
        }
    }
#pragma unroll
    for (int it = 0; it < kIter; ++it) {
        const int e = tid + it * NT;
        if (e < kTotal) {
            int out, pa, pb;
            const float* q;
            bool qjl, rem;
            where(e, out, q, pa, pb, qjl, rem);
            const float sc = qjl ? s2 : s1;
            float a = va[it] * sc, b = vb[it] * sc;
            if (rem) {
                a -= __half2float(__float2half_rn(a));
                b -= __half2float(__float2half_rn(b));
            }
            dst[out] = pack_half2(a, b);
        }
    }
}

// R8 (head_dim 128, at most 8 query rows per unit): the transposed form.
// Scores as S^T = K Q^T with 16 tokens on M and the 8 rows on N (the query
// fragments' registers 0 and 2 are the B operand of rows 0..7; two 8-token
// key tiles' operands are the A operand), outputs as O^T = V^T P^T with 16
// value columns on M: half the MMAs and half the softmax work per token of
// the 16-row form, whose rows 8..15 would be padding.
template <int KB, bool KPROD, bool VGROUP, int VB, int D = kD, bool R8 = false>
__global__ void __launch_bounds__(kThreads, 1) split_mma_kernel(MmaArgs m) {
    static_assert(!R8 || D == kD, "the transposed form at head_dim 128");
    extern __shared__ __align__(128) unsigned char smem[];
    const DecodeArgs& a = m.a;
    const StageLayout& st = m.st;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, j = lane & 3;
    const int Hkv = a.pool.Hkv;
    const int RG = a.plan.row_groups;
    // head_dim D = 128 NH: each CTA takes one 128-column half h2 of the values
    // (the output accumulator of a warp is 16 x 128); every lane decodes NC
    // 32-coordinate chunks of each key (scores need all D coordinates).
    // Head_dim 64 runs in the head_dim-128 layout: lanes j >= 2, whose chunk
    // lies past the vector's end, decode chunk 1 again (finite operands against
    // zero query coordinates for the scores; their output columns 64..127 are
    // not merged).
    static_assert(D == 64 || D % kD == 0, "head_dim 64 or a multiple of 128");
    constexpr int NH = D > kD ? D / kD : 1, NC = D > kD ? D / kD : 1;
    constexpr int DV = D < kD ? kD : D;                       // the fragment layout's head_dim
    const int jc = D < kD ? (j < D / 32 ? j : D / 32 - 1) : j;  // the lane's chunk, clamped
    // grid (KV head x row group x half, sequence, split): CTAs are dispatched
    // split by split, so every unit's full first splits run before the
    // shorter (last, partial) and empty ones, which make up the last wave
    const int split = blockIdx.z;
    const int h2 = blockIdx.x % NH;
    const int h = (blockIdx.x / NH) % Hkv;
    const int rg = blockIdx.x / NH / Hkv;
    const int b = blockIdx.y;
    const int unit = (b * Hkv + h) * RG + rg;
    const int punit = unit * NH + h2;  // the half's partial rows
    const int BT = a.pool.BT;
    const int TT = st.tt;

    // (the rings start past a table at offset 0 in the kernels that keep one there)
    unsigned char* ring = smem + (pair4_wide(D, KB, KPROD, VGROUP, VB) ? st.ring_off : 0) +
                          static_cast<size_t>(warp) * kStages * st.bytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + st.bar_off) + warp * kStages;

    const int N = a.seq_lens[b] + a.len_add;
    // causal window end (local token index): the sequence's end, or a shard's
    const int vis = a.causal_end ? a.causal_end[b] : N;
    const bool bad = N < (a.causal_end ? 0 : a.Lq) || N > a.max_blocks * BT;
    if (bad && split == 0 && threadIdx.x == 0 && rg == 0 && h == 0) atomicOr(a.err, TQ_DEVERR_SEQLEN);
    const int t_begin = split * a.plan.chunk;
    const int t_end = min(t_begin + a.plan.chunk, bad ? 0 : N);
    const int ntiles = t_end > t_begin ? (t_end - t_begin + TT - 1) / TT : 0;
    const int my_n = ntiles > warp ? (ntiles - warp + kWarps - 1) / kWarps : 0;

    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
    }
    __syncwarp();

    // Barrier of the lookup tables (bulk-copied from the codec's prebuilt copy
    // at once) and the query fragments (copied after the wait below): two
    // arrivals, one per copy group.
    uint64_t* tbar = reinterpret_cast<uint64_t*>(smem + st.bar_off) + kWarps * kStages;
    // 2-bit keys decode through the shared quad table, others in registers
    constexpr bool kQuadTab = quad_keys(KB, KPROD, VGROUP);
    // 3-bit MSE values decode through the shared pair table, others in registers
    constexpr bool kPairTab = !VGROUP && VB == 3;
    uint32_t pair_off = 0;  // the pair table's offset: 8 KB-aligned shared address inside its region
    if constexpr (kPairTab) {
        const uint32_t region = smem_u32(smem + st.vt_off);
        pair_off = st.vt_off + (((region + kVPairBytes - 1) & ~static_cast<uint32_t>(kVPairBytes - 1)) - region);
    }
    // 4-bit MSE keys / values through the shared 4-bit pair table (MSE keys)
    constexpr bool kP4K = pair4_keys(D, KB, KPROD), kP4V = pair4_values(D, KPROD, VGROUP, VB);
    // both: one table of 256-byte entries at offset 0 (keys copy set 0, values set 1)
    constexpr bool kP4W = pair4_wide(D, KB, KPROD, VGROUP, VB);
    const bool quad_copy = kQuadTab && a.kc.quad, pair_copy = kPairTab && a.vc.pair;
    const bool p4k_copy = kP4K && !kP4W && a.kc.pair4, p4v_copy = kP4V && !kP4W && a.vc.pair4;
    const bool p4w_copy = kP4W && a.kc.pair4w && a.kc.pair4w == a.vc.pair4w;   // one codebook
    if (threadIdx.x == 0) {
        mbar_init(tbar, 2);
        mbar_fence_init();
        mbar_expect_tx(tbar, (quad_copy ? kKQuadBytes : 0) + (pair_copy ? kVPairBytes : 0) +
                                 (p4k_copy ? kPair4Bytes : 0) + (p4v_copy ? kPair4Bytes : 0) +
                                 (p4w_copy ? kPair4WBytes : 0));
        if (quad_copy) bulk_g2s(smem + st.kt_off, a.kc.quad, kKQuadBytes, tbar);
        if (pair_copy) bulk_g2s(smem + pair_off, a.vc.pair, kVPairBytes, tbar);
        if (p4k_copy) bulk_g2s(smem + st.kt_off, a.kc.pair4, kPair4Bytes, tbar);
        if (p4v_copy) bulk_g2s(smem + st.vt_off, a.vc.pair4, kPair4Bytes, tbar);
        if (p4w_copy) bulk_g2s(smem, a.kc.pair4w, kPair4WBytes, tbar);
    }
    // a codec without the prebuilt table: build it here
    auto build_pair4 = [&](uint32_t* tab, const float* cq) {
        for (int i = threadIdx.x; i < 256 * 32; i += kThreads) {
            const int e = i >> 5;
            tab[i] = h_bits(__ldg(cq + (e & 15))) | (h_bits(__ldg(cq + (e >> 4))) << 16);
        }
    };
    uint32_t k4_lane = 0, v4_lane = 0;
    if constexpr (kP4W) {
        // the lanes' copies: bytes 4 lane (keys) and 128 + 4 lane (values) of an entry
        k4_lane = 4u * lane;
        v4_lane = 128u + 4u * lane;
        if (!p4w_copy) {   // codecs without one shared prebuilt table: build it here
            uint32_t* tab = reinterpret_cast<uint32_t*>(smem);
            for (int i = threadIdx.x; i < 256 * 64; i += kThreads) {
                const int e = i >> 6;
                const float* cq = (i & 63) < 32 ? a.kc.cq : a.vc.cq;
                tab[i] = h_bits(__ldg(cq + (e & 15))) | (h_bits(__ldg(cq + (e >> 4))) << 16);
            }
        }
    } else {
        if constexpr (kP4K) {
            k4_lane = smem_u32(smem + st.kt_off) + 4u * lane;
            if (!p4k_copy) build_pair4(reinterpret_cast<uint32_t*>(smem + st.kt_off), a.kc.cq);
        }
        if constexpr (kP4V) {
            v4_lane = smem_u32(smem + st.vt_off) + 4u * lane;
            if (!p4v_copy) build_pair4(reinterpret_cast<uint32_t*>(smem + st.vt_off), a.vc.cq);
        }
    }
    typename MseTable<KB>::type ktab{};
    if constexpr (!kQuadTab && !kP4K) ktab = mse_table<KB>(a.kc.cq);
    uint32_t kt_lane = 0;
    if constexpr (kQuadTab) {
        kt_lane = smem_u32(smem + st.kt_off) + 8u * (lane & 15);
        if (!quad_copy) {  // a codec without the prebuilt table: build it here
            uint2* tab = reinterpret_cast<uint2*>(smem + st.kt_off);
            for (int i = threadIdx.x; i < 256 * 16; i += kThreads) {
                const int e = i >> 4;
                const uint32_t c0 = h_bits(__ldg(a.kc.cq + (e & 3))), c1 = h_bits(__ldg(a.kc.cq + ((e >> 2) & 3)));
                const uint32_t c2 = h_bits(__ldg(a.kc.cq + ((e >> 4) & 3))), c3 = h_bits(__ldg(a.kc.cq + (e >> 6)));
                tab[i] = make_uint2(c0 | (c1 << 16), c2 | (c3 << 16));
            }
        }
    }
    // QJL signs of prod keys with 3-bit values: a table of sign nibbles in the
    // slack of the pair table's region (a 2 KB-aligned 2 KB block: the larger
    // slack, before or after the 8 KB-aligned pair table, holds one); entry e
    // (four sign bits, a set bit is +1) copy c at 128 e + 8 c: the fp16 pairs
    // (s0, s1), (s2, s3)
    constexpr bool kNibQ = nibble_qjl(KPROD, VGROUP, VB);
    uint32_t qn_lane = 0;
    if constexpr (kNibQ) {
        const uint32_t region = smem_u32(smem + st.vt_off);
        uint32_t nib;
        if constexpr (kPairTab) {
            const uint32_t pair_at = smem_u32(smem + pair_off);
            nib = pair_at - region >= 4096u ? (region + 2047u) & ~2047u : pair_at + kVPairBytes;
        } else {
            nib = (region + 2047u) & ~2047u;   // group values: a 4 KB region of its own
        }
        qn_lane = nib + 8u * (lane & 15);
        uint2* tab = reinterpret_cast<uint2*>(smem + st.vt_off + (nib - region));
        for (int i = threadIdx.x; i < 16 * 16; i += kThreads) {
            const int e = i >> 4;
            auto pm = [&](int bit) { return (e >> bit) & 1 ? 0x3C00u : 0xBC00u; };
            tab[i] = make_uint2(pm(0) | (pm(1) << 16), pm(2) | (pm(3) << 16));
        }
    }
    typename MseTable<VGROUP ? 2 : VB>::type vtab{};
    if constexpr (!VGROUP && !kPairTab && !kP4V) vtab = mse_table<VB>(a.vc.cq);
    uint32_t vt_lane = 0;
    if constexpr (kPairTab) {
        vt_lane = smem_u32(smem + pair_off) + 4u * lane;
        if (!pair_copy) {
            uint32_t* tab = reinterpret_cast<uint32_t*>(smem + pair_off);
            for (int i = threadIdx.x; i < 64 * 32; i += kThreads) {
                const int e = i >> 5;
                tab[i] = h_bits(__ldg(a.vc.cq + (e & 7))) | (h_bits(__ldg(a.vc.cq + (e >> 3))) << 16);
            }
        }
    }

    // causal limits of this thread's two rows (padding rows see everything)
    // (R8: the lane's rows 2 j and 2 j + 1, its tokens g and g + 8 of each 16)
    const int r0 = R8 ? rg * kRows + 2 * j : rg * kRows + g, r1 = R8 ? r0 + 1 : r0 + 8;
    const int lim0 = r0 < a.plan.rows ? vis - a.Lq + (r0 % a.Lq) : N - 1;
    const int lim1 = r1 < a.plan.rows ? vis - a.Lq + (r1 % a.Lq) : N - 1;
    const int lim_all = vis - a.Lq;  // every row sees the tokens up to here

    // output accumulator: 16 n8 tiles of 8 columns x 16 rows, or (R8) 8 m16
    // tiles of 16 columns x 8 rows
    constexpr int kOT = R8 ? 8 : 16;
    float o[kOT][4];
#pragma unroll
    for (int p = 0; p < kOT; ++p) o[p][0] = o[p][1] = o[p][2] = o[p][3] = 0.0f;
    // group values: groups per token, and the group of this lane's value chunk
    [[maybe_unused]] int vng = 0, vgi = 0;
    if constexpr (VGROUP) {
        vng = D / a.vc.group;
        vgi = (32 * (4 * h2 + jc)) / a.vc.group;
    }
    float mrow0 = kNoMax, mrow1 = kNoMax, lrow0 = 0.0f, lrow1 = 0.0f;
    bool failed = false;

    // Stage copies: lane k < 7 copies record stream k of the tile (one warp
    // instruction for all streams), after lane 0 has posted the stage's bytes.
    // Blocks hold a power-of-two token count, so block index and slot are a
    // shift and a mask. bad_stage bit s marks a stage whose block-table entry
    // was out of range (its copy reads block 0; the tile is flagged and skipped).
    const int bt_shift = __ffs(BT) - 1;
    // A tile of TT tokens spans TT / BT blocks when blocks are shorter than
    // the tile (up to four: 7 streams x 4 blocks fit the warp's lanes), one
    // block otherwise. Lane k copies record stream k % 7 of block k / 7 of the
    // tile into that stream's run of the stage (blocks one after another).
    const int tile_blocks = TT > BT ? TT / BT : 1;
    const int blk_tokens = TT > BT ? BT : TT;   // tokens a lane's copy carries
    const int blk_shift = __ffs(blk_tokens) - 1;   // a power of two
    const int my_stream = lane % 7, my_blk = lane / 7;
    unsigned blk_tx = 0;                         // bytes of one block's part of a stage
    int s_off = -1, s_field = 0;
    int64_t s_src = 0;
#pragma unroll
    for (int k = 0; k < 7; ++k) {
        if (st.off[k] >= 0) blk_tx += blk_tokens * st.field[k];
        if (my_stream == k && my_blk < tile_blocks && st.off[k] >= 0) {
            s_off = st.off[k] + my_blk * blk_tokens * st.field[k];
            s_field = st.field[k];
            s_src = a.pool.off[k];
        }
    }
    const uint64_t pol = policy_evict_first();
    uint32_t bad_stage = 0;
    // The physical block of this lane's block of tile i (its table entry): read
    // a tile ahead of the copy in the main loop, so that the copy does not wait
    // for the load. Blocks of the tile that hold no token of this split (a
    // partial last tile may end before the tile's last block) are not read.
    auto entry = [&](int i) -> int32_t {
        if (!a.table) return 0;   // contiguous: the block follows from the position
        const int t0 = t_begin + (warp + i * kWarps) * TT;
        const int lb = (t0 >> bt_shift) + my_blk;
        const int live = min(tile_blocks, (t_end - t0 + blk_tokens - 1) >> blk_shift);
        if (s_off < 0 || my_blk >= live) return 0;
        return a.table[static_cast<int64_t>(b) * a.max_blocks + lb];
    };
    auto issue = [&](int i, int32_t tab) {
        const int t0 = t_begin + (warp + i * kWarps) * TT;
        const int lb = (t0 >> bt_shift) + my_blk;
        const int slot0 = t0 & (BT - 1);
        const int live = min(tile_blocks, (t_end - t0 + blk_tokens - 1) >> blk_shift);
        const bool mine = s_off >= 0 && my_blk < live;
        int64_t pb = 0;
        bool badb = false;
        if (mine) {
            pb = a.table ? static_cast<int64_t>(tab) : static_cast<int64_t>(b) * a.max_blocks + lb;
            badb = pb < 0 || pb >= a.pool.num_blocks;
            if (badb) pb = 0;
        }
        const int sidx = i % kStages;
        const bool bad_any = __any_sync(0xffffffffu, badb);
        bad_stage = bad_any ? (bad_stage | (1u << sidx)) : (bad_stage & ~(1u << sidx));
        const char* base = a.pool.base + (pb * Hkv + h) * a.pool.sub_bytes;
        unsigned char* dst = ring + static_cast<size_t>(sidx) * st.bytes;
        uint64_t* bar = &bars[sidx];
        if (lane == 0) mbar_expect_tx(bar, blk_tx * live);
        __syncwarp();
        if (mine)
            bulk_g2s_once(dst + s_off, base + s_src + static_cast<int64_t>(slot0) * s_field, blk_tokens * s_field,
                          bar, pol);
    };

    // First stages: fetched before waiting for the kernel this one may overlap,
    // except a tile holding tokens that kernel appended in this step (positions
    // from N - len_add on), which is visible only after the wait. Older records
    // come from kernels complete before this one could start: the query-prep
    // CTAs release it only after waiting for their own predecessor.
    const int pre = my_n < kStages - 1 ? my_n : kStages - 1;
    auto early = [&](int i) {
        return a.len_add == 0 || t_begin + (warp + i * kWarps) * TT + TT <= N - a.len_add;
    };
    for (int i = 0; i < pre; ++i)
        if (early(i)) issue(i, entry(i));
    // query fragments of this unit, shared by all warps: [2][8][32] uint4
    // (written by the query-prep kernel this one may overlap: wait for it)
    const uint4* qsm = reinterpret_cast<const uint4*>(smem + st.qs_off);
    tc::grid_wait_prior();
    for (int i = 0; i < pre; ++i)
        if (!early(i)) issue(i, entry(i));
    if constexpr (D == kD) {
        if (threadIdx.x == 0) {
            tc::fence_proxy_async_global();
            mbar_expect_tx(tbar, kQFragBytes);
            bulk_g2s(smem + st.qs_off, m.qfrag + static_cast<int64_t>(unit) * 2 * 8 * 32, kQFragBytes, tbar);
        }
    } else {
        // from the unit's fp32 q' and q'' rows (the query prep of this head_dim)
        frag_from_rows<KB, frag_order(KB, KPROD, VGROUP, VB), D, kThreads>(
            reinterpret_cast<uint32_t*>(smem + st.qs_off), a.qrot + static_cast<int64_t>(unit) * kRows * D,
            a.qjl + static_cast<int64_t>(unit) * kRows * D, KPROD, a.scale * kLog2e / a.kc.cq_scale,
            a.scale * kLog2e * kSqrtHalfPi / static_cast<float>(D), threadIdx.x);
        if (threadIdx.x == 0) mbar_expect_tx(tbar, 0);
    }
    __syncthreads();  // the barrier's initialisation and any tables and fragments built here
    if (!mbar_wait(tbar, 0)) {
        if (threadIdx.x == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
        (void)mbar_wait(tbar, 0);  // no copy may still be in flight below
    }
    int waited = 0;
    int32_t pb_ahead = kStages - 1 < my_n ? entry(kStages - 1) : 0;   // the next copy's table entry
    for (int i = 0; i < my_n; ++i) {
        if (i + kStages - 1 < my_n) {
            __syncwarp();
            issue(i + kStages - 1, pb_ahead);
            if (i + kStages < my_n) pb_ahead = entry(i + kStages);
        }
        if (!mbar_wait(&bars[i % kStages], (i / kStages) & 1)) {
            failed = true;
            break;
        }
        waited = i + 1;
        const unsigned char* sp = ring + static_cast<size_t>(i % kStages) * st.bytes;
        const uint32_t* kidx = reinterpret_cast<const uint32_t*>(sp + st.off[0]);
        const uint32_t* ksgn = KPROD ? reinterpret_cast<const uint32_t*>(sp + st.off[1]) : nullptr;
        const float* knorm = reinterpret_cast<const float*>(sp + st.off[2]);
        const float* krn = KPROD ? reinterpret_cast<const float*>(sp + st.off[3]) : nullptr;
        const uint32_t* vidx = reinterpret_cast<const uint32_t*>(sp + st.off[4]);
        const float* vnorm = VGROUP ? nullptr : reinterpret_cast<const float*>(sp + st.off[5]);
        const __half* vsc = VGROUP ? reinterpret_cast<const __half*>(sp + st.off[5]) : nullptr;
        const __half* vmn = VGROUP ? reinterpret_cast<const __half*>(sp + st.off[6]) : nullptr;

        const int t0 = t_begin + (warp + i * kWarps) * TT;
        int valid = min(TT, t_end - t0);
        if ((bad_stage >> (i % kStages)) & 1u) {
            if (lane == 0) atomicOr(a.err, TQ_DEVERR_BLOCK);
            valid = 0;
        }

        // rescale threshold lag of this tile (0 if a value norm could overflow P')
        float lag = kLag;
        if constexpr (!VGROUP) {
            float nmax = 0.0f;
            if (2 * lane < valid) nmax = vnorm[2 * lane];
            if (2 * lane + 1 < valid) nmax = fmaxf(nmax, vnorm[2 * lane + 1]);
            if (__any_sync(0xffffffffu, nmax > kLagNorm)) lag = 0.0f;
        }

        // One step = NT n8 tiles of tokens (8 NT tokens): the score MMAs run as
        // 2 NT independent accumulator chains of eight k-steps each (a chain's
        // MMAs wait on one another), so wider steps keep more MMAs in flight.
        auto step = [&](auto ntc, const int base) {
            constexpr int NT = decltype(ntc)::value;
            // QJL signs as exact +-1 operands; the residual norm multiplies the
            // sign products in fp32 below
            [[maybe_unused]] constexpr uint32_t neg2 = 0xBC00BC00u;  // (-1, -1): a set bit gives +1
            // ---------------- scores: S = Q' K^T (+ Q'' sigma^T), key operands
            // decoded two k-steps at a time
            // (R8: MT m16 tiles of 16 tokens, the n8 tiles 2 mt and 2 mt + 1)
            constexpr int MT = R8 ? (NT + 1) / 2 : NT;
            float sc[MT][4], sd[MT][4];
            uint32_t kw[NT][KB];
            uint32_t sw[NT];
#pragma unroll
            for (int nt = 0; nt < MT; ++nt) {
                sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.0f;
                sd[nt][0] = sd[nt][1] = sd[nt][2] = sd[nt][3] = 0.0f;
            }
            // the lane's 32-coordinate chunk j NC + c of each key, k-steps 8 c .. 8 c + 7
#pragma unroll
            for (int c = 0; c < NC; ++c) {
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int tau = base + 8 * nt + g;
                load_words<KB>(kidx + tau * (D / 32 * KB) + (jc * NC + c) * KB, kw[nt]);
                if constexpr (KPROD) sw[nt] = ksgn[tau * (D / 32) + jc * NC + c];
                else sw[nt] = 0u;
            }
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
                uint32_t hk[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if constexpr (kP4W) pair4w_word(smem, kw[nt][q2 < KB ? q2 : 0], k4_lane, hk[nt]);
                    else if constexpr (kP4K) pair4_word(kw[nt][q2 < KB ? q2 : 0], k4_lane, hk[nt]);
                    else key_ks2<KB, kQuadTab>(kw[nt], ktab, kt_lane, q2, hk[nt]);
                }
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int ks = 2 * q2 + e;
                    uint32_t qa[4], qj[4];
                    {
                        const uint4 v = qsm[(8 * c + ks) * 32 + lane];
                        qa[0] = v.x; qa[1] = v.y; qa[2] = v.z; qa[3] = v.w;
                        const uint4 w = qsm[(DV / 16 + 8 * c + ks) * 32 + lane];
                        qj[0] = w.x; qj[1] = w.y; qj[2] = w.z; qj[3] = w.w;
                    }
                    // the QJL sign operands of tile nt, k-step ks (B-operand pairs)
                    auto signs = [&](int nt, uint32_t& b0, uint32_t& b1) {
                        if constexpr (KPROD && kNibQ) {
                            // sign nibble ks of the lane's word at bits 7..10: a table address
                            const uint32_t x = ks == 0 ? shl_f(sw[nt], 7)
                                               : ks == 1 ? shl_f(sw[nt], 3) : (sw[nt] >> (4 * ks - 7));
                            const uint2 sv = lds_u64((x & 0x780u) | qn_lane);
                            b0 = sv.x;
                            b1 = sv.y;
                        } else if constexpr (KPROD) {
                            b0 = dec1(sw[nt], 15 - ks, neg2);
                            b1 = dec1(sw[nt], 7 - ks, neg2);
                        } else {
                            b0 = hk[nt][2 * e];
                            b1 = hk[nt][2 * e + 1];
                        }
                    };
                    if constexpr (R8) {
                        // A: tokens g of tiles 2 mt and 2 mt + 1; B: rows 0..7
                        const uint32_t qb[2] = {qa[0], qa[2]}, jb[2] = {qj[0], qj[2]};
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            const int n0 = 2 * mt, n1 = 2 * mt + 1 < NT ? 2 * mt + 1 : 2 * mt;
                            const uint32_t ka[4] = {hk[n0][2 * e], hk[n1][2 * e], hk[n0][2 * e + 1], hk[n1][2 * e + 1]};
                            mma16816(sc[mt], ka, qb[0], qb[1]);
                            uint32_t s00, s01, s10, s11;
                            signs(n0, s00, s01);
                            signs(n1, s10, s11);
                            const uint32_t sa[4] = {s00, s10, s01, s11};
                            mma16816(sd[mt], sa, jb[0], jb[1]);
                        }
                    } else {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma16816(sc[nt], qa, hk[nt][2 * e], hk[nt][2 * e + 1]);
                            uint32_t b0, b1;
                            signs(nt, b0, b1);
                            mma16816(sd[nt], qj, b0, b1);
                        }
                    }
                }
            }
            }
            // ---------------- values of the first 16 tokens: decoded while the
            // score MMAs are in flight (independent of the scores)
            uint32_t hA[16], hB[16];
            auto decode_values = [&](int kg) {
                const int tA = base + 16 * kg + g, tB = tA + 8;
                uint32_t wA[VB], wB[VB];
                // the lane's 32-coordinate chunk 4 h2 + j of the CTA's value half
                load_words<VB>(vidx + tA * (D / 32 * VB) + (4 * h2 + jc) * VB, wA);
                load_words<VB>(vidx + tB * (D / 32 * VB) + (4 * h2 + jc) * VB, wB);
                if constexpr (VGROUP) {
                    // fp16 pairs (2^VB s, 2^VB s) and (min, min) straight from the
                    // stored halves (the power-of-two product is exact)
                    const __half z = __float2half_rn(0.0f);
                    const __half2 mul = __float2half2_rn(VB == 4 ? 16.0f : 4.0f);
                    const bool okA = tA < valid, okB = tB < valid;
                    const __half2 sA = __hmul2(__half2half2(okA ? vsc[tA * vng + vgi] : z), mul);
                    const __half2 mA = __half2half2(okA ? vmn[tA * vng + vgi] : z);
                    const __half2 sB = __hmul2(__half2half2(okB ? vsc[tB * vng + vgi] : z), mul);
                    const __half2 mB = __half2half2(okB ? vmn[tB * vng + vgi] : z);
                    GroupChunk<VB>::run(wA, h2_bits(sA), h2_bits(mA), hA);
                    GroupChunk<VB>::run(wB, h2_bits(sB), h2_bits(mB), hB);
                } else if constexpr (kPairTab) {
                    pair3_chunk(wA, vt_lane, hA);
                    pair3_chunk(wB, vt_lane, hB);
                } else if constexpr (kP4V) {
#pragma unroll
                    for (int wi = 0; wi < 4; ++wi) {
                        uint32_t ga[4], gb[4];
                        if constexpr (kP4W) {
                            pair4w_word(smem, wA[wi < VB ? wi : 0], v4_lane, ga);
                            pair4w_word(smem, wB[wi < VB ? wi : 0], v4_lane, gb);
                        } else {
                            pair4_word(wA[wi < VB ? wi : 0], v4_lane, ga);
                            pair4_word(wB[wi < VB ? wi : 0], v4_lane, gb);
                        }
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            hA[4 * wi + k] = ga[k];
                            hB[4 * wi + k] = gb[k];
                        }
                    }
                } else {
                    mse_chunk<VB>(wA, vtab, hA);
                    mse_chunk<VB>(wB, vtab, hB);
                }
            };
            decode_values(0);
            if constexpr (R8) {
                // tokens ta (tile 2 mt) and tb = ta + 8 (tile 2 mt + 1) of the lane,
                // rows r0 = 2 j and r1 = 2 j + 1: S^T entries (ta, r0), (ta, r1),
                // (tb, r0), (tb, r1)
                float2 nv8[MT];
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    const int ta = base + 16 * mt + g, tb = ta + 8;
                    if constexpr (KPROD) {
                        // codebook part + residual norm x QJL part
                        const float ga = krn[ta], gb = krn[tb];
                        sc[mt][0] = fmaf(ga, sd[mt][0], sc[mt][0]);
                        sc[mt][1] = fmaf(ga, sd[mt][1], sc[mt][1]);
                        sc[mt][2] = fmaf(gb, sd[mt][2], sc[mt][2]);
                        sc[mt][3] = fmaf(gb, sd[mt][3], sc[mt][3]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) sc[mt][e] += sd[mt][e];
                    }
                    const float kna = knorm[ta], knb = knorm[tb];
                    sc[mt][0] *= kna;
                    sc[mt][1] *= kna;
                    sc[mt][2] *= knb;
                    sc[mt][3] *= knb;
                    if constexpr (!VGROUP) nv8[mt] = make_float2(vnorm[ta], vnorm[tb]);
                    else nv8[mt] = make_float2(0.0f, 0.0f);
                }
                // masks only where the step reaches past the tile's end or a row's
                // causal limit (past the end, the stage holds stale bytes: their
                // value norms become 0)
                if (base + 8 * NT > valid || t0 + base + 8 * NT - 1 > lim_all) {
#pragma unroll
                    for (int mt = 0; mt < MT; ++mt) {
                        const int ta = base + 16 * mt + g, tb = ta + 8;
                        const bool va = ta < valid, vb = tb < valid;
                        if (!(va && t0 + ta <= lim0)) sc[mt][0] = -INFINITY;
                        if (!(va && t0 + ta <= lim1)) sc[mt][1] = -INFINITY;
                        if (!(vb && t0 + tb <= lim0)) sc[mt][2] = -INFINITY;
                        if (!(vb && t0 + tb <= lim1)) sc[mt][3] = -INFINITY;
                        if (!va) nv8[mt].x = 0.0f;
                        if (!vb) nv8[mt].y = 0.0f;
                    }
                }
                const float th0 = mrow0 + lag, th1 = mrow1 + lag;
                bool over = false;
#pragma unroll
                for (int mt = 0; mt < MT; ++mt)
                    over |= sc[mt][0] > th0 || sc[mt][1] > th1 || sc[mt][2] > th0 || sc[mt][3] > th1;
                if (__any_sync(0xffffffffu, over)) {
                    // a score passed m + lag: move m to the exact row maxima (the
                    // lanes g of one j hold the rows' tokens)
                    float mx0 = fmaxf(sc[0][0], sc[0][2]), mx1 = fmaxf(sc[0][1], sc[0][3]);
#pragma unroll
                    for (int mt = 1; mt < MT; ++mt) {
                        mx0 = fmaxf(mx0, fmaxf(sc[mt][0], sc[mt][2]));
                        mx1 = fmaxf(mx1, fmaxf(sc[mt][1], sc[mt][3]));
                    }
#pragma unroll
                    for (int o2 = 4; o2 < 32; o2 <<= 1) {
                        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
                        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
                    }
                    const float mn0 = fmaxf(mrow0, mx0), mn1 = fmaxf(mrow1, mx1);
                    const float al0 = ex2(mrow0 - mn0);
                    const float al1 = ex2(mrow1 - mn1);
                    lrow0 *= al0;
                    lrow1 *= al1;
#pragma unroll
                    for (int p = 0; p < kOT; ++p) {
                        o[p][0] *= al0; o[p][1] *= al1;
                        o[p][2] *= al0; o[p][3] *= al1;
                    }
                    mrow0 = mn0;
                    mrow1 = mn1;
                }
                // P' = fp16(p * value norm) per token; the row sums add P' / norm
                // (a zero norm: its p enters the row sums in the branch below)
                uint32_t pu[MT][2];
                [[maybe_unused]] bool zero = false;
                float2 lsum = make_float2(0.0f, 0.0f);  // this step's (row r0, row r1) sums
#pragma unroll
                for (int mt = 0; mt < MT; ++mt) {
                    float2 wa = make_float2(ex2(sc[mt][0] - mrow0), ex2(sc[mt][1] - mrow1));   // token ta
                    float2 wb = make_float2(ex2(sc[mt][2] - mrow0), ex2(sc[mt][3] - mrow1));   // token tb
                    float ra = 1.0f, rb = 1.0f;
                    if constexpr (!VGROUP) {
                        const float nx = nv8[mt].x, ny = nv8[mt].y;
                        zero |= !(fminf(nx, ny) > 0.0f);
                        ra = rcp_approx(fmaxf(nx, 1e-30f));
                        rb = rcp_approx(fmaxf(ny, 1e-30f));
                        sc[mt][0] = wa.x;  // keep p for the zero-norm branch
                        sc[mt][1] = wa.y;
                        sc[mt][2] = wb.x;
                        sc[mt][3] = wb.y;
                        wa = __fmul2_rn(wa, make_float2(nx, nx));
                        wb = __fmul2_rn(wb, make_float2(ny, ny));
                    }
                    pu[mt][0] = pack_half2(wa.x, wa.y);
                    pu[mt][1] = pack_half2(wb.x, wb.y);
                    const float2 fa = __half22float2(*reinterpret_cast<const __half2*>(&pu[mt][0]));
                    const float2 fb = __half22float2(*reinterpret_cast<const __half2*>(&pu[mt][1]));
                    lsum = __ffma2_rn(fa, make_float2(ra, ra), lsum);
                    lsum = __ffma2_rn(fb, make_float2(rb, rb), lsum);
                }
                lrow0 += lsum.x;
                lrow1 += lsum.y;
                if constexpr (!VGROUP) {
                    if (__any_sync(0xffffffffu, zero)) {
#pragma unroll
                        for (int mt = 0; mt < MT; ++mt) {
                            if (!(nv8[mt].x > 0.0f)) { lrow0 += sc[mt][0]; lrow1 += sc[mt][1]; }
                            if (!(nv8[mt].y > 0.0f)) { lrow0 += sc[mt][2]; lrow1 += sc[mt][3]; }
                        }
                    }
                }
                // ---------------- O^T += V^T P'^T, 16 tokens (one m16 tile) per k-group:
                // A = the value columns of pairs 2 p and 2 p + 1 (16) x the tokens,
                // B = P'^T (tokens x rows) by transposing the lane's (token, row pair)
#pragma unroll
                for (int kg = 0; kg < MT; ++kg) {
                    if (kg > 0) decode_values(kg);
                    const uint32_t b0 = movmatrix_t(pu[kg][0]), b1 = movmatrix_t(pu[kg][1]);
#pragma unroll
                    for (int p = 0; p < kOT; ++p) {
                        const uint32_t va[4] = {movmatrix_t(hA[2 * p]), movmatrix_t(hA[2 * p + 1]),
                                                movmatrix_t(hB[2 * p]), movmatrix_t(hB[2 * p + 1])};
                        mma16816(o[p], va, b0, b1);
                    }
                }
            } else {
    #pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    if constexpr (KPROD) {
                        // codebook part + residual norm x QJL part, per token column
                        const float2 gm = *reinterpret_cast<const float2*>(krn + base + 8 * nt + 2 * j);
                        // (two tokens' columns per packed fp32 pair operation)
                        const float2 lo = __ffma2_rn(gm, make_float2(sd[nt][0], sd[nt][1]), make_float2(sc[nt][0], sc[nt][1]));
                        const float2 hi = __ffma2_rn(gm, make_float2(sd[nt][2], sd[nt][3]), make_float2(sc[nt][2], sc[nt][3]));
                        sc[nt][0] = lo.x; sc[nt][1] = lo.y; sc[nt][2] = hi.x; sc[nt][3] = hi.y;
                    } else {
    #pragma unroll
                        for (int e = 0; e < 4; ++e) sc[nt][e] += sd[nt][e];
                    }
                }
                // ---------------- scale, mask, online softmax (log2 domain)
                float2 nv[NT];
    #pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float2 kn = *reinterpret_cast<const float2*>(knorm + base + 8 * nt + 2 * j);
                    if constexpr (!VGROUP) nv[nt] = *reinterpret_cast<const float2*>(vnorm + base + 8 * nt + 2 * j);
                    else nv[nt] = make_float2(0.0f, 0.0f);
                    const float2 lo = __fmul2_rn(make_float2(sc[nt][0], sc[nt][1]), kn);
                    const float2 hi = __fmul2_rn(make_float2(sc[nt][2], sc[nt][3]), kn);
                    sc[nt][0] = lo.x; sc[nt][1] = lo.y; sc[nt][2] = hi.x; sc[nt][3] = hi.y;
                }
                // masks only where the step reaches past the tile's end or a row's
                // causal limit (past the end, the stage holds stale bytes: their
                // value norms become 0)
                if (base + 8 * NT > valid || t0 + base + 8 * NT - 1 > lim_all) {
    #pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const int tl = base + 8 * nt + 2 * j;
                        const int pos = t0 + tl;
                        const bool v0 = tl < valid, v1 = tl + 1 < valid;
                        if (!(v0 && pos <= lim0)) sc[nt][0] = -INFINITY;
                        if (!(v1 && pos + 1 <= lim0)) sc[nt][1] = -INFINITY;
                        if (!(v0 && pos <= lim1)) sc[nt][2] = -INFINITY;
                        if (!(v1 && pos + 1 <= lim1)) sc[nt][3] = -INFINITY;
                        if (!v0) nv[nt].x = 0.0f;
                        if (!v1) nv[nt].y = 0.0f;
                    }
                }
                const float th0 = mrow0 + lag, th1 = mrow1 + lag;
                bool over = false;
    #pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    over |= sc[nt][0] > th0 || sc[nt][1] > th0 || sc[nt][2] > th1 || sc[nt][3] > th1;
                if (__any_sync(0xffffffffu, over)) {
                    // a score passed m + lag: move m to the exact row maxima
                    float mx0 = fmaxf(sc[0][0], sc[0][1]), mx1 = fmaxf(sc[0][2], sc[0][3]);
    #pragma unroll
                    for (int nt = 1; nt < NT; ++nt) {
                        mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
                        mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
                    }
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
                    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
                    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
                    const float mn0 = fmaxf(mrow0, mx0), mn1 = fmaxf(mrow1, mx1);
                    const float al0 = ex2(mrow0 - mn0);
                    const float al1 = ex2(mrow1 - mn1);
                    lrow0 *= al0;
                    lrow1 *= al1;
    #pragma unroll
                    for (int p = 0; p < 16; ++p) {
                        o[p][0] *= al0; o[p][1] *= al0;
                        o[p][2] *= al1; o[p][3] *= al1;
                    }
                    mrow0 = mn0;
                    mrow1 = mn1;
                }
                // P' = fp16(p * value norm); the row sums add the weights actually
                // multiplied (P' / norm), so the rounding of P' cancels in o = sum/L.
                // A zero norm gives P' = 0 and a huge finite 1/norm (nothing added);
                // its p enters the row sums in the rare branch below.
                uint32_t pa[NT][2];
                [[maybe_unused]] bool zero = false;
                const float2 nm0 = make_float2(-mrow0, -mrow0), nm1 = make_float2(-mrow1, -mrow1);
                float2 lsum = make_float2(0.0f, 0.0f);  // this step's (row g, row g + 8) sums
    #pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const float2 x0 = __fadd2_rn(make_float2(sc[nt][0], sc[nt][1]), nm0);
                    const float2 x1 = __fadd2_rn(make_float2(sc[nt][2], sc[nt][3]), nm1);
                    float2 w01 = make_float2(ex2(x0.x), ex2(x0.y));
                    float2 w23 = make_float2(ex2(x1.x), ex2(x1.y));
                    float r0 = 1.0f, r1 = 1.0f;
                    if constexpr (!VGROUP) {
                        const float nx = nv[nt].x, ny = nv[nt].y;
                        zero |= !(fminf(nx, ny) > 0.0f);
                        r0 = rcp_approx(fmaxf(nx, 1e-30f));
                        r1 = rcp_approx(fmaxf(ny, 1e-30f));
                        sc[nt][0] = w01.x;  // keep p for the zero-norm branch
                        sc[nt][1] = w01.y;
                        sc[nt][2] = w23.x;
                        sc[nt][3] = w23.y;
                        w01 = __fmul2_rn(w01, nv[nt]);
                        w23 = __fmul2_rn(w23, nv[nt]);
                    }
                    pa[nt][0] = pack_half2(w01.x, w01.y);
                    pa[nt][1] = pack_half2(w23.x, w23.y);
                    const float2 f0 = __half22float2(*reinterpret_cast<const __half2*>(&pa[nt][0]));
                    const float2 f1 = __half22float2(*reinterpret_cast<const __half2*>(&pa[nt][1]));
                    lsum = __ffma2_rn(make_float2(f0.x, f1.x), make_float2(r0, r0), lsum);
                    lsum = __ffma2_rn(make_float2(f0.y, f1.y), make_float2(r1, r1), lsum);
                }
                lrow0 += lsum.x;
                lrow1 += lsum.y;
                if constexpr (!VGROUP) {
                    if (__any_sync(0xffffffffu, zero)) {
    #pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            if (!(nv[nt].x > 0.0f)) { lrow0 += sc[nt][0]; lrow1 += sc[nt][2]; }
                            if (!(nv[nt].y > 0.0f)) { lrow0 += sc[nt][1]; lrow1 += sc[nt][3]; }
                        }
                    }
                }
                // ---------------- O += P' V, 16 tokens per k-group
    #pragma unroll
                for (int kg = 0; kg < NT / 2; ++kg) {
                    if (kg > 0) decode_values(kg);
                    const uint32_t pk[4] = {pa[2 * kg][0], pa[2 * kg][1], pa[2 * kg + 1][0], pa[2 * kg + 1][1]};
    #pragma unroll
                    for (int p = 0; p < 16; ++p) mma16816(o[p], pk, movmatrix_t(hA[p]), movmatrix_t(hB[p]));
                }
            }
        };
        if (TT >= 32) {
            for (int u = 0; u < TT / 32; ++u) {
                if (32 * u >= valid) break;
                step(std::integral_constant<int, 4>{}, 32 * u);
            }
        } else if (valid > 0) {
            step(std::integral_constant<int, 2>{}, 0);
        }
    }
    tc::grid_release_dependents();  // the next kernel may start; it waits for this one before the workspace
    if (mrow0 == kNoMax) mrow0 = -INFINITY;  // no score seen by this thread's rows
    if (mrow1 == kNoMax) mrow1 = -INFINITY;
    if (failed && lane == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
    // drain copies that were issued but never waited for (only after a timeout)
    if (failed) {
        const int issued = my_n < waited + kStages - 1 ? my_n : waited + kStages - 1;
        for (int i = waited; i < issued; ++i) (void)mbar_wait(&bars[i % kStages], (i / kStages) & 1);
    }

    __syncwarp();
    if (lane == 0)
        for (int s = 0; s < kStages; ++s) mbar_inval(&bars[s]);
    if (threadIdx.x == 0) mbar_inval(tbar);

    // ---------------- merge the warps of this CTA
    // row sums over the lanes that share the thread's rows (R8: the lanes g of
    // one j; else the lanes j of one g)
#pragma unroll
    for (int o2 = R8 ? 4 : 1; o2 < (R8 ? 32 : 4); o2 <<= 1) {
        lrow0 += __shfl_xor_sync(0xffffffffu, lrow0, o2);
        lrow1 += __shfl_xor_sync(0xffffffffu, lrow1, o2);
    }
    __syncthreads();
    constexpr int kStride = kCoStride;  // column d at d + d / 32
    float* cm = reinterpret_cast<float*>(smem);
    float* cl = cm + kWarps * kRows;
    float* co = cl + kWarps * kRows;
    const int lr0 = r0 - rg * kRows, lr1 = r1 - rg * kRows;   // the thread's rows in the group
    if (R8 ? g == 0 : j == 0) {
        cm[warp * kRows + lr0] = mrow0;
        cm[warp * kRows + lr1] = mrow1;
        cl[warp * kRows + lr0] = lrow0;
        cl[warp * kRows + lr1] = lrow1;
    }
    if constexpr (R8) {
        // o[p]: O^T of value pairs 2 p (entries 0, 1) and 2 p + 1 (2, 3), column g
        // of the pair's eight (chunk g / 2, element g % 2), rows lr0 (0, 2) and lr1
#pragma unroll
        for (int p = 0; p < kOT; ++p) {
#pragma unroll
            for (int hp = 0; hp < 2; ++hp) {
                int pa_, pb_;
                if constexpr (VGROUP) group_pair(VB, 2 * p + hp, pa_, pb_);
                else mse_pair(VB, 2 * p + hp, pa_, pb_);
                const int d = 33 * (g >> 1) + ((g & 1) ? pb_ : pa_);
                co[(warp * kRows + lr0) * kStride + d] = o[p][2 * hp];
                co[(warp * kRows + lr1) * kStride + d] = o[p][2 * hp + 1];
            }
        }
    } else {
#pragma unroll
        for (int p = 0; p < kOT; ++p) {
            int pa_, pb_;
            if constexpr (VGROUP) group_pair(VB, p, pa_, pb_);
            else mse_pair(VB, p, pa_, pb_);
            const int d0 = 33 * j + pa_, d1 = 33 * j + pb_;
            co[(warp * kRows + lr0) * kStride + d0] = o[p][0];
            co[(warp * kRows + lr0) * kStride + d1] = o[p][1];
            co[(warp * kRows + lr1) * kStride + d0] = o[p][2];
            co[(warp * kRows + lr1) * kStride + d1] = o[p][3];
        }
    }
    __syncthreads();
    const int S = a.plan.splits;
    const int tid = threadIdx.x;
    const int r = tid >> 4;
    const int dbase = (tid & 15) * 8;
    const bool merger = tid < (R8 ? 8 : kRows) * 16;  // 16 threads per row, 8 columns each
    if (merger) {
        float M = -INFINITY;
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, cm[w * kRows + r]);
        float L = 0.0f, acc[8] = {};
        if (M != -INFINITY) {
            for (int w = 0; w < kWarps; ++w) {
                const float mw = cm[w * kRows + r];
                if (mw == -INFINITY) continue;
                const float wt = ex2(mw - M);
                L = fmaf(wt, cl[w * kRows + r], L);
                for (int k = 0; k < 8; ++k)
                    acc[k] = fmaf(wt, co[(w * kRows + r) * kStride + dbase + dbase / 32 + k], acc[k]);
            }
        }
        float* dst = m.part + ((static_cast<int64_t>(punit) * S + split) * kRows + r) * kD + dbase;
        reinterpret_cast<float4*>(dst)[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        if ((tid & 15) == 0) {
            float* mlp = m.ml + ((static_cast<int64_t>(punit) * S + split) * kRows + r) * 2;
            mlp[0] = M;
            mlp[1] = L;
        }
    }
}

// Query prep fused with the short encode of a decode step's new tokens
// (decode_step.cu): one launch in place of the append and the query prep.
cudaError_t launch_step_prep(int kb, int ord, const MmaArgs& m, const EncodeAppendArgs& e, cudaStream_t s);

// The merge kernel after a split kernel: one CTA per (unit, row).
template <bool VGROUP, int D = kD>
cudaError_t launch_merge(const MmaArgs& m, cudaStream_t s) {
    const DecodeArgs& a = m.a;
    const bool rotate = !VGROUP && !a.part_acc;
    const size_t smem = merge_rows_smem<VGROUP, D>(rotate);
    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        const cudaError_t e = cudaFuncSetAttribute(merge_rows_kernel<VGROUP, D>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(merge_rows_smem<VGROUP, D>(true)));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        attr_set.fetch_or(bit);
    }
    const int units = a.batch * a.pool.Hkv * a.plan.row_groups;
    const cudaError_t e = launch_overlapped(merge_rows_kernel<VGROUP, D>, dim3(units, kRows), dim3(merge_threads<VGROUP, D>()), smem, s, m);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e;
}

// Opt-in of a split kernel to the largest dynamic shared memory the device
// allows next to its static shared memory (once per device); the result is
// that limit, or -1 with the error in *err.
template <typename K>
int split_smem_limit(K kernel, std::atomic<uint64_t>& attr_set, std::atomic<int>* max_dyn, cudaError_t* err) {
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        int optin = 0;
        cudaFuncAttributes fa{};
        cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, kernel);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();  // do not leave the error for the next launch
            *err = e;
            return -1;
        }
        attr_set.fetch_or(bit);
        max_dyn[dev & 63].store(optin - static_cast<int>(fa.sharedSizeBytes));
    }
    return max_dyn[dev & 63].load();
}

// Query prep of head dims above 128: q' = R_k q and, for prod keys,
// q'' = (S_k R_k) q (S_k q' up to rounding: the product is a codec table), in
// fp32 into [unit][16][D]. CTA (unit, 32-column slice, matrix): the slice of
// the transposed matrix (D rows of 128 B, one bulk copy each) and the unit's 16
// query rows (contiguous in q) are staged in shared memory at once; lane c
// owns column c of the slice, warp w rows 2 w and 2 w + 1, and each output is
// one fp32 chain of fused multiply-adds over ascending k.
constexpr int kQRThreads = 256;

template <int D>
__global__ void __launch_bounds__(kQRThreads) qrows_kernel(DecodeArgs a) {
    static_assert(D % 32 == 0 && D <= kQRThreads, "one bulk copy per matrix row and thread");
    extern __shared__ __align__(128) float qr_smem[];
    float* ms = qr_smem;        // [D][32] the matrix slice
    float* qs = ms + D * 32;    // [16][D] query rows
    __shared__ uint64_t bar;
    // This kernel is a plain launch (it starts after everything before it on
    // the stream is complete, the records included), so the split kernel may
    // start its prologue (tables, first record copies) at once; it waits for
    // this grid before it reads the rows written below.
    tc::grid_release_dependents();
    const int unit = blockIdx.x, c0 = 32 * blockIdx.y;
    const bool qjl = blockIdx.z != 0;
    const float* M = qjl ? a.kc.SRt : a.kc.Rt;
    const int tid = threadIdx.x;
    if (tid == 0) {
        mbar_init(&bar, 1);
        mbar_fence_init();
        mbar_expect_tx(&bar, D * 32 * 4);
    }
    __syncthreads();
    if (tid < D) bulk_g2s(ms + tid * 32, M + static_cast<int64_t>(tid) * D + c0, 32 * 4, &bar);
    const int RG = a.plan.row_groups;
    const int rg = unit % RG, bh = unit / RG;
    const int b = bh / a.pool.Hkv, h = bh % a.pool.Hkv;
    // row r of the group: query head h G + r / Lq, position r % Lq, at
    // (b Hq + h G) Lq + r rows into q
    const int64_t q0 = (static_cast<int64_t>(b) * a.Hq + h * a.G) * a.Lq + rg * kRows;
    const int nrows = min(kRows, a.plan.rows - rg * kRows);
#pragma unroll 4
    for (int e = tid; e < kRows * D; e += kQRThreads) {
        const int rr = e / D;
        float v = 0.0f;
        if (rr < nrows) {
            const int64_t src = q0 * D + e;
            if (a.q_dtype == TQ_F32) v = static_cast<const float*>(a.q)[src];
            else if (a.q_dtype == TQ_BF16) v = __bfloat162float(static_cast<const __nv_bfloat16*>(a.q)[src]);
            else v = __half2float(static_cast<const __half*>(a.q)[src]);
        }
        qs[e] = v;
    }
    __syncthreads();
    if (!mbar_wait(&bar, 0)) {
        if (tid == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
        (void)mbar_wait(&bar, 0);  // no copy may still be in flight below
    }
    const int lane = tid & 31, w = tid >> 5;
    const float4* x0 = reinterpret_cast<const float4*>(qs + (2 * w) * D);
    const float4* x1 = reinterpret_cast<const float4*>(qs + (2 * w + 1) * D);
    float y0 = 0.0f, y1 = 0.0f;
#pragma unroll 4
    for (int k4 = 0; k4 < D / 4; ++k4) {
        const float4 u = x0[k4], v = x1[k4];
        const float m0 = ms[(4 * k4) * 32 + lane], m1 = ms[(4 * k4 + 1) * 32 + lane];
        const float m2 = ms[(4 * k4 + 2) * 32 + lane], m3 = ms[(4 * k4 + 3) * 32 + lane];
        y0 = fmaf(m0, u.x, y0);
        y1 = fmaf(m0, v.x, y1);
        y0 = fmaf(m1, u.y, y0);
        y1 = fmaf(m1, v.y, y1);
        y0 = fmaf(m2, u.z, y0);
        y1 = fmaf(m2, v.z, y1);
        y0 = fmaf(m3, u.w, y0);
        y1 = fmaf(m3, v.w, y1);
    }
    float* out = (qjl ? a.qjl : a.qrot) + static_cast<int64_t>(unit) * kRows * D + c0 + lane;
    out[(2 * w) * D] = y0;       // padding rows: zero queries give zeros
    out[(2 * w + 1) * D] = y1;
    if (tid == 0) mbar_inval(&bar);
}

template <int D>
constexpr size_t qrows_smem() { return static_cast<size_t>(D) * 32 * 4 + static_cast<size_t>(kRows) * D * 4; }

// Head dims other than 128 (above it two 128-column value halves per unit;
// 64 in the head_dim-128 layout): the query prep writes the fp32 q' and q''
// rows, the split kernel builds its fragments from them, then the merge.
template <int KB, bool KPROD, bool VGROUP, int VB, int D>
cudaError_t launch_mma_wide(const MmaArgs& m, size_t smem, cudaStream_t s) {
    static_assert(D == 64 || (D > kD && D % kD == 0), "head_dim 64 or a multiple of 128 above 128");
    const DecodeArgs& a = m.a;
    static std::atomic<uint64_t> attr_set{0}, qr_set{0};
    static std::atomic<int> max_dyn[64];
    cudaError_t e = cudaSuccess;
    const int lim = split_smem_limit(split_mma_kernel<KB, KPROD, VGROUP, VB, D>, attr_set, max_dyn, &e);
    if (lim < 0) return e;
    if (static_cast<int>(smem) > lim) return cudaErrorInvalidValue;
    if (KPROD && !a.kc.SRt) return cudaErrorInvalidValue;
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(qr_set.load() & bit)) {
        e = cudaFuncSetAttribute(qrows_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(qrows_smem<D>()));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        qr_set.fetch_or(bit);
    }
    const int units = a.batch * a.pool.Hkv * a.plan.row_groups;
    qrows_kernel<D><<<dim3(units, D / 32, KPROD ? 2 : 1), kQRThreads, qrows_smem<D>(), s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = launch_overlapped(split_mma_kernel<KB, KPROD, VGROUP, VB, D>,
                          dim3(a.pool.Hkv * a.plan.row_groups * (D > kD ? D / kD : 1), a.batch, a.plan.splits),
                          dim3(kThreads),
                          smem, s, m);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (e != cudaSuccess) return e;
    return launch_merge<VGROUP, D>(m, s);
}

// R8: the transposed split kernel (head_dim 128, at most 8 query rows per unit).
template <int KB, bool KPROD, bool VGROUP, int VB, bool R8 = false>
cudaError_t launch_mma(const MmaArgs& m, size_t smem, cudaStream_t s, const EncodeAppendArgs* step) {
    const DecodeArgs& a = m.a;
    static std::atomic<uint64_t> attr_set{0};
    static std::atomic<int> max_dyn[64];
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        // opt in once to the largest dynamic size the device allows next to the
        // kernel's static shared memory: later calls may need larger stages
        int optin = 0;
        cudaFuncAttributes fa{};
        cudaError_t e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
        if (e == cudaSuccess) e = cudaFuncGetAttributes(&fa, split_mma_kernel<KB, KPROD, VGROUP, VB, kD, R8>);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(split_mma_kernel<KB, KPROD, VGROUP, VB, kD, R8>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     optin - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();  // do not leave the error for the next launch
            return e;
        }
        attr_set.fetch_or(bit);
        max_dyn[dev & 63].store(optin - static_cast<int>(fa.sharedSizeBytes));
    }
    if (static_cast<int>(smem) > max_dyn[dev & 63].load()) return cudaErrorInvalidValue;
    const int RG = a.plan.row_groups;
    cudaError_t e = cudaSuccess;
    if (step) {
        e = launch_step_prep(KB, frag_order(KB, KPROD, VGROUP, VB), m, *step, s);
        if (e != cudaSuccess) return e;
        e = launch_overlapped(split_mma_kernel<KB, KPROD, VGROUP, VB, kD, R8>, dim3(a.pool.Hkv * RG, a.batch, a.plan.splits),
                              dim3(kThreads), smem, s, m);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        if (e != cudaSuccess) return e;
        return launch_merge<VGROUP>(m, s);
    }
    static std::atomic<uint64_t> qattr_set{0};
    if (!(qattr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(qfrag_kernel<KB, frag_order(KB, KPROD, VGROUP, VB)>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(sizeof(QSmem)));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        qattr_set.fetch_or(bit);
    }
    e = launch_overlapped(qfrag_kernel<KB, frag_order(KB, KPROD, VGROUP, VB)>, dim3(qfrag_grid(a.batch * a.pool.Hkv * RG)),
                          dim3(kQThreads),
                          sizeof(QSmem), s, m);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (e != cudaSuccess) return e;
    e = launch_overlapped(split_mma_kernel<KB, KPROD, VGROUP, VB, kD, R8>, dim3(a.pool.Hkv * RG, a.batch, a.plan.splits),
                          dim3(kThreads), smem, s, m);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (e != cudaSuccess) return e;
    return launch_merge<VGROUP>(m, s);
}

}  // namespace mmadec
}  // namespace tq

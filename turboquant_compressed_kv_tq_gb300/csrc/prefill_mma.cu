// Prefill attention over the compressed cache on the tensor cores (head_dim 128).
//
// The function is the decode attention's for any query length: a chunk of
// q_len positions, already appended, attends to its sequence's compressed
// prefix and causally to itself (query l sees keys t <= N - q_len + l). What
// changes is the work split: one CTA owns 8 row groups of 16 query rows (one
// warp each) and walks the key/value tiles its rows can see. Each 64-token
// tile is fetched once (1-D bulk copies, double-buffered), decoded once by the
// whole CTA into fp16 operand tiles in shared memory -- key levels c_k[idx]
// and +-rnorm signs in the query fragments' coordinate order, value levels (or
// group-dequantised values) in natural order -- and then used by all 8 warps:
// scores on mma.sync against the tile, online softmax in log2 units, P.V on
// mma.sync with the value tile transposed by ldmatrix. No split-K: each CTA
// finishes its rows, divides by the row sums and applies the inverse value
// rotation from a shared-memory copy of R_v.
//
// Query fragments come from the decode path's query-prep kernel (workspace).
#include "decode_mma_impl.cuh"

namespace tq {
namespace mmadec {
namespace {

constexpr int kPWarps = 8;
constexpr int kPThreads = kPWarps * 32;
constexpr int kPTok = 64;            // tokens per tile (at most)
constexpr int kOpStride = kD + 8;    // halves per operand row: conflict-free fragment loads

struct PrefillArgs {
    DecodeArgs a;
    StageLayout st;                  // record streams of one tile (st.tt tokens)
    const uint4* qfrag;              // [unit][2][8][32] uint4
    int op_off;                      // 3 operand tiles [kPTok][kOpStride] halves
    int norm_off;                    // key and value norms [2][kPTok] floats
    int rv_off;                      // R_v [kD][kD] floats
    int bar_off;                     // 3 mbarriers + the CTA's key limit
};

__device__ __forceinline__ void ldsm_x4_trans(uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3, const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(smem_u32(p)));
}

template <int KB, bool KPROD, bool VGROUP, int VB>
__global__ void __launch_bounds__(kPThreads, 1) prefill_kernel(PrefillArgs P) {
    extern __shared__ __align__(128) unsigned char smem[];
    const DecodeArgs& a = P.a;
    const StageLayout& st = P.st;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int g = lane >> 2, j = lane & 3;
    const int Hkv = a.pool.Hkv, RG = a.plan.row_groups, BT = a.pool.BT, TT = st.tt;
    const int h = blockIdx.y, b = blockIdx.z;
    const int rg = blockIdx.x + warp * gridDim.x;
    const bool active = rg < RG;
    const int unit = (b * Hkv + h) * RG + rg;

    __half* Kop = reinterpret_cast<__half*>(smem + P.op_off);
    __half* Sop = Kop + kPTok * kOpStride;
    __half* Vop = Sop + kPTok * kOpStride;
    float* kn = reinterpret_cast<float*>(smem + P.norm_off);
    float* vn = kn + kPTok;
    float* Rv = reinterpret_cast<float*>(smem + P.rv_off);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bar_off);  // [0,1] tiles, [2] R_v
    int* s_lim = reinterpret_cast<int*>(bars + 3);

    const int N = a.seq_lens[b];
    const bool bad = N < a.Lq || N > a.max_blocks * BT;
    if (bad && tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(a.err, TQ_DEVERR_SEQLEN);
    const int r0 = rg * kRows + g, r1 = r0 + 8;
    const bool ok0 = active && r0 < a.plan.rows, ok1 = active && r1 < a.plan.rows;
    const int lim0 = ok0 ? N - a.Lq + (r0 % a.Lq) : -1;
    const int lim1 = ok1 ? N - a.Lq + (r1 % a.Lq) : -1;

    if (tid == 0) {
        *s_lim = -1;
        for (int s = 0; s < 3; ++s) mbar_init(&bars[s], 1);
        mbar_fence_init();
        if constexpr (!VGROUP) {
            mbar_expect_tx(&bars[2], kD * kD * 4);
            bulk_g2s(Rv, a.vc.R, kD * kD * 4, &bars[2]);
        }
    }
    __syncthreads();
    {
        int ml = max(lim0, lim1);
        for (int o = 16; o > 0; o >>= 1) ml = max(ml, __shfl_xor_sync(0xffffffffu, ml, o));
        if (lane == 0) atomicMax(s_lim, ml);
    }
    __syncthreads();
    const int kend = bad ? 0 : min(*s_lim + 1, N);
    const int ntiles = kend > 0 ? (kend + TT - 1) / TT : 0;

    uint32_t qa[8][4], qj[8][4];
    {
        const uint4* qf = P.qfrag + static_cast<int64_t>(active ? unit : 0) * 2 * 8 * 32;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            const uint4 v = active ? qf[ks * 32 + lane] : make_uint4(0, 0, 0, 0);
            const uint4 w = active ? qf[(8 + ks) * 32 + lane] : make_uint4(0, 0, 0, 0);
            qa[ks][0] = v.x; qa[ks][1] = v.y; qa[ks][2] = v.z; qa[ks][3] = v.w;
            qj[ks][0] = w.x; qj[ks][1] = w.y; qj[ks][2] = w.z; qj[ks][3] = w.w;
        }
    }
    const auto ktab = mse_table<KB>(a.kc.c);
    typename MseTable<VGROUP ? 2 : VB>::type vtab{};
    if constexpr (!VGROUP) vtab = mse_table<VB>(a.vc.c);

    // records are shared by all query blocks of a KV head: default L2 policy
    auto issue = [&](int i) {
        const int t0 = i * TT;
        const int lb = t0 / BT;
        const int slot0 = t0 - lb * BT;
        int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(b) * a.max_blocks + lb])
                             : static_cast<int64_t>(b) * a.max_blocks + lb;
        if (pb < 0 || pb >= a.pool.num_blocks) pb = 0;  // flagged and masked when decoded
        const char* base = a.pool.base + (pb * Hkv + h) * a.pool.sub_bytes;
        unsigned char* dst = smem + static_cast<size_t>(i & 1) * st.bytes;
        uint64_t* bar = &bars[i & 1];
        unsigned total = 0;
        for (int k = 0; k < 7; ++k)
            if (st.off[k] >= 0) total += TT * st.field[k];
        mbar_expect_tx(bar, total);
        for (int k = 0; k < 7; ++k)
            if (st.off[k] >= 0)
                bulk_g2s(dst + st.off[k], base + a.pool.off[k] + static_cast<int64_t>(slot0) * st.field[k],
                         TT * st.field[k], bar);
    };
    if (tid == 0 && ntiles > 0) issue(0);

    float o[16][4];
#pragma unroll
    for (int p = 0; p < 16; ++p) o[p][0] = o[p][1] = o[p][2] = o[p][3] = 0.0f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.0f, l1 = 0.0f;
    bool failed = false;
    int waited = 0;

    for (int i = 0; i < ntiles; ++i) {
        if (tid == 0 && i + 1 < ntiles) issue(i + 1);   // its stage was consumed in iteration i - 1
        const bool ok = mbar_wait(&bars[i & 1], (i >> 1) & 1);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        waited = i + 1;
        const unsigned char* sp = smem + static_cast<size_t>(i & 1) * st.bytes;
        const int t0 = i * TT;
        int valid = min(TT, kend - t0);
        {
            const int lb = t0 / BT;
            const int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(b) * a.max_blocks + lb])
                                       : static_cast<int64_t>(b) * a.max_blocks + lb;
            if (pb < 0 || pb >= a.pool.num_blocks) {
                if (tid == 0) atomicOr(a.err, TQ_DEVERR_BLOCK);
                valid = 0;
            }
        }

        // ---------------- decode the tile once: thread -> (token, 32-coordinate quarter)
        {
            const int tok = tid >> 2, qt = tid & 3;
            uint32_t* krow = reinterpret_cast<uint32_t*>(Kop + tok * kOpStride);
            uint32_t* srow = reinterpret_cast<uint32_t*>(Sop + tok * kOpStride);
            __half* vrow = Vop + tok * kOpStride;
            if (tok < TT && tok < valid) {
                const uint32_t* kidx = reinterpret_cast<const uint32_t*>(sp + st.off[0]);
                uint32_t kw[KB], hk[16];
                load_words<KB>(kidx + tok * (4 * KB) + qt * KB, kw);
                mse_chunk<KB>(kw, ktab, hk);
#pragma unroll
                for (int ks = 0; ks < 8; ++ks) {
                    krow[8 * ks + qt] = hk[2 * ks];          // halves 16ks + 2qt
                    krow[8 * ks + 4 + qt] = hk[2 * ks + 1];  // halves 16ks + 8 + 2qt
                }
                if constexpr (KPROD) {
                    const uint32_t sw = reinterpret_cast<const uint32_t*>(sp + st.off[1])[tok * 4 + qt];
                    const uint32_t hg = h_bits(-reinterpret_cast<const float*>(sp + st.off[3])[tok]);
                    const uint32_t neg2 = hg | (hg << 16);
#pragma unroll
                    for (int ks = 0; ks < 8; ++ks) {
                        srow[8 * ks + qt] = dec1(sw, 15 - ks, neg2);
                        srow[8 * ks + 4 + qt] = dec1(sw, 7 - ks, neg2);
                    }
                }
                const uint32_t* vidx = reinterpret_cast<const uint32_t*>(sp + st.off[4]);
                uint32_t vw[VB], hv[16];
                load_words<VB>(vidx + tok * (4 * VB) + qt * VB, vw);
                if constexpr (VGROUP) {
                    const int ng = kD / a.vc.group;
                    const int gi = (32 * qt) / a.vc.group;
                    const float sc = __half2float(reinterpret_cast<const __half*>(sp + st.off[5])[tok * ng + gi]);
                    const float mn = __half2float(reinterpret_cast<const __half*>(sp + st.off[6])[tok * ng + gi]);
                    GroupChunk<VB>::run(vw, pack_half2(sc * (VB == 4 ? 16.0f : 4.0f), sc * (VB == 4 ? 16.0f : 4.0f)),
                                        pack_half2(mn, mn), hv);
#pragma unroll
                    for (int p = 0; p < 16; ++p) {
                        int pa, pb;
                        group_pair(VB, p, pa, pb);
                        vrow[32 * qt + pa] = __ushort_as_half(static_cast<unsigned short>(hv[p] & 0xFFFFu));
                        vrow[32 * qt + pb] = __ushort_as_half(static_cast<unsigned short>(hv[p] >> 16));
                    }
                } else {
                    mse_chunk<VB>(vw, vtab, hv);
#pragma unroll
                    for (int p = 0; p < 16; ++p) {
                        int pa, pb;
                        mse_pair(VB, p, pa, pb);
                        vrow[32 * qt + pa] = __ushort_as_half(static_cast<unsigned short>(hv[p] & 0xFFFFu));
                        vrow[32 * qt + pb] = __ushort_as_half(static_cast<unsigned short>(hv[p] >> 16));
                    }
                }
                if (qt == 0) {
                    kn[tok] = reinterpret_cast<const float*>(sp + st.off[2])[tok];
                    vn[tok] = VGROUP ? 1.0f : reinterpret_cast<const float*>(sp + st.off[5])[tok];
                }
            } else if (tok < kPTok) {
                // rows the scores mask out still meet P = 0 in P.V: keep them finite
#pragma unroll
                for (int q = 0; q < 16; ++q) {
                    krow[4 * q + qt] = 0u;
                    srow[4 * q + qt] = 0u;
                    reinterpret_cast<uint32_t*>(vrow)[4 * q + qt] = 0u;
                }
                if (qt == 0) {
                    kn[tok] = 0.0f;
                    vn[tok] = 0.0f;
                }
            }
        }
        __syncthreads();

        if (active) {
            // ---------------- scores of the warp's 16 rows against the tile
            float sc[8][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.0f;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
                for (int nt = 0; nt < 8; ++nt) {
                    if (8 * nt < TT) {
                        const uint32_t* kr = reinterpret_cast<const uint32_t*>(Kop + (8 * nt + g) * kOpStride);
                        const uint32_t b0 = kr[8 * ks + j], b1 = kr[8 * ks + 4 + j];
                        mma16816(sc[nt], qa[ks], b0, b1);
                        if constexpr (KPROD) {
                            const uint32_t* sr = reinterpret_cast<const uint32_t*>(Sop + (8 * nt + g) * kOpStride);
                            mma16816(sc[nt], qj[ks], sr[8 * ks + j], sr[8 * ks + 4 + j]);
                        } else {
                            mma16816(sc[nt], qj[ks], b0, b1);
                        }
                    }
                }
            }
            // scale by the key norm, mask, online softmax (log2 domain)
            float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                if (8 * nt < TT) {
                    const int tl = 8 * nt + 2 * j;
                    const int pos = t0 + tl;
                    const float k0 = kn[tl], k1 = kn[tl + 1];
                    sc[nt][0] = (tl < valid && pos <= lim0) ? sc[nt][0] * k0 : -INFINITY;
                    sc[nt][1] = (tl + 1 < valid && pos + 1 <= lim0) ? sc[nt][1] * k1 : -INFINITY;
                    sc[nt][2] = (tl < valid && pos <= lim1) ? sc[nt][2] * k0 : -INFINITY;
                    sc[nt][3] = (tl + 1 < valid && pos + 1 <= lim1) ? sc[nt][3] * k1 : -INFINITY;
                    mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
                    mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
                }
            }
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            if (__any_sync(0xffffffffu, mn0 != m0 || mn1 != m1)) {
                const float al0 = mn0 == -INFINITY ? 1.0f : ex2(m0 - mn0);
                const float al1 = mn1 == -INFINITY ? 1.0f : ex2(m1 - mn1);
                l0 *= al0;
                l1 *= al1;
#pragma unroll
                for (int p = 0; p < 16; ++p) {
                    o[p][0] *= al0; o[p][1] *= al0;
                    o[p][2] *= al1; o[p][3] *= al1;
                }
                m0 = mn0;
                m1 = mn1;
            }
            // P' = fp16(p * value norm) as A fragments; row sums from the rounded
            // weights divided back (a zero-norm value contributes p directly)
            uint32_t pa[4][4];
#pragma unroll
            for (int nt = 0; nt < 8; ++nt) {
                if (8 * nt < TT) {
                    const int tl = 8 * nt + 2 * j;
                    const float v0 = vn[tl], v1 = vn[tl + 1];
                    const float p0 = m0 == -INFINITY ? 0.0f : ex2(sc[nt][0] - m0);
                    const float p1 = m0 == -INFINITY ? 0.0f : ex2(sc[nt][1] - m0);
                    const float p2 = m1 == -INFINITY ? 0.0f : ex2(sc[nt][2] - m1);
                    const float p3 = m1 == -INFINITY ? 0.0f : ex2(sc[nt][3] - m1);
                    const bool z0 = !(v0 > 0.0f), z1 = !(v1 > 0.0f);
                    const uint32_t w01 = pack_half2(z0 ? 0.0f : p0 * v0, z1 ? 0.0f : p1 * v1);
                    const uint32_t w23 = pack_half2(z0 ? 0.0f : p2 * v0, z1 ? 0.0f : p3 * v1);
                    const float2 f01 = __half22float2(*reinterpret_cast<const __half2*>(&w01));
                    const float2 f23 = __half22float2(*reinterpret_cast<const __half2*>(&w23));
                    l0 += (z0 ? p0 : f01.x * __fdividef(1.0f, v0)) + (z1 ? p1 : f01.y * __fdividef(1.0f, v1));
                    l1 += (z0 ? p2 : f23.x * __fdividef(1.0f, v0)) + (z1 ? p3 : f23.y * __fdividef(1.0f, v1));
                    pa[nt >> 1][(nt & 1) * 2] = w01;
                    pa[nt >> 1][(nt & 1) * 2 + 1] = w23;
                }
            }
            // ---------------- P' . V on the tile: B fragments by transposing loads
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                if (16 * kk < TT) {
                    const int mi = lane >> 3, rr = lane & 7;
                    const __half* base = Vop + (16 * kk + (mi & 1) * 8 + rr) * kOpStride + (mi >> 1) * 8;
#pragma unroll
                    for (int dn = 0; dn < 8; ++dn) {
                        uint32_t v0, v1, v2, v3;
                        ldsm_x4_trans(v0, v1, v2, v3, base + 16 * dn);
                        mma16816(o[2 * dn], pa[kk], v0, v1);
                        mma16816(o[2 * dn + 1], pa[kk], v2, v3);
                    }
                }
            }
        }
        __syncthreads();  // the tile's operands and its ring stage are free again
    }
    if (failed) {
        if (tid == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
        const int issued = min(ntiles, waited + 2);
        for (int i = waited; i < issued; ++i) (void)mbar_wait(&bars[i & 1], (i >> 1) & 1);
    }
    bool rv_ok = true;
    if constexpr (!VGROUP) rv_ok = mbar_wait(&bars[2], 0);
    if (__syncthreads_or(!rv_ok)) {
        if (tid == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
        (void)mbar_wait(&bars[2], 0);
    }

    // ---------------- rows: o / l in shared memory (over the ring and operands)
    float* orot = reinterpret_cast<float*>(smem);   // [kPWarps][16][kD]
    if (active) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
        const float i0 = l0 > 0.0f ? 1.0f / l0 : 0.0f, i1 = l1 > 0.0f ? 1.0f / l1 : 0.0f;
        float* w0 = orot + (warp * kRows + g) * kD;
        float* w1 = w0 + 8 * kD;
#pragma unroll
        for (int dn = 0; dn < 16; ++dn) {
            w0[8 * dn + 2 * j] = o[dn][0] * i0;
            w0[8 * dn + 2 * j + 1] = o[dn][1] * i0;
            w1[8 * dn + 2 * j] = o[dn][2] * i1;
            w1[8 * dn + 2 * j + 1] = o[dn][3] * i1;
        }
    }
    __syncthreads();
    // output rows: MSE values rotated back (x = o_rot @ R_v), group values as they are
    for (int e = tid; e < kPWarps * kRows * (kD / 8); e += kPThreads) {
        const int wr = e / (kRows * (kD / 8));
        const int rr = (e / (kD / 8)) % kRows;
        const int d0 = 8 * (e % (kD / 8));
        const int rgw = blockIdx.x + wr * gridDim.x;
        const int row = rgw * kRows + rr;
        if (rgw >= RG || row >= a.plan.rows) continue;
        const float* orow = orot + (wr * kRows + rr) * kD;
        float res[8];
        if constexpr (!VGROUP) {
#pragma unroll
            for (int k = 0; k < 8; ++k) res[k] = 0.0f;
            for (int i2 = 0; i2 < kD; ++i2) {
                const float ov = orow[i2];
                const float4 ra = *reinterpret_cast<const float4*>(Rv + i2 * kD + d0);
                const float4 rb = *reinterpret_cast<const float4*>(Rv + i2 * kD + d0 + 4);
                res[0] = fmaf(ov, ra.x, res[0]); res[1] = fmaf(ov, ra.y, res[1]);
                res[2] = fmaf(ov, ra.z, res[2]); res[3] = fmaf(ov, ra.w, res[3]);
                res[4] = fmaf(ov, rb.x, res[4]); res[5] = fmaf(ov, rb.y, res[5]);
                res[6] = fmaf(ov, rb.z, res[6]); res[7] = fmaf(ov, rb.w, res[7]);
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) res[k] = orow[d0 + k];
        }
        const int gq = row / a.Lq, l = row % a.Lq;
        float* dst = a.out + ((static_cast<int64_t>(b) * a.Hq + h * a.G + gq) * a.Lq + l) * kD + d0;
        reinterpret_cast<float4*>(dst)[0] = make_float4(res[0], res[1], res[2], res[3]);
        reinterpret_cast<float4*>(dst)[1] = make_float4(res[4], res[5], res[6], res[7]);
    }
    if (tid == 0)
        for (int s = 0; s < 3; ++s) mbar_inval(&bars[s]);
}

template <int KB, bool KPROD, bool VGROUP, int VB>
cudaError_t launch_prefill_t(const PrefillArgs& P, size_t smem, cudaStream_t s) {
    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel<KB, KPROD, VGROUP, VB>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(qfrag_kernel<KB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     static_cast<int>(sizeof(QSmem)));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        attr_set.fetch_or(bit);
    }
    const DecodeArgs& a = P.a;
    const int RG = a.plan.row_groups;
    MmaArgs m{};
    m.a = a;
    m.qfrag = P.qfrag;
    m.cnt = nullptr;
    qfrag_kernel<KB><<<dim3(a.batch * a.pool.Hkv, RG), kQThreads, sizeof(QSmem), s>>>(m);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const int gx = (RG + kPWarps - 1) / kPWarps;
    prefill_kernel<KB, KPROD, VGROUP, VB><<<dim3(gx, a.pool.Hkv, a.batch), kPThreads, smem, s>>>(P);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
}

}  // namespace

// Codec combinations built for prefill attention.
bool prefill_supported(int kb, bool kprod, bool vgroup, int vb) {
    if (kprod && kb == 2 && !vgroup && (vb == 3 || vb == 4)) return true;
    if (kprod && kb == 2 && vgroup && vb == 4) return true;
    if (!kprod && kb == 4 && !vgroup && vb == 4) return true;
    return false;
}

cudaError_t launch_prefill(const DecodeArgs& a, const uint4* qfrag, cudaStream_t s) {
    const DecodePlan& p = a.plan;
    PrefillArgs P{};
    P.a = a;
    P.qfrag = qfrag;
    P.st.tt = p.tile;
    P.st.bytes = p.st_bytes;
    for (int k = 0; k < 7; ++k) {
        P.st.off[k] = p.st_off[k];
        P.st.field[k] = p.st_field[k];
    }
    const size_t ring = 2 * static_cast<size_t>(p.st_bytes);
    const size_t ops = 3 * static_cast<size_t>(kPTok) * kOpStride * 2;
    const size_t orot = static_cast<size_t>(kPWarps) * kRows * kD * 4;
    size_t off = ring + ops;
    if (off < orot) off = orot;  // the output rows reuse the ring and operand tiles
    P.op_off = static_cast<int>(ring);
    P.norm_off = static_cast<int>((off + 15) / 16 * 16);
    P.rv_off = P.norm_off + 2 * kPTok * 4;
    P.bar_off = P.rv_off + kD * kD * 4;
    const size_t smem = static_cast<size_t>(P.bar_off) + 32;
    if (p.kprod && p.kb == 2 && !p.vgroup && p.vb == 3) return launch_prefill_t<2, true, false, 3>(P, smem, s);
    if (p.kprod && p.kb == 2 && !p.vgroup && p.vb == 4) return launch_prefill_t<2, true, false, 4>(P, smem, s);
    if (p.kprod && p.kb == 2 && p.vgroup && p.vb == 4) return launch_prefill_t<2, true, true, 4>(P, smem, s);
    if (!p.kprod && p.kb == 4 && !p.vgroup && p.vb == 4) return launch_prefill_t<4, false, false, 4>(P, smem, s);
    return cudaErrorInvalidValue;
}

}  // namespace mmadec
}  // namespace tq

// Prefill attention over the compressed cache on the 5th-generation tensor
// cores (tcgen05.mma, TMEM accumulators), head_dim 128.
//
// The function is the decode attention's for any query length: a chunk of
// q_len positions, already appended, attends to its sequence's compressed
// prefix and causally to itself (query l sees keys t <= N - q_len + l). One
// CTA owns 128 query rows (8 groups of 16) of one KV head -- TMEM lane = row,
// four threads per row (column quarters of its scores and output) -- and walks
// the key/value tiles its rows can see; each tile is fetched once (1-D bulk
// copies, double-buffered) and decoded once for all 128 rows. Per 64-token
// tile:
//   decode   the CTA decodes the tile once (one token and 32-coordinate
//            quarter per thread; half the threads take the keys and signs,
//            half the values) into shared-memory operands in the canonical
//            no-swizzle K-major layout: key levels c_k[idx] and +-rnorm signs
//            (64 tokens x 128, decoder pair p of quarter q at position
//            32q + 2p, the query operands permuted to match), values in the
//            same pair order, then transposed 8x8 block by 8x8 block
//            (ldmatrix.trans + stmatrix) into V^T (128 columns x 64 tokens);
//   scores   S = Q' K^T (+ Q'' sigma^T) as tcgen05.mma M 128, N 64, K 16 into 64
//            TMEM columns;
//   softmax  each thread reads its quarter row of S (tcgen05.ld), scales by
//            the key norms, masks, exchanges the row maximum with the row's
//            other threads,
//            keeps a running row maximum that only moves when the tile maximum
//            exceeds it by 8 (log2 units: weights stay <= 2^8 and the output
//            accumulator is rescaled rarely), writes its quarter row of
//            P' = p * value norm (fp16) as the K-major A operand;
//   values   O += P' V as tcgen05.mma M 128, N 128, K 16 into 128 TMEM columns,
//            running while the next tile is decoded (its V^T and P' are
//            written only after this MMA has completed).
// At the end the four threads of a row read its row of O, divide by the row
// sum and apply the inverse value rotation from a shared-memory copy of R_v.
// Query fragments come from the decode path's query-prep kernel (workspace).
#include <climits>

#include "decode_mma_impl.cuh"
#include "tc_ptx.cuh"

namespace tq {
namespace mmadec {
namespace {

constexpr int kTRows = 128;       // query rows per CTA = MMA M = TMEM lanes
constexpr int kTSplit = 4;        // threads per row: column quarters of its scores and output
constexpr int kTCompute = kTRows * kTSplit;   // the decode and softmax warps
constexpr int kTThreads = kTCompute + 64;     // plus a warp that issues the MMAs and one for the copies
constexpr int kCtlWarp = kTCompute / 32, kLoadWarp = kCtlWarp + 1;
constexpr int kBarCompute = 1;    // named barrier of the compute warps
constexpr int kTTok = 64;         // tokens per tile
constexpr int kVStride = kD + 8;  // halves per row of the row-major value scratch
constexpr float kRescaleGap = 8.0f;
// per-tile stash: key norms, value weights [64] floats each, 1/weight hi and
// lo [64] fp16 each, then whether a weight of each half tile exceeds 256 [2]
constexpr int kStashBytes = 2 * kTTok * 4 + 2 * kTTok * 2 + 16;
// TMEM columns: output [O | row sums] (144), scores of even and odd tiles (64
// each), P' (32 of fp16 pairs), the query operands Q' and Q'' (64 each, fp16 pairs)
constexpr uint32_t kColO = 0, kColS1 = 192, kColS0 = 256, kColP = 320, kColQa = 384, kColQj = 448;

struct TcPrefillArgs {
    DecodeArgs a;
    StageLayout st;               // record streams of one tile
    const uint4* qfrag;           // [unit][2][8][32] uint4 (query-prep output)
    int k_off[2], s_off[2];       // key levels and sign operands of even / odd tiles: 64 x 128 fp16
    int vt_off[2];                // V^T operands: 144 x 64 fp16 (value rows, 1/weight hi and lo, zero rows)
    int vs_off[2];                // value scratch [64][kVStride] fp16
    int norm_off;                 // three stashes: key norms, value weights [2][64] floats; 1/weight [2][64] fp16
    int sx_off;                   // row-maximum exchange [2][kTSplit][128] floats
    int orow_off;                 // output staging [128][kD + 1] floats (over the operands, after the last tile)
    int rv_off;                   // R_v [kD][kD] floats (MSE values only)
    int bar_off;                  // mbarriers (7); then the TMEM slot, the row limits and the consumed-tile count
};

// Byte offset of (row, k) in a K-major operand whose K extent is KX.
template <int KX>
__device__ __forceinline__ int kmaj(int row, int k) {
    return ((row >> 3) * (KX / 8) + (k >> 3)) * 128 + (row & 7) * 16 + (k & 7) * 2;
}

template <int KB, bool KPROD, bool VGROUP, int VB>
__global__ void __launch_bounds__(kTThreads, 1) prefill_tc_kernel(TcPrefillArgs P) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const DecodeArgs& a = P.a;
    const StageLayout& st = P.st;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const bool ctl = warp == kCtlWarp, loader = warp == kLoadWarp;
    const int Hkv = a.pool.Hkv, RG = a.plan.row_groups, BT = a.pool.BT, TT = st.tt;
    const int h = blockIdx.y, b = blockIdx.z;
    // mbarriers: [0,1] tile records, [2] scores done, [3] R_v, [4] P' written by
    // the 16 compute warps, [5] output MMA done, [6] operands written by the 16 compute warps
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + P.bar_off);
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 7);
    int* s_lim = reinterpret_cast<int*>(s_tmem + 1);                    // largest and smallest row limit
    int* s_consumed = s_lim + 2;   // tiles whose records every compute warp has decoded (control -> loader)
    float* Rv = reinterpret_cast<float*>(smem + P.rv_off);
    const uint32_t sbase = tc::smem_addr(smem);
    // per-tile values, three deep (tile t in stash t % 3: a warp may be a
    // tile's decode ahead of another's softmax): key norms, value weights,
    // 1/weight as fp16 hi, lo
    auto stash_kn = [&](int t) { return reinterpret_cast<float*>(smem + P.norm_off + (t % 3) * kStashBytes); };
    auto s_x = [&](int t) { return reinterpret_cast<float*>(smem + P.sx_off) + (t & 1) * kTSplit * kTRows; };

    // a compute thread's row (its warp's TMEM lane quarter) and column quarter
    const int row = 32 * (warp & 3) + lane, cq = (warp >> 2) & 3;
    const int w8 = row >> 4;                        // row group slot of the CTA
    // row blocks in reverse launch order: the later query positions see more
    // keys, so the longest CTAs start first and the last wave holds short ones
    const int bx = gridDim.x - 1 - blockIdx.x;
    const int rg = bx + w8 * gridDim.x;
    const int r = rg * kRows + (row & 15);
    const bool compute = warp < kCtlWarp;
    const bool row_ok = compute && rg < RG && r < a.plan.rows;
    const int N = a.seq_lens[b];
    const bool bad = N < a.Lq || N > a.max_blocks * BT;
    if (bad && tid == 0 && blockIdx.x == 0 && h == 0) atomicOr(a.err, TQ_DEVERR_SEQLEN);
    const int lim = row_ok ? N - a.Lq + (r % a.Lq) : -1;

    if (warp == 0) {
        tc::tmem_alloc(s_tmem, 512);
        tc::tmem_relinquish();
    }
    if (tid == 0) {
        s_lim[0] = -1;
        s_lim[1] = INT_MAX;
        *s_consumed = 0;
        for (int s = 0; s < 4; ++s) tc::mbar_init(&bars[s], 1);
        tc::mbar_init(&bars[4], kTCompute / 32);
        tc::mbar_init(&bars[5], 1);
        tc::mbar_init(&bars[6], kTCompute / 32);
        tc::mbar_fence_init();
        if constexpr (!VGROUP) {
            tc::mbar_expect_tx(&bars[3], kD * kD * 4);
            tc::bulk_g2s(Rv, a.vc.R, kD * kD * 4, &bars[3]);
        }
    }
    // rows kD and kD+1 of the value operands hold 1 / weight (fp16 hi, lo) per
    // token, so that their output columns accumulate the row sum of P' / weight;
    // rows kD+2..kD+15 stay zero
    for (int e = tid; e < 2 * 16 * (kTTok / 8); e += kTThreads) {
        const int bi = e >> 7, n = kD + ((e >> 3) & 15), kc = e & 7;
        *reinterpret_cast<uint4*>(smem + P.vt_off[bi] + kmaj<kTTok>(n, 8 * kc)) = make_uint4(0u, 0u, 0u, 0u);
    }
    tc::fence_proxy_async_smem();
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    if (compute) {
        atomicMax(&s_lim[0], lim);
        if (row_ok) atomicMin(&s_lim[1], lim);
    }
    const uint32_t tmem = *s_tmem;
    const uint32_t t_row = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
    constexpr int HC = kTTok / kTSplit, OC = kD / kTSplit;   // score and output columns per thread
    const uint32_t tO = t_row + kColO + OC * cq, tL = t_row + kColO + kD;
    // the query operands of this thread's row into TMEM: coordinate quarter cq
    // (pairs p of the query fragments, column 16 cq + p) of Q' and of Q''
    if (compute) {
        const int rgs = bx + w8 * gridDim.x;
        const uint32_t* qf = reinterpret_cast<const uint32_t*>(P.qfrag) +
                             static_cast<int64_t>((b * Hkv + h) * RG + rgs) * 2048;
        const int ln = 4 * (row & 7) + cq, rbit = (row >> 3) & 1;
        uint32_t qa[16], qj[16];
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            const int x = (p >> 1) * 128 + ln * 4 + rbit + 2 * (p & 1);   // fragment (ks, lane, reg)
            qa[p] = rgs < RG ? qf[x] : 0u;
            qj[p] = rgs < RG ? qf[1024 + x] : 0u;
        }
        tc::tmem_st16u(t_row + kColQa + 16 * cq, qa);
        tc::tmem_st16u(t_row + kColQj + 16 * cq, qj);
    }
    tc::tc_fence_before();
    __syncthreads();
    tc::tc_fence_after();
    const int kend = bad ? 0 : min(s_lim[0] + 1, N);
    const int minlim = s_lim[1];   // tiles ending at or below it are visible to every valid row
    const int ntiles = kend > 0 ? (kend + TT - 1) / TT : 0;

    bool failed = false, o_started = false;
    if (loader) {
        // ---------------- the load thread: tile records into the two ring stages;
        // tile j + 2 goes into tile j's stage once every compute warp has decoded it
        if (lane == 0) {
            auto issue = [&](int i) {
                const int t0 = i * TT;
                const int lb = t0 / BT;
                const int slot0 = t0 - lb * BT;
                int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(b) * a.max_blocks + lb])
                                     : static_cast<int64_t>(b) * a.max_blocks + lb;
                if (pb < 0 || pb >= a.pool.num_blocks) pb = 0;   // flagged and masked by the compute warps
                const char* base = a.pool.base + (pb * Hkv + h) * a.pool.sub_bytes;
                unsigned char* dst = smem + static_cast<size_t>(i & 1) * st.bytes;
                unsigned total = 0;
                for (int k = 0; k < 7; ++k)
                    if (st.off[k] >= 0) total += TT * st.field[k];
                tc::mbar_expect_tx(&bars[i & 1], total);
                for (int k = 0; k < 7; ++k)
                    if (st.off[k] >= 0)
                        tc::bulk_g2s(dst + st.off[k],
                                     base + a.pool.off[k] + static_cast<int64_t>(slot0) * st.field[k],
                                     TT * st.field[k], &bars[i & 1]);
            };
            int issued = 0;
            bool ok = true;
            for (; issued < 2 && issued < ntiles; ++issued) issue(issued);
            while (issued < ntiles) {
                unsigned it = 0;
                while (tc::ld_acquire(s_consumed) < issued - 1 && ++it < tc::kSpinLimit) __nanosleep(32);
                if (it >= tc::kSpinLimit) {
                    ok = false;
                    break;
                }
                issue(issued++);
            }
            if (!ok) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
            // drain the last copies (after a timeout elsewhere they may not have been waited for)
            for (int t = issued > 2 ? issued - 2 : 0; t < issued; ++t) (void)tc::mbar_wait(&bars[t & 1], (t >> 1) & 1);
        }
        __syncwarp();
    } else if (ctl) {
        // ---------------- the control thread: the MMAs. Tile j's scores go to
        // TMEM columns S[j & 1] from the operand buffers j & 1
        if (lane == 0) {
            constexpr uint32_t idS = tc::idesc_f16_f32(kTRows, kTTok);
            constexpr uint32_t idO = tc::idesc_f16_f32(kTRows, kD + 16);
            // descriptor words of the operand buffers; a 256-byte step of the start
            // address adds 16 to the low word
            auto lo_of = [&](int off, int lbo) {
                return static_cast<uint32_t>(tc::smem_desc(sbase + off, lbo, 0) & 0xFFFFFFFFu);
            };
            const uint32_t hiK = static_cast<uint32_t>(tc::smem_desc(0, 0, 2048) >> 32);
            const uint32_t hiV = static_cast<uint32_t>(tc::smem_desc(0, 0, 1024) >> 32);
            const uint32_t loK0 = lo_of(P.k_off[0], 128), loK1 = lo_of(P.k_off[1], 128);
            const uint32_t loS0 = KPROD ? lo_of(P.s_off[0], 128) : loK0;
            const uint32_t loS1 = KPROD ? lo_of(P.s_off[1], 128) : loK1;
            const uint32_t loV0 = lo_of(P.vt_off[0], 128), loV1 = lo_of(P.vt_off[1], 128);
            bool ok = true;
            int s_commits = 0, o_commits = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int bj = j & 1;
                ok = tc::mbar_wait(&bars[6], j & 1);   // tile j's operands are in shared memory
                if (!ok) break;
                tc::st_release(s_consumed, j + 1);    // and its records are free
                tc::tc_fence_after();
                const uint32_t dS = tmem + (bj ? kColS1 : kColS0);
                const uint32_t k0 = bj ? loK1 : loK0, s0 = bj ? loS1 : loS0;
#pragma unroll
                for (int s = 0; s < kD / 16; ++s) {
                    if (s == 0) tc::mma_f16_ta_w<false>(dS, tmem + kColQa, k0, hiK, idS);
                    else tc::mma_f16_ta_w<true>(dS, tmem + kColQa + 8 * s, k0 + 16 * s, hiK, idS);
                    tc::mma_f16_ta_w<true>(dS, tmem + kColQj + 8 * s, s0 + 16 * s, hiK, idS);
                }
                tc::mma_commit(&bars[2]);
                ++s_commits;
                ok = tc::mbar_wait(&bars[4], j & 1);   // P' (and the rescaled O) of tile j are in TMEM
                if (!ok) break;
                tc::tc_fence_after();
                const uint32_t v0 = bj ? loV1 : loV0;
                if (j == 0) tc::mma_f16_ta_w<false>(tmem + kColO, tmem + kColP, v0, hiV, idO);
                else tc::mma_f16_ta_w<true>(tmem + kColO, tmem + kColP, v0, hiV, idO);
#pragma unroll
                for (int s = 1; s < kTTok / 16; ++s)
                    tc::mma_f16_ta_w<true>(tmem + kColO, tmem + kColP + 8 * s, v0 + 16 * s, hiV, idO);
                tc::mma_commit(&bars[5]);
                ++o_commits;
            }
            if (!ok) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
            // drain the last MMAs issued (after a timeout), whose phases are the
            // most recent of their barriers
            if (s_commits) (void)tc::mbar_wait(&bars[2], (s_commits - 1) & 1);
            if (o_commits) (void)tc::mbar_wait(&bars[5], (o_commits - 1) & 1);
        }
        __syncwarp();
    } else {
        const auto ktab = mse_table<KB>(a.kc.cq);
        typename MseTable<VGROUP ? 2 : VB>::type vtab{};
        if constexpr (!VGROUP) vtab = mse_table<VB>(a.vc.cq);
        float m = -INFINITY;

        // ---------------- decode tile t into the operand buffers t & 1: one
        // (token, 32-coordinate quarter) unit per thread, lanes on consecutive
        // tokens; pair p of quarter qt goes to operand position 32 qt + 2p, so each
        // operand row is written as four 16-byte chunks (no bank conflicts).
        // Returns whether the tile's records arrived; `valid` = its valid tokens.
        auto decode_tile = [&](int t, int& valid) -> bool {
            const int bt = t & 1;
            const bool ring_ok = tc::mbar_wait(&bars[bt], (t >> 1) & 1);
            const unsigned char* sp = smem + static_cast<size_t>(bt) * st.bytes;
            const int t0 = t * TT;
            valid = min(TT, kend - t0);
            {
                const int lb = t0 / BT;
                const int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(b) * a.max_blocks + lb])
                                           : static_cast<int64_t>(b) * a.max_blocks + lb;
                if (pb < 0 || pb >= a.pool.num_blocks) {
                    if (tid == 0) atomicOr(a.err, TQ_DEVERR_BLOCK);
                    valid = 0;
                }
            }
            float* kn = stash_kn(t);
            float* vw = kn + kTTok;
            __half* rhi = reinterpret_cast<__half*>(vw + kTTok);
            __half* rlo = rhi + kTTok;
            static_assert(kTTok * 4 * 2 == kTCompute, "one key unit and one value unit per thread pair");
            const bool vside = tid >= kTCompute / 2;   // first half: keys and signs; second: values
            const int wd = warp & 7;
            const int tok = 32 * (wd & 1) + lane, qt = wd >> 1;
            __half* vrow = reinterpret_cast<__half*>(smem + P.vs_off[bt]) + tok * kVStride + 32 * qt;
            auto kchunk = [&](int off, int c) {
                return reinterpret_cast<uint4*>(smem + off + kmaj<kD>(tok, 32 * qt + 8 * c));
            };
            float wt = 0.0f;   // the value thread's weight (0 for a masked token)
            if (tok < valid && !vside) {
                const uint32_t* kidx = reinterpret_cast<const uint32_t*>(sp + st.off[0]);
                uint32_t kw[KB], hk[16];
                load_words<KB>(kidx + tok * (4 * KB) + qt * KB, kw);
                mse_chunk<KB>(kw, ktab, hk);
#pragma unroll
                for (int c = 0; c < 4; ++c) *kchunk(P.k_off[bt], c) = make_uint4(hk[4 * c], hk[4 * c + 1], hk[4 * c + 2], hk[4 * c + 3]);
                if constexpr (KPROD) {
                    const uint32_t sw = reinterpret_cast<const uint32_t*>(sp + st.off[1])[tok * 4 + qt];
                    const uint32_t hg = h_bits(-reinterpret_cast<const float*>(sp + st.off[3])[tok]);
                    const uint32_t neg2 = hg | (hg << 16);
                    uint32_t hs[16];
#pragma unroll
                    for (int k2 = 0; k2 < 8; ++k2) {
                        hs[2 * k2] = dec1(sw, 15 - k2, neg2);
                        hs[2 * k2 + 1] = dec1(sw, 7 - k2, neg2);
                    }
#pragma unroll
                    for (int c = 0; c < 4; ++c) *kchunk(P.s_off[bt], c) = make_uint4(hs[4 * c], hs[4 * c + 1], hs[4 * c + 2], hs[4 * c + 3]);
                }
                if (qt == 0) kn[tok] = reinterpret_cast<const float*>(sp + st.off[2])[tok];
            } else if (tok < valid) {
                const uint32_t* vidx = reinterpret_cast<const uint32_t*>(sp + st.off[4]);
                uint32_t vwd[VB], hv[16];
                load_words<VB>(vidx + tok * (4 * VB) + qt * VB, vwd);
                if constexpr (VGROUP) {
                    const int ng = kD / a.vc.group;
                    const int gi = (32 * qt) / a.vc.group;
                    const float sc = __half2float(reinterpret_cast<const __half*>(sp + st.off[5])[tok * ng + gi]);
                    const float mn = __half2float(reinterpret_cast<const __half*>(sp + st.off[6])[tok * ng + gi]);
                    const float mul = sc * (VB == 4 ? 16.0f : 4.0f);
                    GroupChunk<VB>::run(vwd, pack_half2(mul, mul), pack_half2(mn, mn), hv);
                } else {
                    mse_chunk<VB>(vwd, vtab, hv);
                }
                // P' carries the weight (the value norm; 1 for a zero vector, whose
                // operand row is zero), and rows kD, kD+1 of V^T carry 1 / weight
                wt = 1.0f;
                if constexpr (!VGROUP) {
                    const float nv = reinterpret_cast<const float*>(sp + st.off[5])[tok];
                    if (nv > 0.0f) {
                        wt = nv;
                    } else {
#pragma unroll
                        for (int p = 0; p < 16; ++p) hv[p] = 0u;
                    }
                }
                if (qt == 0) {
                    const float rw = 1.0f / wt;
                    const __half h1 = __float2half_rn(rw);
                    vw[tok] = wt;
                    rhi[tok] = h1;
                    rlo[tok] = __float2half_rn(rw - __half2float(h1));
                }
                // values in pair order; the epilogue maps columns back to coordinates
#pragma unroll
                for (int c = 0; c < 4; ++c)
                    reinterpret_cast<uint4*>(vrow)[c] = make_uint4(hv[4 * c], hv[4 * c + 1], hv[4 * c + 2], hv[4 * c + 3]);
            } else {
                // masked tokens meet P' = 0: keep every operand finite
                const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (vside) {
                        reinterpret_cast<uint4*>(vrow)[c] = z;
                    } else {
                        *kchunk(P.k_off[bt], c) = z;
                        if constexpr (KPROD) *kchunk(P.s_off[bt], c) = z;
                    }
                }
                if (qt == 0) {
                    if (vside) {
                        vw[tok] = 0.0f;
                        rhi[tok] = rlo[tok] = __float2half_rn(0.0f);
                    } else {
                        kn[tok] = 0.0f;
                    }
                }
            }
            if (vside && qt == 0) {   // whole warps: does a weight of these 32 tokens exceed 256?
                const bool big = __any_sync(0xffffffffu, wt > 256.0f);
                if (lane == 0) reinterpret_cast<int*>(rlo + kTTok)[wd & 1] = big;
            }
            return ring_ok;
        };
        // ---------------- tile t's values to V^T (8x8 blocks, four per
        // instruction) and its 1/weight rows; then hand the operands to the
        // control thread. Every warp's decode of tile t precedes this (barrier).
        auto transpose_tile = [&](int t) {
            const int bt = t & 1;
            const __half* vs = reinterpret_cast<const __half*>(smem + P.vs_off[bt]);
            for (int it = warp; it < (kD / 8) * (kTTok / 8) / 4; it += kTCompute / 32) {
                const int mi = lane >> 3, rr = lane & 7;
                const int blk = 4 * it + mi;
                const int db = blk >> 3, tb = blk & 7;
                uint32_t x0, x1, x2, x3;
                tc::ldmatrix_x4_trans(x0, x1, x2, x3, vs + (8 * tb + rr) * kVStride + 8 * db);
                tc::stmatrix_x4(smem + P.vt_off[bt] + kmaj<kTTok>(8 * db + rr, 8 * tb), x0, x1, x2, x3);
            }
            if (tid < 2 * (kTTok / 8)) {   // rows kD (hi) and kD+1 (lo), 8 tokens per chunk
                const __half* rhi = reinterpret_cast<const __half*>(stash_kn(t) + 2 * kTTok);
                const int n = tid >> 3, kc = tid & 7;
                const uint4 v = reinterpret_cast<const uint4*>(n ? rhi + kTTok : rhi)[kc];
                *reinterpret_cast<uint4*>(smem + P.vt_off[bt] + kmaj<kTTok>(kD + n, 8 * kc)) = v;
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[6]);
        };

        // tile i's scores run on the tensor cores while tile i + 1 is decoded;
        // its output MMA while tile i + 1 is transposed and tile i + 2 decoded
        int valid_cur = 0;
        bool late = false;   // a wait that failed after this tile's barrier
        if (ntiles > 0) {
            const bool ok0 = decode_tile(0, valid_cur);
            if (tc::bar_or(kBarCompute, kTCompute, !ok0)) failed = true;
            else transpose_tile(0);
        }
        for (int i = 0; i < ntiles && !failed; ++i) {
            const bool more = i + 1 < ntiles;
            int valid_next = 0;
            const bool ring_ok = more ? decode_tile(i + 1, valid_next) : true;

            // ---------------- softmax of this thread's quarter row (log2 units); the
            // row maximum is exchanged with the row's other threads through shared memory
            const bool s_ok = tc::mbar_wait(&bars[2], i & 1);
            tc::tc_fence_after();
            const float* kn = stash_kn(i);
            const float* vw = kn + kTTok;
            const int t0 = i * TT;
            float sv[HC];
            tc::tmem_ld16(t_row + ((i & 1) ? kColS1 : kColS0) + HC * cq, sv);
            // scores relative to the running maximum, y = s * norm - m, in one fused
            // multiply-add (absolute, m taken as 0, while the row has no maximum yet)
            const bool first = m == -INFINITY;
            const float mneg = first ? 0.0f : -m;
            {
                const float4* k4 = reinterpret_cast<const float4*>(kn + HC * cq);
#pragma unroll
                for (int q = 0; q < HC / 4; ++q) {
                    const float4 n4 = k4[q];
                    sv[4 * q] = fmaf(sv[4 * q], n4.x, mneg);
                    sv[4 * q + 1] = fmaf(sv[4 * q + 1], n4.y, mneg);
                    sv[4 * q + 2] = fmaf(sv[4 * q + 2], n4.z, mneg);
                    sv[4 * q + 3] = fmaf(sv[4 * q + 3], n4.w, mneg);
                }
            }
            // a tile whose 64 operand columns are all valid tokens below every
            // row's causal limit needs no mask (blocks shorter than 64 tokens
            // leave zero columns, which the mask must keep out of the row sums)
            const bool open = valid_cur == kTTok && t0 + kTTok - 1 <= minlim;
            if (!open) {
#pragma unroll
                for (int c = 0; c < HC; ++c) {
                    const int tc_ = HC * cq + c;
                    if (!(tc_ < valid_cur && t0 + tc_ <= lim)) sv[c] = -INFINITY;
                }
            }
            float mx = sv[0];
#pragma unroll
            for (int c = 1; c < HC; ++c) mx = fmaxf(mx, sv[c]);
            float* sx = s_x(i);
            sx[cq * kTRows + row] = mx;
            // every warp has decoded tile i + 1 and published its row maxima
            if (tc::bar_or(kBarCompute, kTCompute, !s_ok || !ring_ok || late)) {
                failed = true;
                break;
            }
#pragma unroll
            for (int o = 1; o < kTSplit; ++o) mx = fmaxf(mx, sx[((cq + o) & (kTSplit - 1)) * kTRows + row]);
            // the previous tile's output MMA reads P' and the V^T buffers of tile i + 1
            if (i > 0) {
                late = !tc::mbar_wait(&bars[5], (i - 1) & 1);
                tc::tc_fence_after();
            }
            // move the running maximum only when this tile exceeds it by the gap
            // (the row's threads take the same decision from the same values)
            // the gap is 8, or less when a value weight of the tile exceeds 256, so
            // that P' = p * weight <= 2^15.8 stays inside fp16
            const int* big = reinterpret_cast<const int*>(reinterpret_cast<const __half*>(vw + kTTok) + 2 * kTTok);
            float gap = kRescaleGap;
            if (big[0] | big[1]) {   // rare: the tile's largest weight
                float wmax = 0.0f;
                for (int t = 0; t < kTTok; ++t) wmax = fmaxf(wmax, vw[t]);
                gap = fminf(kRescaleGap, 15.8f - __log2f(wmax));
            }
            // mx is the row's largest y: relative to m, or absolute for a first row
            const bool move = first ? mx != -INFINITY : mx > gap;
            const float alpha = move ? (first ? 0.0f : ex2(-mx)) : 1.0f;
            // y - sub is the score relative to the new maximum
            const float sub = move ? mx : 0.0f;
            if (move) m = first ? mx : m + mx;
            if (__any_sync(0xffffffffu, move) && o_started) {
                float v[32];
                tc::tmem_ld32(tO, v);
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] *= alpha;
                tc::tmem_st32(tO, v);
                if (cq == 0) {   // the row-sum columns
                    float w[16];
                    tc::tmem_ld16(tL, w);
#pragma unroll
                    for (int e = 0; e < 16; ++e) w[e] *= alpha;
                    tc::tmem_st16(tL, w);
                }
            }
            // P' = fp16(p * weight) into TMEM (the A operand of the output MMA);
            // the rows kD, kD+1 of V^T divide each rounded P' back by its weight
            // for the row sum, so the rounding of P' cancels in O / l
            const float4* w4 = reinterpret_cast<const float4*>(vw + HC * cq);
            const bool steady = __all_sync(0xffffffffu, !move && !first);
            uint32_t pw[HC / 2];
#pragma unroll
            for (int q = 0; q < HC / 4; ++q) {
                const float4 n4 = w4[q];
                const int c = 4 * q;
                float p0, p1, p2, p3;
                if (steady) {   // no row of the warp moved its maximum or starts here
                    p0 = ex2(sv[c]);
                    p1 = ex2(sv[c + 1]);
                    p2 = ex2(sv[c + 2]);
                    p3 = ex2(sv[c + 3]);
                } else {        // a row with no score yet keeps p = 0
                    const bool none = m == -INFINITY;
                    p0 = none ? 0.0f : ex2(sv[c] - sub);
                    p1 = none ? 0.0f : ex2(sv[c + 1] - sub);
                    p2 = none ? 0.0f : ex2(sv[c + 2] - sub);
                    p3 = none ? 0.0f : ex2(sv[c + 3] - sub);
                }
                pw[2 * q] = pack_half2(p0 * n4.x, p1 * n4.y);
                pw[2 * q + 1] = pack_half2(p2 * n4.z, p3 * n4.w);
            }
            tc::tmem_st8u(t_row + kColP + (HC / 2) * cq, pw);
            // hand P' and the rescaled O to the control thread
            tc::tc_fence_before();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(&bars[4]);
            o_started = true;
            if (more) transpose_tile(i + 1);
            valid_cur = valid_next;
        }
        if (!failed && o_started) {
            const bool done = tc::mbar_wait(&bars[5], (ntiles - 1) & 1);
            tc::tc_fence_after();
            if (tc::bar_or(kBarCompute, kTCompute, !done || late)) failed = true;
        }
        if (failed && tid == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
    }
    tc::tc_fence_before();
    __syncthreads();   // the control thread has drained every copy and MMA
    tc::tc_fence_after();

    // ---------------- output rows: O / l staged in shared memory (over the
    // operand buffers, idle now), then rotated back by R_v, each thread writing
    // its quarter of the row's dimensions
    failed = __syncthreads_or(failed);
    float* orow = reinterpret_cast<float*>(smem + P.orow_off) + row * (kD + 1);
    if (compute) {
        float l = 0.0f;
        if (o_started && !failed) {
            float w[16];
            tc::tmem_ld16(tL, w);
            l = w[0] + w[1];
        }
        // MSE values were multiplied as fp16(op_scale * level): divide op_scale out
        const float vs = VGROUP ? 1.0f : a.vc.cq_scale;
        const float inv = (o_started && !failed && l > 0.0f) ? 1.0f / (l * vs) : 0.0f;
        float v[32];
        tc::tmem_ld32(tO, v);
        // column 32 qt + 2p + odd holds coordinate 32 qt + (odd ? b : a) of value pair p
        const int qbase = OC * cq;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            int pa, pb;
            if constexpr (VGROUP) group_pair(VB, e >> 1, pa, pb);
            else mse_pair(VB, e >> 1, pa, pb);
            orow[qbase + ((e & 1) ? pb : pa)] = (o_started && !failed) ? v[e] * inv : 0.0f;  // TMEM unwritten otherwise
        }
    }
    bool rv_ok = true;
    if constexpr (!VGROUP) rv_ok = tc::mbar_wait(&bars[3], 0);
    if (__syncthreads_or(!rv_ok) && tid == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
    if (row_ok) {
        const int gq = r / a.Lq, lq = r % a.Lq;
        float* dst = a.out + ((static_cast<int64_t>(b) * a.Hq + h * a.G + gq) * a.Lq + lq) * kD;
        const int d0 = OC * cq;
        float acc[32];
        if constexpr (VGROUP) {
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = orow[d0 + e];
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) acc[e] = 0.0f;
#pragma unroll 2
            for (int i2 = 0; i2 < kD; ++i2) {
                const float ov = orow[i2];
                const float4* rr = reinterpret_cast<const float4*>(Rv + i2 * kD + d0);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 r4 = rr[q];
                    acc[4 * q] = fmaf(ov, r4.x, acc[4 * q]);
                    acc[4 * q + 1] = fmaf(ov, r4.y, acc[4 * q + 1]);
                    acc[4 * q + 2] = fmaf(ov, r4.z, acc[4 * q + 2]);
                    acc[4 * q + 3] = fmaf(ov, r4.w, acc[4 * q + 3]);
                }
            }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q)
            *reinterpret_cast<float4*>(dst + d0 + 4 * q) =
                make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
    }
    tc::tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc::tc_fence_after();
        tc::tmem_dealloc(tmem, 512);
    }
    if (tid == 0)
        for (int s = 0; s < 7; ++s) tc::mbar_inval(&bars[s]);
}

template <int KB, bool KPROD, bool VGROUP, int VB>
cudaError_t launch_prefill_tc_t(const TcPrefillArgs& P, size_t smem, cudaStream_t s) {
    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(prefill_tc_kernel<KB, KPROD, VGROUP, VB>,
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
    qfrag_kernel<KB><<<dim3(qfrag_grid(a.batch * a.pool.Hkv * RG)), kQThreads, sizeof(QSmem), s>>>(m);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const int gx = (RG + 7) / 8;
    prefill_tc_kernel<KB, KPROD, VGROUP, VB><<<dim3(gx, a.pool.Hkv, a.batch), kTThreads, smem, s>>>(P);
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
    TcPrefillArgs P{};
    P.a = a;
    P.qfrag = qfrag;
    // a stage holds one tile of one block: the decode plan's tile, or the
    // block when blocks are shorter (the decode gathers several short blocks
    // into one stage; this kernel copies one block per stage)
    const int TT = p.tile > a.pool.BT ? a.pool.BT : p.tile;
    P.st.tt = TT;
    int so = 0;
    for (int k = 0; k < 7; ++k) {
        P.st.field[k] = p.st_field[k];
        P.st.off[k] = p.st_off[k] >= 0 ? so : -1;
        if (p.st_off[k] >= 0) so += TT * p.st_field[k];
    }
    P.st.bytes = (so + 127) / 128 * 128;
    int off = 2 * P.st.bytes;
    off = (off + 1023) / 1024 * 1024;
    const int ops_begin = off;
    for (int i = 0; i < 2; ++i) { P.k_off[i] = off; off += kTTok * kD * 2; }
    for (int i = 0; i < 2; ++i) { P.s_off[i] = off; off += p.kprod ? kTTok * kD * 2 : 0; }   // prod keys only
    for (int i = 0; i < 2; ++i) { P.vt_off[i] = off; off += (kD + 16) * kTTok * 2; }       // V^T, 1/weight and zero rows
    const int ops_end = off;
    for (int i = 0; i < 2; ++i) { P.vs_off[i] = off; off += kTTok * kVStride * 2; }
    P.norm_off = off; off += 3 * kStashBytes;
    P.sx_off = off; off += 2 * kTSplit * kTRows * 4;
    P.rv_off = off; off += p.vgroup ? 0 : kD * kD * 4;       // group values are not rotated
    P.bar_off = off; off += 128;
    P.orow_off = ops_begin;                                  // after the last tile
    if (ops_end - ops_begin < kTRows * (kD + 1) * 4) return cudaErrorInvalidValue;
    const size_t smem = static_cast<size_t>(off);
    if (smem > 232448) return cudaErrorInvalidValue;   // the largest dynamic shared memory a CTA can opt into
    if (p.kprod && p.kb == 2 && !p.vgroup && p.vb == 3) return launch_prefill_tc_t<2, true, false, 3>(P, smem, s);
    if (p.kprod && p.kb == 2 && !p.vgroup && p.vb == 4) return launch_prefill_tc_t<2, true, false, 4>(P, smem, s);
    if (p.kprod && p.kb == 2 && p.vgroup && p.vb == 4) return launch_prefill_tc_t<2, true, true, 4>(P, smem, s);
    if (!p.kprod && p.kb == 4 && !p.vgroup && p.vb == 4) return launch_prefill_tc_t<4, false, false, 4>(P, smem, s);
    return cudaErrorInvalidValue;
}

}  // namespace mmadec
}  // namespace tq

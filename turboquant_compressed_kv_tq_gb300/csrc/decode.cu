// TurboQuant decode attention over the compressed cache.
//
// "lightning-mlx/plan.md" asks for a fused attention kernel that works on the
// Lloyd-Max codes directly instead of dequantising the cache; the validation
// script of "turboquant/validate_moe_phase2.py" scores queries against
// compressed keys (attention_score). In the rotated domain, with q' = R_k q
// and q'' = S_k q',
//   <q, k_hat_t> = n_t (<q', c[idx_t]> + sqrt(pi/2)/D * rnorm_t <q'', sign_t>)
// and for MSE values sum_t p_t v_hat_t = (sum_t p_t n_t c_v[idx_t]) @ R_v, so the
// cache is never rotated back: the query is rotated once and the output once.
//
// Three kernels per call:
//   qprep  : q' (and q'' for prod keys) for every query row, fp32;
//   split  : one CTA per (token split, kv head x row group, sequence) runs an
//            online softmax over its tokens and writes (max, sum, acc[D]);
//   merge  : log-sum-exp merge of the splits, 1/sum, inverse value rotation.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cfloat>
#include <cmath>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kTile = 32;   // tokens per tile
constexpr int kSimtMinChunk = 256;   // fewest tokens per split of the SIMT decode
constexpr int kRows = 16;   // query rows per CTA (one row group)
constexpr int kThreads = 128;

__device__ __forceinline__ float load_q(const void* p, int dtype, int64_t i) {
    if (dtype == TQ_F32) return static_cast<const float*>(p)[i];
    if (dtype == TQ_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    return __half2float(static_cast<const __half*>(p)[i]);
}

__device__ __forceinline__ unsigned extract_code(const uint32_t* words, int i, int b) {
    const int p = i * b;
    const int w = p >> 5;
    const int sh = p & 31;
    uint32_t v = words[w] >> sh;
    if (sh + b > 32) v |= words[w + 1] << (32 - sh);
    return v & ((1u << b) - 1u);
}

// q' = R q and q'' = S q' for the 16 rows of one (sequence, kv head, row
// group): one pass over each matrix for all 16 rows (a matrix element is
// loaded once and used for every row).
template <int D>
__global__ void qprep_kernel(DecodeArgs a) {
    __shared__ float qs[kRows][D];
    __shared__ float q1[kRows][D];
    const int Hkv = a.pool.Hkv;
    const int bh = blockIdx.x;
    const int b = bh / Hkv, h = bh % Hkv;
    const int rg = blockIdx.y;
    const int RG = a.plan.row_groups;
    const int i = threadIdx.x;
    for (int rr = 0; rr < kRows; ++rr) {
        const int r = rg * kRows + rr;
        float v = 0.0f;
        if (r < a.plan.rows) {
            const int g = r / a.Lq, l = r % a.Lq;
            v = load_q(a.q, a.q_dtype, ((static_cast<int64_t>(b) * a.Hq + h * a.G + g) * a.Lq + l) * D + i);
        }
        qs[rr][i] = v;
    }
    __syncthreads();
    float t[kRows] = {};
    for (int k = 0; k < D; ++k) {
        const float rk = __ldg(a.kc.Rt + k * D + i);
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) t[rr] = fmaf(rk, qs[rr][k], t[rr]);
    }
    float z[kRows] = {};
    if (a.kc.mode == TQ_MODE_PROD) {
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) q1[rr][i] = t[rr];
        __syncthreads();
        for (int k = 0; k < D; ++k) {
            const float sk = __ldg(a.kc.St + k * D + i);
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) z[rr] = fmaf(sk, q1[rr][k], z[rr]);
        }
    }
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) {
        const bool live = rg * kRows + rr < a.plan.rows;
        const int64_t o = ((static_cast<int64_t>(bh) * RG + rg) * kRows + rr) * D + i;
        a.qrot[o] = live ? t[rr] : 0.0f;
        a.qjl[o] = live ? z[rr] : 0.0f;
    }
}

template <int D>
struct SplitSmem {
    float qr[kRows][D];
    float qj[kRows][D];
    float kh[kTile][D + 1];
    float vh[kTile][D + 1];
    uint32_t sg[kTile][D / 32 + 1];   // padded: the lanes of a warp read different banks
    float kn[kTile], kr[kTile], vn[kTile];
    float sc[kRows][kTile + 1];
    float m[kRows], l[kRows], alpha[kRows];
};

template <int D>
__global__ void __launch_bounds__(kThreads) split_kernel(DecodeArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SplitSmem<D>& sm = *reinterpret_cast<SplitSmem<D>*>(smem_raw);
    constexpr int kDPer = (D + kThreads - 1) / kThreads;
    const int tid = threadIdx.x;
    const int Hkv = a.pool.Hkv;
    const int RG = a.plan.row_groups;
    const int split = blockIdx.x;
    const int h = blockIdx.y % Hkv;
    const int rg = blockIdx.y / Hkv;
    const int b = blockIdx.z;
    const int bh = b * Hkv + h;
    const int rows = a.plan.rows;
    const int BT = a.pool.BT;
    const float kappa = 1.2533141373155003f / static_cast<float>(D);  // sqrt(pi/2)/D

    const int N = a.seq_lens[b] + a.len_add;
    const int cap = a.max_blocks * BT;
    // causal window end (local token index): the sequence's end, or a shard's
    const int vis = a.causal_end ? a.causal_end[b] : N;
    const bool bad = N < (a.causal_end ? 0 : a.Lq) || N > cap;
    if (bad && split == 0 && tid == 0 && rg == 0 && h == 0) atomicOr(a.err, TQ_DEVERR_SEQLEN);
    const int t_begin = split * a.plan.chunk;
    int t_end = t_begin + a.plan.chunk;
    const int n_eff = bad ? 0 : N;
    if (t_end > n_eff) t_end = n_eff;

    for (int e = tid; e < kRows * D; e += kThreads) {
        const int rr = e / D, i = e % D;
        const int64_t o = ((static_cast<int64_t>(bh) * RG + rg) * kRows + rr) * D + i;
        sm.qr[rr][i] = a.qrot[o];
        sm.qj[rr][i] = a.qjl[o];
    }
    if (tid < kRows) {
        sm.m[tid] = -INFINITY;
        sm.l[tid] = 0.0f;
    }
    float acc[kRows][kDPer];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
#pragma unroll
        for (int j = 0; j < kDPer; ++j) acc[r][j] = 0.0f;
    __syncthreads();

    const int kb = a.kc.ib, vb = a.vc.mode == TQ_MODE_GROUP ? a.vc.bits : a.vc.ib;
    // A tile never crosses a block: TT divides BT and every split starts on a
    // multiple of kTile.
    const int TT = BT < kTile ? BT : kTile;
    for (int tile = t_begin; tile < t_end; tile += TT) {
        const int nt = min(TT, t_end - tile);
        const int lb = tile / BT;
        const int slot0 = tile - lb * BT;
        const int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(b) * a.max_blocks + lb])
                                   : static_cast<int64_t>(b) * a.max_blocks + lb;
        const bool pb_ok = pb >= 0 && pb < a.pool.num_blocks;
        if (!pb_ok && tid == 0) atomicOr(a.err, TQ_DEVERR_BLOCK);
        const char* base = a.pool.base + (pb_ok ? (pb * Hkv + h) * a.pool.sub_bytes : 0);
        const uint32_t* kidx = reinterpret_cast<const uint32_t*>(base + a.pool.off[0]) + static_cast<int64_t>(slot0) * a.kc.W;
        const uint32_t* vidx = reinterpret_cast<const uint32_t*>(base + a.pool.off[4]) + static_cast<int64_t>(slot0) * a.vc.W;
        for (int e = tid; e < nt * D; e += kThreads) {
            const int t = e / D, i = e % D;
            sm.kh[t][i] = __ldg(a.kc.c + extract_code(kidx + t * a.kc.W, i, kb));
            const unsigned vcode = extract_code(vidx + t * a.vc.W, i, vb);
            if (a.vc.mode == TQ_MODE_GROUP) {
                const int ng = D / a.vc.group;
                const __half* sc = reinterpret_cast<const __half*>(base + a.pool.off[5]) + static_cast<int64_t>(slot0 + t) * ng;
                const __half* mn = reinterpret_cast<const __half*>(base + a.pool.off[6]) + static_cast<int64_t>(slot0 + t) * ng;
                sm.vh[t][i] = fmaf(static_cast<float>(vcode), __half2float(sc[i / a.vc.group]),
                                   __half2float(mn[i / a.vc.group]));
            } else {
                sm.vh[t][i] = __ldg(a.vc.c + vcode);
            }
        }
        if (a.kc.mode == TQ_MODE_PROD) {
            const uint32_t* sgn = reinterpret_cast<const uint32_t*>(base + a.pool.off[1]) + static_cast<int64_t>(slot0) * a.kc.Ws;
            for (int e = tid; e < nt * (D / 32); e += kThreads) sm.sg[e / (D / 32)][e % (D / 32)] = sgn[e];
        }
        if (tid < nt) {
            sm.kn[tid] = reinterpret_cast<const float*>(base + a.pool.off[2])[slot0 + tid];
            sm.kr[tid] = a.kc.mode == TQ_MODE_PROD ? reinterpret_cast<const float*>(base + a.pool.off[3])[slot0 + tid] : 0.0f;
            sm.vn[tid] = a.vc.mode == TQ_MODE_GROUP ? 1.0f : reinterpret_cast<const float*>(base + a.pool.off[5])[slot0 + tid];
        }
        __syncthreads();
        // scores
        {
            const int t = tid & (kTile - 1);
            for (int rr = tid / kTile; rr < kRows; rr += kThreads / kTile) {
                const int r = rg * kRows + rr;
                float s = -INFINITY;
                if (t < nt && r < rows && pb_ok) {
                    const int l = r % a.Lq;
                    const int pos = tile + t;
                    if (pos <= vis - a.Lq + l) {
                        float dot = 0.0f;
                        for (int i = 0; i < D; ++i) dot = fmaf(sm.qr[rr][i], sm.kh[t][i], dot);
                        if (a.kc.mode == TQ_MODE_PROD) {
                            float sd = 0.0f;
                            for (int w = 0; w < D / 32; ++w) {
                                const uint32_t word = sm.sg[t][w];
#pragma unroll 8
                                for (int k = 0; k < 32; ++k) {
                                    const float qv = sm.qj[rr][32 * w + k];
                                    sd += ((word >> k) & 1u) ? qv : -qv;
                                }
                            }
                            dot = fmaf(kappa * sm.kr[t], sd, dot);
                        }
                        s = a.scale * sm.kn[t] * dot;
                    }
                }
                sm.sc[rr][t] = s;
            }
        }
        __syncthreads();
        if (tid < kRows) {
            const int rr = tid;
            float mt = -INFINITY;
            for (int t = 0; t < kTile; ++t) mt = fmaxf(mt, sm.sc[rr][t]);
            const float mo = sm.m[rr];
            const float mn = fmaxf(mo, mt);
            float alpha = 1.0f, sum = 0.0f;
            if (mn != -INFINITY) {
                alpha = expf(mo - mn);
                for (int t = 0; t < kTile; ++t) {
                    const float p = expf(sm.sc[rr][t] - mn);
                    sum += p;
                    sm.sc[rr][t] = p * sm.vn[t < nt ? t : 0];
                }
            } else {
                for (int t = 0; t < kTile; ++t) sm.sc[rr][t] = 0.0f;
            }
            sm.l[rr] = sm.l[rr] * alpha + sum;
            sm.m[rr] = mn;
            sm.alpha[rr] = alpha;
        }
        __syncthreads();
#pragma unroll
        for (int j = 0; j < kDPer; ++j) {
            const int d = tid + j * kThreads;
            if (d < D) {
#pragma unroll
                for (int r = 0; r < kRows; ++r) acc[r][j] *= sm.alpha[r];
                // one value load per token, used for all 16 rows
                for (int t = 0; t < nt; ++t) {
                    const float vv = sm.vh[t][d];
#pragma unroll
                    for (int r = 0; r < kRows; ++r) acc[r][j] = fmaf(sm.sc[r][t], vv, acc[r][j]);
                }
            }
        }
        __syncthreads();
    }
    const int64_t pbase = ((static_cast<int64_t>(bh) * RG + rg) * a.plan.splits + split) * kRows;
#pragma unroll
    for (int j = 0; j < kDPer; ++j) {
        const int d = tid + j * kThreads;
        if (d < D) {
#pragma unroll
            for (int r = 0; r < kRows; ++r) a.part[(pbase + r) * D + d] = acc[r][j];
        }
    }
    if (tid < kRows) {
        a.ml[(pbase + tid) * 2] = sm.m[tid];
        a.ml[(pbase + tid) * 2 + 1] = sm.l[tid];
    }
}

// Merge the splits of one (sequence, kv head, row group) and rotate back:
// first every row's merged accumulator, then one pass over R_v for all rows.
template <int D>
__global__ void merge_kernel(DecodeArgs a) {
    __shared__ float orot[kRows][D];
    const int Hkv = a.pool.Hkv;
    const int bh = blockIdx.x;
    const int b = bh / Hkv, h = bh % Hkv;
    const int rg = blockIdx.y;
    const int RG = a.plan.row_groups;
    const int S = a.plan.splits;
    const int i = threadIdx.x;
    const int64_t base = (static_cast<int64_t>(bh) * RG + rg) * S;
    for (int rr = 0; rr < kRows; ++rr) {
        float M = -INFINITY;
        for (int s = 0; s < S; ++s) M = fmaxf(M, a.ml[((base + s) * kRows + rr) * 2]);
        float L = 0.0f, o = 0.0f;
        if (M != -INFINITY) {
            for (int s = 0; s < S; ++s) {
                const float ms = a.ml[((base + s) * kRows + rr) * 2];
                if (ms == -INFINITY) continue;
                const float w = expf(ms - M);
                L = fmaf(w, a.ml[((base + s) * kRows + rr) * 2 + 1], L);
                o = fmaf(w, a.part[((base + s) * kRows + rr) * D + i], o);
            }
        }
        const int r = rg * kRows + rr;
        if (a.part_acc) {
            // a shard's state: max (natural-log units), sum, rotated-domain accumulator
            if (r < a.plan.rows) {
                const int g = r / a.Lq, l = r % a.Lq;
                const int64_t orow = (static_cast<int64_t>(b) * a.Hq + h * a.G + g) * a.Lq + l;
                if (i == 0) {
                    a.part_ml[2 * orow] = M;
                    a.part_ml[2 * orow + 1] = L;
                }
                a.part_acc[orow * D + i] = o;
            }
            continue;
        }
        orot[rr][i] = L > 0.0f ? o / L : 0.0f;
    }
    if (a.part_acc) return;
    __syncthreads();
    float res[kRows];
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) res[rr] = orot[rr][i];
    if (a.vc.mode != TQ_MODE_GROUP) {
#pragma unroll
        for (int rr = 0; rr < kRows; ++rr) res[rr] = 0.0f;
        for (int k = 0; k < D; ++k) {
            const float rk = __ldg(a.vc.R + k * D + i);
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) res[rr] = fmaf(orot[rr][k], rk, res[rr]);
        }
    }
#pragma unroll
    for (int rr = 0; rr < kRows; ++rr) {
        const int r = rg * kRows + rr;
        if (r >= a.plan.rows) break;
        const int g = r / a.Lq, l = r % a.Lq;
        a.out[((static_cast<int64_t>(b) * a.Hq + h * a.G + g) * a.Lq + l) * D + i] = res[rr];
    }
}

// Log-sum-exp merge of the partial states of P sequence shards, row r of
// part p at ml[(p * rows + r) * 2] (max, sum) and acc[(p * rows + r) * D]:
// M = max_p m_p, L = sum_p e^(m_p - M) l_p, o = sum_p e^(m_p - M) acc_p / L,
// rotated back by R_v for MSE values. One CTA of D threads per row.
__global__ void shard_merge_kernel(CodecDev vc, int P, const float* ml, const float* acc, int64_t rows, float* out) {
    __shared__ float orot[256];
    const int D = vc.D;
    const int64_t r = blockIdx.x;
    const int i = threadIdx.x;
    float M = -INFINITY;
    for (int p = 0; p < P; ++p) M = fmaxf(M, ml[(p * rows + r) * 2]);
    float L = 0.0f, o = 0.0f;
    if (M != -INFINITY) {
        for (int p = 0; p < P; ++p) {
            const float mp = ml[(p * rows + r) * 2];
            if (mp == -INFINITY) continue;
            const float w = expf(mp - M);
            L = fmaf(w, ml[(p * rows + r) * 2 + 1], L);
            o = fmaf(w, acc[(p * rows + r) * D + i], o);
        }
    }
    orot[i] = L > 0.0f ? o / L : 0.0f;
    __syncthreads();
    float res = orot[i];
    if (vc.mode != TQ_MODE_GROUP) {
        res = 0.0f;
        for (int k = 0; k < D; ++k) res = fmaf(orot[k], __ldg(vc.R + k * D + i), res);
    }
    out[r * D + i] = res;
}

template <int D>
cudaError_t launch_decode_d(const DecodeArgs& a, cudaStream_t s) {
    const int B = a.batch, Hkv = a.pool.Hkv, RG = a.plan.row_groups;
    qprep_kernel<D><<<dim3(B * Hkv, RG), D, 0, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const size_t smem = sizeof(SplitSmem<D>);
    static std::atomic<uint64_t> attr_set{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(split_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        attr_set.fetch_or(bit);
    }
    split_kernel<D><<<dim3(a.plan.splits, Hkv * RG, B), kThreads, smem, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    merge_kernel<D><<<dim3(B * Hkv, RG), D, 0, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
}

}  // namespace

namespace mmadec {
struct MmaArgs;
}

}  // namespace tq
#include "decode_mma_impl.cuh"
namespace tq {
namespace mmadec {
bool dispatch_a(int, bool, bool, int, const MmaArgs&, size_t, cudaStream_t, const EncodeAppendArgs*, cudaError_t*);
bool dispatch_b(int, bool, bool, int, const MmaArgs&, size_t, cudaStream_t, const EncodeAppendArgs*, cudaError_t*);
bool dispatch_c(int, bool, bool, int, const MmaArgs&, size_t, cudaStream_t, const EncodeAppendArgs*, cudaError_t*);
bool wide_supported(int D, int kb, bool prod, bool vgroup, int vb);
bool dispatch_d(int D, int kb, bool prod, bool vgroup, int vb, const MmaArgs&, size_t, cudaStream_t, cudaError_t*);
bool dispatch_e(int D, int kb, bool prod, bool vgroup, int vb, const MmaArgs&, size_t, cudaStream_t, cudaError_t*);
bool r8_supported(int kb, bool prod, bool vgroup, int vb);
bool dispatch_f(int, bool, bool, int, const MmaArgs&, size_t, cudaStream_t, const EncodeAppendArgs*, cudaError_t*);
}  // namespace mmadec

namespace {

size_t al256(size_t x) { return (x + 255) / 256 * 256; }

// Token splits: enough CTAs to cover the GPU, split length a multiple of the
// tile, and at most `max_chunk` tokens so that many short units still balance.
void choose_splits(DecodePlan& p, int64_t units, int64_t target_ctas, int max_seq_len, int tile, int max_chunk,
                   int min_chunk = 0) {
    const int64_t max_splits = (max_seq_len + (min_chunk > tile ? min_chunk : tile) - 1) / (min_chunk > tile ? min_chunk : tile);
    int64_t splits = (target_ctas + units - 1) / units;
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    int64_t chunk = (max_seq_len + splits - 1) / splits;
    chunk = (chunk + tile - 1) / tile * tile;
    if (chunk > max_chunk) chunk = max_chunk;
    if (chunk < tile) chunk = tile;
    splits = (max_seq_len + chunk - 1) / chunk;
    p.splits = static_cast<int>(splits < 1 ? 1 : splits);
    p.chunk = static_cast<int>(chunk);
}

bool mma_supported(const tq_cache_desc* d, DecodePlan& p) {
    if (d->head_dim != mmadec::kD && d->head_dim != 2 * mmadec::kD && d->head_dim != mmadec::kD / 2) return false;
    p.kprod = d->key_mode == TQ_MODE_PROD;
    p.kb = p.kprod ? d->key_bits - 1 : d->key_bits;
    if (p.kprod ? (p.kb < 1 || p.kb > 3) : (p.kb < 2 || p.kb > 4)) return false;
    p.vgroup = d->value_mode == TQ_MODE_GROUP;
    p.vb = d->value_bits;
    if (p.vgroup) {
        if ((p.vb != 2 && p.vb != 4) || d->value_group < 32) return false;
    } else if (p.vb < 2 || p.vb > 4) {
        return false;
    }
    // head_dim 64 and 256: the instantiated codec pairs only
    return d->head_dim == mmadec::kD || mmadec::wide_supported(d->head_dim, p.kb, p.kprod, p.vgroup, p.vb);
}

}  // namespace

DecodePlan make_decode_plan(const tq_cache_desc* d, int batch, int G, int Lq, int max_seq_len, int num_sms) {
    DecodePlan p{};
    const int D = d->head_dim;
    const int Hkv = d->num_kv_heads;
    p.rows = G * Lq;
    p.row_groups = (p.rows + kRows - 1) / kRows;
    const int64_t units = static_cast<int64_t>(batch) * Hkv * p.row_groups;
    if (mma_supported(d, p)) {
        p.kind = 1;
        const int NH = D > mmadec::kD ? D / mmadec::kD : 1;  // 128-column value halves: CTAs per (unit, split)
        // stage layout for a tile size; the tile halves (down to 16 tokens)
        // while the split kernel's shared memory would exceed the budget
        auto layout = [&](int tile) {
            p.tile = tile;
            int o = 0;
            for (int k = 0; k < 7; ++k) {
                const int64_t so = d->stream_offset[k];
                int64_t next = d->subblock_bytes;
                for (int k2 = k + 1; k2 < 7; ++k2)
                    if (d->stream_offset[k2] >= 0) { next = d->stream_offset[k2]; break; }
                if (so < 0) {
                    p.st_off[k] = -1;
                    p.st_field[k] = 0;
                    continue;
                }
                p.st_field[k] = static_cast<int>((next - so) / d->block_tokens);
                p.st_off[k] = o;
                o += p.tile * p.st_field[k];
            }
            p.st_bytes = (o + 127) / 128 * 128;
            // 4-bit MSE keys and values: their one table of 256-byte entries at offset 0
            const bool wide = mmadec::pair4_wide(D, p.kb, p.kprod, p.vgroup, p.vb);
            p.ring_off = wide ? mmadec::kPair4WBytes : 0;
            const size_t ring = p.ring_off + static_cast<size_t>(mmadec::kWarps) * mmadec::kStages * p.st_bytes;
            p.qs_off = static_cast<int>(ring);
            size_t ringq = ring + static_cast<size_t>(mmadec::kQFragBytes) * NH;
            p.vt_off = wide ? 0 : -1;
            if (!p.vgroup && p.vb == 3) {  // pair table of 3-bit value codes (aligned inside the region)
                p.vt_off = static_cast<int>(ringq);
                ringq += mmadec::kVPairRegion;
            }
            if (p.vgroup && mmadec::nibble_qjl(p.kprod, p.vgroup, p.vb)) {  // QJL sign nibbles (aligned inside)
                p.vt_off = static_cast<int>(ringq);
                ringq += mmadec::kQNibRegion;
            }
            if (!wide && mmadec::pair4_values(D, p.kprod, p.vgroup, p.vb)) {  // pair table of 4-bit value codes
                p.vt_off = static_cast<int>(ringq);
                ringq += mmadec::kPair4Bytes;
            }
            p.kt_off = wide ? 0 : -1;
            if (!wide && mmadec::pair4_keys(D, p.kb, p.kprod)) {  // pair table of 4-bit key codes
                p.kt_off = static_cast<int>(ringq);
                ringq += mmadec::kPair4Bytes;
            }
            if (mmadec::quad_keys(p.kb, p.kprod, p.vgroup)) {  // quad table of 2-bit key codes
                p.kt_off = static_cast<int>(ringq);
                ringq += mmadec::kKQuadBytes;
            }
            const size_t combine = mmadec::kWarpMergeBytes;
            const size_t body = ((ringq > combine ? ringq : combine) + 127) / 128 * 128;
            p.bar_off = static_cast<int>(body);
            p.smem = body + sizeof(uint64_t) * (mmadec::kWarps * mmadec::kStages + 1);  // + the tables' barrier
        };
        // 64-token tiles; a tile gathers up to four shorter blocks (one copy per
        // block and record stream)
        int tile = mmadec::kMaxTile;
        if (d->block_tokens < 16) tile = d->block_tokens;
        layout(tile);
        while (p.smem > mmadec::kSmemBudget && tile > 16) {
            tile /= 2;
            layout(tile);
        }
        // At most 16384 tokens per split; where the units alone fill the GPU
        // (several waves of CTAs) at most 12288, so that the last wave's CTAs,
        // the grid's tail, are short.
        const int max_chunk = units * NH >= num_sms ? 12288 : 16384;
        choose_splits(p, units * NH, num_sms, max_seq_len, p.tile, max_chunk);
        // A CTA's time is its busiest warp's: ceil(tiles of a split / warps)
        // tiles. Where 64-token tiles leave that warp a tile more than the
        // average (short splits), 32-token tiles (each about 0.52 of a 64-token
        // tile's time, per-tile overheads included) can balance better.
        if (tile == 64) {
            auto busiest = [&](const DecodePlan& q) {
                const int tiles = (q.chunk + q.tile - 1) / q.tile;
                return (tiles + mmadec::kWarps - 1) / mmadec::kWarps;
            };
            const DecodePlan h = p;   // the 64-token plan
            layout(32);
            choose_splits(p, units * NH, num_sms, max_seq_len, 32, max_chunk);
            if (100 * busiest(h) <= 52 * busiest(p) || p.smem > mmadec::kSmemBudget) p = h;
        }
        // at most 8 query rows per unit at head_dim 128: the transposed kernel
        p.r8 = D == mmadec::kD && p.rows <= 8 && mmadec::r8_supported(p.kb, p.kprod, p.vgroup, p.vb) ? 1 : 0;
        // head_dim 128: the units' query fragments; otherwise the fp32 q' and
        // q'' rows of the query prep (two arrays of q_bytes)
        p.q_bytes = D == mmadec::kD ? al256(static_cast<size_t>(units) * 2 * 8 * 32 * 16)
                                    : al256(static_cast<size_t>(units) * kRows * D * sizeof(float));
    } else {
        p.kind = 0;
        p.tile = kTile;
        // at least kSimtMinChunk tokens per split: the merge reads every
        // split's partials once per output row, so many short splits cost
        // more in the merge than they gain in the split kernel
        choose_splits(p, units, static_cast<int64_t>(num_sms) * 4, max_seq_len, kTile, 1 << 30, kSimtMinChunk);
        p.q_bytes = al256(static_cast<size_t>(units) * kRows * D * sizeof(float));
    }
    // the tensor-core kernels write 128-column partial rows at head_dim 64
    const int part_cols = p.kind == 1 && D < mmadec::kD ? mmadec::kD : D;
    p.part_bytes = al256(static_cast<size_t>(units) * p.splits * kRows * part_cols * sizeof(float));
    // (max, sum) rows: one set per value half of the tensor-core path
    const int ml_sets = p.kind == 1 && D > mmadec::kD ? D / mmadec::kD : 1;
    p.ml_bytes = al256(static_cast<size_t>(units) * ml_sets * p.splits * kRows * 2 * sizeof(float));
    p.total = (p.kind == 1 && D == mmadec::kD ? p.q_bytes : 2 * p.q_bytes) + p.part_bytes + p.ml_bytes;
    return p;
}

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s, const EncodeAppendArgs* step) {
    if (a.batch == 0) return cudaSuccess;
    if (a.plan.kind == 1) {
        if (a.plan.splits > 65535) return cudaErrorInvalidValue;  // the split kernel's grid z
        mmadec::MmaArgs m{};
        m.a = a;
        m.st.tt = a.plan.tile;
        m.st.bytes = a.plan.st_bytes;
        m.st.bar_off = a.plan.bar_off;
        m.st.qs_off = a.plan.qs_off;
        m.st.vt_off = a.plan.vt_off;
        m.st.kt_off = a.plan.kt_off;
        m.st.ring_off = a.plan.ring_off;
        for (int k = 0; k < 7; ++k) {
            m.st.off[k] = a.plan.st_off[k];
            m.st.field[k] = a.plan.st_field[k];
        }
        char* ws = static_cast<char*>(a.ws);
        cudaError_t e = cudaErrorInvalidValue;
        const DecodePlan& p = a.plan;
        if (a.kc.D != mmadec::kD) {
            // fp32 query rows at a.qrot / a.qjl, partials after both
            m.part = a.part;
            m.ml = a.ml;
            if (step) return cudaErrorInvalidValue;  // the step's append runs before
            if (mmadec::dispatch_d(a.kc.D, p.kb, p.kprod, p.vgroup, p.vb, m, p.smem, s, &e)) return e;
            if (mmadec::dispatch_e(a.kc.D, p.kb, p.kprod, p.vgroup, p.vb, m, p.smem, s, &e)) return e;
            return cudaErrorInvalidValue;
        }
        m.qfrag = reinterpret_cast<const uint4*>(ws);
        m.part = reinterpret_cast<float*>(ws + a.plan.q_bytes);
        m.ml = reinterpret_cast<float*>(ws + a.plan.q_bytes + a.plan.part_bytes);
        if (p.r8) {
            if (mmadec::dispatch_f(p.kb, p.kprod, p.vgroup, p.vb, m, p.smem, s, step, &e)) return e;
            return cudaErrorInvalidValue;
        }
        if (mmadec::dispatch_a(p.kb, p.kprod, p.vgroup, p.vb, m, p.smem, s, step, &e)) return e;
        if (mmadec::dispatch_b(p.kb, p.kprod, p.vgroup, p.vb, m, p.smem, s, step, &e)) return e;
        if (mmadec::dispatch_c(p.kb, p.kprod, p.vgroup, p.vb, m, p.smem, s, step, &e)) return e;
        return cudaErrorInvalidValue;
    }
    switch (a.kc.D) {
        case 64: return launch_decode_d<64>(a, s);
        case 128: return launch_decode_d<128>(a, s);
        case 256: return launch_decode_d<256>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_shard_merge(const CodecDev& vc, int parts, const float* ml, const float* acc, int64_t rows,
                               float* out, cudaStream_t s) {
    shard_merge_kernel<<<static_cast<unsigned>(rows), vc.D, 0, s>>>(vc, parts, ml, acc, rows, out);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
}

}  // namespace tq

// Decode attention over split states: each key and value vector of head_dim
// D is held as two TurboQuant states ("omlx/turboquant_kv.py",
// TurboQuantSplitState(low, high), carried through every batch operation by
// _filter_state and _concat_state_batch): the low coordinates [0, DL) under
// one codec pair and the high coordinates [DL, D) under another, each with its
// own norm, rotation, codebook and bit width. The attention score of a token
// is the sum of the two halves' scores,
//   <q, k_hat> = <q_low, k_hat_low> + <q_high, k_hat_high>,
// each half in its own rotated domain (q'_half = R_half q_half,
// q''_half = S_half q'_half), and the output is [o_low | o_high], each half
// rotated back by its own value rotation.
//
// Three kernels, as the SIMT decode: query prep, split-K online softmax,
// merge of the splits with the inverse rotations.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <atomic>
#include <cmath>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kTile = 32;   // tokens per tile
constexpr int kRows = 16;   // query rows per CTA
constexpr int kThreads = 128;

__device__ __forceinline__ float q_elem(const void* p, int dtype, int64_t i) {
    if (dtype == TQ_F32) return static_cast<const float*>(p)[i];
    if (dtype == TQ_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    return __half2float(static_cast<const __half*>(p)[i]);
}

// Code i of b bits from a packed word stream (codes may straddle words).
__device__ __forceinline__ unsigned code_at(const uint32_t* words, int i, int b) {
    const int p = i * b;
    const int w = p >> 5, sh = p & 31;
    uint32_t v = words[w] >> sh;
    if (sh + b > 32) v |= words[w + 1] << (32 - sh);
    return v & ((1u << b) - 1u);
}

// q' = R q, q'' = S q' of each half for the 16 rows of one (sequence, kv
// head, row group); one thread per coordinate of the whole vector.
template <int DL, int DH>
__global__ void split_state_qprep_kernel(SplitStateArgs a) {
    constexpr int D = DL + DH;
    __shared__ float qs[D];
    __shared__ float q1[D];
    const int bh = blockIdx.x;
    const int b = bh / a.Hkv, h = bh % a.Hkv;
    const int rg = blockIdx.y;
    const int i = threadIdx.x;
    const bool lo = i < DL;
    const CodecDev& kc = lo ? a.klo : a.khi;
    const int n = lo ? DL : DH, ii = lo ? i : i - DL, k0 = lo ? 0 : DL;
    for (int rr = 0; rr < kRows; ++rr) {
        const int r = rg * kRows + rr;
        const int64_t o = ((static_cast<int64_t>(bh) * a.row_groups + rg) * kRows + rr) * D + i;
        if (r >= a.rows) {
            a.qrot[o] = 0.0f;
            a.qjl[o] = 0.0f;
            continue;
        }
        const int g = r / a.Lq, l = r % a.Lq;
        qs[i] = q_elem(a.q, a.q_dtype, ((static_cast<int64_t>(b) * a.Hq + h * a.G + g) * a.Lq + l) * D + i);
        __syncthreads();
        float t = 0.0f;
        for (int k = 0; k < n; ++k) t = fmaf(__ldg(kc.Rt + k * n + ii), qs[k0 + k], t);
        q1[i] = t;
        a.qrot[o] = t;
        __syncthreads();
        float z = 0.0f;
        if (kc.mode == TQ_MODE_PROD)
            for (int k = 0; k < n; ++k) z = fmaf(__ldg(kc.St + k * n + ii), q1[k0 + k], z);
        a.qjl[o] = z;
        __syncthreads();
    }
}

template <int DL, int DH>
struct SplitStateSmem {
    static constexpr int D = DL + DH;
    float qr[kRows][D];
    float qj[kRows][D];
    float kh[kTile][D + 1];   // key level x key norm of its half
    float vh[kTile][D + 1];   // value, norm of its half folded in
    uint32_t sg[kTile][D / 32];
    float kq[kTile][2];       // sqrt(pi/2)/D_half x residual norm x norm (prod halves)
    float sc[kRows][kTile + 1];
    float m[kRows], l[kRows], alpha[kRows];
};

template <int DL, int DH>
__global__ void __launch_bounds__(kThreads) split_state_kernel(SplitStateArgs a) {
    constexpr int D = DL + DH;
    constexpr int kDPer = (D + kThreads - 1) / kThreads;
    extern __shared__ __align__(16) unsigned char smem_raw[];
    SplitStateSmem<DL, DH>& sm = *reinterpret_cast<SplitStateSmem<DL, DH>*>(smem_raw);
    const int tid = threadIdx.x;
    const int split = blockIdx.x;
    const int h = blockIdx.y % a.Hkv;
    const int rg = blockIdx.y / a.Hkv;
    const int b = blockIdx.z;
    const int bh = b * a.Hkv + h;
    const int BT = a.plo.BT;
    const int N = a.seq_lens[b];
    const bool bad = N < a.Lq || N > a.max_blocks * BT;
    if (bad && split == 0 && tid == 0 && rg == 0 && h == 0) atomicOr(a.err, TQ_DEVERR_SEQLEN);
    const int t_begin = split * a.chunk;
    const int t_end = min(t_begin + a.chunk, bad ? 0 : N);

    for (int e = tid; e < kRows * D; e += kThreads) {
        const int rr = e / D, i = e % D;
        const int64_t o = ((static_cast<int64_t>(bh) * a.row_groups + rg) * kRows + rr) * D + i;
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

    const int TT = BT < kTile ? BT : kTile;
    for (int tile = t_begin; tile < t_end; tile += TT) {
        const int nt = min(TT, t_end - tile);
        const int lb = tile / BT;
        const int slot0 = tile - lb * BT;
        const int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(b) * a.max_blocks + lb])
                                   : static_cast<int64_t>(b) * a.max_blocks + lb;
        const bool pb_ok = pb >= 0 && pb < a.plo.num_blocks;
        if (!pb_ok && tid == 0) atomicOr(a.err, TQ_DEVERR_BLOCK);
        const char* blo = a.plo.base + (pb_ok ? (pb * a.Hkv + h) * a.plo.sub_bytes : 0);
        const char* bhi = a.phi.base + (pb_ok ? (pb * a.Hkv + h) * a.phi.sub_bytes : 0);
        for (int e = tid; e < nt * D; e += kThreads) {
            const int t = e / D, i = e % D;
            const bool lo = i < DL;
            const int ii = lo ? i : i - DL;
            const CodecDev& kc = lo ? a.klo : a.khi;
            const CodecDev& vc = lo ? a.vlo : a.vhi;
            const PoolDev& pl = lo ? a.plo : a.phi;
            const char* base = lo ? blo : bhi;
            const uint32_t* kidx = reinterpret_cast<const uint32_t*>(base + pl.off[0]) + static_cast<int64_t>(slot0 + t) * kc.W;
            const float kn = reinterpret_cast<const float*>(base + pl.off[2])[slot0 + t];
            sm.kh[t][i] = kn * __ldg(kc.c + code_at(kidx, ii, kc.ib));
            const uint32_t* vidx = reinterpret_cast<const uint32_t*>(base + pl.off[4]) + static_cast<int64_t>(slot0 + t) * vc.W;
            const unsigned vcode = code_at(vidx, ii, vc.mode == TQ_MODE_GROUP ? vc.bits : vc.ib);
            if (vc.mode == TQ_MODE_GROUP) {
                const int ng = (lo ? DL : DH) / vc.group;
                const __half* sc = reinterpret_cast<const __half*>(base + pl.off[5]) + static_cast<int64_t>(slot0 + t) * ng;
                const __half* mn = reinterpret_cast<const __half*>(base + pl.off[6]) + static_cast<int64_t>(slot0 + t) * ng;
                sm.vh[t][i] = fmaf(static_cast<float>(vcode), __half2float(sc[ii / vc.group]), __half2float(mn[ii / vc.group]));
            } else {
                const float vn = reinterpret_cast<const float*>(base + pl.off[5])[slot0 + t];
                sm.vh[t][i] = vn * __ldg(vc.c + vcode);
            }
        }
        for (int e = tid; e < nt * (D / 32); e += kThreads) {
            const int t = e / (D / 32), wd = e % (D / 32);
            const bool lo = wd < DL / 32;
            const CodecDev& kc = lo ? a.klo : a.khi;
            const PoolDev& pl = lo ? a.plo : a.phi;
            const char* base = lo ? blo : bhi;
            sm.sg[t][wd] = kc.mode == TQ_MODE_PROD
                               ? reinterpret_cast<const uint32_t*>(base + pl.off[1])[static_cast<int64_t>(slot0 + t) * kc.Ws + (lo ? wd : wd - DL / 32)]
                               : 0u;
        }
        if (tid < 2 * nt) {
            const int t = tid >> 1, half = tid & 1;
            const CodecDev& kc = half ? a.khi : a.klo;
            const PoolDev& pl = half ? a.phi : a.plo;
            const char* base = half ? bhi : blo;
            float v = 0.0f;
            if (kc.mode == TQ_MODE_PROD) {
                const float kn = reinterpret_cast<const float*>(base + pl.off[2])[slot0 + t];
                const float rn = reinterpret_cast<const float*>(base + pl.off[3])[slot0 + t];
                v = 1.2533141373155003f / static_cast<float>(half ? DH : DL) * rn * kn;
            }
            sm.kq[t][half] = v;
        }
        __syncthreads();
        // scores
        {
            const int t = tid & (kTile - 1);
            for (int rr = tid / kTile; rr < kRows; rr += kThreads / kTile) {
                const int r = rg * kRows + rr;
                float s = -INFINITY;
                if (t < nt && r < a.rows && pb_ok) {
                    const int l = r % a.Lq;
                    if (tile + t <= N - a.Lq + l) {
                        float dot = 0.0f;
                        for (int i = 0; i < D; ++i) dot = fmaf(sm.qr[rr][i], sm.kh[t][i], dot);
                        float s0 = 0.0f, s1 = 0.0f;
                        for (int i = 0; i < DL; ++i) {
                            const float qv = sm.qj[rr][i];
                            s0 += ((sm.sg[t][i >> 5] >> (i & 31)) & 1u) ? qv : -qv;
                        }
                        for (int i = DL; i < D; ++i) {
                            const float qv = sm.qj[rr][i];
                            s1 += ((sm.sg[t][i >> 5] >> (i & 31)) & 1u) ? qv : -qv;
                        }
                        dot = fmaf(sm.kq[t][0], s0, dot);
                        dot = fmaf(sm.kq[t][1], s1, dot);
                        s = a.scale * dot;
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
                    sm.sc[rr][t] = p;
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
                for (int r = 0; r < kRows; ++r) {
                    float v = acc[r][j] * sm.alpha[r];
                    for (int t = 0; t < nt; ++t) v = fmaf(sm.sc[r][t], sm.vh[t][d], v);
                    acc[r][j] = v;
                }
            }
        }
        __syncthreads();
    }
    const int64_t pbase = ((static_cast<int64_t>(bh) * a.row_groups + rg) * a.splits + split) * kRows;
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

// Merge the splits, 1 / sum, and rotate each half back by its value rotation.
template <int DL, int DH>
__global__ void split_state_merge_kernel(SplitStateArgs a) {
    constexpr int D = DL + DH;
    __shared__ float orot[D];
    const int bh = blockIdx.x;
    const int b = bh / a.Hkv, h = bh % a.Hkv;
    const int rg = blockIdx.y;
    const int S = a.splits;
    const int i = threadIdx.x;
    const bool lo = i < DL;
    const CodecDev& vc = lo ? a.vlo : a.vhi;
    const int n = lo ? DL : DH, ii = lo ? i : i - DL, k0 = lo ? 0 : DL;
    for (int rr = 0; rr < kRows; ++rr) {
        const int r = rg * kRows + rr;
        if (r >= a.rows) break;
        const int64_t base = (static_cast<int64_t>(bh) * a.row_groups + rg) * S;
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
        orot[i] = L > 0.0f ? o / L : 0.0f;
        __syncthreads();
        float res = orot[i];
        if (vc.mode != TQ_MODE_GROUP) {
            res = 0.0f;
            for (int k = 0; k < n; ++k) res = fmaf(orot[k0 + k], __ldg(vc.R + k * n + ii), res);
        }
        const int g = r / a.Lq, l = r % a.Lq;
        a.out[((static_cast<int64_t>(b) * a.Hq + h * a.G + g) * a.Lq + l) * D + i] = res;
        __syncthreads();
    }
}

template <int DL, int DH>
cudaError_t launch_split_state_d(const SplitStateArgs& a, cudaStream_t s) {
    constexpr int D = DL + DH;
    split_state_qprep_kernel<DL, DH><<<dim3(a.batch * a.Hkv, a.row_groups), D, 0, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    const size_t smem = sizeof(SplitStateSmem<DL, DH>);
    static std::atomic<uint64_t> attr_set{0};  // one bit per device
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(split_state_kernel<DL, DH>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        attr_set.fetch_or(bit);
    }
    split_state_kernel<DL, DH><<<dim3(a.splits, a.Hkv * a.row_groups, a.batch), kThreads, smem, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    split_state_merge_kernel<DL, DH><<<dim3(a.batch * a.Hkv, a.row_groups), D, 0, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
}

}  // namespace

void split_state_plan(SplitStateArgs& a, int max_seq_len, int num_sms) {
    a.rows = a.G * a.Lq;
    a.row_groups = (a.rows + kRows - 1) / kRows;
    const int64_t units = static_cast<int64_t>(a.batch) * a.Hkv * a.row_groups;
    const int64_t max_splits = (max_seq_len + kTile - 1) / kTile;
    int64_t splits = (static_cast<int64_t>(num_sms) * 4 + units - 1) / (units > 0 ? units : 1);
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    int64_t chunk = (max_seq_len + splits - 1) / splits;
    chunk = (chunk + kTile - 1) / kTile * kTile;
    if (chunk < kTile) chunk = kTile;
    splits = (max_seq_len + chunk - 1) / chunk;
    a.splits = static_cast<int>(splits < 1 ? 1 : splits);
    a.chunk = static_cast<int>(chunk);
}

size_t split_state_workspace(const SplitStateArgs& a, int D) {
    const int64_t units = static_cast<int64_t>(a.batch) * a.Hkv * a.row_groups;
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t q = al(static_cast<size_t>(units) * kRows * D * sizeof(float));
    const size_t part = al(static_cast<size_t>(units) * a.splits * kRows * D * sizeof(float));
    const size_t ml = al(static_cast<size_t>(units) * a.splits * kRows * 2 * sizeof(float));
    return 2 * q + part + ml;
}

void split_state_bind_workspace(SplitStateArgs& a, void* ws, int D) {
    const int64_t units = static_cast<int64_t>(a.batch) * a.Hkv * a.row_groups;
    auto al = [](size_t x) { return (x + 255) / 256 * 256; };
    const size_t q = al(static_cast<size_t>(units) * kRows * D * sizeof(float));
    const size_t part = al(static_cast<size_t>(units) * a.splits * kRows * D * sizeof(float));
    char* p = static_cast<char*>(ws);
    a.qrot = reinterpret_cast<float*>(p);
    a.qjl = reinterpret_cast<float*>(p + q);
    a.part = reinterpret_cast<float*>(p + 2 * q);
    a.ml = reinterpret_cast<float*>(p + 2 * q + part);
}

cudaError_t launch_split_state(const SplitStateArgs& a, cudaStream_t s) {
    if (a.batch == 0) return cudaSuccess;
    const int dl = a.klo.D, dh = a.khi.D;
    if (dl == 64 && dh == 64) return launch_split_state_d<64, 64>(a, s);
    if (dl == 64 && dh == 128) return launch_split_state_d<64, 128>(a, s);
    if (dl == 128 && dh == 64) return launch_split_state_d<128, 64>(a, s);
    if (dl == 128 && dh == 128) return launch_split_state_d<128, 128>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace tq

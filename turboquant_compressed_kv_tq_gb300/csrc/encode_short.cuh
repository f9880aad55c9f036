// Short appends (decode steps, n_new < 32) of rotated codecs, head_dim <= 128.
//
// One CTA per (head, sequence, tensor) encodes all NV >= n_new vectors with one
// thread per coordinate. The transposed rotation (and QJL matrix) is staged in
// shared memory by one bulk copy, so the specification's sequential fma chains
// (identical order, bit-exact with the one-vector encoder) run at
// shared-memory latency, NV independent chains per thread. The body runs in a
// block of at least D threads: threads past D only take part in the barriers,
// so a wider kernel (the fused decode-step preparation) can host it.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tc_ptx.cuh"
#include "tq_internal.h"

namespace tq {

__device__ __forceinline__ float load_elem(const void* p, int dtype, int64_t i) {
    if (dtype == TQ_F32) return static_cast<const float*>(p)[i];
    if (dtype == TQ_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    return __half2float(static_cast<const __half*>(p)[i]);
}

// Dynamic shared memory of the body: the larger of the key and value layouts.
template <int D, int NV>
constexpr size_t encode_short_smem(bool two_tables) {
    return (two_tables ? 2 : 1) * static_cast<size_t>(D) * D * 4 +
           static_cast<size_t>(2 * NV * D + NV) * 4 + 8 + static_cast<size_t>(NV) * D;
}

template <int D, int NV>
__device__ __forceinline__ void encode_short_body(const EncodeAppendArgs& a, int h, int bq, int is_v,
                                                  unsigned char* smem_raw) {
    const CodecDev& cd = is_v ? a.vc : a.kc;
    const bool prod = cd.mode == TQ_MODE_PROD;
    float* Rt = reinterpret_cast<float*>(smem_raw);        // [D][D]
    float* St = Rt + D * D;                                 // [D][D] (prod)
    float* xs = St + (prod ? D * D : 0);                    // [NV][D]
    float* rs = xs + NV * D;                                // [NV][D] residuals (prod)
    float* ns = rs + NV * D;                                // [NV] norms
    uint64_t* bar = reinterpret_cast<uint64_t*>(ns + NV);  // 8-byte aligned (NV even)
    unsigned char* codes = reinterpret_cast<unsigned char*>(bar + 1);  // [NV][D]
    const int i = threadIdx.x;
    const bool act = i < D;
    const int n = a.n_new;
    // the next kernel may start its prologue now; this grid completes only
    // after the grid before it has (the wait at the end), so completion still
    // orders everything earlier in the stream
    tc::grid_release_dependents();

    if (i == 0) {
        tc::mbar_init(bar, 1);
        tc::mbar_fence_init();
        tc::mbar_expect_tx(bar, (prod ? 2u : 1u) * D * D * 4u);
        tc::bulk_g2s(Rt, cd.Rt, D * D * 4, bar);
        if (prod) tc::bulk_g2s(St, cd.St, D * D * 4, bar);
    }
    const void* src = is_v ? a.v : a.k;
    const int64_t base = (static_cast<int64_t>(bq) * a.pool.Hkv + h) * n * D;
    if (act) {
#pragma unroll
        for (int v = 0; v < NV; ++v) xs[v * D + i] = v < n ? load_elem(src, a.dtype, base + v * D + i) : 0.0f;
    }
    __syncthreads();
    if (i < n) {
        float n2 = 0.0f;
        for (int k = 0; k < D; ++k) n2 = __fmaf_rn(xs[i * D + k], xs[i * D + k], n2);
        ns[i] = __fsqrt_rn(n2);
    }
    const bool ok = tc::mbar_wait(bar, 0);
    if (__syncthreads_or(!ok)) {
        if (i == 0) atomicOr(a.err, TQ_DEVERR_TIMEOUT);
        (void)tc::mbar_wait(bar, 0);  // the copy may still land: bounded second wait
        tc::grid_wait_prior();
        return;
    }

    // rotation: NV chains, each in ascending k
    const int b = cd.ib;
    if (act) {
        float acc[NV];
#pragma unroll
        for (int v = 0; v < NV; ++v) acc[v] = 0.0f;
#pragma unroll 4
        for (int k = 0; k < D; ++k) {
            const float rt = Rt[k * D + i];
#pragma unroll
            for (int v = 0; v < NV; ++v) acc[v] = __fmaf_rn(rt, xs[v * D + k], acc[v]);
        }
        const int nm = (1 << b) - 1;
#pragma unroll
        for (int v = 0; v < NV; ++v) {
            const float nv = ns[v < n ? v : 0];
            const float y = (nv > 0.0f) ? __fdiv_rn(acc[v], nv) : 0.0f;
            int code = 0;
            for (int j = 0; j < nm; ++j) code += (y > __ldg(cd.m + j)) ? 1 : 0;
            codes[v * D + i] = static_cast<unsigned char>(code);
            if (prod) rs[v * D + i] = __fsub_rn(y, __ldg(cd.c + code));
        }
    }
    __syncthreads();

    // destinations (per vector; out-of-range positions are flagged and skipped)
    const int BT = a.pool.BT;
    auto sub_of = [&](int v, int& slot) -> char* {
        const int pos = a.seq_lens[bq] + v;
        const int lb = pos / BT;
        slot = pos - lb * BT;
        if (pos < 0 || lb >= a.max_blocks) {
            if (i == 0 && !is_v) atomicOr(a.err, TQ_DEVERR_CAPACITY);
            return nullptr;
        }
        const int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(bq) * a.max_blocks + lb])
                                   : static_cast<int64_t>(bq) * a.max_blocks + lb;
        if (pb < 0 || pb >= a.pool.num_blocks) {
            if (i == 0 && !is_v) atomicOr(a.err, TQ_DEVERR_BLOCK);
            return nullptr;
        }
        return a.pool.base + (pb * a.pool.Hkv + h) * a.pool.sub_bytes;
    };
    const int64_t o_idx = is_v ? a.pool.off[4] : a.pool.off[0];
    const int64_t o_norm = is_v ? a.pool.off[5] : a.pool.off[2];

    float z[NV];
#pragma unroll
    for (int v = 0; v < NV; ++v) z[v] = 0.0f;
    if (prod && act) {
#pragma unroll 4
        for (int k = 0; k < D; ++k) {
            const float st = St[k * D + i];
#pragma unroll
            for (int v = 0; v < NV; ++v) z[v] = __fmaf_rn(st, rs[v * D + k], z[v]);
        }
    }
    // residual norms: thread v chains vector v (ascending k)
    float g2 = 0.0f;
    if (prod && i < n)
        for (int k = 0; k < D; ++k) g2 = __fmaf_rn(rs[i * D + k], rs[i * D + k], g2);
    const int W = cd.W;
    for (int v = 0; v < n; ++v) {
        int slot = 0;
        char* sub = sub_of(v, slot);
        if (prod) {
            const unsigned bal = __ballot_sync(0xffffffffu, z[v] >= 0.0f);
            if (sub && act && (i & 31) == 0)
                reinterpret_cast<uint32_t*>(sub + a.pool.off[1])[static_cast<int64_t>(slot) * cd.Ws + (i >> 5)] = bal;
        }
        if (!sub) continue;
        if (i < W) {
            const int bit0 = 32 * i;
            const int first = bit0 / b;
            int last = (bit0 + 31) / b;
            if (last > D - 1) last = D - 1;
            uint32_t word = 0;
            for (int c = first; c <= last; ++c) {
                const int sh = c * b - bit0;
                const uint32_t cv = codes[v * D + c];
                word |= (sh >= 0) ? (cv << sh) : (cv >> (-sh));
            }
            reinterpret_cast<uint32_t*>(sub + o_idx)[static_cast<int64_t>(slot) * W + i] = word;
        }
        if (i == D - 1) reinterpret_cast<float*>(sub + o_norm)[slot] = ns[v];
        if (prod && i == v) reinterpret_cast<float*>(sub + a.pool.off[3])[slot] = __fsqrt_rn(g2);
    }
    __syncthreads();
    if (i == 0) tc::mbar_inval(bar);
    tc::grid_wait_prior();
}

}  // namespace tq

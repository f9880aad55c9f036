// Register-blocked encode for large appends (chunked prefill), MSE and prod
// codecs.
//
// Same fp32 specification as the per-vector kernel in encode.cu -- each output
// coordinate is a chain of fused multiply-adds in ascending k followed by an
// IEEE division by the norm -- so indices, signs and norms are bit-identical.
// Only the schedule differs: one CTA encodes VB vectors of one (sequence, head,
// tensor); the rotation (then the QJL matrix) streams through shared memory in
// k-chunks; each thread keeps a 4-vector x 8-coordinate block of accumulators in
// registers, so three shared-memory loads feed thirty-two fused multiply-adds.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kThreads = 256;
constexpr int kTV = 4;   // vectors per thread
constexpr int kTI = 8;   // coordinates per thread
constexpr int kKC = 32;  // matrix rows per shared-memory chunk

template <int D>
struct BlockShape {
    static constexpr int IG = D / kTI;        // coordinate groups
    static constexpr int VG = kThreads / IG;  // vector groups
    static constexpr int VB = VG * kTV;       // vectors per CTA
};

template <int D>
struct BlockSmem {
    static constexpr int VB = BlockShape<D>::VB;
    float xT[D][VB];  // inputs, then residuals (prod), transposed
    float mT[kKC][D]; // chunk of the transposed matrix
    float norm[VB];
    float rnorm[VB];
    unsigned char code[VB][D];
    unsigned char sbit[VB][D];
};

__device__ __forceinline__ float load_elem(const void* p, int dtype, int64_t i) {
    if (dtype == TQ_F32) return static_cast<const float*>(p)[i];
    if (dtype == TQ_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
    return __half2float(static_cast<const __half*>(p)[i]);
}

// acc[v][ii] = sum_k M[i0+ii][k] * xT[k][v0+v], fused multiply-adds in ascending k.
// MT is the transposed matrix in global memory (MT[k*D + i] = M[i][k]).
template <int D>
__device__ __forceinline__ void block_gemm(BlockSmem<D>& sm, const float* __restrict__ MT, int v0, int i0,
                                           float (&acc)[kTV][kTI]) {
#pragma unroll
    for (int v = 0; v < kTV; ++v)
#pragma unroll
        for (int ii = 0; ii < kTI; ++ii) acc[v][ii] = 0.0f;
    for (int k0 = 0; k0 < D; k0 += kKC) {
        __syncthreads();
        for (int e = threadIdx.x * 4; e < kKC * D; e += kThreads * 4)
            *reinterpret_cast<float4*>(&sm.mT[0][0] + e) = __ldg(reinterpret_cast<const float4*>(MT + k0 * D + e));
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kKC; ++kk) {
            const float4 xv = *reinterpret_cast<const float4*>(&sm.xT[k0 + kk][v0]);
            const float4 m0 = *reinterpret_cast<const float4*>(&sm.mT[kk][i0]);
            const float4 m1 = *reinterpret_cast<const float4*>(&sm.mT[kk][i0 + 4]);
            const float xs[4] = {xv.x, xv.y, xv.z, xv.w};
            const float ms[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
#pragma unroll
            for (int v = 0; v < kTV; ++v)
#pragma unroll
                for (int ii = 0; ii < kTI; ++ii) acc[v][ii] = __fmaf_rn(ms[ii], xs[v], acc[v][ii]);
        }
    }
}

template <int D>
__global__ void __launch_bounds__(kThreads) encode_block_kernel(EncodeAppendArgs a, int is_v) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    BlockSmem<D>& sm = *reinterpret_cast<BlockSmem<D>*>(smem_raw);
    constexpr int VB = BlockShape<D>::VB;
    constexpr int IG = BlockShape<D>::IG;
    const CodecDev& cd = is_v ? a.vc : a.kc;
    const int tid = threadIdx.x;
    const int t0 = blockIdx.x * VB;
    const int h = blockIdx.y;
    const int bq = blockIdx.z;
    const int nv = min(VB, a.n_new - t0);
    const int i0 = (tid % IG) * kTI, v0 = (tid / IG) * kTV;

    // inputs, transposed; vectors past the end are zero (never written out)
    const void* src = is_v ? a.v : a.k;
    const int64_t base = ((static_cast<int64_t>(bq) * a.pool.Hkv + h) * a.n_new + t0) * D;
    for (int e = tid; e < VB * D; e += kThreads) {
        const int v = e / D, k = e % D;
        sm.xT[k][v] = v < nv ? load_elem(src, a.dtype, base + static_cast<int64_t>(v) * D + k) : 0.0f;
    }
    __syncthreads();
    if (tid < VB) {
        float n2 = 0.0f;
        for (int k = 0; k < D; ++k) n2 = __fmaf_rn(sm.xT[k][tid], sm.xT[k][tid], n2);
        sm.norm[tid] = __fsqrt_rn(n2);
    }
    float acc[kTV][kTI];
    block_gemm<D>(sm, cd.Rt, v0, i0, acc);  // its first barrier publishes the norms

    const int b = cd.ib;
    const int nm = (1 << b) - 1;
    float res[kTV][kTI];
#pragma unroll
    for (int v = 0; v < kTV; ++v) {
        const float n = sm.norm[v0 + v];
#pragma unroll
        for (int ii = 0; ii < kTI; ++ii) {
            const float y = (n > 0.0f) ? __fdiv_rn(acc[v][ii], n) : 0.0f;
            int code = 0;
            for (int jm = 0; jm < nm; ++jm) code += (y > __ldg(cd.m + jm)) ? 1 : 0;
            sm.code[v0 + v][i0 + ii] = static_cast<unsigned char>(code);
            res[v][ii] = __fsub_rn(y, __ldg(cd.c + code));
        }
    }
    if (cd.mode == TQ_MODE_PROD) {
        __syncthreads();  // every thread is done reading the inputs
#pragma unroll
        for (int v = 0; v < kTV; ++v)
#pragma unroll
            for (int ii = 0; ii < kTI; ++ii) sm.xT[i0 + ii][v0 + v] = res[v][ii];
        __syncthreads();
        if (tid < VB) {
            float g2 = 0.0f;
            for (int k = 0; k < D; ++k) g2 = __fmaf_rn(sm.xT[k][tid], sm.xT[k][tid], g2);
            sm.rnorm[tid] = __fsqrt_rn(g2);
        }
        block_gemm<D>(sm, cd.St, v0, i0, acc);
#pragma unroll
        for (int v = 0; v < kTV; ++v)
#pragma unroll
            for (int ii = 0; ii < kTI; ++ii) sm.sbit[v0 + v][i0 + ii] = acc[v][ii] >= 0.0f ? 1 : 0;
    }
    __syncthreads();

    // records of the valid vectors: index words, sign words, then the norms
    const int W = cd.W;
    const int Ws = cd.mode == TQ_MODE_PROD ? D / 32 : 0;
    const int per = W + Ws + 1;
    const int BT = a.pool.BT;
    const int64_t o_idx = is_v ? a.pool.off[4] : a.pool.off[0];
    const int64_t o_norm = is_v ? a.pool.off[5] : a.pool.off[2];
    for (int e = tid; e < nv * per; e += kThreads) {
        const int v = e / per, f = e % per;
        const int pos = a.seq_lens[bq] + t0 + v;
        const int lb = pos / BT;
        const int slot = pos - lb * BT;
        if (pos < 0 || lb >= a.max_blocks) {
            if (f == 0) atomicOr(a.err, TQ_DEVERR_CAPACITY);
            continue;
        }
        const int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(bq) * a.max_blocks + lb])
                                   : static_cast<int64_t>(bq) * a.max_blocks + lb;
        if (pb < 0 || pb >= a.pool.num_blocks) {
            if (f == 0) atomicOr(a.err, TQ_DEVERR_BLOCK);
            continue;
        }
        char* sub = a.pool.base + (pb * a.pool.Hkv + h) * a.pool.sub_bytes;
        if (f < W) {
            const int bit0 = 32 * f;
            const int first = bit0 / b;
            int last = (bit0 + 31) / b;
            if (last > D - 1) last = D - 1;
            uint32_t word = 0;
            for (int c = first; c <= last; ++c) {
                const int sh = c * b - bit0;
                const uint32_t cv = sm.code[v][c];
                word |= (sh >= 0) ? (cv << sh) : (cv >> (-sh));
            }
            reinterpret_cast<uint32_t*>(sub + o_idx)[static_cast<int64_t>(slot) * W + f] = word;
        } else if (f < W + Ws) {
            const int w = f - W;
            uint32_t word = 0;
            for (int k = 0; k < 32; ++k) word |= static_cast<uint32_t>(sm.sbit[v][32 * w + k]) << k;
            reinterpret_cast<uint32_t*>(sub + a.pool.off[1])[static_cast<int64_t>(slot) * Ws + w] = word;
        } else {
            reinterpret_cast<float*>(sub + o_norm)[slot] = sm.norm[v];
            if (cd.mode == TQ_MODE_PROD) reinterpret_cast<float*>(sub + a.pool.off[3])[slot] = sm.rnorm[v];
        }
    }
}

template <int D>
cudaError_t launch_block(const EncodeAppendArgs& a, int is_v, cudaStream_t s) {
    const size_t smem = sizeof(BlockSmem<D>);
    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(encode_block_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(smem));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        attr_set.fetch_or(bit);
    }
    constexpr int VB = BlockShape<D>::VB;
    const dim3 grid((a.n_new + VB - 1) / VB, a.pool.Hkv, a.batch);
    encode_block_kernel<D><<<grid, kThreads, smem, s>>>(a, is_v);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
}

}  // namespace

// Blocked encode of one tensor (keys: is_v = 0, values: is_v = 1), MSE or prod codec.
cudaError_t launch_encode_block(const EncodeAppendArgs& a, int is_v, cudaStream_t s) {
    switch (a.kc.D) {
        case 64: return launch_block<64>(a, is_v, s);
        case 128: return launch_block<128>(a, is_v, s);
        case 256: return launch_block<256>(a, is_v, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace tq

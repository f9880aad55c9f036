// TurboQuant encode kernels: per-token append into the paged pool and the
// codec-only quantise.
//
// One CTA encodes one vector with one thread per coordinate. The arithmetic is
// the fp32 specification of the codec, written with explicit IEEE intrinsics
// so that no compiler contraction or reassociation can change a bit:
//   norm  n   = sqrt(sum_k x_k^2)                 (sequential fma, k ascending)
//   rotate y_i = (sum_k R_ik x_k) / n, 0 if n == 0  (sequential fma, k ascending)
//   index  i  = #{ j : y_i > m_j }                 (Lloyd-Max midpoints)
// prod keys ("turboquant/validate_moe_phase2.py", TurboQuantProd fields):
//   r = y - c[index], rnorm = sqrt(sum r_i^2), sign_j = ((S r)_j >= 0)
// group values ("turboquant/validate_moe_phase2.py", quantize_values):
//   scale = f16((max - min) / (2^b - 1)), zero = f16(min),
//   code = clamp(rint((x - zero) / scale), 0, 2^b - 1)
// Packing follows "omlx/turboquant_kv.py" (_infer_head_dim): index i occupies
// bits [i*b, i*b + b) of ceil(D*b/32) uint32 words, least significant first.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "encode_short.cuh"
#include "tc_ptx.cuh"
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kMaxD = 256;

struct VecSmem {
    float x[kMaxD];
    float r[kMaxD];
    unsigned char code[kMaxD];
    __half gscale[kMaxD / 8];
    __half gmin[kMaxD / 8];
};

// Record destinations for one vector. Unused pointers are null.
struct RecordOut {
    uint32_t* idx;
    uint32_t* sgn;
    float* norm;
    float* rnorm;
    __half* scale;
    __half* zero;
};

// Encode the vector in sm.x (blockDim.x == D threads).
__device__ void encode_vector(const CodecDev& cd, VecSmem& sm, const RecordOut& out) {
    const int D = cd.D;
    const int i = threadIdx.x;
    int b;
    if (cd.mode == TQ_MODE_GROUP) {
        b = cd.bits;
        const int g = cd.group;
        const int qmax = (1 << b) - 1;
        if (i < D / g) {
            float lo = sm.x[i * g], hi = sm.x[i * g];
            for (int k = 1; k < g; ++k) {
                const float t = sm.x[i * g + k];
                lo = (t < lo) ? t : lo;
                hi = (t > hi) ? t : hi;
            }
            const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), static_cast<float>(qmax)));
            const __half mh = __float2half_rn(lo);
            sm.gscale[i] = sh;
            sm.gmin[i] = mh;
            if (out.scale) out.scale[i] = sh;
            if (out.zero) out.zero[i] = mh;
        }
        __syncthreads();
        const float sf = __half2float(sm.gscale[i / g]);
        const float mf = __half2float(sm.gmin[i / g]);
        int q = 0;
        if (sf != 0.0f) {
            const float r = rintf(__fdiv_rn(__fsub_rn(sm.x[i], mf), sf));
            q = !(r > 0.0f) ? 0 : (r > static_cast<float>(qmax) ? qmax : static_cast<int>(r));
        }
        sm.code[i] = static_cast<unsigned char>(q);
    } else {
        b = cd.ib;
        float n2 = 0.0f;
        for (int k = 0; k < D; ++k) n2 = __fmaf_rn(sm.x[k], sm.x[k], n2);
        const float n = __fsqrt_rn(n2);
        float t = 0.0f;
#pragma unroll 32
        for (int k = 0; k < D; ++k) t = __fmaf_rn(__ldg(cd.Rt + k * D + i), sm.x[k], t);
        const float y = (n > 0.0f) ? __fdiv_rn(t, n) : 0.0f;
        const int nm = (1 << b) - 1;
        int code = 0;
        for (int j = 0; j < nm; ++j) code += (y > __ldg(cd.m + j)) ? 1 : 0;
        sm.code[i] = static_cast<unsigned char>(code);
        if (i == 0 && out.norm) *out.norm = n;
        if (cd.mode == TQ_MODE_PROD) {
            sm.r[i] = __fsub_rn(y, __ldg(cd.c + code));
            __syncthreads();
            float g2 = 0.0f;
            for (int k = 0; k < D; ++k) g2 = __fmaf_rn(sm.r[k], sm.r[k], g2);
            if (i == 0 && out.rnorm) *out.rnorm = __fsqrt_rn(g2);
            float z = 0.0f;
#pragma unroll 32
            for (int k = 0; k < D; ++k) z = __fmaf_rn(__ldg(cd.St + k * D + i), sm.r[k], z);
            const unsigned bal = __ballot_sync(0xffffffffu, z >= 0.0f);
            if ((i & 31) == 0 && out.sgn) out.sgn[i >> 5] = bal;
        }
    }
    __syncthreads();
    // pack: thread w assembles word w from the codes overlapping bits [32w, 32w+32)
    const int W = (D * b + 31) / 32;
    if (i < W && out.idx) {
        const int bit0 = 32 * i;
        const int first = bit0 / b;
        int last = (bit0 + 31) / b;
        if (last > D - 1) last = D - 1;
        uint32_t word = 0;
        for (int c = first; c <= last; ++c) {
            const int sh = c * b - bit0;
            const uint32_t v = sm.code[c];
            word |= (sh >= 0) ? (v << sh) : (v >> (-sh));
        }
        out.idx[i] = word;
    }
}

// which: 0 = keys and values (grid z = 2 * batch), 1 = keys only, 2 = values only.
__global__ void encode_append_kernel(EncodeAppendArgs a, int which) {
    __shared__ VecSmem sm;
    const int t = blockIdx.x;
    const int h = blockIdx.y;
    const int bq = which == 0 ? (blockIdx.z >> 1) : blockIdx.z;
    const bool is_v = which == 0 ? (blockIdx.z & 1) : which == 2;
    const CodecDev& cd = is_v ? a.vc : a.kc;
    const int D = cd.D;
    const int i = threadIdx.x;

    const int pos = a.seq_lens[bq] + t;
    const int BT = a.pool.BT;
    const int lb = pos / BT;
    const int slot = pos - lb * BT;
    if (pos < 0 || lb >= a.max_blocks) {
        if (i == 0 && !is_v) atomicOr(a.err, TQ_DEVERR_CAPACITY);
        return;
    }
    const int64_t pb = a.table ? static_cast<int64_t>(a.table[static_cast<int64_t>(bq) * a.max_blocks + lb])
                               : static_cast<int64_t>(bq) * a.max_blocks + lb;
    if (pb < 0 || pb >= a.pool.num_blocks) {
        if (i == 0 && !is_v) atomicOr(a.err, TQ_DEVERR_BLOCK);
        return;
    }
    const int64_t src = ((static_cast<int64_t>(bq) * a.pool.Hkv + h) * a.n_new + t) * D;
    sm.x[i] = load_elem(is_v ? a.v : a.k, a.dtype, src + i);
    __syncthreads();

    char* base = a.pool.base + (pb * a.pool.Hkv + h) * a.pool.sub_bytes;
    RecordOut o{};
    if (!is_v) {
        o.idx = reinterpret_cast<uint32_t*>(base + a.pool.off[0]) + static_cast<int64_t>(slot) * cd.W;
        if (cd.mode == TQ_MODE_PROD) {
            o.sgn = reinterpret_cast<uint32_t*>(base + a.pool.off[1]) + static_cast<int64_t>(slot) * cd.Ws;
            o.rnorm = reinterpret_cast<float*>(base + a.pool.off[3]) + slot;
        }
        o.norm = reinterpret_cast<float*>(base + a.pool.off[2]) + slot;
    } else {
        o.idx = reinterpret_cast<uint32_t*>(base + a.pool.off[4]) + static_cast<int64_t>(slot) * cd.W;
        if (cd.mode == TQ_MODE_GROUP) {
            const int ng = D / cd.group;
            o.scale = reinterpret_cast<__half*>(base + a.pool.off[5]) + static_cast<int64_t>(slot) * ng;
            o.zero = reinterpret_cast<__half*>(base + a.pool.off[6]) + static_cast<int64_t>(slot) * ng;
        } else {
            o.norm = reinterpret_cast<float*>(base + a.pool.off[5]) + slot;
        }
    }
    encode_vector(cd, sm, o);
}

__global__ void quantize_kernel(QuantizeArgs a) {
    __shared__ VecSmem sm;
    const CodecDev& cd = a.cd;
    const int D = cd.D;
    const int64_t v = blockIdx.x + static_cast<int64_t>(blockIdx.y) * gridDim.x;
    if (v >= a.n) return;
    sm.x[threadIdx.x] = load_elem(a.x, a.dtype, v * D + threadIdx.x);
    __syncthreads();
    RecordOut o{};
    o.idx = a.idx ? a.idx + v * cd.W : nullptr;
    if (cd.mode == TQ_MODE_GROUP) {
        const int ng = D / cd.group;
        o.scale = a.aux0 ? static_cast<__half*>(a.aux0) + v * ng : nullptr;
        o.zero = a.aux1 ? static_cast<__half*>(a.aux1) + v * ng : nullptr;
    } else {
        o.norm = a.aux0 ? static_cast<float*>(a.aux0) + v : nullptr;
        if (cd.mode == TQ_MODE_PROD) {
            o.sgn = a.aux1 ? static_cast<uint32_t*>(a.aux1) + v * cd.Ws : nullptr;
            o.rnorm = a.aux2 ? static_cast<float*>(a.aux2) + v : nullptr;
        }
    }
    encode_vector(cd, sm, o);
}

// Short appends: the body lives in encode_short.cuh (shared with the fused
// decode-step preparation kernel).
template <int D, int NV>
__global__ void __launch_bounds__(D) encode_short_kernel(EncodeAppendArgs a) {
    extern __shared__ __align__(16) unsigned char smem_raw[];
    encode_short_body<D, NV>(a, blockIdx.x, blockIdx.y, blockIdx.z, smem_raw);
}

template <int D, int NV>
cudaError_t launch_short(const EncodeAppendArgs& a, bool values_rotated, cudaStream_t s) {
    const bool two = a.kc.mode == TQ_MODE_PROD || (values_rotated && a.vc.mode == TQ_MODE_PROD);
    const size_t smem = encode_short_smem<D, NV>(two);
    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        cudaError_t e = cudaFuncSetAttribute(encode_short_kernel<D, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             static_cast<int>(encode_short_smem<D, NV>(true)));
        if (e != cudaSuccess) {
            (void)cudaGetLastError();
            return e;
        }
        attr_set.fetch_or(bit);
    }
    const dim3 grid(a.pool.Hkv, a.batch, values_rotated ? 2 : 1);
    const cudaError_t e = launch_overlapped(encode_short_kernel<D, NV>, grid, dim3(D), smem, s, a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return e;
}

template <int D>
cudaError_t launch_short_nv(const EncodeAppendArgs& a, bool values_rotated, cudaStream_t s) {
    if (a.n_new <= 2) return launch_short<D, 2>(a, values_rotated, s);
    if (a.n_new <= 8) return launch_short<D, 8>(a, values_rotated, s);
    return launch_short<D, 32>(a, values_rotated, s);
}

}  // namespace

cudaError_t launch_encode_append(const EncodeAppendArgs& a, cudaStream_t s) {
    if (a.batch == 0 || a.n_new == 0) return cudaSuccess;
    // Short appends (decode steps): one CTA per vector. Long appends (prefill
    // chunks): the register-blocked kernel for rotated codecs.
    constexpr int kBlockedFrom = 32;
    if (a.n_new < kBlockedFrom) {
        // rotated keys (and values) with head_dim <= 128: tables staged in shared memory
        const bool vrot = a.vc.mode != TQ_MODE_GROUP;
        if (a.kc.mode != TQ_MODE_GROUP && a.kc.D <= 128) {
            cudaError_t e = a.kc.D == 64 ? launch_short_nv<64>(a, vrot, s) : launch_short_nv<128>(a, vrot, s);
            if (e != cudaSuccess || vrot) return e;
            dim3 grid(a.n_new, a.pool.Hkv, a.batch);
            encode_append_kernel<<<grid, a.vc.D, 0, s>>>(a, 2);
            g_launches.fetch_add(1, std::memory_order_relaxed);
            return cudaGetLastError();
        }
        dim3 grid(a.n_new, a.pool.Hkv, a.batch * 2);
        encode_append_kernel<<<grid, a.kc.D, 0, s>>>(a, 0);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        return cudaGetLastError();
    }
    // Chunks of >= 64 tokens rotate on the tensor cores unless the caller asked
    // for the sequential fp32 order (inputs must be 16-byte aligned rows).
    constexpr int kTensorFrom = 64;
    const bool aligned = (reinterpret_cast<uintptr_t>(a.k) % 16 == 0) && (reinterpret_cast<uintptr_t>(a.v) % 16 == 0);
    const bool tc_ok = !a.exact && a.n_new >= kTensorFrom && aligned;
    if (tc_ok && encode_tc_supported(a, 0) && encode_tc_supported(a, 1)) {
        cudaError_t pe = cudaSuccess;
        if (launch_encode_tc_pair(a, s, &pe)) return pe;   // keys and values in one launch
    }
    cudaError_t e = (tc_ok && encode_tc_supported(a, 0)) ? launch_encode_tc(a, 0, s) : launch_encode_block(a, 0, s);
    if (e != cudaSuccess) return e;
    if (a.vc.mode == TQ_MODE_GROUP) {
        dim3 grid(a.n_new, a.pool.Hkv, a.batch);
        encode_append_kernel<<<grid, a.vc.D, 0, s>>>(a, 2);
        g_launches.fetch_add(1, std::memory_order_relaxed);
        return cudaGetLastError();
    }
    return (tc_ok && encode_tc_supported(a, 1)) ? launch_encode_tc(a, 1, s) : launch_encode_block(a, 1, s);
}

cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t s) {
    if (a.n == 0) return cudaSuccess;
    const int64_t gx = a.n < 65535 ? a.n : 65535;
    const int64_t gy = (a.n + gx - 1) / gx;
    quantize_kernel<<<dim3(static_cast<unsigned>(gx), static_cast<unsigned>(gy)), a.cd.D, 0, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
}

}  // namespace tq

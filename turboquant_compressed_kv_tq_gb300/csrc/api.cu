// C ABI of libtq: codec lifetime, cache layout, argument checks and launches.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <new>

#include "tq_internal.h"

namespace tq {

std::atomic<uint64_t> g_launches{0};

namespace {

// Per-device error word written by the kernels (see tq_device_error).
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;
unsigned* g_err_ptr[kMaxDevices] = {};
int g_num_sms[kMaxDevices] = {};
std::mutex g_dev_mu;

tq_status device_state(unsigned** err, int* num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_err_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return TQ_ERR_CUDA;
        // the allocation-free decode's fixed scratch array is reserved here, when
        // the library is first set up on the device, not by that entry point
        if (noalloc_reserve() != TQ_OK) return TQ_ERR_CUDA;
        int sms = 0;
        if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return TQ_ERR_CUDA;
        g_err_ptr[dev] = static_cast<unsigned*>(p);
        g_num_sms[dev] = sms;
    }
    if (err) *err = g_err_ptr[dev];
    if (num_sms) *num_sms = g_num_sms[dev];
    return TQ_OK;
}

// The bounded-wait error path, on its own: one thread waits on an mbarrier
// that nothing arrives on (mbarrier.try_wait.parity in a loop, as the kernels
// wait for their bulk copies), bounded by a deadline on the global timer (and,
// as a backstop, by an iteration count); when the deadline passes it sets
// TQ_DEVERR_TIMEOUT, invalidates the barrier and returns.
__global__ void wait_timeout_kernel(unsigned* err, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t a = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;\n" ::"r"(a) : "memory");
    unsigned long long t0, t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t0));
    bool done = false;
    for (unsigned it = 0; it < (1u << 24) && !done; ++it) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(a), "r"(0u), "r"(1000u)
            : "memory");
        done = ok != 0;
        asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
        if (t - t0 > limit_ns) break;
    }
    if (!done) atomicOr(err, TQ_DEVERR_TIMEOUT);
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(a) : "memory");
}

int index_bits_of(int bits, int mode) { return mode == TQ_MODE_PROD ? bits - 1 : bits; }

int record_bytes_of(int D, int bits, int mode, int group) {
    const int w = (D * index_bits_of(bits, mode) + 31) / 32;
    if (mode == TQ_MODE_MSE) return 4 * w + 4;
    if (mode == TQ_MODE_PROD) return 4 * w + 4 * (D / 32) + 8;
    return 4 * w + 4 * (D / group);
}

bool head_dim_ok(int D) { return D == 64 || D == 128 || D == 256; }

void free_codec(tq_codec* c) {
    if (!c) return;
    int prev = -1;
    cudaGetDevice(&prev);
    if (c->device >= 0) cudaSetDevice(c->device);
    cudaFree(c->d_R);
    cudaFree(c->d_Rt);
    cudaFree(c->d_St);
    cudaFree(c->d_SRt);
    cudaFree(c->d_c);
    cudaFree(c->d_m);
    cudaFree(c->d_cq);
    cudaFree(c->d_Rtc);
    cudaFree(c->d_Stc);
    cudaFree(c->d_quad);
    cudaFree(c->d_pair);
    cudaFree(c->d_pair4);
    cudaFree(c->d_pair4w);
    if (prev >= 0) cudaSetDevice(prev);
    delete c;
}

template <typename T>
tq_status upload(T** dst, const std::vector<T>& src) {
    if (src.empty()) return TQ_OK;
    if (cudaMalloc(reinterpret_cast<void**>(dst), src.size() * sizeof(T)) != cudaSuccess) return TQ_ERR_OOM;
    if (cudaMemcpy(*dst, src.data(), src.size() * sizeof(T), cudaMemcpyHostToDevice) != cudaSuccess)
        return TQ_ERR_CUDA;
    return TQ_OK;
}

// fp16 bits of a float that is exactly an fp16 value (the operand levels are)
uint32_t half_bits_exact(float f) {
    uint32_t u;
    std::memcpy(&u, &f, 4);
    const uint32_t sign = (u >> 16) & 0x8000u;
    const int e = static_cast<int>((u >> 23) & 0xFFu) - 127;
    const uint32_t mant = u & 0x7FFFFFu;
    if ((u & 0x7FFFFFFFu) == 0) return sign;
    if (e >= -14) return sign | (static_cast<uint32_t>(e + 15) << 10) | (mant >> 13);
    return sign | ((mant | 0x800000u) >> (-e - 1));  // subnormal half: value 2^-24 x m
}

// Decode lookup tables of an MSE codebook in the split kernel's shared-memory
// layout (bank copies included): code quads for 2 index bits, code pairs for 3.
std::vector<uint32_t> quad_table(const std::vector<float>& cq) {
    std::vector<uint32_t> t(256 * 16 * 2);
    for (int i = 0; i < 256 * 16; ++i) {
        const int e = i >> 4;
        t[2 * i] = half_bits_exact(cq[e & 3]) | (half_bits_exact(cq[(e >> 2) & 3]) << 16);
        t[2 * i + 1] = half_bits_exact(cq[(e >> 4) & 3]) | (half_bits_exact(cq[e >> 6]) << 16);
    }
    return t;
}

std::vector<uint32_t> pair_table(const std::vector<float>& cq) {
    std::vector<uint32_t> t(64 * 32);
    for (int i = 0; i < 64 * 32; ++i) {
        const int e = i >> 5;
        t[i] = half_bits_exact(cq[e & 7]) | (half_bits_exact(cq[e >> 3]) << 16);
    }
    return t;
}

// 4-bit code pairs: entry e (a byte of two codes) at 128 e + 4 c for bank copy c < 32.
std::vector<uint32_t> pair4_table(const std::vector<float>& cq) {
    std::vector<uint32_t> t(256 * 32);
    for (int i = 0; i < 256 * 32; ++i) {
        const int e = i >> 5;
        t[i] = half_bits_exact(cq[e & 15]) | (half_bits_exact(cq[e >> 4]) << 16);
    }
    return t;
}

// The same pairs in 256-byte entries: entry e at 256 e + 4 c for c < 64 (the
// byte of codes itself times 256 is the entry's offset: one byte permute
// forms a lane's address).
std::vector<uint32_t> pair4w_table(const std::vector<float>& cq) {
    std::vector<uint32_t> t(256 * 64);
    for (int i = 0; i < 256 * 64; ++i) {
        const int e = i >> 6;
        t[i] = half_bits_exact(cq[e & 15]) | (half_bits_exact(cq[e >> 4]) << 16);
    }
    return t;
}

std::vector<float> transpose(const std::vector<float>& a, int D) {
    std::vector<float> t(a.size());
    for (int i = 0; i < D; ++i)
        for (int k = 0; k < D; ++k) t[static_cast<size_t>(k) * D + i] = a[static_cast<size_t>(i) * D + k];
    return t;
}

// Transposed product (S R)^T of two D x D row-major matrices, accumulated in
// fp64 over ascending k and rounded once to fp32: entry [k][i] = sum_j S[i][j] R[j][k].
std::vector<float> product_transposed(const std::vector<float>& S, const std::vector<float>& R, int D) {
    std::vector<float> t(S.size());
    std::vector<double> row(D);
    for (int i = 0; i < D; ++i) {
        for (int k = 0; k < D; ++k) row[k] = 0.0;
        for (int j = 0; j < D; ++j) {
            const double sij = S[static_cast<size_t>(i) * D + j];
            const float* rj = R.data() + static_cast<size_t>(j) * D;
            for (int k = 0; k < D; ++k) row[k] += sij * rj[k];
        }
        for (int k = 0; k < D; ++k) t[static_cast<size_t>(k) * D + i] = static_cast<float>(row[k]);
    }
    return t;
}

CodecDev dev_view(const tq_codec* c) {
    CodecDev d{};
    d.R = c->d_R;
    d.Rt = c->d_Rt;
    d.St = c->d_St;
    d.SRt = c->d_SRt;
    d.c = c->d_c;
    d.m = c->d_m;
    d.cq = c->d_cq;
    d.cq_scale = c->host.op_scale;
    d.Rtc = c->d_Rtc;
    d.Stc = c->d_Stc;
    d.quad = c->d_quad;
    d.pair = c->d_pair;
    d.pair4 = c->d_pair4;
    d.pair4w = c->d_pair4w;
    d.D = c->head_dim;
    d.mode = c->mode;
    d.bits = c->bits;
    d.ib = c->index_bits;
    d.W = c->index_words;
    d.Ws = c->sign_words;
    d.group = c->group;
    return d;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

tq_status check_codecs_vs_cache(const tq_codec* kc, const tq_codec* vc, const tq_cache_desc* d) {
    if (!kc || !vc || !d) return TQ_ERR_INVALID_ARG;
    if (kc->mode == TQ_MODE_GROUP || vc->mode == TQ_MODE_PROD) return TQ_ERR_UNSUPPORTED;
    if (kc->head_dim != d->head_dim || vc->head_dim != d->head_dim) return TQ_ERR_CONFIG_MISMATCH;
    if (kc->mode != d->key_mode || kc->bits != d->key_bits || kc->seed != d->key_seed)
        return TQ_ERR_CONFIG_MISMATCH;
    if (vc->mode != d->value_mode || vc->bits != d->value_bits) return TQ_ERR_CONFIG_MISMATCH;
    if (vc->mode == TQ_MODE_GROUP ? vc->group != d->value_group : vc->seed != d->value_seed)
        return TQ_ERR_CONFIG_MISMATCH;
    if (!d->pool || !aligned16(d->pool) || d->num_blocks <= 0 || d->num_kv_heads <= 0) return TQ_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (kc->device != dev || vc->device != dev) return TQ_ERR_INVALID_ARG;
    return TQ_OK;
}

PoolDev pool_view(const tq_cache_desc* d, int layer) {
    PoolDev p{};
    p.base = static_cast<char*>(d->pool) + d->layer_stride * layer;
    p.sub_bytes = d->subblock_bytes;
    for (int i = 0; i < 7; ++i) p.off[i] = d->stream_offset[i];
    p.Hkv = d->num_kv_heads;
    p.BT = d->block_tokens;
    p.num_blocks = d->num_blocks;
    return p;
}

// The mixed-configuration guard of BatchTurboQuantKVCache.merge ("omlx/
// turboquant_kv.py"): caches share blocks only under one layout and codec
// configuration.
bool same_config(const tq_cache_desc* a, const tq_cache_desc* b) {
    return a->head_dim == b->head_dim && a->num_kv_heads == b->num_kv_heads && a->block_tokens == b->block_tokens &&
           a->num_layers == b->num_layers && a->key_mode == b->key_mode && a->key_bits == b->key_bits &&
           a->key_seed == b->key_seed && a->value_mode == b->value_mode && a->value_bits == b->value_bits &&
           a->value_group == b->value_group && a->value_seed == b->value_seed &&
           a->subblock_bytes == b->subblock_bytes;
}

bool same_pool(const tq_cache_desc* a, const tq_cache_desc* b) {
    return a->pool == b->pool && a->layer_stride == b->layer_stride && a->num_blocks == b->num_blocks;
}

bool ranges_overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Host checks common to the batch operations: a usable view of a batch.
tq_status check_batch(const tq_batch* t) {
    if (!t || !t->cache || !t->block_table || !t->seq_lens) return TQ_ERR_INVALID_ARG;
    const tq_cache_desc* c = t->cache;
    if (!c->pool || c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->num_layers <= 0 || c->num_layers > 65535 ||
        c->block_tokens < 16 || (c->block_tokens & (c->block_tokens - 1)) != 0 || c->subblock_bytes <= 0 ||
        c->subblock_bytes % 16 != 0)
        return TQ_ERR_INVALID_ARG;
    if (t->batch < 0 || t->capacity < t->batch || t->max_blocks <= 0) return TQ_ERR_INVALID_ARG;
    if (static_cast<int64_t>(t->max_blocks) * c->block_tokens > 2147483647) return TQ_ERR_INVALID_ARG;
    return TQ_OK;
}

bool batch_arrays_overlap(const tq_batch* a, const tq_batch* b) {
    const size_t ta = static_cast<size_t>(a->capacity) * a->max_blocks * 4, tb = static_cast<size_t>(b->capacity) * b->max_blocks * 4;
    const size_t la = static_cast<size_t>(a->capacity) * 4, lb = static_cast<size_t>(b->capacity) * 4;
    return ranges_overlap(a->block_table, ta, b->block_table, tb) || ranges_overlap(a->seq_lens, la, b->seq_lens, lb) ||
           ranges_overlap(a->block_table, ta, b->seq_lens, lb) || ranges_overlap(a->seq_lens, la, b->block_table, tb);
}

// Rows [0, n) of src (from row src_row0) appended to dst at dst_row0, in
// chunks; blocks copied from the free list unless the two share a pool.
tq_status append_rows(const tq_batch* src, int src_row0, int n, tq_batch* dst, int dst_row0,
                      const int32_t* free_blocks, int n_free, int32_t* n_used, cudaStream_t s) {
    const bool copy = !same_pool(src->cache, dst->cache);
    if (copy && (!n_used || (n_free > 0 && !free_blocks) || n_free < 0)) return TQ_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (device_state(&err, nullptr) != TQ_OK) return TQ_ERR_CUDA;
    for (int c = 0; c < n; c += kBatchRowChunk) {
        const int m = n - c < kBatchRowChunk ? n - c : kBatchRowChunk;
        if (launch_batch_rows(src, dst, m, nullptr, src_row0 + c, dst_row0 + c, copy, free_blocks, n_free, n_used,
                              0, nullptr, nullptr, nullptr, false, err, s) != cudaSuccess)
            return TQ_ERR_CUDA;
    }
    return TQ_OK;
}

}  // namespace
}  // namespace tq

using namespace tq;

extern "C" {

int tq_abi_version(void) { return TQ_ABI_VERSION; }

uint64_t tq_launch_count(void) { return g_launches.load(); }

const char* tq_status_string(tq_status s) {
    switch (s) {
        case TQ_OK: return "ok";
        case TQ_ERR_INVALID_ARG: return "invalid argument";
        case TQ_ERR_UNSUPPORTED: return "unsupported head_dim/bits/mode";
        case TQ_ERR_CONFIG_MISMATCH: return "codec does not match the cache descriptor";
        case TQ_ERR_CAPACITY: return "capacity exceeded";
        case TQ_ERR_OOM: return "out of device memory";
        case TQ_ERR_CUDA: return "CUDA error";
        case TQ_ERR_DEVICE_BOUNDS: return "device reported an out-of-range index";
    }
    return "unknown status";
}

tq_status tq_codec_create(int head_dim, int bits, tq_mode mode, uint64_t seed, tq_codec** out) {
    if (!out) return TQ_ERR_INVALID_ARG;
    *out = nullptr;
    if (!head_dim_ok(head_dim)) return TQ_ERR_UNSUPPORTED;
    if (mode == TQ_MODE_MSE) {
        if (bits < 1 || bits > 4) return TQ_ERR_UNSUPPORTED;
    } else if (mode == TQ_MODE_PROD) {
        if (bits < 2 || bits > 5) return TQ_ERR_UNSUPPORTED;
    } else {
        return TQ_ERR_UNSUPPORTED;
    }
    tq_codec* c = new (std::nothrow) tq_codec();
    if (!c) return TQ_ERR_OOM;
    c->head_dim = head_dim;
    c->bits = bits;
    c->mode = mode;
    c->seed = seed;
    c->index_bits = index_bits_of(bits, mode);
    c->index_words = (head_dim * c->index_bits + 31) / 32;
    c->sign_words = mode == TQ_MODE_PROD ? head_dim / 32 : 0;
    c->record_bytes = record_bytes_of(head_dim, bits, mode, 0);
    if (cudaGetDevice(&c->device) != cudaSuccess) {
        delete c;
        return TQ_ERR_CUDA;
    }
    build_codec_tables(head_dim, c->index_bits, mode == TQ_MODE_PROD, seed, c->host);
    tq_status st = upload(&c->d_R, c->host.rotation);
    if (st == TQ_OK) st = upload(&c->d_Rt, transpose(c->host.rotation, head_dim));
    if (st == TQ_OK && mode == TQ_MODE_PROD) st = upload(&c->d_St, transpose(c->host.qjl, head_dim));
    // q'' = (S R) q in one pass with q' = R q: the query prep of the tensor-core
    // decode at head_dims other than 128
    if (st == TQ_OK && mode == TQ_MODE_PROD && head_dim != 128)
        st = upload(&c->d_SRt, product_transposed(c->host.qjl, c->host.rotation, head_dim));
    if (st == TQ_OK) st = upload(&c->d_c, c->host.centroids);
    if (st == TQ_OK) st = upload(&c->d_m, c->host.midpoints);
    if (st == TQ_OK) st = upload(&c->d_cq, c->host.op_levels);
    if (st == TQ_OK && c->index_bits == 2) st = upload(&c->d_quad, quad_table(c->host.op_levels));
    if (st == TQ_OK && c->index_bits == 3) st = upload(&c->d_pair, pair_table(c->host.op_levels));
    if (st == TQ_OK && c->index_bits == 4 && mode == TQ_MODE_MSE)
        st = upload(&c->d_pair4, pair4_table(c->host.op_levels));
    if (st == TQ_OK && c->index_bits == 4 && mode == TQ_MODE_MSE)
        st = upload(&c->d_pair4w, pair4w_table(c->host.op_levels));
    if (st == TQ_OK && head_dim <= 128) {
        // tensor-core operands for the chunked-prefill encoder: 16 R and S, fp16 hi + lo
        std::vector<uint16_t> op;
        build_tc_operand(c->host.rotation, head_dim, 16.0, op);
        st = upload(&c->d_Rtc, op);
        if (st == TQ_OK && mode == TQ_MODE_PROD) {
            build_tc_operand(c->host.qjl, head_dim, 1.0, op);
            st = upload(&c->d_Stc, op);
        }
    }
    if (st == TQ_OK && device_state(nullptr, nullptr) != TQ_OK) st = TQ_ERR_CUDA;
    if (st != TQ_OK) {
        free_codec(c);
        return st;
    }
    *out = c;
    return TQ_OK;
}

tq_status tq_bits_split(double bits, int* key_bits, int* value_bits) {
    if (!key_bits || !value_bits) return TQ_ERR_INVALID_ARG;
    *key_bits = *value_bits = 0;
    if (!(bits > -1e9 && bits < 1e9)) return TQ_ERR_UNSUPPORTED;  // NaN, infinities, absurd widths
    int kb, vb;
    if (std::fabs(bits - std::nearbyint(bits)) <= 1e-6) {
        kb = vb = static_cast<int>(bits);  // an integer width converts by truncation, as printed
    } else {
        kb = static_cast<int>(std::floor(bits));
        vb = static_cast<int>(std::ceil(bits));
    }
    if (kb < 1 || vb > 4) return TQ_ERR_UNSUPPORTED;
    *key_bits = kb;
    *value_bits = vb;
    return TQ_OK;
}

tq_status tq_codec_pair_for_bits(int head_dim, double bits, uint64_t seed, tq_codec** key_codec,
                                 tq_codec** value_codec) {
    if (!key_codec || !value_codec) return TQ_ERR_INVALID_ARG;
    *key_codec = *value_codec = nullptr;
    int kb = 0, vb = 0;
    tq_status st = tq_bits_split(bits, &kb, &vb);
    if (st != TQ_OK) return st;
    tq_codec* kc = nullptr;
    tq_codec* vc = nullptr;
    st = tq_codec_create(head_dim, kb, TQ_MODE_MSE, seed, &kc);
    if (st == TQ_OK) st = tq_codec_create(head_dim, vb, TQ_MODE_MSE, seed + 1, &vc);
    if (st != TQ_OK) {
        tq_codec_destroy(kc);
        tq_codec_destroy(vc);
        return st;
    }
    *key_codec = kc;
    *value_codec = vc;
    return TQ_OK;
}

tq_status tq_codec_create_group(int head_dim, int bits, int group_size, tq_codec** out) {
    if (!out) return TQ_ERR_INVALID_ARG;
    *out = nullptr;
    if (!head_dim_ok(head_dim)) return TQ_ERR_UNSUPPORTED;
    if (bits != 2 && bits != 4) return TQ_ERR_UNSUPPORTED;
    if (group_size != 32 && group_size != 64 && group_size != 128) return TQ_ERR_UNSUPPORTED;
    if (head_dim % group_size != 0) return TQ_ERR_UNSUPPORTED;
    tq_codec* c = new (std::nothrow) tq_codec();
    if (!c) return TQ_ERR_OOM;
    c->head_dim = head_dim;
    c->bits = bits;
    c->mode = TQ_MODE_GROUP;
    c->group = group_size;
    c->index_bits = bits;
    c->index_words = (head_dim * bits + 31) / 32;
    c->record_bytes = record_bytes_of(head_dim, bits, TQ_MODE_GROUP, group_size);
    if (cudaGetDevice(&c->device) != cudaSuccess || device_state(nullptr, nullptr) != TQ_OK) {
        delete c;
        return TQ_ERR_CUDA;
    }
    *out = c;
    return TQ_OK;
}

void tq_codec_destroy(tq_codec* codec) { free_codec(codec); }

tq_status tq_codec_info(const tq_codec* c, tq_codec_info_t* out) {
    if (!c || !out) return TQ_ERR_INVALID_ARG;
    out->head_dim = c->head_dim;
    out->bits = c->bits;
    out->mode = c->mode;
    out->group_size = c->group;
    out->seed = c->seed;
    out->index_bits = c->index_bits;
    out->index_words = c->index_words;
    out->sign_words = c->sign_words;
    out->record_bytes = c->record_bytes;
    out->device = c->device;
    return TQ_OK;
}

tq_status tq_codec_build_host(int head_dim, int bits, tq_mode mode, uint64_t seed, float* rotation, float* qjl,
                              float* centroids, float* midpoints) {
    if (!head_dim_ok(head_dim)) return TQ_ERR_UNSUPPORTED;
    if (mode == TQ_MODE_MSE ? (bits < 1 || bits > 4) : mode == TQ_MODE_PROD ? (bits < 2 || bits > 5) : true)
        return TQ_ERR_UNSUPPORTED;
    HostTables t;
    build_codec_tables(head_dim, index_bits_of(bits, mode), mode == TQ_MODE_PROD, seed, t);
    if (rotation) std::memcpy(rotation, t.rotation.data(), t.rotation.size() * sizeof(float));
    if (qjl && !t.qjl.empty()) std::memcpy(qjl, t.qjl.data(), t.qjl.size() * sizeof(float));
    if (centroids) std::memcpy(centroids, t.centroids.data(), t.centroids.size() * sizeof(float));
    if (midpoints) std::memcpy(midpoints, t.midpoints.data(), t.midpoints.size() * sizeof(float));
    return TQ_OK;
}

tq_status tq_codec_export(const tq_codec* c, float* rotation, float* qjl, float* centroids, float* midpoints) {
    if (!c || c->mode == TQ_MODE_GROUP) return TQ_ERR_INVALID_ARG;
    const auto& h = c->host;
    if (rotation) std::memcpy(rotation, h.rotation.data(), h.rotation.size() * sizeof(float));
    if (qjl) {
        if (h.qjl.empty()) return TQ_ERR_INVALID_ARG;
        std::memcpy(qjl, h.qjl.data(), h.qjl.size() * sizeof(float));
    }
    if (centroids) std::memcpy(centroids, h.centroids.data(), h.centroids.size() * sizeof(float));
    if (midpoints) std::memcpy(midpoints, h.midpoints.data(), h.midpoints.size() * sizeof(float));
    return TQ_OK;
}

tq_status tq_cache_desc_init(tq_cache_desc* d, const tq_codec* kc, const tq_codec* vc, int num_layers,
                             int num_blocks, int block_tokens, int num_kv_heads, void* pool,
                             size_t pool_bytes, size_t* required_bytes) {
    if (!d || !kc || !vc) return TQ_ERR_INVALID_ARG;
    if (kc->head_dim != vc->head_dim) return TQ_ERR_CONFIG_MISMATCH;
    if (kc->mode == TQ_MODE_GROUP || vc->mode == TQ_MODE_PROD) return TQ_ERR_UNSUPPORTED;
    if (num_layers <= 0 || num_blocks <= 0 || num_kv_heads <= 0) return TQ_ERR_INVALID_ARG;
    if (block_tokens < 16 || block_tokens > 65536 || (block_tokens & (block_tokens - 1)) != 0)
        return TQ_ERR_INVALID_ARG;
    if (pool && !aligned16(pool)) return TQ_ERR_INVALID_ARG;
    std::memset(d, 0, sizeof(*d));
    const int D = kc->head_dim;
    const int64_t BT = block_tokens;
    int64_t o = 0;
    d->encode_policy = TQ_ENCODE_AUTO;
    for (int i = 0; i < 7; ++i) d->stream_offset[i] = -1;
    d->stream_offset[0] = o;
    o += BT * 4 * kc->index_words;
    if (kc->mode == TQ_MODE_PROD) {
        d->stream_offset[1] = o;
        o += BT * 4 * kc->sign_words;
    }
    d->stream_offset[2] = o;
    o += BT * 4;
    if (kc->mode == TQ_MODE_PROD) {
        d->stream_offset[3] = o;
        o += BT * 4;
    }
    d->stream_offset[4] = o;
    o += BT * 4 * vc->index_words;
    if (vc->mode == TQ_MODE_MSE) {
        d->stream_offset[5] = o;
        o += BT * 4;
    } else {
        const int64_t ng = D / vc->group;
        d->stream_offset[5] = o;
        o += BT * 2 * ng;
        d->stream_offset[6] = o;
        o += BT * 2 * ng;
    }
    d->subblock_bytes = o;
    d->layer_stride = o * num_kv_heads * static_cast<int64_t>(num_blocks);
    d->num_layers = num_layers;
    d->num_blocks = num_blocks;
    d->block_tokens = block_tokens;
    d->num_kv_heads = num_kv_heads;
    d->head_dim = D;
    d->key_mode = kc->mode;
    d->key_bits = kc->bits;
    d->key_seed = kc->seed;
    d->value_mode = vc->mode;
    d->value_bits = vc->bits;
    d->value_group = vc->group;
    d->value_seed = vc->seed;
    d->pool = pool;
    const size_t total = static_cast<size_t>(d->layer_stride) * num_layers;
    if (required_bytes) *required_bytes = total;
    if (pool && pool_bytes < total) return TQ_ERR_CAPACITY;
    return TQ_OK;
}

tq_status tq_batch_filter(const tq_batch* batch, const int32_t* keep, int n_keep, tq_batch* out, int32_t* freed,
                          int32_t* n_freed, tq_stream_t stream) {
    tq_status st = check_batch(batch);
    if (st == TQ_OK) st = check_batch(out);
    if (st != TQ_OK) return st;
    if (!same_config(batch->cache, out->cache) || !same_pool(batch->cache, out->cache)) return TQ_ERR_CONFIG_MISMATCH;
    if (n_keep < 0 || n_keep > batch->batch || (n_keep > 0 && !keep) || out->capacity < n_keep || !n_freed ||
        out->max_blocks != batch->max_blocks || batch_arrays_overlap(batch, out))
        return TQ_ERR_INVALID_ARG;
    const int n_drop = batch->batch - n_keep;
    if (n_drop > 0 && !freed) return TQ_ERR_INVALID_ARG;
    std::vector<char> kept(static_cast<size_t>(batch->batch), 0);
    for (int i = 0; i < n_keep; ++i) {
        if (keep[i] < 0 || keep[i] >= batch->batch || kept[keep[i]]) return TQ_ERR_INVALID_ARG;
        kept[keep[i]] = 1;
    }
    std::vector<int> drop;
    for (int r = 0; r < batch->batch; ++r)
        if (!kept[r]) drop.push_back(r);
    unsigned* err = nullptr;
    if (device_state(&err, nullptr) != TQ_OK) return TQ_ERR_CUDA;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int rounds = std::max(1, (std::max(n_keep, n_drop) + kBatchRowChunk - 1) / kBatchRowChunk);
    for (int c = 0; c < rounds; ++c) {
        const int r0 = c * kBatchRowChunk;
        const int m = std::max(0, std::min(kBatchRowChunk, n_keep - r0));
        const int md = std::max(0, std::min(kBatchRowChunk, n_drop - r0));
        if (launch_batch_rows(batch, out, m, m ? keep + r0 : nullptr, 0, r0, false, nullptr, 0, nullptr, md,
                              md ? drop.data() + r0 : nullptr, freed, n_freed, c == 0, err, s) != cudaSuccess)
            return TQ_ERR_CUDA;
    }
    out->batch = n_keep;
    return TQ_OK;
}

tq_status tq_batch_extend(tq_batch* dst, const tq_batch* src, const int32_t* free_blocks, int n_free,
                          int32_t* n_used, tq_stream_t stream) {
    tq_status st = check_batch(dst);
    if (st == TQ_OK) st = check_batch(src);
    if (st != TQ_OK) return st;
    if (!same_config(src->cache, dst->cache)) return TQ_ERR_CONFIG_MISMATCH;
    if (batch_arrays_overlap(src, dst)) return TQ_ERR_INVALID_ARG;
    if (static_cast<int64_t>(dst->batch) + src->batch > dst->capacity) return TQ_ERR_CAPACITY;
    st = append_rows(src, 0, src->batch, dst, dst->batch, free_blocks, n_free, n_used,
                     reinterpret_cast<cudaStream_t>(stream));
    if (st == TQ_OK) dst->batch += src->batch;
    return st;
}

tq_status tq_batch_merge(tq_batch* dst, const tq_batch* srcs, int n_srcs, const int32_t* free_blocks, int n_free,
                         int32_t* n_used, tq_stream_t stream) {
    tq_status st = check_batch(dst);
    if (st != TQ_OK) return st;
    if (n_srcs < 0 || (n_srcs > 0 && !srcs)) return TQ_ERR_INVALID_ARG;
    int64_t rows = dst->batch;
    for (int i = 0; i < n_srcs; ++i) {
        st = check_batch(&srcs[i]);
        if (st != TQ_OK) return st;
        if (!same_config(srcs[i].cache, dst->cache)) return TQ_ERR_CONFIG_MISMATCH;
        if (batch_arrays_overlap(&srcs[i], dst)) return TQ_ERR_INVALID_ARG;
        rows += srcs[i].batch;
    }
    if (rows > dst->capacity) return TQ_ERR_CAPACITY;
    for (int i = 0; i < n_srcs; ++i) {
        st = tq_batch_extend(dst, &srcs[i], free_blocks, n_free, n_used, stream);
        if (st != TQ_OK) return st;
    }
    return TQ_OK;
}

tq_status tq_batch_extract(const tq_batch* src, int idx, tq_batch* dst, const int32_t* free_blocks, int n_free,
                           int32_t* n_used, tq_stream_t stream) {
    tq_status st = check_batch(src);
    if (st == TQ_OK) st = check_batch(dst);
    if (st != TQ_OK) return st;
    if (!same_config(src->cache, dst->cache)) return TQ_ERR_CONFIG_MISMATCH;
    if (idx < 0 || idx >= src->batch || batch_arrays_overlap(src, dst)) return TQ_ERR_INVALID_ARG;
    if (dst->capacity < 1) return TQ_ERR_CAPACITY;
    st = append_rows(src, idx, 1, dst, 0, free_blocks, n_free, n_used, reinterpret_cast<cudaStream_t>(stream));
    if (st == TQ_OK) dst->batch = 1;
    return st;
}

tq_status tq_cache_copy_blocks(const tq_cache_desc* src, const tq_cache_desc* dst, const int32_t* src_blocks,
                               const int32_t* dst_blocks, int n, tq_stream_t stream) {
    if (!src || !dst || n < 0) return TQ_ERR_INVALID_ARG;
    if (!same_config(src, dst)) return TQ_ERR_CONFIG_MISMATCH;
    if (n == 0) return TQ_OK;
    if (!src->pool || !dst->pool || !src_blocks || !dst_blocks) return TQ_ERR_INVALID_ARG;
    if (n > 2147483647 / 2 || src->num_layers > 65535) return TQ_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (device_state(&err, nullptr) != TQ_OK) return TQ_ERR_CUDA;
    return launch_copy_blocks(src, dst, src_blocks, dst_blocks, n, err, reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? TQ_OK
               : TQ_ERR_CUDA;
}

namespace {

// Checks of tq_encode_append and its launch arguments. *run = false when there
// is nothing to append (batch or n_new zero) and the call is complete.
tq_status append_args(const tq_codec* kc, const tq_codec* vc, const tq_cache_desc* cache, int layer, const void* k,
                      const void* v, tq_dtype dtype, int batch, int n_new, const int32_t* seq_lens,
                      const int32_t* block_table, int max_blocks, EncodeAppendArgs* out, bool* run) {
    *run = false;
    tq_status st = check_codecs_vs_cache(kc, vc, cache);
    if (st != TQ_OK) return st;
    if (layer < 0 || layer >= cache->num_layers || batch < 0 || n_new < 0 || max_blocks <= 0)
        return TQ_ERR_INVALID_ARG;
    if (dtype != TQ_F32 && dtype != TQ_BF16 && dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
    if (cache->encode_policy != TQ_ENCODE_AUTO && cache->encode_policy != TQ_ENCODE_EXACT) return TQ_ERR_INVALID_ARG;
    if (static_cast<int64_t>(n_new) > static_cast<int64_t>(max_blocks) * cache->block_tokens) return TQ_ERR_CAPACITY;
    if (!block_table && static_cast<int64_t>(batch) * max_blocks > cache->num_blocks) return TQ_ERR_CAPACITY;
    if (batch == 0 || n_new == 0) return TQ_OK;
    if (!k || !v || !seq_lens) return TQ_ERR_INVALID_ARG;
    if (batch > 32767) return TQ_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (device_state(&err, nullptr) != TQ_OK) return TQ_ERR_CUDA;
    EncodeAppendArgs& a = *out;
    a = EncodeAppendArgs{};
    a.kc = dev_view(kc);
    a.vc = dev_view(vc);
    a.pool = pool_view(cache, layer);
    a.k = k;
    a.v = v;
    a.dtype = dtype;
    a.batch = batch;
    a.n_new = n_new;
    a.seq_lens = seq_lens;
    a.table = block_table;
    a.max_blocks = max_blocks;
    a.exact = cache->encode_policy == TQ_ENCODE_EXACT;
    a.err = err;
    *run = true;
    return TQ_OK;
}

}  // namespace

tq_status tq_encode_append(const tq_codec* kc, const tq_codec* vc, const tq_cache_desc* cache, int layer,
                           const void* k, const void* v, tq_dtype dtype, int batch, int n_new,
                           const int32_t* seq_lens, const int32_t* block_table, int max_blocks,
                           tq_stream_t stream) {
    EncodeAppendArgs a{};
    bool run = false;
    const tq_status st = append_args(kc, vc, cache, layer, k, v, dtype, batch, n_new, seq_lens, block_table,
                                     max_blocks, &a, &run);
    if (st != TQ_OK || !run) return st;
    return launch_encode_append(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_quantize(const tq_codec* c, const void* x, tq_dtype dtype, int64_t n, uint32_t* idx, void* aux0,
                      void* aux1, void* aux2, tq_stream_t stream) {
    if (!c || n < 0) return TQ_ERR_INVALID_ARG;
    if (dtype != TQ_F32 && dtype != TQ_BF16 && dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
    if (n == 0) return TQ_OK;
    if (!x) return TQ_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (dev != c->device) return TQ_ERR_INVALID_ARG;
    if (n > static_cast<int64_t>(65535) * 65535) return TQ_ERR_INVALID_ARG;
    QuantizeArgs a{};
    a.cd = dev_view(c);
    a.x = x;
    a.dtype = dtype;
    a.n = n;
    a.idx = idx;
    a.aux0 = aux0;
    a.aux1 = aux1;
    a.aux2 = aux2;
    return launch_quantize(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_decode_plan(const tq_cache_desc* cache, int batch, int num_q_heads, int q_len, int max_seq_len,
                         int num_sms, tq_decode_plan_info* info) {
    if (!cache || !info || batch < 0 || q_len <= 0 || max_seq_len < q_len || num_sms <= 0) return TQ_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || cache->num_kv_heads <= 0 || num_q_heads % cache->num_kv_heads != 0)
        return TQ_ERR_INVALID_ARG;
    if (cache->block_tokens < 16 || (cache->block_tokens & (cache->block_tokens - 1)) != 0) return TQ_ERR_INVALID_ARG;
    const int G = num_q_heads / cache->num_kv_heads;
    if (G * q_len > 64) return TQ_ERR_UNSUPPORTED;
    const DecodePlan p = make_decode_plan(cache, batch, G, q_len, max_seq_len, num_sms);
    info->tensor_cores = p.kind == 1 ? 1 : 0;
    info->row_groups = p.row_groups;
    info->splits = p.splits;
    info->chunk_tokens = p.chunk;
    info->tile_tokens = p.tile;
    info->smem_bytes = p.kind == 1 ? p.smem : 0;
    info->workspace_bytes = p.total;
    info->transposed = p.kind == 1 && p.r8 ? 1 : 0;
    return TQ_OK;
}

tq_status tq_decode_workspace_bytes(const tq_cache_desc* cache, int batch, int num_q_heads, int q_len,
                                    int max_seq_len, size_t* bytes) {
    if (!cache || !bytes || batch < 0 || q_len <= 0 || max_seq_len < q_len) return TQ_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || cache->num_kv_heads <= 0 || num_q_heads % cache->num_kv_heads != 0)
        return TQ_ERR_INVALID_ARG;
    if (cache->block_tokens < 16 || (cache->block_tokens & (cache->block_tokens - 1)) != 0) return TQ_ERR_INVALID_ARG;
    const int G = num_q_heads / cache->num_kv_heads;
    if (G * q_len > 64) return TQ_ERR_UNSUPPORTED;
    int sms = 0;
    if (device_state(nullptr, &sms) != TQ_OK) return TQ_ERR_CUDA;
    *bytes = make_decode_plan(cache, batch, G, q_len, max_seq_len, sms).total;
    return TQ_OK;
}

namespace {

// Checks of tq_decode_attention and its launch arguments (*run = false: batch
// zero, nothing to do).
tq_status decode_args(const tq_codec* kc, const tq_codec* vc, const tq_cache_desc* cache, int layer, const void* q,
                      tq_dtype q_dtype, int batch, int num_q_heads, int q_len, const int32_t* seq_lens,
                      const int32_t* block_table, int max_blocks, int max_seq_len, float scale, float* out,
                      void* workspace, size_t workspace_bytes, DecodeArgs* args, bool* run,
                      const int32_t* causal_end = nullptr, float* part_ml = nullptr, float* part_acc = nullptr) {
    const bool shard = part_acc != nullptr;
    *run = false;
    tq_status st = check_codecs_vs_cache(kc, vc, cache);
    if (st != TQ_OK) return st;
    if (layer < 0 || layer >= cache->num_layers || batch < 0 || q_len <= 0 || max_blocks <= 0)
        return TQ_ERR_INVALID_ARG;
    if (q_dtype != TQ_F32 && q_dtype != TQ_BF16 && q_dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
    if (num_q_heads <= 0 || num_q_heads % cache->num_kv_heads != 0) return TQ_ERR_INVALID_ARG;
    if (max_seq_len < (shard ? 1 : q_len)) return TQ_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks) * cache->block_tokens)
        return TQ_ERR_CAPACITY;
    if (!block_table && static_cast<int64_t>(batch) * max_blocks > cache->num_blocks) return TQ_ERR_CAPACITY;
    const int G = num_q_heads / cache->num_kv_heads;
    if (G * q_len > 64) return TQ_ERR_UNSUPPORTED;
    if (batch == 0) return TQ_OK;
    if (batch > 65535) return TQ_ERR_INVALID_ARG;
    if (!q || !seq_lens || !workspace) return TQ_ERR_INVALID_ARG;
    if (shard ? (!part_ml || !aligned16(part_acc) || (reinterpret_cast<uintptr_t>(part_ml) & 7u) != 0) : !out)
        return TQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TQ_ERR_INVALID_ARG;
    if (!shard && !aligned16(out)) return TQ_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    int sms = 0;
    if (device_state(&err, &sms) != TQ_OK) return TQ_ERR_CUDA;
    const DecodePlan plan = make_decode_plan(cache, batch, G, q_len, max_seq_len, sms);
    if (workspace_bytes < plan.total) return TQ_ERR_CAPACITY;
    DecodeArgs& a = *args;
    a = DecodeArgs{};
    a.kc = dev_view(kc);
    a.vc = dev_view(vc);
    // 4-bit MSE keys and values of one codebook (the levels depend on the head
    // dimension and the width only): one wide pair table serves both
    if (kc->d_pair4w && vc->d_pair4w && kc->host.op_levels.size() == vc->host.op_levels.size() &&
        std::memcmp(kc->host.op_levels.data(), vc->host.op_levels.data(),
                    kc->host.op_levels.size() * sizeof(float)) == 0)
        a.vc.pair4w = a.kc.pair4w;
    a.pool = pool_view(cache, layer);
    a.q = q;
    a.q_dtype = q_dtype;
    a.batch = batch;
    a.Hq = num_q_heads;
    a.Lq = q_len;
    a.G = G;
    a.seq_lens = seq_lens;
    a.table = block_table;
    a.max_blocks = max_blocks;
    a.scale = scale == 0.0f ? 1.0f / std::sqrt(static_cast<float>(cache->head_dim)) : scale;
    a.out = out;
    a.causal_end = causal_end;
    a.part_ml = part_ml;
    a.part_acc = part_acc;
    char* ws = static_cast<char*>(workspace);
    a.qrot = reinterpret_cast<float*>(ws);
    a.qjl = reinterpret_cast<float*>(ws + plan.q_bytes);
    a.part = reinterpret_cast<float*>(ws + 2 * plan.q_bytes);
    a.ml = reinterpret_cast<float*>(ws + 2 * plan.q_bytes + plan.part_bytes);
    a.ws = workspace;
    a.plan = plan;
    a.err = err;
    *run = true;
    return TQ_OK;
}

}  // namespace

tq_status tq_decode_attention(const tq_codec* kc, const tq_codec* vc, const tq_cache_desc* cache, int layer,
                              const void* q, tq_dtype q_dtype, int batch, int num_q_heads, int q_len,
                              const int32_t* seq_lens, const int32_t* block_table, int max_blocks,
                              int max_seq_len, float scale, float* out, void* workspace,
                              size_t workspace_bytes, tq_stream_t stream) {
    DecodeArgs a{};
    bool run = false;
    const tq_status st = decode_args(kc, vc, cache, layer, q, q_dtype, batch, num_q_heads, q_len, seq_lens,
                                     block_table, max_blocks, max_seq_len, scale, out, workspace, workspace_bytes,
                                     &a, &run);
    if (st != TQ_OK || !run) return st;
    return launch_decode(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_decode_partials(const tq_codec* kc, const tq_codec* vc, const tq_cache_desc* cache, int layer,
                             const void* q, tq_dtype q_dtype, int batch, int num_q_heads, int q_len,
                             const int32_t* seq_lens, const int32_t* causal_end, const int32_t* block_table,
                             int max_blocks, int max_seq_len, float scale, float* part_ml, float* part_acc,
                             void* workspace, size_t workspace_bytes, tq_stream_t stream) {
    if (!part_acc) return TQ_ERR_INVALID_ARG;
    DecodeArgs a{};
    bool run = false;
    const tq_status st = decode_args(kc, vc, cache, layer, q, q_dtype, batch, num_q_heads, q_len, seq_lens,
                                     block_table, max_blocks, max_seq_len, scale, nullptr, workspace,
                                     workspace_bytes, &a, &run, causal_end, part_ml, part_acc);
    if (st != TQ_OK || !run) return st;
    return launch_decode(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_decode_merge(const tq_codec* value_codec, int num_parts, const float* parts_ml, const float* parts_acc,
                          int64_t rows, float* out, tq_stream_t stream) {
    if (!value_codec || num_parts < 0 || rows < 0) return TQ_ERR_INVALID_ARG;
    if (rows == 0) return TQ_OK;
    if (num_parts == 0 || !parts_ml || !parts_acc || !out) return TQ_ERR_INVALID_ARG;
    if (rows > 2147483647) return TQ_ERR_INVALID_ARG;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return TQ_ERR_CUDA;
    if (dev != value_codec->device) return TQ_ERR_INVALID_ARG;
    return launch_shard_merge(dev_view(value_codec), num_parts, parts_ml, parts_acc, rows, out,
                              reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? TQ_OK
               : TQ_ERR_CUDA;
}

namespace {

// The two halves of a split state: codecs matching their caches, and caches
// of one layout shape (addressed by one block table).
tq_status check_split(const tq_split_state* st) {
    if (!st || !st->low || !st->high) return TQ_ERR_INVALID_ARG;
    tq_status e = check_codecs_vs_cache(st->key_low, st->value_low, st->low);
    if (e == TQ_OK) e = check_codecs_vs_cache(st->key_high, st->value_high, st->high);
    if (e != TQ_OK) return e;
    const tq_cache_desc *a = st->low, *b = st->high;
    if (a->num_layers != b->num_layers || a->num_blocks != b->num_blocks || a->block_tokens != b->block_tokens ||
        a->num_kv_heads != b->num_kv_heads)
        return TQ_ERR_CONFIG_MISMATCH;
    const int dl = a->head_dim, dh = b->head_dim;
    if ((dl != 64 && dl != 128) || (dh != 64 && dh != 128)) return TQ_ERR_UNSUPPORTED;
    return TQ_OK;
}

}  // namespace

tq_status tq_encode_append_split(const tq_split_state* st, int layer, const void* k_low, const void* v_low,
                                 const void* k_high, const void* v_high, tq_dtype dtype, int batch, int n_new,
                                 const int32_t* seq_lens, const int32_t* block_table, int max_blocks,
                                 tq_stream_t stream) {
    tq_status e = check_split(st);
    if (e != TQ_OK) return e;
    // both halves are checked before either is launched
    EncodeAppendArgs lo{}, hi{};
    bool run_lo = false, run_hi = false;
    e = append_args(st->key_low, st->value_low, st->low, layer, k_low, v_low, dtype, batch, n_new, seq_lens,
                    block_table, max_blocks, &lo, &run_lo);
    if (e == TQ_OK)
        e = append_args(st->key_high, st->value_high, st->high, layer, k_high, v_high, dtype, batch, n_new,
                        seq_lens, block_table, max_blocks, &hi, &run_hi);
    if (e != TQ_OK) return e;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (run_lo && launch_encode_append(lo, s) != cudaSuccess) return TQ_ERR_CUDA;
    if (run_hi && launch_encode_append(hi, s) != cudaSuccess) return TQ_ERR_CUDA;
    return TQ_OK;
}

namespace {

tq_status split_args(const tq_split_state* st, int batch, int num_q_heads, int q_len, int max_seq_len,
                     SplitStateArgs* a) {
    tq_status e = check_split(st);
    if (e != TQ_OK) return e;
    const tq_cache_desc* c = st->low;
    if (batch < 0 || q_len <= 0 || max_seq_len < q_len || num_q_heads <= 0 || num_q_heads % c->num_kv_heads != 0)
        return TQ_ERR_INVALID_ARG;
    const int G = num_q_heads / c->num_kv_heads;
    if (G * q_len > 64) return TQ_ERR_UNSUPPORTED;
    unsigned* err = nullptr;
    int sms = 0;
    if (device_state(&err, &sms) != TQ_OK) return TQ_ERR_CUDA;
    *a = SplitStateArgs{};
    a->klo = dev_view(st->key_low);
    a->vlo = dev_view(st->value_low);
    a->khi = dev_view(st->key_high);
    a->vhi = dev_view(st->value_high);
    a->batch = batch;
    a->Hq = num_q_heads;
    a->Lq = q_len;
    a->G = G;
    a->Hkv = c->num_kv_heads;
    a->err = err;
    split_state_plan(*a, max_seq_len, sms);
    return TQ_OK;
}

}  // namespace

tq_status tq_decode_workspace_bytes_split(const tq_split_state* st, int batch, int num_q_heads, int q_len,
                                          int max_seq_len, size_t* bytes) {
    if (!bytes) return TQ_ERR_INVALID_ARG;
    SplitStateArgs a{};
    const tq_status e = split_args(st, batch, num_q_heads, q_len, max_seq_len, &a);
    if (e != TQ_OK) return e;
    *bytes = split_state_workspace(a, st->low->head_dim + st->high->head_dim);
    return TQ_OK;
}

tq_status tq_decode_attention_split(const tq_split_state* st, int layer, const void* q, tq_dtype q_dtype,
                                    int batch, int num_q_heads, int q_len, const int32_t* seq_lens,
                                    const int32_t* block_table, int max_blocks, int max_seq_len, float scale,
                                    float* out, void* workspace, size_t workspace_bytes, tq_stream_t stream) {
    SplitStateArgs a{};
    tq_status e = split_args(st, batch, num_q_heads, q_len, max_seq_len, &a);
    if (e != TQ_OK) return e;
    const tq_cache_desc* c = st->low;
    if (layer < 0 || layer >= c->num_layers || max_blocks <= 0) return TQ_ERR_INVALID_ARG;
    if (q_dtype != TQ_F32 && q_dtype != TQ_BF16 && q_dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
    if (static_cast<int64_t>(max_seq_len) > static_cast<int64_t>(max_blocks) * c->block_tokens)
        return TQ_ERR_CAPACITY;
    if (!block_table && static_cast<int64_t>(batch) * max_blocks > c->num_blocks) return TQ_ERR_CAPACITY;
    if (batch == 0) return TQ_OK;
    if (batch > 65535) return TQ_ERR_INVALID_ARG;
    if (!q || !out || !seq_lens || !workspace) return TQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TQ_ERR_INVALID_ARG;
    const int D = c->head_dim + st->high->head_dim;
    if (workspace_bytes < split_state_workspace(a, D)) return TQ_ERR_CAPACITY;
    a.plo = pool_view(st->low, layer);
    a.phi = pool_view(st->high, layer);
    a.q = q;
    a.q_dtype = q_dtype;
    a.seq_lens = seq_lens;
    a.table = block_table;
    a.max_blocks = max_blocks;
    a.scale = scale == 0.0f ? 1.0f / std::sqrt(static_cast<float>(D)) : scale;
    a.out = out;
    split_state_bind_workspace(a, workspace, D);
    return launch_split_state(a, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_decode_step(const tq_codec* kc, const tq_codec* vc, const tq_cache_desc* cache, int layer,
                         const void* k_new, const void* v_new, tq_dtype kv_dtype, int n_new, const void* q,
                         tq_dtype q_dtype, int batch, int num_q_heads, int q_len, const int32_t* seq_lens,
                         const int32_t* block_table, int max_blocks, int max_seq_len, float scale, float* out,
                         void* workspace, size_t workspace_bytes, tq_stream_t stream) {
    EncodeAppendArgs e{};
    bool run_e = false;
    tq_status st = append_args(kc, vc, cache, layer, k_new, v_new, kv_dtype, batch, n_new, seq_lens, block_table,
                               max_blocks, &e, &run_e);
    if (st != TQ_OK) return st;
    DecodeArgs a{};
    bool run_d = false;
    st = decode_args(kc, vc, cache, layer, q, q_dtype, batch, num_q_heads, q_len, seq_lens, block_table, max_blocks,
                     max_seq_len, scale, out, workspace, workspace_bytes, &a, &run_d);
    if (st != TQ_OK || !run_d) return st;
    a.len_add = run_e ? n_new : 0;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // one launch for the append and the query prep where the tensor-core path
    // and the short rotated encoder both apply; else the two calls in order
    const bool fused = run_e && a.plan.kind == 1 && n_new <= 8 && cache->head_dim == 128 &&
                       kc->mode != TQ_MODE_GROUP && vc->mode != TQ_MODE_GROUP;
    if (fused) return launch_decode(a, s, &e) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
    if (run_e && launch_encode_append(e, s) != cudaSuccess) return TQ_ERR_CUDA;
    return launch_decode(a, s) == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

namespace {

// Plan of a prefill call: the decode plan's record layout and codec class, with
// the query rows of the whole chunk; returns TQ_OK or the reason it cannot run.
tq_status prefill_plan(const tq_cache_desc* cache, int batch, int num_q_heads, int q_len, DecodePlan* plan,
                       size_t* ws) {
    if (!cache || batch < 0 || q_len <= 0 || num_q_heads <= 0) return TQ_ERR_INVALID_ARG;
    if (num_q_heads % cache->num_kv_heads != 0) return TQ_ERR_INVALID_ARG;
    const int G = num_q_heads / cache->num_kv_heads;
    const int64_t rows = static_cast<int64_t>(G) * q_len;
    if ((rows + 15) / 16 > 65535) return TQ_ERR_UNSUPPORTED;
    const DecodePlan p = make_decode_plan(cache, batch > 0 ? batch : 1, G, q_len, q_len, 1);
    if (p.kind != 1 || !mmadec::prefill_supported(p.kb, p.kprod, p.vgroup, p.vb)) return TQ_ERR_UNSUPPORTED;
    if (plan) *plan = p;
    if (ws) *ws = (static_cast<size_t>(batch) * cache->num_kv_heads * p.row_groups * 2 * 8 * 32 * 16 + 255) / 256 * 256;
    return TQ_OK;
}

}  // namespace

tq_status tq_prefill_workspace_bytes(const tq_cache_desc* cache, int batch, int num_q_heads, int q_len,
                                     size_t* bytes) {
    if (!bytes) return TQ_ERR_INVALID_ARG;
    return prefill_plan(cache, batch, num_q_heads, q_len, nullptr, bytes);
}

tq_status tq_prefill_attention(const tq_codec* kc, const tq_codec* vc, const tq_cache_desc* cache, int layer,
                               const void* q, tq_dtype q_dtype, int batch, int num_q_heads, int q_len,
                               const int32_t* seq_lens, const int32_t* block_table, int max_blocks, float scale,
                               float* out, void* workspace, size_t workspace_bytes, tq_stream_t stream) {
    tq_status st = check_codecs_vs_cache(kc, vc, cache);
    if (st != TQ_OK) return st;
    if (layer < 0 || layer >= cache->num_layers || batch < 0 || q_len <= 0 || max_blocks <= 0)
        return TQ_ERR_INVALID_ARG;
    if (q_dtype != TQ_F32 && q_dtype != TQ_BF16 && q_dtype != TQ_F16) return TQ_ERR_INVALID_ARG;
    if (static_cast<int64_t>(q_len) > static_cast<int64_t>(max_blocks) * cache->block_tokens) return TQ_ERR_CAPACITY;
    if (!block_table && static_cast<int64_t>(batch) * max_blocks > cache->num_blocks) return TQ_ERR_CAPACITY;
    DecodePlan plan{};
    size_t need = 0;
    st = prefill_plan(cache, batch, num_q_heads, q_len, &plan, &need);
    if (st != TQ_OK) return st;
    if (batch == 0) return TQ_OK;
    if (batch > 65535) return TQ_ERR_INVALID_ARG;
    if (!q || !out || !seq_lens || !workspace) return TQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TQ_ERR_INVALID_ARG;
    if (!aligned16(out)) return TQ_ERR_INVALID_ARG;
    if (workspace_bytes < need) return TQ_ERR_CAPACITY;
    unsigned* err = nullptr;
    if (device_state(&err, nullptr) != TQ_OK) return TQ_ERR_CUDA;
    DecodeArgs a{};
    a.kc = dev_view(kc);
    a.vc = dev_view(vc);
    a.pool = pool_view(cache, layer);
    a.q = q;
    a.q_dtype = q_dtype;
    a.batch = batch;
    a.Hq = num_q_heads;
    a.Lq = q_len;
    a.G = num_q_heads / cache->num_kv_heads;
    a.seq_lens = seq_lens;
    a.table = block_table;
    a.max_blocks = max_blocks;
    a.scale = scale == 0.0f ? 1.0f / std::sqrt(static_cast<float>(cache->head_dim)) : scale;
    a.out = out;
    a.ws = workspace;
    a.plan = plan;
    a.err = err;
    return mmadec::launch_prefill(a, static_cast<const uint4*>(workspace), reinterpret_cast<cudaStream_t>(stream)) ==
                   cudaSuccess
               ? TQ_OK
               : TQ_ERR_CUDA;
}

tq_status tq_selftest_wait_timeout(double seconds, tq_stream_t stream) {
    if (!(seconds > 0.0 && seconds <= 1.0)) return TQ_ERR_INVALID_ARG;
    unsigned* err = nullptr;
    if (device_state(&err, nullptr) != TQ_OK) return TQ_ERR_CUDA;
    wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(
        err, static_cast<unsigned long long>(seconds * 1e9));
    ++g_launches;
    return cudaGetLastError() == cudaSuccess ? TQ_OK : TQ_ERR_CUDA;
}

tq_status tq_device_error(uint32_t* flags) {
    unsigned* err = nullptr;
    if (device_state(&err, nullptr) != TQ_OK) return TQ_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return TQ_ERR_CUDA;
    unsigned v = 0;
    if (cudaMemcpy(&v, err, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess) return TQ_ERR_CUDA;
    const unsigned zero = 0;
    if (cudaMemcpy(err, &zero, sizeof(zero), cudaMemcpyHostToDevice) != cudaSuccess) return TQ_ERR_CUDA;
    if (flags) *flags = v;
    return v ? TQ_ERR_DEVICE_BOUNDS : TQ_OK;
}

}  // extern "C"

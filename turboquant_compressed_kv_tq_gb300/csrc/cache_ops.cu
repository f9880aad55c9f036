// Block copies between paged caches of one codec configuration.
//
// A block holds block_tokens tokens of one sequence for every KV head: the
// sub-blocks (p * Hkv + h), h = 0..Hkv-1, are one contiguous run of
// Hkv * subblock_bytes bytes in each layer pool. The batch operations of
// "omlx/turboquant_kv.py" (BatchTurboQuantKVCache.merge, extend, extract,
// filter) become block-table edits plus copies of such runs.
#include "tq_internal.h"

namespace tq {
namespace {

constexpr int kCopyThreads = 256;

struct CopyArgs {
    const char* src;
    char* dst;
    int64_t src_layer_stride, dst_layer_stride;
    int64_t block_bytes;         // Hkv * subblock_bytes (multiple of 16)
    int src_blocks_total, dst_blocks_total;
    const int32_t* src_ids;
    const int32_t* dst_ids;
    unsigned* err;
};

// grid (pairs, layers): one CTA copies one block of one layer with 16-byte accesses.
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(CopyArgs a) {
    const int i = blockIdx.x, layer = blockIdx.y;
    const int sb = a.src_ids[i], db = a.dst_ids[i];
    if (sb < 0 || sb >= a.src_blocks_total || db < 0 || db >= a.dst_blocks_total) {
        if (threadIdx.x == 0 && layer == 0) atomicOr(a.err, TQ_DEVERR_BLOCK);
        return;
    }
    const uint4* s = reinterpret_cast<const uint4*>(a.src + layer * a.src_layer_stride + sb * a.block_bytes);
    uint4* d = reinterpret_cast<uint4*>(a.dst + layer * a.dst_layer_stride + db * a.block_bytes);
    const int64_t n16 = a.block_bytes / 16;
    for (int64_t k = threadIdx.x; k < n16; k += kCopyThreads) d[k] = __ldcs(s + k);
}

}  // namespace

cudaError_t launch_copy_blocks(const tq_cache_desc* src, const tq_cache_desc* dst, const int32_t* src_ids,
                               const int32_t* dst_ids, int n, unsigned* err, cudaStream_t s) {
    CopyArgs a{};
    a.src = static_cast<const char*>(src->pool);
    a.dst = static_cast<char*>(dst->pool);
    a.src_layer_stride = src->layer_stride;
    a.dst_layer_stride = dst->layer_stride;
    a.block_bytes = src->subblock_bytes * src->num_kv_heads;
    a.src_blocks_total = src->num_blocks;
    a.dst_blocks_total = dst->num_blocks;
    a.src_ids = src_ids;
    a.dst_ids = dst_ids;
    a.err = err;
    copy_blocks_kernel<<<dim3(n, src->num_layers), kCopyThreads, 0, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
}

}  // namespace tq

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

// ------------------------------------------------------------------ batch operations
//
// BatchTurboQuantKVCache.filter / extend / merge / extract ("omlx/turboquant_kv.py")
// on the paged layout: a single-CTA kernel rewrites a chunk of block-table
// rows (and, for filter, lists the blocks of the dropped rows), then, where a
// sequence moves to another pool, a copy kernel moves its blocks.

namespace tq {
namespace {

constexpr int kRowChunk = 256;   // rows per launch (lists travel as kernel parameters)

struct RowsArgs {
    const int32_t* src_table;
    const int32_t* src_lens;
    int src_mb, src_rows;
    int32_t* dst_table;
    int32_t* dst_lens;
    int dst_mb, dst_row0;
    int n;                        // rows written by this launch
    int list_mode;                // 1: source row of output i is rows[i]; 0: src_row0 + i
    int src_row0;
    int copy;                     // 1: blocks taken from the free list; 0: ids kept
    const int32_t* free_blocks;
    int n_free;
    int32_t* cursor;              // device: next free-list index (read, advanced)
    int BT, src_num_blocks;
    int n_drop;                   // filter: rows whose blocks are listed as freed
    int32_t* freed;
    int32_t* n_freed;
    int reset_freed;
    unsigned* err;
    int rows[kRowChunk];
    int drop[kRowChunk];
};

// Exclusive prefix sum of v over the block (kRowChunk threads); returns the total.
__device__ int block_scan(int v, int* s_tmp, int* excl) {
    const int t = threadIdx.x;
    s_tmp[t] = v;
    __syncthreads();
    for (int off = 1; off < kRowChunk; off <<= 1) {
        const int x = t >= off ? s_tmp[t - off] : 0;
        __syncthreads();
        s_tmp[t] += x;
        __syncthreads();
    }
    *excl = s_tmp[t] - v;
    const int total = s_tmp[kRowChunk - 1];
    __syncthreads();
    return total;
}

__global__ void __launch_bounds__(kRowChunk) batch_rows_kernel(RowsArgs a) {
    __shared__ int s_tmp[kRowChunk];
    __shared__ int s_base, s_fbase;
    const int i = threadIdx.x;
    if (i == 0) {
        s_base = a.copy ? *a.cursor : 0;
        s_fbase = a.reset_freed ? 0 : (a.n_freed ? *a.n_freed : 0);
    }
    __syncthreads();
    // ---- rows: length, token blocks, destination ids
    int s = -1, len = 0, need = 0;
    if (i < a.n) {
        s = a.list_mode ? a.rows[i] : a.src_row0 + i;
        len = a.src_lens[s];
        if (len < 0 || len > a.src_mb * a.BT) {
            atomicOr(a.err, TQ_DEVERR_SEQLEN);
            len = len < 0 ? 0 : a.src_mb * a.BT;
        }
        need = (len + a.BT - 1) / a.BT;
        if (a.copy && need > a.dst_mb) {
            atomicOr(a.err, TQ_DEVERR_CAPACITY);
            need = a.dst_mb;
        }
    }
    int off = 0;
    const int total = block_scan(a.copy ? need : 0, s_tmp, &off);
    if (i < a.n) {
        int32_t* drow = a.dst_table + static_cast<int64_t>(a.dst_row0 + i) * a.dst_mb;
        const int32_t* srow = a.src_table + static_cast<int64_t>(s) * a.src_mb;
        int got = 0;
        for (int lb = 0; lb < a.dst_mb; ++lb) {
            int32_t id = -1;
            if (a.copy) {
                if (lb < need) {
                    const int k = s_base + off + lb;
                    if (k < a.n_free) {
                        id = a.free_blocks[k];
                        const int32_t sid = srow[lb];
                        if (sid < 0 || sid >= a.src_num_blocks) atomicOr(a.err, TQ_DEVERR_BLOCK);
                        ++got;
                    } else {
                        atomicOr(a.err, TQ_DEVERR_CAPACITY);
                    }
                }
            } else if (lb < a.src_mb) {
                id = srow[lb];
            }
            drow[lb] = id;
        }
        // a copied sequence keeps only the tokens whose blocks it received
        a.dst_lens[a.dst_row0 + i] = a.copy ? min(len, got * a.BT) : len;
    }
    if (i == 0 && a.copy) *a.cursor = min(s_base + total, a.n_free);
    // ---- filter: ids of the dropped rows, in row then entry order
    int cnt = 0;
    const int32_t* drow = nullptr;
    if (i < a.n_drop) {
        drow = a.src_table + static_cast<int64_t>(a.drop[i]) * a.src_mb;
        for (int lb = 0; lb < a.src_mb; ++lb) cnt += drow[lb] >= 0;
    }
    int foff = 0;
    const int ftotal = block_scan(cnt, s_tmp, &foff);
    if (i < a.n_drop) {
        int k = s_fbase + foff;
        for (int lb = 0; lb < a.src_mb; ++lb)
            if (drow[lb] >= 0) a.freed[k++] = drow[lb];
    }
    if (i == 0 && a.n_freed) *a.n_freed = s_fbase + ftotal;
}

struct MoveArgs {
    const char* src;
    char* dst;
    int64_t src_layer_stride, dst_layer_stride;
    int64_t block_bytes;
    const int32_t* src_table;
    const int32_t* dst_table;
    const int32_t* dst_lens;
    int src_mb, dst_mb, src_row0, dst_row0, BT;
    int src_num_blocks, dst_num_blocks;
};

constexpr int kMoveSplit = 8;

// grid (rows, layers, kMoveSplit): the blocks holding a moved sequence's tokens.
__global__ void __launch_bounds__(kCopyThreads) batch_move_kernel(MoveArgs a) {
    const int r = blockIdx.x, layer = blockIdx.y;
    const int len = a.dst_lens[a.dst_row0 + r];
    const int nb = (len + a.BT - 1) / a.BT;
    const int32_t* srow = a.src_table + static_cast<int64_t>(a.src_row0 + r) * a.src_mb;
    const int32_t* drow = a.dst_table + static_cast<int64_t>(a.dst_row0 + r) * a.dst_mb;
    const int64_t n16 = a.block_bytes / 16;
    for (int lb = blockIdx.z; lb < nb; lb += kMoveSplit) {
        const int sb = srow[lb], db = drow[lb];
        if (sb < 0 || sb >= a.src_num_blocks || db < 0 || db >= a.dst_num_blocks) continue;  // flagged by the row kernel
        const uint4* s = reinterpret_cast<const uint4*>(a.src + layer * a.src_layer_stride + sb * a.block_bytes);
        uint4* d = reinterpret_cast<uint4*>(a.dst + layer * a.dst_layer_stride + db * a.block_bytes);
        for (int64_t k = threadIdx.x; k < n16; k += kCopyThreads) d[k] = __ldcs(s + k);
    }
}

}  // namespace

cudaError_t launch_batch_rows(const tq_batch* src, tq_batch* dst, int n, const int* rows, int src_row0, int dst_row0,
                              bool copy, const int32_t* free_blocks, int n_free, int32_t* n_used, int n_drop,
                              const int* drop, int32_t* freed, int32_t* n_freed, bool reset_freed, unsigned* err,
                              cudaStream_t s) {
    RowsArgs a{};
    a.src_table = src->block_table;
    a.src_lens = src->seq_lens;
    a.src_mb = src->max_blocks;
    a.src_rows = src->batch;
    a.dst_table = dst->block_table;
    a.dst_lens = dst->seq_lens;
    a.dst_mb = dst->max_blocks;
    a.dst_row0 = dst_row0;
    a.n = n;
    a.list_mode = rows ? 1 : 0;
    a.src_row0 = src_row0;
    a.copy = copy ? 1 : 0;
    a.free_blocks = free_blocks;
    a.n_free = n_free;
    a.cursor = n_used;
    a.BT = src->cache->block_tokens;
    a.src_num_blocks = src->cache->num_blocks;
    a.n_drop = n_drop;
    a.freed = freed;
    a.n_freed = n_freed;
    a.reset_freed = reset_freed ? 1 : 0;
    a.err = err;
    for (int i = 0; rows && i < n; ++i) a.rows[i] = rows[i];
    for (int i = 0; drop && i < n_drop; ++i) a.drop[i] = drop[i];
    batch_rows_kernel<<<1, kRowChunk, 0, s>>>(a);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || !copy || n == 0) return e;
    MoveArgs m{};
    m.src = static_cast<const char*>(src->cache->pool);
    m.dst = static_cast<char*>(dst->cache->pool);
    m.src_layer_stride = src->cache->layer_stride;
    m.dst_layer_stride = dst->cache->layer_stride;
    m.block_bytes = src->cache->subblock_bytes * src->cache->num_kv_heads;
    m.src_table = src->block_table;
    m.dst_table = dst->block_table;
    m.dst_lens = dst->seq_lens;
    m.src_mb = src->max_blocks;
    m.dst_mb = dst->max_blocks;
    m.src_row0 = src_row0;
    m.dst_row0 = dst_row0;
    m.BT = a.BT;
    m.src_num_blocks = src->cache->num_blocks;
    m.dst_num_blocks = dst->cache->num_blocks;
    batch_move_kernel<<<dim3(n, src->cache->num_layers, kMoveSplit), kCopyThreads, 0, s>>>(m);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return cudaGetLastError();
}

}  // namespace tq

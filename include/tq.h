/*
 * tq.h -- C ABI of the GB300 TurboQuant compressed-KV library (libtq.so).
 *
 * TurboQuant stores each key/value vector of a KV cache as its norm plus the
 * Lloyd-Max codebook indices of its randomly rotated unit vector, bit-packed
 * into uint32 words; "prod" keys add a 1-bit QJL sign sketch of the rotated
 * residual and the residual norm; values may instead use per-group affine
 * quantisation. Decode attention reads that compressed cache directly.
 *
 * Sources, by page title:
 *   "lightning-mlx/plan.md"               -- codec outline (rotation, Lloyd-Max,
 *       norm separation, group denormalise, inverse rotation `rotated @ Q` in
 *       fp32), incremental append for decode, the fused decode-attention kernel
 *       over Lloyd-Max codes, and the bandwidth-bound decode model.
 *   "omlx/turboquant_kv.py"               -- packed_width = ceil(head_dim*bits/32),
 *       prod keys pack bits-1 index bits, codecs rebuilt from (head_dim, bits,
 *       seed) with the value codec on seed+1, append at the written end rather
 *       than the allocated capacity, refusal to batch caches of mixed (bits,
 *       seed), state fields of MSE and prod states.
 *   "turboquant/validate_moe_phase2.py"   -- TurboQuantProd fields (mse_indices,
 *       qjl_signs, residual_norms, norms; norms in float32), head_dim x head_dim
 *       fp32 rotation Pi and QJL matrix S, value group quantisation with
 *       scales and zeros, attention scale 1/sqrt(head_dim), direct scoring of
 *       queries against compressed keys (attention_score).
 *
 * Conventions for every call:
 *   - Pointers named "device" are CUDA device pointers on the device that was
 *     current when the codecs were created; "host" pointers are host memory.
 *   - Calls that take a stream only enqueue work on it (asynchronous, no host
 *     synchronisation, no allocation); arguments are checked on the host first.
 *   - Errors are returned as tq_status; nothing is thrown across the ABI.
 *     Violations that only the GPU can see (a sequence longer than its block
 *     table, a block id outside the pool) skip the offending access and set
 *     bits in a per-device error word read by tq_device_error().
 *   - Shapes are row-major and contiguous.
 *   - Consecutive calls on one stream overlap at their boundaries (programmatic
 *     dependent launch): a call's first kernel may start, and read its plain
 *     inputs (q, k, v, k_new, v_new), while the previous call's last kernel
 *     is still finishing. Every read of cache records, block tables, lengths
 *     and workspaces waits for the kernels before it; the plain inputs do not.
 *     So q, k, v, k_new and v_new must not be the output (out, or a shard's
 *     state) of the immediately preceding decode call (tq_decode_attention,
 *     tq_decode_attention_noalloc, tq_decode_step, tq_decode_partials) on the
 *     same stream: any other kernel or memory copy enqueued between the two
 *     calls (as a model's projections are) restores plain stream order.
 */
#ifndef TQ_H
#define TQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define TQ_ABI_VERSION 2

/* A cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *tq_stream_t;

typedef enum { TQ_MODE_MSE = 0, TQ_MODE_PROD = 1, TQ_MODE_GROUP = 2 } tq_mode;
typedef enum { TQ_F32 = 0, TQ_BF16 = 1, TQ_F16 = 2 } tq_dtype;

/* How tq_encode_append rotates long appends (tq_cache_desc.encode_policy). */
typedef enum {
    TQ_ENCODE_AUTO = 0,  /* tensor cores for appends of >= 64 tokens (see tq_encode_append) */
    TQ_ENCODE_EXACT = 1  /* always the sequential fp32 specification, bit for bit          */
} tq_encode_policy;

typedef enum {
    TQ_OK = 0,
    TQ_ERR_INVALID_ARG = 1,     /* null pointer, negative size, misaligned buffer  */
    TQ_ERR_UNSUPPORTED = 2,     /* head_dim/bits/mode combination not built         */
    TQ_ERR_CONFIG_MISMATCH = 3, /* codec does not match the cache descriptor         */
    TQ_ERR_CAPACITY = 4,        /* pool or workspace too small for the request       */
    TQ_ERR_OOM = 5,             /* codec table allocation failed                      */
    TQ_ERR_CUDA = 6,            /* a CUDA runtime call or kernel launch failed        */
    TQ_ERR_DEVICE_BOUNDS = 7    /* reported by tq_device_error: GPU saw a bad index   */
} tq_status;

/* Device error bits (tq_device_error). */
#define TQ_DEVERR_CAPACITY 1u   /* append past a sequence's block-table capacity */
#define TQ_DEVERR_BLOCK 2u      /* block id outside [0, num_blocks)              */
#define TQ_DEVERR_SEQLEN 4u     /* decode seq_len outside [q_len, capacity]      */
#define TQ_DEVERR_TIMEOUT 8u    /* a bounded wait for a bulk copy ran out         */

/* ------------------------------------------------------------------ */
/* Codecs                                                               */
/* ------------------------------------------------------------------ */

typedef struct tq_codec tq_codec; /* opaque; immutable after creation */

typedef struct {
    int head_dim;
    int bits;          /* total bits per coordinate (prod: MSE bits + 1)      */
    int mode;          /* tq_mode                                              */
    int group_size;    /* group mode only                                      */
    uint64_t seed;
    int index_bits;    /* bits per packed index: bits, or bits-1 for prod      */
    int index_words;   /* packed_width = ceil(head_dim * index_bits / 32)      */
    int sign_words;    /* prod: head_dim/32 QJL sign words, else 0             */
    int record_bytes;  /* bytes stored per token for this codec                */
    int device;        /* CUDA device holding the tables                       */
} tq_codec_info_t;

/*
 * Build an MSE or prod codec from (head_dim, bits, seed) alone, as the codec
 * rebuild of "omlx/turboquant_kv.py" (_rebuild_codecs) requires:
 *   rotation R (head_dim x head_dim, fp32): Q factor with positive diagonal of
 *     the QR factorisation of a seeded Gaussian matrix (SplitMix64 stream
 *     2*seed, Box-Muller normals, Householder QR in fp64), y = R x;
 *   QJL matrix S (prod only, fp32): i.i.d. N(0,1), stream 2*seed+1;
 *   codebook: 2^index_bits Lloyd-Max levels for the density of one coordinate
 *     of a uniform unit vector in R^head_dim, (1-t^2)^((head_dim-3)/2), with
 *     the midpoints between levels as decision thresholds.
 * head_dim in {64, 128, 256}; MSE bits 1..4; prod bits 2..5. The tables live
 * on the current CUDA device (plus a host copy). Returns TQ_ERR_UNSUPPORTED
 * for other values. *out receives a codec owned by the caller
 * (tq_codec_destroy). Thread-safe.
 */
tq_status tq_codec_create(int head_dim, int bits, tq_mode mode, uint64_t seed, tq_codec **out);

/*
 * Fractional bit widths, as the codec rebuild of "omlx/turboquant_kv.py"
 * (_rebuild_codecs) reads them: a width b that is not an integer (further
 * than 1e-6 from round(b)) gives keys floor(b) bits and values ceil(b) bits,
 * so that the pair averages b over a token (b = 3.5: 3-bit keys, 4-bit
 * values); an integer width (within 1e-6) gives both (int)b, truncated as the
 * page converts it (2.9999995 -> 2). tq_bits_split is host arithmetic only
 * (no CUDA device needed); widths whose key or value bits fall outside 1..4,
 * and non-finite b, return TQ_ERR_UNSUPPORTED with both outputs 0;
 * TQ_ERR_INVALID_ARG for NULL outputs.
 * tq_codec_pair_for_bits builds the two MSE codecs of that rule with
 * tq_codec_create: keys (head_dim, key bits, seed), values (head_dim, value
 * bits, seed + 1). On any error neither codec is created and both outputs
 * are NULL; on success the caller owns both (tq_codec_destroy).
 */
tq_status tq_bits_split(double bits, int *key_bits, int *value_bits);
tq_status tq_codec_pair_for_bits(int head_dim, double bits, uint64_t seed, tq_codec **key_codec,
                                 tq_codec **value_codec);

/*
 * Group codec ("turboquant/validate_moe_phase2.py", quantize_values): per
 * group of group_size consecutive coordinates an fp16 scale
 * (max-min)/(2^bits-1) and an fp16 minimum; codes round((x-min)/scale)
 * clamped to [0, 2^bits-1]; no rotation. bits in {2, 4}; group_size in
 * {32, 64, 128} dividing head_dim.
 */
tq_status tq_codec_create_group(int head_dim, int bits, int group_size, tq_codec **out);

void tq_codec_destroy(tq_codec *codec);
tq_status tq_codec_info(const tq_codec *codec, tq_codec_info_t *out);

/*
 * Build the fp32 tables of an MSE or prod codec on the host only, without a
 * CUDA device (the same construction as tq_codec_create): R and S are
 * head_dim*head_dim row-major (S only for prod, may be NULL), centroids
 * 2^index_bits, midpoints 2^index_bits - 1. Lets a table be reproduced and
 * inspected offline.
 */
tq_status tq_codec_build_host(int head_dim, int bits, tq_mode mode, uint64_t seed, float *rotation,
                              float *qjl, float *centroids, float *midpoints);

/* Host copies of the fp32 tables. Any pointer may be NULL. R and S are
 * head_dim*head_dim row-major; centroids 2^index_bits; midpoints
 * 2^index_bits - 1. Group codecs have no tables (TQ_ERR_INVALID_ARG). */
tq_status tq_codec_export(const tq_codec *codec, float *rotation, float *qjl, float *centroids,
                          float *midpoints);

/* ------------------------------------------------------------------ */
/* Cache layout                                                         */
/* ------------------------------------------------------------------ */

/*
 * Paged compressed cache. Each layer owns a pool of num_blocks blocks; a
 * block holds block_tokens consecutive tokens of one sequence for every KV
 * head. The (block p, head h) sub-block starts at byte
 *     (p * num_kv_heads + h) * subblock_bytes
 * of the layer pool and stores its streams one after another, each
 * token-major: key indices [BT][index_words] u32, key QJL signs
 * [BT][head_dim/32] u32 (prod), key norms [BT] f32, key residual norms [BT]
 * f32 (prod), value indices [BT][index_words] u32, then value norms [BT] f32
 * (MSE) or value scales and minima [BT][head_dim/group] f16 (group).
 * A contiguous cache is the special case of one sequence whose block table
 * is the identity (or NULL, see below).
 */
typedef struct {
    void *pool;              /* device, 16-byte aligned: pool of layer 0             */
    int64_t layer_stride;    /* bytes between consecutive layer pools               */
    int num_layers;
    int num_blocks;          /* physical blocks per layer pool                      */
    int block_tokens;        /* power of two, 16..65536                             */
    int num_kv_heads;
    int head_dim;
    int key_mode, key_bits;
    uint64_t key_seed;
    int value_mode, value_bits, value_group;
    uint64_t value_seed;
    int64_t subblock_bytes;  /* block_tokens * (key + value record bytes)           */
    int64_t stream_offset[7];/* byte offsets of the streams in a sub-block (-1 = none):
                                key idx, key signs, key norm, key rnorm,
                                value idx, value norm | value scale, value min     */
    int encode_policy;       /* tq_encode_policy; tq_cache_desc_init sets AUTO      */
} tq_cache_desc;

/*
 * Fill *desc for a pool of num_layers layers laid out back to back
 * (layer_stride = num_blocks * num_kv_heads * subblock_bytes). If pool_bytes
 * is smaller than that total, returns TQ_ERR_CAPACITY. pool may be NULL to
 * query sizes only (pool_bytes is then ignored); *required_bytes (optional)
 * receives the total.
 */
tq_status tq_cache_desc_init(tq_cache_desc *desc, const tq_codec *key_codec,
                             const tq_codec *value_codec, int num_layers, int num_blocks,
                             int block_tokens, int num_kv_heads, void *pool, size_t pool_bytes,
                             size_t *required_bytes);

/*
 * Copy whole blocks of compressed records, every layer, from cache `src` to
 * cache `dst`: block src_blocks[i] of src becomes block dst_blocks[i] of dst.
 * The batch operations of "omlx/turboquant_kv.py" (BatchTurboQuantKVCache.merge,
 * extend, extract, filter) become, on a paged cache, block-table edits plus
 * this copy: merge and extend copy the joining sequences' blocks into the
 * batch's pool and append their table rows, extract copies one sequence's
 * blocks into a cache of its own, filter keeps table rows and copies nothing.
 * Ragged lengths need no padding (seq_lens are per sequence), so the pages'
 * left/right-padding realignment (prepare, finalize) has no counterpart.
 *   src_blocks, dst_blocks device int32 [n]; when src and dst share a pool,
 *   the two sets must not overlap.
 * Errors: TQ_ERR_CONFIG_MISMATCH unless both caches have the same head_dim,
 * heads, block size, layer count and codec configuration (the mixed-config
 * guard of BatchTurboQuantKVCache.merge); TQ_ERR_INVALID_ARG for bad
 * pointers or n < 0. Ids outside [0, num_blocks) are skipped and flagged
 * (TQ_DEVERR_BLOCK).
 */
tq_status tq_cache_copy_blocks(const tq_cache_desc *src, const tq_cache_desc *dst, const int32_t *src_blocks,
                               const int32_t *dst_blocks, int n, tq_stream_t stream);

/*
 * A batch of sequences in a paged cache: the state that
 * "omlx/turboquant_kv.py" (BatchTurboQuantKVCache) keeps per batch, on the
 * paged layout. Row b of the block table lists the physical blocks of
 * sequence b in token order (-1 = no block); seq_lens[b] counts its cached
 * tokens, which occupy its first ceil(seq_lens[b] / block_tokens) blocks.
 * Entries past those may hold blocks reserved for later appends.
 */
typedef struct {
    const tq_cache_desc *cache; /* pool and layout holding the batch's blocks     */
    int32_t *block_table;       /* device [capacity][max_blocks]                   */
    int32_t *seq_lens;          /* device [capacity]                               */
    int batch;                  /* sequences in use: rows 0 .. batch-1             */
    int capacity;               /* rows that block_table and seq_lens hold         */
    int max_blocks;             /* entries per block-table row                     */
} tq_batch;

/*
 * The batch operations of "omlx/turboquant_kv.py" (BatchTurboQuantKVCache
 * .filter, .extend, .merge, .extract) on the paged layout. Each checks the
 * mixed-configuration guard of .merge on the host (TQ_ERR_CONFIG_MISMATCH
 * unless every cache involved has the same head_dim, KV heads, block size,
 * layer count and key/value codec configuration), then rewrites block-table
 * rows and sequence lengths on the device and, where a sequence moves to
 * another pool, copies its blocks (every layer). Ragged lengths need no
 * padding, so the pages' left-padding realignment (prepare, finalize, the
 * padding arithmetic of extend and extract) has no counterpart here.
 *
 * Blocks taken in a destination pool come from the caller's free list:
 * free_blocks (device int32 [n_free]) is consumed in order from index
 * *n_used (device int32, read and advanced by the call; zero it before a
 * first call). A sequence whose blocks do not fit gets -1 entries and sets
 * TQ_DEVERR_CAPACITY; a source block id outside its pool is skipped and
 * sets TQ_DEVERR_BLOCK; a length beyond its row's blocks sets
 * TQ_DEVERR_SEQLEN (tq_device_error). Where source and destination share a
 * pool (the same pool pointer), rows keep their block ids and nothing is
 * copied: the blocks change owner.
 * Table and length arrays of the two sides must not overlap; all calls are
 * asynchronous on the stream and update the host fields batch as stated.
 */

/*
 * filter (BatchTurboQuantKVCache.filter): out rows 0..n_keep-1 become rows
 * keep[0..n_keep-1] (host int32, distinct, each in [0, batch->batch)) of
 * `batch`, whole rows with their reserved entries; out->batch = n_keep.
 * `out` describes the same pool. Every block id (>= 0) of the rows not kept
 * is written to freed (device int32, room for (batch->batch - n_keep) *
 * max_blocks ids) in row then entry order, and *n_freed (device int32) is set
 * to their count. Nothing is copied.
 * Errors: TQ_ERR_INVALID_ARG for bad pointers, sizes, repeated or
 * out-of-range keep entries, or out->capacity < n_keep;
 * TQ_ERR_CONFIG_MISMATCH if out->cache is not the same pool and layout.
 */
tq_status tq_batch_filter(const tq_batch *batch, const int32_t *keep, int n_keep, tq_batch *out, int32_t *freed,
                          int32_t *n_freed, tq_stream_t stream);

/*
 * extend (BatchTurboQuantKVCache.extend): the sequences of `src` become rows
 * dst->batch .. dst->batch + src->batch - 1 of `dst`, in order; each keeps
 * its length, and its blocks are copied into blocks taken from the free list
 * of dst's pool (entries past its last token's block become -1), unless both
 * batches share a pool. dst->batch grows by src->batch.
 * Errors: TQ_ERR_CAPACITY if dst->capacity is too small; TQ_ERR_INVALID_ARG
 * for bad pointers or sizes; the mixed-configuration guard.
 */
tq_status tq_batch_extend(tq_batch *dst, const tq_batch *src, const int32_t *free_blocks, int n_free,
                          int32_t *n_used, tq_stream_t stream);

/*
 * merge (BatchTurboQuantKVCache.merge): tq_batch_extend of dst by srcs[0],
 * srcs[1], ... in order (each src usually one sequence in a cache of its
 * own). The guard covers every source before anything is launched.
 */
tq_status tq_batch_merge(tq_batch *dst, const tq_batch *srcs, int n_srcs, const int32_t *free_blocks, int n_free,
                         int32_t *n_used, tq_stream_t stream);

/*
 * extract (BatchTurboQuantKVCache.extract): sequence idx (host, in
 * [0, src->batch)) of `src` becomes the only sequence of `dst` (row 0,
 * dst->batch = 1), its blocks copied into blocks from dst's free list unless
 * the two share a pool.
 * Errors: as tq_batch_extend; TQ_ERR_INVALID_ARG for idx out of range.
 */
tq_status tq_batch_extract(const tq_batch *src, int idx, tq_batch *dst, const int32_t *free_blocks, int n_free,
                           int32_t *n_used, tq_stream_t stream);

/* ------------------------------------------------------------------ */
/* Encode                                                               */
/* ------------------------------------------------------------------ */

/*
 * Append n_new tokens per sequence to layer `layer` of the cache: compress
 * keys with key_codec and values with value_codec and write them at
 * positions seq_lens[b] .. seq_lens[b]+n_new-1 -- the written end of each
 * sequence, never the allocated capacity ("omlx/turboquant_kv.py",
 * BatchTurboQuantKVCache._phys_end) -- incremental per-token append as
 * "lightning-mlx/plan.md" asks of update_and_fetch.
 *   k, v        device [batch][num_kv_heads][n_new][head_dim], dtype f32/bf16/f16
 *   seq_lens    device int32 [batch], tokens already cached (not modified)
 *   block_table device int32 [batch][max_blocks] of physical block ids, or NULL:
 *               then sequence b owns blocks b*max_blocks .. b*max_blocks+max_blocks-1
 * The fp32 specification (sequential fused multiply-adds, IEEE division and
 * square root): norm = sqrt(sum x_k^2), y = (R x)/norm,
 * index_i = #{midpoints < y_i}; prod residual r = y - c[index], rnorm = |r|,
 * sign_j = ((S r)_j >= 0). Short appends (decode steps), group codecs, f32
 * inputs, head_dim 256 and TQ_ENCODE_EXACT follow it bit for bit. With
 * TQ_ENCODE_AUTO, appends of >= 64 tokens of bf16/f16 MSE or prod vectors
 * with head_dim 64 or 128 rotate on the tensor cores, as the pages plan for
 * chunked prefill: norms stay bit-exact, y and S r are computed with errors
 * far below the specification's own fp32 rounding bound, so an index or a
 * sign differs from the specification only where the exact value lies within
 * that bound of a decision threshold (a midpoint, or 0), and the residual
 * norm then follows the differing index. Tokens past a sequence's capacity
 * are skipped and flagged (TQ_DEVERR_CAPACITY).
 * Errors: TQ_ERR_CONFIG_MISMATCH if a codec's (head_dim, bits, mode, seed,
 * group) differs from the descriptor (the mixed-config guard of
 * BatchTurboQuantKVCache.merge); TQ_ERR_CAPACITY if n_new exceeds
 * max_blocks*block_tokens; TQ_ERR_INVALID_ARG for bad pointers or sizes or an
 * unknown encode_policy.
 */
tq_status tq_encode_append(const tq_codec *key_codec, const tq_codec *value_codec,
                           const tq_cache_desc *cache, int layer, const void *k, const void *v,
                           tq_dtype dtype, int batch, int n_new, const int32_t *seq_lens,
                           const int32_t *block_table, int max_blocks, tq_stream_t stream);

/*
 * Codec-only quantise of n vectors x (device [n][head_dim]) into plain record
 * arrays (the codec's quantize): idx [n][index_words] u32; for MSE norm [n]
 * f32; for prod also signs [n][head_dim/32] u32 and rnorm [n] f32; for group
 * scale and min [n][head_dim/group] f16 (passed in aux0/aux1). Unused
 * outputs may be NULL. Same arithmetic as tq_encode_append.
 *   mse : aux0 = norm,  aux1 = unused, aux2 = unused
 *   prod: aux0 = norm,  aux1 = signs,  aux2 = rnorm
 *   group: aux0 = scale, aux1 = min,   aux2 = unused
 */
tq_status tq_quantize(const tq_codec *codec, const void *x, tq_dtype dtype, int64_t n,
                      uint32_t *idx, void *aux0, void *aux1, void *aux2, tq_stream_t stream);

/* ------------------------------------------------------------------ */
/* Decode attention                                                     */
/* ------------------------------------------------------------------ */

/* Workspace (device bytes) tq_decode_attention needs for these sizes. */
tq_status tq_decode_workspace_bytes(const tq_cache_desc *cache, int batch, int num_q_heads,
                                    int q_len, int max_seq_len, size_t *bytes);

/* Launch shape tq_decode_attention would use (host arithmetic only; the pages
 * have no counterpart: this exists so callers can inspect and size a decode). */
typedef struct {
    int tensor_cores;    /* 1: tensor-core split kernel (head_dim 128; 64 and 256 with prod *
                          *    3-bit keys and group 2/4-bit or MSE 3/4-bit values, or MSE  *
                          *    4-bit keys and values); 0: SIMT kernels                     */
    int row_groups;      /* 16-row groups per (sequence, KV head): ceil(G * q_len / 16)    */
    int splits;          /* token splits per (sequence, KV head, row group)               */
    int chunk_tokens;    /* tokens per split (a multiple of tile_tokens)                  */
    int tile_tokens;     /* tokens per shared-memory stage: divides block_tokens, or      *
                          * gathers up to four whole blocks; 64 unless 32 balances the    *
                          * CTA's warps better or the stages would not fit next to the    *
                          * lookup tables                                                 */
    size_t smem_bytes;   /* dynamic shared memory of the split kernel (tensor cores)     */
    size_t workspace_bytes; /* as tq_decode_workspace_bytes for num_sms SMs              */
    int transposed;      /* 1: the tensor-core split kernel in its transposed form        *
                          * (head_dim 128, at most 8 query rows per KV head, the codec    *
                          * pairs of the head_dim-64/256 set): tokens on the MMA's M       */
} tq_decode_plan_info;

/*
 * The plan tq_decode_attention makes for these sizes on a GPU of num_sms SMs
 * (the split count targets one CTA per SM). cache: the descriptor's layout
 * fields (head_dim, modes, bits, group, block_tokens, num_kv_heads,
 * subblock_bytes, stream_offset); no device is touched. Returns
 * TQ_ERR_INVALID_ARG or TQ_ERR_UNSUPPORTED as tq_decode_workspace_bytes does.
 */
tq_status tq_decode_plan(const tq_cache_desc *cache, int batch, int num_q_heads, int q_len,
                         int max_seq_len, int num_sms, tq_decode_plan_info *info);

/*
 * Decode attention over layer `layer` of the compressed cache
 * ("lightning-mlx/plan.md": fused attention over Lloyd-Max codes;
 * "turboquant/validate_moe_phase2.py": attention_score scores queries against
 * compressed keys). For every sequence b, query head hq (KV head
 * hq / (num_q_heads/num_kv_heads)) and query position l < q_len:
 *   q' = R_k q, q'' = S_k q' (once per query);
 *   score_t = scale * n_t * (<q', c_k[idx_t]> + sqrt(pi/2)/D * rnorm_t <q'', sign_t>)
 *             (the second term for prod keys only), for keys t <= N - q_len + l
 *             where N = seq_lens[b] (the q_len query tokens are the newest,
 *             already appended);
 *   out = softmax(score) . V, with MSE values accumulated in the rotated domain
 *         as n^v_t c_v[idx^v_t] and rotated back once (x = (sum) @ R_v), group
 *         values as code*scale+min.
 *   q    device [batch][num_q_heads][q_len][head_dim], f32/bf16/f16
 *   out  device [batch][num_q_heads][q_len][head_dim] f32
 *   seq_lens device int32 [batch] in [q_len, capacity]; max_seq_len (host) must
 *        bound every seq_lens[b]; it sizes the split-K grid.
 *   scale 0 means 1/sqrt(head_dim).
 *   workspace device, >= tq_decode_workspace_bytes(...), 256-byte aligned;
 *        only this call uses it while it runs (calls that overlap on the GPU
 *        must use distinct workspaces).
 * (num_q_heads/num_kv_heads) * q_len <= 64.
 */
tq_status tq_decode_attention(const tq_codec *key_codec, const tq_codec *value_codec,
                              const tq_cache_desc *cache, int layer, const void *q,
                              tq_dtype q_dtype, int batch, int num_q_heads, int q_len,
                              const int32_t *seq_lens, const int32_t *block_table, int max_blocks,
                              int max_seq_len, float scale, float *out, void *workspace,
                              size_t workspace_bytes, tq_stream_t stream);

/*
 * One decode step of one layer: tq_encode_append of the step's n_new tokens
 * followed by tq_decode_attention over the grown sequences
 * ("lightning-mlx/plan.md", the minimum work list: an incremental append that
 * quantizes only the new tokens, and attention over the compressed cache;
 * running both from one call, with the append inside the decode's first
 * launch, is this library's). Results are those of the two calls in sequence:
 * the same cache bytes and the same outputs.
 *   k_new, v_new device [batch][num_kv_heads][n_new][head_dim], kv_dtype
 *        f32/bf16/f16; n_new >= 0 (0: a plain decode).
 *   seq_lens device int32 [batch]: tokens in the cache BEFORE the step (not
 *        modified); the new tokens go to positions seq_lens[b] ..
 *        seq_lens[b] + n_new - 1 and sequence b then attends over
 *        seq_lens[b] + n_new tokens, its q_len queries being the newest.
 *   max_seq_len (host) bounds every seq_lens[b] + n_new; the workspace is
 *        tq_decode_workspace_bytes(cache, batch, num_q_heads, q_len,
 *        max_seq_len).
 *   q, out, block_table, max_blocks, scale, workspace: as tq_decode_attention.
 * With head_dim 128, rotated keys and values (MSE or prod), n_new <= 8 and the
 * tensor-core decode, the append runs inside the query-prep launch (two
 * launches per step instead of three); otherwise the two calls run in order.
 * Errors: those of tq_encode_append and tq_decode_attention, checked before
 * anything is launched.
 */
tq_status tq_decode_step(const tq_codec *key_codec, const tq_codec *value_codec,
                         const tq_cache_desc *cache, int layer, const void *k_new,
                         const void *v_new, tq_dtype kv_dtype, int n_new, const void *q,
                         tq_dtype q_dtype, int batch, int num_q_heads, int q_len,
                         const int32_t *seq_lens, const int32_t *block_table, int max_blocks,
                         int max_seq_len, float scale, float *out, void *workspace,
                         size_t workspace_bytes, tq_stream_t stream);

/* ------------------------------------------------------------------ */
/* Sequence-sharded decode                                              */
/* ------------------------------------------------------------------ */

/*
 * Decode attention over one shard of each sequence's tokens, when a KV cache
 * is split by sequence position across GPUs ("turboquant/validate_moe_phase2.py",
 * TEST 3: with tensor parallelism each GPU holds a shard of the KV cache).
 * Each shard yields, per query row, the unnormalised softmax state of its
 * keys; tq_decode_merge combines the shards' states. Scores and values are
 * those of tq_decode_attention.
 *   seq_lens   device int32 [batch]: tokens of this shard (0 allowed).
 *   causal_end device int32 [batch] or NULL: the end of the queries' causal
 *              window in this shard's local token indices, i.e. the global
 *              sequence length minus the global index of the shard's first
 *              token; query l (of q_len) sees local keys t <= causal_end -
 *              q_len + l. NULL means the shard's own length (the queries are
 *              its newest tokens).
 *   part_ml    device float [batch][num_q_heads][q_len][2] (8-byte aligned):
 *              m (a reference maximum of the scores, natural-log units) and
 *              l = sum_t exp(s_t - m) over the visible keys; a row with no
 *              visible key gets m = -inf, l = 0.
 *   part_acc   device float [batch][num_q_heads][q_len][head_dim] (16-byte
 *              aligned): sum_t exp(s_t - m) v_t, with v_t in the rotated
 *              domain for MSE values (n c[index], before the inverse
 *              rotation) and dequantised for group values.
 *   m is any reference value the kernels keep (the state is defined up to it:
 *   m + ln l and acc / l are unique).
 *   max_seq_len >= 1 bounds every seq_lens[b]; workspace as
 *   tq_decode_workspace_bytes(cache, batch, num_q_heads, q_len, max_seq_len).
 * Other arguments and errors as tq_decode_attention.
 */
tq_status tq_decode_partials(const tq_codec *key_codec, const tq_codec *value_codec,
                             const tq_cache_desc *cache, int layer, const void *q, tq_dtype q_dtype,
                             int batch, int num_q_heads, int q_len, const int32_t *seq_lens,
                             const int32_t *causal_end, const int32_t *block_table, int max_blocks,
                             int max_seq_len, float scale, float *part_ml, float *part_acc,
                             void *workspace, size_t workspace_bytes, tq_stream_t stream);

/*
 * Log-sum-exp merge of num_parts shards' states of `rows` query rows:
 * parts_ml [num_parts][rows][2] and parts_acc [num_parts][rows][head_dim]
 * (device, in the layout tq_decode_partials writes, one part after another;
 * rows = batch * num_q_heads * q_len). out [rows][head_dim] (device fp32) =
 * (sum_p e^(m_p - M) acc_p) / (sum_p e^(m_p - M) l_p), M = max_p m_p, then
 * `@ R_v` for MSE values (value_codec's rotation; "lightning-mlx/plan.md",
 * the inverse rotation `rotated @ Q`); rows no part sees are 0. The parts
 * may come from different GPUs (gathered by the caller).
 */
tq_status tq_decode_merge(const tq_codec *value_codec, int num_parts, const float *parts_ml,
                          const float *parts_acc, int64_t rows, float *out, tq_stream_t stream);

/* ------------------------------------------------------------------ */
/* Split (low/high) states                                              */
/* ------------------------------------------------------------------ */

/*
 * Split states ("omlx/turboquant_kv.py": TurboQuantSplitState(low, high),
 * carried through the batch operations by _filter_state and
 * _concat_state_batch): each key and value vector of head_dim D is stored as
 * two TurboQuant states, the low coordinates [0, DL) under one codec pair and
 * the high coordinates [DL, D) under another, each with its own norm,
 * rotation, Lloyd-Max codebook and bit width (for example more bits on the
 * high channels, the outlier channels of a mixed width). The two halves live
 * in two caches of the same layout shape (layers, blocks, block size, KV
 * heads) addressed by one block table and one set of lengths; each cache is
 * an ordinary cache of its half's head_dim (batch operations apply to both).
 */
typedef struct {
    const tq_codec *key_low, *value_low;    /* head_dim DL                         */
    const tq_codec *key_high, *value_high;  /* head_dim DH                         */
    const tq_cache_desc *low, *high;        /* caches of the two halves            */
} tq_split_state;

/*
 * Append n_new tokens per sequence to both halves: tq_encode_append of the
 * low halves k_low, v_low [batch][num_kv_heads][n_new][DL] into `low` and of
 * k_high, v_high [batch][num_kv_heads][n_new][DH] into `high` (device,
 * contiguous, one dtype). Errors: those of tq_encode_append;
 * TQ_ERR_CONFIG_MISMATCH if the two caches differ in layers, blocks, block
 * size or KV heads.
 */
tq_status tq_encode_append_split(const tq_split_state *state, int layer, const void *k_low, const void *v_low,
                                 const void *k_high, const void *v_high, tq_dtype dtype, int batch, int n_new,
                                 const int32_t *seq_lens, const int32_t *block_table, int max_blocks,
                                 tq_stream_t stream);

/* Workspace (device bytes) of tq_decode_attention_split for these sizes. */
tq_status tq_decode_workspace_bytes_split(const tq_split_state *state, int batch, int num_q_heads, int q_len,
                                          int max_seq_len, size_t *bytes);

/*
 * Decode attention over split states: score_t = scale * (<q_low, k_hat_low_t>
 * + <q_high, k_hat_high_t>), each half scored in its own rotated domain as
 * tq_decode_attention scores a whole vector, softmax over the visible keys
 * (the causal rule of tq_decode_attention), out = [o_low | o_high] with each
 * half's value sum rotated back by its own value rotation (group halves are
 * not rotated).
 *   q    device [batch][num_q_heads][q_len][D], D = DL + DH; scale 0 means
 *        1/sqrt(D). out device [batch][num_q_heads][q_len][D] fp32.
 * DL, DH in {64, 128}; (num_q_heads/num_kv_heads) * q_len <= 64. Other
 * arguments and errors as tq_decode_attention.
 */
tq_status tq_decode_attention_split(const tq_split_state *state, int layer, const void *q, tq_dtype q_dtype,
                                    int batch, int num_q_heads, int q_len, const int32_t *seq_lens,
                                    const int32_t *block_table, int max_blocks, int max_seq_len, float scale,
                                    float *out, void *workspace, size_t workspace_bytes, tq_stream_t stream);

/* ------------------------------------------------------------------ */
/* Prefill attention                                                    */
/* ------------------------------------------------------------------ */

/* Workspace (device bytes) tq_prefill_attention needs for these sizes. */
tq_status tq_prefill_workspace_bytes(const tq_cache_desc *cache, int batch, int num_q_heads,
                                     int q_len, size_t *bytes);

/*
 * Prefill attention over layer `layer` of the compressed cache: the function
 * of tq_decode_attention for a long query chunk ("omlx/turboquant_kv.py":
 * BatchTurboQuantKVCache inherits prefill_attention from the cache it wraps,
 * with the causal mask offset by the written end, make_mask). The q_len
 * query positions are the newest of each sequence, already appended; query
 * l attends to keys t <= seq_lens[b] - q_len + l, scores and values exactly
 * as tq_decode_attention defines them. Each key/value tile is decoded once
 * for 128 query rows (8 groups of 16) instead of once per 16, and no split-K
 * is needed.
 *   q, out, seq_lens, block_table, max_blocks, scale: as tq_decode_attention.
 *   workspace device, >= tq_prefill_workspace_bytes(...), 256-byte aligned
 *        (query fragments, 8 KB per 16 query rows of a KV head).
 * head_dim 128; keys prod 3-bit with MSE 3/4-bit or group 4-bit values, or
 * keys and values MSE 4-bit (TQ_ERR_UNSUPPORTED otherwise);
 * (num_q_heads/num_kv_heads) * q_len / 16 <= 65535.
 */
tq_status tq_prefill_attention(const tq_codec *key_codec, const tq_codec *value_codec,
                               const tq_cache_desc *cache, int layer, const void *q,
                               tq_dtype q_dtype, int batch, int num_q_heads, int q_len,
                               const int32_t *seq_lens, const int32_t *block_table, int max_blocks,
                               float scale, float *out, void *workspace, size_t workspace_bytes,
                               tq_stream_t stream);

/*
 * Decode attention without a caller-provided workspace. (The pages have no
 * counterpart; this exists for callers of this library.)
 *
 * For callers that cannot allocate device memory: hosts that own all of the
 * GPU's memory and expose no allocator to plug-ins, and serving loops that must
 * not allocate once running (an allocation can block on the device or fail
 * under memory pressure mid-request). Arguments and results are those of
 * tq_decode_attention; the scratch it needs lives instead in a fixed device
 * array of TQ_NOALLOC_SCRATCH_BYTES that every GPU where this library is set
 * up keeps until the process exits. Nothing is allocated by this call.
 *   - The array is reserved, and its device address looked up, when the
 *     library is first set up on a device: by the first tq_codec_create,
 *     tq_codec_create_group or tq_codec_pair_for_bits with that device
 *     current. On a device never set up, this call fails as
 *     tq_decode_attention does with no workspace (TQ_ERR_INVALID_ARG).
 *   - Returns the statuses of tq_decode_attention for the same arguments,
 *     checked in the same order, with TQ_ERR_CAPACITY (nothing launched)
 *     when tq_decode_workspace_bytes() for these sizes exceeds
 *     TQ_NOALLOC_SCRATCH_BYTES (use tq_decode_attention instead).
 *   - All calls on a device share the one array, which keeps the last call's
 *     contents: calls that overlap on the GPU (other streams, or other host
 *     threads) race and corrupt each other's results. Serialise them.
 *   - The cached address belongs to the device's primary context: resetting
 *     the device (cudaDeviceReset) while this library is loaded is not
 *     supported, by this call or by any other (the per-device error word's
 *     address is cached the same way).
 */
#define TQ_NOALLOC_SCRATCH_BYTES (16u << 20)
tq_status tq_decode_attention_noalloc(const tq_codec *key_codec, const tq_codec *value_codec,
                                      const tq_cache_desc *cache, int layer, const void *q,
                                      tq_dtype q_dtype, int batch, int num_q_heads, int q_len,
                                      const int32_t *seq_lens, const int32_t *block_table,
                                      int max_blocks, int max_seq_len, float scale, float *out,
                                      tq_stream_t stream);

/* ------------------------------------------------------------------ */
/* Diagnostics                                                          */
/* ------------------------------------------------------------------ */

const char *tq_status_string(tq_status status);
/* Synchronises the current device, returns its error word in *flags and
 * clears it. Returns TQ_ERR_DEVICE_BOUNDS if any bit was set. */
tq_status tq_device_error(uint32_t *flags);
/* Number of kernels this library has launched since it was loaded. */
uint64_t tq_launch_count(void);
/* Self-test of the bounded-wait error path (the kernels wait for their bulk
 * copies on mbarriers, each wait bounded; a wait that runs out sets
 * TQ_DEVERR_TIMEOUT and the kernel returns). Launches one kernel on `stream`
 * whose single thread waits on an mbarrier nothing arrives on, with a deadline
 * of `seconds` (0 < seconds <= 1, else TQ_ERR_INVALID_ARG, nothing launched)
 * on the GPU's global timer; when it passes, the kernel sets
 * TQ_DEVERR_TIMEOUT in the device error word, invalidates the barrier and
 * returns. No fault and no hang: the device stays usable, and the next
 * tq_device_error() reports and clears the bit. Returns TQ_ERR_CUDA if the
 * launch fails. */
tq_status tq_selftest_wait_timeout(double seconds, tq_stream_t stream);
int tq_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* TQ_H */

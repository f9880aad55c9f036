// Internal declarations shared by the libtq translation units.
#pragma once

#include <atomic>
#include <cstdint>
#include <vector>

#include "tq.h"

#ifdef __CUDACC__
#include <cuda_runtime.h>
#endif

namespace tq {

struct HostTables {
    std::vector<float> rotation;   // D x D row-major, y = R x
    std::vector<float> qjl;        // D x D row-major (prod only)
    std::vector<float> centroids;  // 2^index_bits, ascending, antisymmetric
    std::vector<float> midpoints;  // 2^index_bits - 1
    // Half-precision operand levels of the tensor-core kernels: op_levels[j]
    // is the fp16 number nearest to op_scale * centroids[j] (stored as fp32,
    // exactly), with op_scale in [1, 2) chosen so that the largest relative
    // rounding error over the levels is as small as a search finds; kernels
    // divide op_scale out again in fp32.
    std::vector<float> op_levels;
    float op_scale = 1.0f;
};

// Deterministic codec tables from (D, index bits, seed) (host, fp64 -> fp32).
void build_codec_tables(int D, int index_bits, bool with_qjl, uint64_t seed, HostTables& out);

// Tensor-core operand of scale * M (D x D row-major): fp16 bits of the hi part
// then of the lo remainder, each in the no-swizzle K-major core-matrix layout
// (row = output coordinate, K = input coordinate).
void build_tc_operand(const std::vector<float>& M, int D, double scale, std::vector<uint16_t>& out);

// Device view of one codec.
struct CodecDev {
    const float* R;    // [D][D] row-major
    const float* Rt;   // [D][D] transposed rotation (Rt[k*D+i] = R[i][k])
    const float* St;   // [D][D] transposed QJL matrix (prod) or nullptr
    const float* SRt;  // [D][D] transposed product S R (prod, head_dim other than 128) or nullptr
    const float* c;    // centroids
    const float* m;    // midpoints
    const float* cq;   // fp16-exact operand levels op_scale * c (see HostTables)
    float cq_scale;    // op_scale
    const uint16_t* Rtc;  // tensor-core operand of 16 R (hi, lo), or nullptr
    const uint16_t* Stc;  // tensor-core operand of S (hi, lo) (prod), or nullptr
    // decode lookup tables in their shared-memory layout (copied as they are),
    // or nullptr: 2-bit code quads, entry e (a byte of four codes) at
    // 128 e + 8 c for bank copy c < 16, fp16 pairs (cq[e & 3], cq[(e >> 2) & 3]),
    // (cq[(e >> 4) & 3], cq[e >> 6]); 3-bit code pairs, entry e (six bits) at
    // 128 e + 4 c for bank copy c < 32, fp16 pair (cq[e & 7], cq[e >> 3])
    const uint32_t* quad;
    const uint32_t* pair;
    const uint32_t* pair4;  // 4-bit code pairs, entry e (a byte) at 128 e + 4 c for bank copy c < 32:
                            // fp16 pair (cq[e & 15], cq[e >> 4]); or nullptr
    const uint32_t* pair4w; // the same pairs in 256-byte entries (e at 256 e + 4 c for c < 64: two
                            // sets of bank copies, for keys and values), or nullptr
    int D;
    int mode;          // tq_mode
    int bits;          // total bits
    int ib;            // index bits
    int W;             // index words
    int Ws;            // sign words (prod)
    int group;         // group size (group mode)
};

// Device view of one layer pool.
struct PoolDev {
    char* base;          // layer pool
    int64_t sub_bytes;   // bytes per (block, head) sub-block
    int64_t off[7];      // stream offsets inside a sub-block
    int Hkv;
    int BT;              // tokens per block
    int num_blocks;
};

struct EncodeAppendArgs {
    CodecDev kc, vc;
    PoolDev pool;
    const void* k;
    const void* v;
    int dtype;
    int batch, n_new;
    const int32_t* seq_lens;
    const int32_t* table;
    int max_blocks;
    int exact;           // 1: sequential fp32 order only (no tensor-core rotation)
    unsigned* err;
};

struct QuantizeArgs {
    CodecDev cd;
    const void* x;
    int dtype;
    int64_t n;
    uint32_t* idx;
    void* aux0;
    void* aux1;
    void* aux2;
};

// Decode plan shared by workspace sizing and the launch.
struct DecodePlan {
    int kind;         // 0: SIMT kernels (any shape), 1: tensor-core kernels (head_dim 128, some 64 and 256)
    int r8;           // tensor-core kernels in the transposed form (head_dim 128, at most 8 rows per unit)
    int rows;         // G * Lq
    int row_groups;   // ceil(rows / 16)
    int splits;       // token splits per (sequence, kv head, row group)
    int chunk;        // tokens per split (multiple of the tile)
    int tile;         // tokens per tile / shared-memory stage
    int kb, vb;       // key / value index bits (tensor-core path)
    bool kprod, vgroup;
    int st_off[7];    // stage layout (tensor-core path)
    int st_field[7];
    int st_bytes;
    int bar_off;      // shared-memory offset of the stage barriers
    int qs_off;       // shared-memory offset of the query fragments
    int vt_off;       // shared-memory offset of the 3-bit value pair table region (-1: unused)
    int kt_off;       // shared-memory offset of the 2-bit key quad table (-1: unused)
    int ring_off;     // shared-memory offset of the stage rings (after a table at offset 0)
    size_t smem;      // dynamic shared memory of the split kernel
    size_t q_bytes;   // SIMT and head_dim 256: q' and q'' buffers (each); tensor cores at 128: query fragments
    size_t part_bytes;// partial accumulators
    size_t ml_bytes;  // partial (max, sum)
    size_t total;
};

struct DecodeArgs {
    CodecDev kc, vc;
    PoolDev pool;
    const void* q;
    int q_dtype;
    int batch, Hq, Lq, G;
    const int32_t* seq_lens;
    int len_add;   // tokens appended in the same step: sequence b attends seq_lens[b] + len_add
    const int32_t* table;
    int max_blocks;
    float scale;
    float* out;
    // Sequence shards (tq_decode_partials): causal_end[b] (device, or null:
    // the sequence's own length) is where the queries' causal window ends in
    // the shard's local token indices; with part_ml / part_acc set, the final
    // merge writes each row's unnormalised softmax state (max in natural-log
    // units, sum, accumulator in the rotated domain) there instead of out.
    const int32_t* causal_end;
    float* part_ml;    // [B][Hq][Lq][2]
    float* part_acc;   // [B][Hq][Lq][D]
    float* qrot;   // [B][Hkv][RG*16][D]
    float* qjl;    // [B][Hkv][RG*16][D]
    float* part;   // [B][Hkv][RG][splits][16][D]
    float* ml;     // [B][Hkv][RG][splits][16][2]
    void* ws;      // workspace base
    DecodePlan plan;
    unsigned* err;
};

// Decode over split (low/high) states (decode_split.cu): two codec pairs and
// two pools holding the low coordinates [0, DL) and the high [DL, D).
struct SplitStateArgs {
    CodecDev klo, vlo, khi, vhi;
    PoolDev plo, phi;
    const void* q;
    int q_dtype;
    int batch, Hq, Lq, G, Hkv;
    const int32_t* seq_lens;
    const int32_t* table;
    int max_blocks;
    float scale;
    float* out;
    float* qrot;   // [B][Hkv][RG*16][D]
    float* qjl;
    float* part;   // [B][Hkv][RG][splits][16][D]
    float* ml;
    int rows, row_groups, splits, chunk;
    unsigned* err;
};
void split_state_plan(SplitStateArgs& a, int max_seq_len, int num_sms);
size_t split_state_workspace(const SplitStateArgs& a, int D);
void split_state_bind_workspace(SplitStateArgs& a, void* ws, int D);

DecodePlan make_decode_plan(const tq_cache_desc* d, int batch, int G, int Lq, int max_seq_len, int num_sms);

#ifdef __CUDACC__
// Launch with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream finishes; it must call griddepcontrol.wait
// before it touches what that kernel (or anything before it) writes.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args... args) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

cudaError_t launch_encode_append(const EncodeAppendArgs& a, cudaStream_t s);
cudaError_t launch_encode_block(const EncodeAppendArgs& a, int is_v, cudaStream_t s);
bool encode_tc_supported(const EncodeAppendArgs& a, int is_v);
cudaError_t launch_encode_tc(const EncodeAppendArgs& a, int is_v, cudaStream_t s);
bool launch_encode_tc_pair(const EncodeAppendArgs& a, cudaStream_t s, cudaError_t* err);
cudaError_t launch_quantize(const QuantizeArgs& a, cudaStream_t s);
// `step` (tensor-core path only): the decode step's append, fused into the
// query-prep launch; null for a plain decode.
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t s, const EncodeAppendArgs* step = nullptr);
// Log-sum-exp merge of sequence shards' partial states, then 1 / sum and
// the inverse value rotation (MSE values): decode.cu.
cudaError_t launch_shard_merge(const CodecDev& vc, int parts, const float* ml, const float* acc, int64_t rows,
                               float* out, cudaStream_t s);
cudaError_t launch_split_state(const SplitStateArgs& a, cudaStream_t s);
cudaError_t launch_copy_blocks(const tq_cache_desc* src, const tq_cache_desc* dst, const int32_t* src_ids,
                               const int32_t* dst_ids, int n, unsigned* err, cudaStream_t s);
// Block-table rows of a batch operation (cache_ops.cu): n output rows from
// src rows `rows` (host list, <= 256) or src_row0.., written at dst_row0..;
// copy: blocks moved into ids from the free list; n_drop rows (host list)
// whose block ids go to `freed`.
cudaError_t launch_batch_rows(const tq_batch* src, tq_batch* dst, int n, const int* rows, int src_row0, int dst_row0,
                              bool copy, const int32_t* free_blocks, int n_free, int32_t* n_used, int n_drop,
                              const int* drop, int32_t* freed, int32_t* n_freed, bool reset_freed, unsigned* err,
                              cudaStream_t s);
constexpr int kBatchRowChunk = 256;
namespace mmadec {
bool prefill_supported(int kb, bool kprod, bool vgroup, int vb);
cudaError_t launch_prefill(const DecodeArgs& a, const uint4* qfrag, cudaStream_t s);
}  // namespace mmadec
#endif

extern std::atomic<uint64_t> g_launches;

// Looks up, once per device with that device current, the device address of
// the fixed scratch array of tq_decode_attention_noalloc; loading the array's
// module is what reserves its memory on the device.
tq_status noalloc_reserve();

}  // namespace tq

// Opaque codec handle behind the C ABI.
struct tq_codec {
    int head_dim = 0;
    int bits = 0;
    int mode = 0;
    int group = 0;
    uint64_t seed = 0;
    int index_bits = 0;
    int index_words = 0;
    int sign_words = 0;
    int record_bytes = 0;
    int device = -1;
    tq::HostTables host;
    float* d_R = nullptr;
    float* d_Rt = nullptr;
    float* d_St = nullptr;
    float* d_SRt = nullptr;  // transposed S R (prod codecs with head_dim other than 128)
    float* d_c = nullptr;
    float* d_m = nullptr;
    float* d_cq = nullptr;
    uint16_t* d_Rtc = nullptr;
    uint16_t* d_Stc = nullptr;
    uint32_t* d_quad = nullptr;  // decode lookup table of 2-bit code quads (index bits 2)
    uint32_t* d_pair = nullptr;  // decode lookup table of 3-bit code pairs (index bits 3)
    uint32_t* d_pair4 = nullptr;  // decode lookup table of 4-bit code pairs (MSE, index bits 4)
    uint32_t* d_pair4w = nullptr; // the same in 256-byte entries
};

// tq_decode_attention_noalloc: decode attention for callers that cannot
// allocate device memory.
//
// Some hosts of this library own all of the GPU's memory and hand out no
// allocator (an engine that carves HBM into fixed pools at start-up, a plugin
// running inside such an engine), and some serving loops must not allocate
// once they are running, because an allocation can block on the device or fail
// under memory pressure in the middle of a request. Such callers cannot provide
// the scratch workspace that tq_decode_attention takes. This entry point runs
// the same decode with its scratch in a fixed, file-scope device array instead:
// every GPU that loads the library reserves kScratchBytes for it until the
// process exits, and no call here allocates. The array is reserved when the
// library is first set up on a device (the first codec created there): CUDA
// loads a module's device arrays lazily, so the set-up looks up the array's
// address then, and this entry point only reuses it.
#include <cuda_runtime.h>

#include <mutex>

#include "tq_internal.h"

namespace {

constexpr size_t kScratchBytes = TQ_NOALLOC_SCRATCH_BYTES;  // 16 MiB per device

// Device-side scratch shared by every call of the entry point on a device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device, looked up once
// per device with that device current (the array's name is only a host-side
// stand-in in host code).
tq_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TQ_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return TQ_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return TQ_OK;
}

}  // namespace

namespace tq {
tq_status noalloc_reserve() {
    void* p = nullptr;
    return scratch_address(&p);
}
}  // namespace tq

extern "C" {

tq_status tq_decode_attention_noalloc(const tq_codec* key_codec, const tq_codec* value_codec,
                                      const tq_cache_desc* cache, int layer, const void* q, tq_dtype q_dtype,
                                      int batch, int num_q_heads, int q_len, const int32_t* seq_lens,
                                      const int32_t* block_table, int max_blocks, int max_seq_len, float scale,
                                      float* out, tq_stream_t stream) {
    // The array's address was looked up when the library was set up on this
    // device; a device never set up (no codec created there) has none, and
    // the call then fails as the regular entry point does without a workspace.
    void* scratch = nullptr;
    int dev = -1;
    if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices) {
        std::lock_guard<std::mutex> lk(g_scratch_mu);
        scratch = g_scratch_ptr[dev];
    } else {
        (void)cudaGetLastError();  // no device: the checks below refuse the call
    }
    // The regular entry point checks every argument first, in its own order,
    // and returns TQ_ERR_CAPACITY without launching anything when the decode
    // needs more scratch than the array holds. Every decode kernel writes each
    // scratch value (query rows or fragments, split partials) before any
    // kernel of the same call reads it, so the previous call's contents of the
    // array need no clearing here.
    return tq_decode_attention(key_codec, value_codec, cache, layer, q, q_dtype, batch, num_q_heads, q_len,
                               seq_lens, block_table, max_blocks, max_seq_len, scale, out, scratch,
                               scratch ? kScratchBytes : 0, stream);
}

}  // extern "C"

// Decode-step preparation in one launch: the short encode of the step's new
// tokens (the append of the TurboQuant codec to the cache) and the query prep
// of the tensor-core decode, fused into one grid.
//
// CTAs [0, nq) are the persistent query-prep CTAs; CTAs [nq, nq + 2 Hkv B)
// each encode the n_new <= 8 new keys or values of one (head, sequence) into
// their cache slots, bit-exact with the separate append (the same body). The
// split kernel that follows waits for this whole grid before it fetches any
// record, so it reads the appended tokens.
#include "decode_mma_impl.cuh"
#include "encode_short.cuh"

namespace tq {
namespace mmadec {

// the encoder body needs one thread per coordinate
static_assert(kQThreads >= kD, "the preparation block must cover head_dim threads");

template <int KB, int NV, int ORD>
__global__ void __launch_bounds__(kQThreads) step_prep_kernel(MmaArgs m, EncodeAppendArgs e, int nq) {
    extern __shared__ __align__(16) unsigned char smem[];
    if (static_cast<int>(blockIdx.x) < nq) {
        qfrag_body<KB, ORD>(m, smem, blockIdx.x, nq);
        return;
    }
    const int u = blockIdx.x - nq;
    const int Hkv = e.pool.Hkv;
    const int h = u % Hkv;
    const int bq = (u / Hkv) % e.batch;
    const int is_v = u / (Hkv * e.batch);
    encode_short_body<kD, NV>(e, h, bq, is_v, smem);
}

namespace {

template <int KB, int NV, int ORD>
cudaError_t launch_prep(const MmaArgs& m, const EncodeAppendArgs& e, cudaStream_t s) {
    const size_t enc = encode_short_smem<kD, NV>(true);
    const size_t smem = sizeof(QSmem) > enc ? sizeof(QSmem) : enc;
    static std::atomic<uint64_t> attr_set{0};
    int dev = 0;
    cudaGetDevice(&dev);
    const uint64_t bit = 1ull << (dev & 63);
    if (!(attr_set.load() & bit)) {
        const cudaError_t r = cudaFuncSetAttribute(step_prep_kernel<KB, NV, ORD>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   static_cast<int>(smem));
        if (r != cudaSuccess) {
            (void)cudaGetLastError();
            return r;
        }
        attr_set.fetch_or(bit);
    }
    const DecodeArgs& a = m.a;
    const int units = a.batch * a.pool.Hkv * a.plan.row_groups;
    const int ne = 2 * a.pool.Hkv * a.batch;
    // query-prep CTAs: one per unit, up to the SMs the encode CTAs leave free
    int nq = qfrag_grid(units + ne) - ne;
    if (nq > units) nq = units;
    if (nq < 1) nq = 1;
    const cudaError_t r = launch_overlapped(step_prep_kernel<KB, NV, ORD>, dim3(nq + ne), dim3(kQThreads), smem, s, m, e, nq);
    g_launches.fetch_add(1, std::memory_order_relaxed);
    return r;
}

template <int KB, int ORD>
cudaError_t launch_prep_nv(const MmaArgs& m, const EncodeAppendArgs& e, cudaStream_t s) {
    if (e.n_new <= 2) return launch_prep<KB, 2, ORD>(m, e, s);
    if (e.n_new <= 8) return launch_prep<KB, 8, ORD>(m, e, s);
    return cudaErrorInvalidValue;
}

}  // namespace

// ord: the query fragments' coordinate order (frag_order).
cudaError_t launch_step_prep(int kb, int ord, const MmaArgs& m, const EncodeAppendArgs& e, cudaStream_t s) {
    switch (kb * 4 + ord) {
        case 1 * 4 + 0: return launch_prep_nv<1, 0>(m, e, s);
        case 1 * 4 + 2: return launch_prep_nv<1, 2>(m, e, s);
        case 2 * 4 + 0: return launch_prep_nv<2, 0>(m, e, s);
        case 2 * 4 + 1: return launch_prep_nv<2, 1>(m, e, s);
        case 2 * 4 + 3: return launch_prep_nv<2, 3>(m, e, s);
        case 3 * 4 + 0: return launch_prep_nv<3, 0>(m, e, s);
        case 3 * 4 + 2: return launch_prep_nv<3, 2>(m, e, s);
        case 4 * 4 + 0: return launch_prep_nv<4, 0>(m, e, s);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace mmadec
}  // namespace tq

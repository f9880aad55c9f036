// Instantiations of the tensor-core decode kernel for head_dim 256: 2-bit key
// indices (prod 3-bit keys) with 2-bit group values or 3-bit MSE values.
#include "decode_mma_impl.cuh"

namespace tq {
namespace mmadec {

bool wide_supported(int D, int kb, bool prod, bool vgroup, int vb) {
    return D == 256 && kb == 2 && prod && ((vgroup && vb == 2) || (!vgroup && vb == 3));
}

bool dispatch_d(int D, int kb, bool prod, bool vgroup, int vb, const MmaArgs& m, size_t smem, cudaStream_t s,
                cudaError_t* err) {
    if (D == 256 && kb == 2 && prod && vgroup && vb == 2) {
        *err = launch_mma_wide<2, true, true, 2, 256>(m, smem, s);
        return true;
    }
    if (D == 256 && kb == 2 && prod && !vgroup && vb == 3) {
        *err = launch_mma_wide<2, true, false, 3, 256>(m, smem, s);
        return true;
    }
    return false;
}

}  // namespace mmadec
}  // namespace tq

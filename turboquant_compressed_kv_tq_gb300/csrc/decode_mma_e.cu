// Instantiations of the tensor-core decode kernel for head_dim 64 (run in the
// head_dim-128 layout): prod 3-bit keys (2-bit indices) with 2- or 4-bit group
// values or 3- or 4-bit MSE values, and 4-bit MSE keys with 4-bit MSE values.
#include "decode_mma_impl.cuh"

namespace tq {
namespace mmadec {

bool dispatch_e(int D, int kb, bool prod, bool vgroup, int vb, const MmaArgs& m, size_t smem, cudaStream_t s,
                cudaError_t* err) {
    if (D != 64) return false;
    if (kb == 2 && prod && vgroup && vb == 2) {
        *err = launch_mma_wide<2, true, true, 2, 64>(m, smem, s);
        return true;
    }
    if (kb == 2 && prod && vgroup && vb == 4) {
        *err = launch_mma_wide<2, true, true, 4, 64>(m, smem, s);
        return true;
    }
    if (kb == 2 && prod && !vgroup && vb == 3) {
        *err = launch_mma_wide<2, true, false, 3, 64>(m, smem, s);
        return true;
    }
    if (kb == 2 && prod && !vgroup && vb == 4) {
        *err = launch_mma_wide<2, true, false, 4, 64>(m, smem, s);
        return true;
    }
    if (kb == 4 && !prod && !vgroup && vb == 4) {
        *err = launch_mma_wide<4, false, false, 4, 64>(m, smem, s);
        return true;
    }
    return false;
}

}  // namespace mmadec
}  // namespace tq

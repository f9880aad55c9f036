// Instantiations of the tensor-core decode kernel in its transposed form
// (head_dim 128, at most 8 query rows per unit): prod 3-bit keys (2-bit
// indices) with 2- or 4-bit group values or 3- or 4-bit MSE values, and 4-bit
// MSE keys with 4-bit MSE values.
#include "decode_mma_impl.cuh"

namespace tq {
namespace mmadec {

bool r8_supported(int kb, bool prod, bool vgroup, int vb) {
    if (kb == 2 && prod) return vgroup ? (vb == 2 || vb == 4) : (vb == 3 || vb == 4);
    return kb == 4 && !prod && !vgroup && vb == 4;
}

bool dispatch_f(int kb, bool prod, bool vgroup, int vb, const MmaArgs& m, size_t smem, cudaStream_t s,
                const EncodeAppendArgs* step, cudaError_t* err) {
    if (kb == 2 && prod && vgroup && vb == 2) {
        *err = launch_mma<2, true, true, 2, true>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod && vgroup && vb == 4) {
        *err = launch_mma<2, true, true, 4, true>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod && !vgroup && vb == 3) {
        *err = launch_mma<2, true, false, 3, true>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod && !vgroup && vb == 4) {
        *err = launch_mma<2, true, false, 4, true>(m, smem, s, step);
        return true;
    }
    if (kb == 4 && !prod && !vgroup && vb == 4) {
        *err = launch_mma<4, false, false, 4, true>(m, smem, s, step);
        return true;
    }
    return false;
}

}  // namespace mmadec
}  // namespace tq

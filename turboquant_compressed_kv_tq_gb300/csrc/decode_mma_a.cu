// Instantiations of the tensor-core decode kernel, key index bits 1, 2.
#include "decode_mma_impl.cuh"

namespace tq {
namespace mmadec {

bool dispatch_a(int kb, bool prod, bool vgroup, int vb, const MmaArgs& m, size_t smem, cudaStream_t s,
                const EncodeAppendArgs* step, cudaError_t* err) {
    if (kb == 1 && prod == true && vgroup == false && vb == 2) {
        *err = launch_mma<1, true, false, 2>(m, smem, s, step);
        return true;
    }
    if (kb == 1 && prod == true && vgroup == false && vb == 3) {
        *err = launch_mma<1, true, false, 3>(m, smem, s, step);
        return true;
    }
    if (kb == 1 && prod == true && vgroup == false && vb == 4) {
        *err = launch_mma<1, true, false, 4>(m, smem, s, step);
        return true;
    }
    if (kb == 1 && prod == true && vgroup == true && vb == 2) {
        *err = launch_mma<1, true, true, 2>(m, smem, s, step);
        return true;
    }
    if (kb == 1 && prod == true && vgroup == true && vb == 4) {
        *err = launch_mma<1, true, true, 4>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == true && vgroup == false && vb == 2) {
        *err = launch_mma<2, true, false, 2>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == true && vgroup == false && vb == 3) {
        *err = launch_mma<2, true, false, 3>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == true && vgroup == false && vb == 4) {
        *err = launch_mma<2, true, false, 4>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == true && vgroup == true && vb == 2) {
        *err = launch_mma<2, true, true, 2>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == true && vgroup == true && vb == 4) {
        *err = launch_mma<2, true, true, 4>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == false && vgroup == false && vb == 2) {
        *err = launch_mma<2, false, false, 2>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == false && vgroup == false && vb == 3) {
        *err = launch_mma<2, false, false, 3>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == false && vgroup == false && vb == 4) {
        *err = launch_mma<2, false, false, 4>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == false && vgroup == true && vb == 2) {
        *err = launch_mma<2, false, true, 2>(m, smem, s, step);
        return true;
    }
    if (kb == 2 && prod == false && vgroup == true && vb == 4) {
        *err = launch_mma<2, false, true, 4>(m, smem, s, step);
        return true;
    }
    return false;
}

}  // namespace mmadec
}  // namespace tq

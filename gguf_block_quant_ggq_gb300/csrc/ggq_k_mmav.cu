// ggq_k_mmav.cu -- instantiations of the tensor-path decode GEMV (3-8 tokens).
#include "ggq_mmav.cuh"

namespace ggq {

cudaError_t launch_mmav(int fmt, const MmavParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_mmav_one<F_Q8_0, false>(p, grid, smem, s);
    case F_Q4_K: return launch_mmav_one<F_Q4_K, false>(p, grid, smem, s);
    case F_Q5_K: return launch_mmav_one<F_Q5_K, false>(p, grid, smem, s);
    case F_Q6_K: return launch_mmav_one<F_Q6_K, false>(p, grid, smem, s);
    case F_MXFP4: return launch_mmav_one<F_MXFP4, false>(p, grid, smem, s);
    case F_Q2_K: return launch_mmav_one<F_Q2_K, false>(p, grid, smem, s);
    case F_Q3_K: return launch_mmav_one<F_Q3_K, false>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ggq

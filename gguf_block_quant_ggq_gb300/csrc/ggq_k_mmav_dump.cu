// ggq_k_mmav_dump.cu -- the tensor-path decode GEMV in its integer-core dump form.
#include "ggq_mmav.cuh"

namespace ggq {

cudaError_t launch_mmav_dump(int fmt, const MmavParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_mmav_one<F_Q8_0, true>(p, grid, smem, s);
    case F_Q4_K: return launch_mmav_one<F_Q4_K, true>(p, grid, smem, s);
    case F_Q5_K: return launch_mmav_one<F_Q5_K, true>(p, grid, smem, s);
    case F_Q6_K: return launch_mmav_one<F_Q6_K, true>(p, grid, smem, s);
    case F_MXFP4: return launch_mmav_one<F_MXFP4, true>(p, grid, smem, s);
    case F_Q2_K: return launch_mmav_one<F_Q2_K, true>(p, grid, smem, s);
    case F_Q3_K: return launch_mmav_one<F_Q3_K, true>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ggq

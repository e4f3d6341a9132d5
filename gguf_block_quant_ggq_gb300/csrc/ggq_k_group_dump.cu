// ggq_k_group_dump.cu -- the grouped int8 tensor-core kernel in its integer-core dump form.
#include "ggq_group.cuh"

namespace ggq {

template <int KIND>
static cudaError_t launch_group_fmt(int fmt, const GroupParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_group_one<KIND, F_Q8_0, true>(p, grid, smem, s);
    case F_Q4_K: return launch_group_one<KIND, F_Q4_K, true>(p, grid, smem, s);
    case F_Q5_K: return launch_group_one<KIND, F_Q5_K, true>(p, grid, smem, s);
    case F_Q6_K: return launch_group_one<KIND, F_Q6_K, true>(p, grid, smem, s);
    case F_MXFP4: return launch_group_one<KIND, F_MXFP4, true>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_group_dump(int kind, int fmt, const GroupParams& p, int grid, int smem, cudaStream_t s) {
    switch (kind) {
    case G_GEMV: return launch_group_fmt<G_GEMV>(fmt, p, grid, smem, s);
    case G_GATEUP: return launch_group_fmt<G_GATEUP>(fmt, p, grid, smem, s);
    default: return launch_group_fmt<G_DOWN>(fmt, p, grid, smem, s);
    }
}

}  // namespace ggq

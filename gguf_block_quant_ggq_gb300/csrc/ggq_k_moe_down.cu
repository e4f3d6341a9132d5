// ggq_k_moe_down.cu -- instantiations of the streaming kernel: decode MoE down stage.
#include "ggq_stream.cuh"

namespace ggq {

cudaError_t launch_moe_down(int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_nt<KIND_DOWN, F_Q8_0>(nt, p, grid, smem, s);
    case F_Q4_K: return launch_nt<KIND_DOWN, F_Q4_K>(nt, p, grid, smem, s);
    case F_Q5_K: return launch_nt<KIND_DOWN, F_Q5_K>(nt, p, grid, smem, s);
    case F_Q6_K: return launch_nt<KIND_DOWN, F_Q6_K>(nt, p, grid, smem, s);
    case F_MXFP4: return launch_nt<KIND_DOWN, F_MXFP4>(nt, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ggq

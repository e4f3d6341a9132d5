// ggq_k_gemv_a.cu -- instantiations of the streaming kernel: GEMV and block-dot dump.
#include "ggq_stream.cuh"

namespace ggq {

cudaError_t launch_gemv_a(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q4_0:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_Q4_0, 8>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_Q4_0>(nt, p, grid, smem, s);
    case F_Q8_0:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_Q8_0, 8>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_Q8_0>(nt, p, grid, smem, s);
    case F_MXFP4:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_MXFP4, 8>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_MXFP4>(nt, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ggq

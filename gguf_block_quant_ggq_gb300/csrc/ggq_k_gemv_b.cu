// ggq_k_gemv_b.cu -- instantiations of the streaming kernel: GEMV and block-dot dump.
#include "ggq_stream.cuh"

namespace ggq {

cudaError_t launch_gemv_b(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q4_K:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_Q4_K, 8>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_Q4_K>(nt, p, grid, smem, s);
    case F_Q5_K:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_Q5_K, 8>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_Q5_K>(nt, p, grid, smem, s);
    case F_Q6_K:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_Q6_K, 8>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_Q6_K>(nt, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ggq

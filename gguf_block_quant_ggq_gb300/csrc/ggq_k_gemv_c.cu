// ggq_k_gemv_c.cu -- instantiations of the streaming kernel for the 2- and 3-bit
// K-quants (Q2_K, Q3_K): GEMV and block-dot dump.
#include "ggq_stream.cuh"

namespace ggq {

cudaError_t launch_gemv_c(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q2_K:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_Q2_K, 8>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_Q2_K>(nt, p, grid, smem, s);
    case F_Q3_K:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_Q3_K, 8>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_Q3_K>(nt, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ggq

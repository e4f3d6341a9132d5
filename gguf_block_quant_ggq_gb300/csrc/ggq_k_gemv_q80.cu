// ggq_k_gemv_q80.cu -- the streaming kernel (GEMV and block-dot dump) with Q8_0
// activation blocks: Q4_0 x Q8_0 and Q8_0 x Q8_0.
#include "ggq_stream.cuh"

namespace ggq {

cudaError_t launch_gemv_q80(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q4_0:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_Q4_0, 8, 1>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_Q4_0, 1>(nt, p, grid, smem, s);
    case F_Q8_0:
        return kind == KIND_DUMP ? launch_one<KIND_DUMP, F_Q8_0, 8, 1>(p, grid, smem, s)
                                 : launch_nt<KIND_GEMV, F_Q8_0, 1>(nt, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ggq

// ggq_k_moe_downf.cu -- instantiations of the direct tiny-batch MoE route: fused down kernel.
#include "ggq_direct.cuh"

namespace ggq {

template <int F>
static cudaError_t launch_downf_nt(int nt, const DirectParams& p, int grid, int smem, cudaStream_t s) {
    switch (nt) {  // the direct route serves at most 4 tokens
    case 1: return launch_direct_one<KIND_DOWNF, F, 1>(p, grid, smem, s);
    case 2: return launch_direct_one<KIND_DOWNF, F, 2>(p, grid, smem, s);
    case 4: return launch_direct_one<KIND_DOWNF, F, 4>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_direct_downf(int fmt, int nt, const DirectParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_downf_nt<F_Q8_0>(nt, p, grid, smem, s);
    case F_Q4_K: return launch_downf_nt<F_Q4_K>(nt, p, grid, smem, s);
    case F_Q5_K: return launch_downf_nt<F_Q5_K>(nt, p, grid, smem, s);
    case F_Q6_K: return launch_downf_nt<F_Q6_K>(nt, p, grid, smem, s);
    case F_MXFP4: return launch_downf_nt<F_MXFP4>(nt, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ggq

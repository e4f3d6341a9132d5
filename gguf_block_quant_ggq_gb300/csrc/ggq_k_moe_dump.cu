// ggq_k_moe_dump.cu -- the direct tiny-batch MoE kernels (gate/up and per-pair
// down) in their integer-core dump form.
#include "ggq_direct.cuh"

namespace ggq {

template <int KIND, int F>
static cudaError_t launch_dump_nt(int nt, const DirectParams& p, int grid, int smem, cudaStream_t s) {
    switch (nt) {  // the direct route serves at most 4 tokens
    case 1: return launch_direct_one<KIND, F, 1, true>(p, grid, smem, s);
    case 2: return launch_direct_one<KIND, F, 2, true>(p, grid, smem, s);
    case 4: return launch_direct_one<KIND, F, 4, true>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

template <int KIND>
static cudaError_t launch_dump_fmt(int fmt, int nt, const DirectParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_dump_nt<KIND, F_Q8_0>(nt, p, grid, smem, s);
    case F_Q4_K: return launch_dump_nt<KIND, F_Q4_K>(nt, p, grid, smem, s);
    case F_Q5_K: return launch_dump_nt<KIND, F_Q5_K>(nt, p, grid, smem, s);
    case F_Q6_K: return launch_dump_nt<KIND, F_Q6_K>(nt, p, grid, smem, s);
    case F_MXFP4: return launch_dump_nt<KIND, F_MXFP4>(nt, p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_direct_gateup_dump(int fmt, int nt, const DirectParams& p, int grid, int smem, cudaStream_t s) {
    return launch_dump_fmt<KIND_GATEUP>(fmt, nt, p, grid, smem, s);
}

cudaError_t launch_direct_down_dump(int fmt, int nt, const DirectParams& p, int grid, int smem, cudaStream_t s) {
    return launch_dump_fmt<KIND_DOWN>(fmt, nt, p, grid, smem, s);
}

}  // namespace ggq

// ggq_k_gmm.cu -- instantiations of the grouped f16 tensor-core GEMM.
#include "ggq_gmm.cuh"

namespace ggq {

int gmm_supported(int fmt) { return fmt == F_Q8_0 || fmt == F_Q4_K; }
int gmm_smem_bytes() { return GmmSmem::kTotal; }

template <int KIND>
static cudaError_t launch_gmm_fmt(int fmt, const GmmParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_gmm_one<KIND, F_Q8_0>(p, grid, smem, s);
    case F_Q4_K: return launch_gmm_one<KIND, F_Q4_K>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gmm(int kind, int fmt, const GmmParams& p, int grid, int smem, cudaStream_t s) {
    if (smem != GmmSmem::kTotal) return cudaErrorInvalidValue;
    return kind == G_GATEUP ? launch_gmm_fmt<G_GATEUP>(fmt, p, grid, smem, s)
                            : launch_gmm_fmt<G_DOWN>(fmt, p, grid, smem, s);
}

}  // namespace ggq

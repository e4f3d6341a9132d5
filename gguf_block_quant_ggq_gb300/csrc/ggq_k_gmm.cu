// ggq_k_gmm.cu -- instantiations of the grouped f16 tensor-core GEMM.
#include <cudaTypedefs.h>

#include "ggq_gmm.cuh"

namespace ggq {

namespace {

// The driver's tensor-map encoder, looked up once (a function-local static is
// initialised exactly once even when several host threads get here together).
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        return nullptr;
    }();
    return fn;
}

}  // namespace

// Row-major 2-D tensor [dim1][dim0] of one element type, rows stride1 bytes apart.
int encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t dim0, uint64_t dim1, uint64_t stride1,
              uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz) {
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn) return CUDA_ERROR_NOT_FOUND;
    const cuuint64_t dims[2] = {dim0, dim1};
    const cuuint64_t strides[1] = {stride1};
    const cuuint32_t box[2] = {box0, box1};
    const cuuint32_t es[2] = {1, 1};
    return static_cast<int>(fn(m, type, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                               swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE));
}

int gmm_encode(GmmParams& p, int kind, int fmt, const uint8_t* W, const uint8_t* W2, int64_t rowbytes, int64_t wrows,
               const __half* x16, const float* dx, int64_t dx_pitch, const __half* bs16, int64_t P, int K) {
    const uint64_t k = static_cast<uint64_t>(K), np = static_cast<uint64_t>(P);
    int r = encode_tmap_2d(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, k, np, k * 2, kGmmBK, kGmmBN,
                      CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r) r = encode_tmap_2d(&p.tm_dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dx, static_cast<uint64_t>(dx_pitch), np,
                          static_cast<uint64_t>(dx_pitch) * 4, 4, kGmmBN, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!r) r = encode_tmap_2d(&p.tm_bs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bs16, k / 16, np, k / 8, 16, kGmmBN,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    const uint32_t rows = kind == G_GATEUP ? kGmmBM / 2 : kGmmBM;
    const int nm = kind == G_GATEUP ? 2 : 1;
    for (int m = 0; m < nm && !r; ++m) {
        const uint8_t* w = m ? W2 : W;
        const uint64_t rb = static_cast<uint64_t>(rowbytes), nr = static_cast<uint64_t>(wrows);
        if (fmt == F_Q8_0) {
            r = encode_tmap_2d(&p.tm_w[m][0], CU_TENSOR_MAP_DATA_TYPE_UINT8, w, rb, nr, rb, kGmmRaw, rows, CU_TENSOR_MAP_SWIZZLE_NONE);
        } else {
            r = encode_tmap_2d(&p.tm_w[m][0], CU_TENSOR_MAP_DATA_TYPE_UINT8, w, rb, nr, rb, 16, rows, CU_TENSOR_MAP_SWIZZLE_NONE);
            if (!r) r = encode_tmap_2d(&p.tm_w[m][1], CU_TENSOR_MAP_DATA_TYPE_UINT8, w, rb, nr, rb, 32, rows, CU_TENSOR_MAP_SWIZZLE_NONE);
        }
    }
    return r;
}

int gmm_supported(int fmt) { return fmt == F_Q8_0 || fmt == F_Q4_K; }
int gmm_smem_bytes() { return GmmSmem::kTotal; }

template <int KIND, bool DUMP>
static cudaError_t launch_gmm_fmt(int fmt, const GmmParams& p, int grid, int smem, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_gmm_one<KIND, F_Q8_0, DUMP>(p, grid, smem, s);
    case F_Q4_K: return launch_gmm_one<KIND, F_Q4_K, DUMP>(p, grid, smem, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gmm(int kind, int fmt, const GmmParams& p, int grid, int smem, cudaStream_t s) {
    if (smem != GmmSmem::kTotal) return cudaErrorInvalidValue;
    return kind == G_GATEUP ? launch_gmm_fmt<G_GATEUP, false>(fmt, p, grid, smem, s)
                            : launch_gmm_fmt<G_DOWN, false>(fmt, p, grid, smem, s);
}

cudaError_t launch_gmm_dump(int kind, int fmt, const GmmParams& p, int grid, int smem, cudaStream_t s) {
    if (smem != GmmSmem::kTotal) return cudaErrorInvalidValue;
    return kind == G_GATEUP ? launch_gmm_fmt<G_GATEUP, true>(fmt, p, grid, smem, s)
                            : launch_gmm_fmt<G_DOWN, true>(fmt, p, grid, smem, s);
}

}  // namespace ggq

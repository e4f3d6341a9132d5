// ggq_k_gmmtc.cu -- tensor maps and launch of the tcgen05 grouped GEMM (Q8_0, Q4_K and MXFP4 banks).
#include "ggq_gmmtc.cuh"

#include <atomic>

namespace ggq {

int gmmtc_encode(GmmTcParams& p, int fmt, const uint8_t* W, const uint8_t* W2, int64_t rowbytes, int64_t wrows,
                 const __half* x16, const float* dx, int64_t dx_pitch, const __half* bs16, int64_t P, int K) {
    const uint64_t k = static_cast<uint64_t>(K), np = static_cast<uint64_t>(P);
    int r = encode_tmap_2d(&p.tm_b, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, k, np, k * 2, kTcBK, kTcBN,
                           CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r) r = encode_tmap_2d(&p.tm_b32, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, x16, k, np, k * 2, kTcBK, kTcNarrow,
                               CU_TENSOR_MAP_SWIZZLE_128B);
    if (!r) r = encode_tmap_2d(&p.tm_dx, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, dx, static_cast<uint64_t>(dx_pitch), np,
                               static_cast<uint64_t>(dx_pitch) * 4, 4, kTcBN, CU_TENSOR_MAP_SWIZZLE_NONE);
    if (!r) r = encode_tmap_2d(&p.tm_bs, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, bs16 ? bs16 : x16, k / 16, np, k / 8, 16, kTcBN,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    const uint64_t rb = static_cast<uint64_t>(rowbytes), nr = static_cast<uint64_t>(wrows);
    if (fmt == F_Q8_0 || fmt == F_MXFP4) {
        const int box = fmt == F_Q8_0 ? kTcRaw : kTcRawMx;
        for (int m = 0; m < 2 && !r; ++m)
            r = encode_tmap_2d(&p.tm_w[m], CU_TENSOR_MAP_DATA_TYPE_UINT8, m ? (W2 ? W2 : W) : W, rb, nr, rb, box, kTcBM,
                               CU_TENSOR_MAP_SWIZZLE_NONE);
    } else {
        if (!r) r = encode_tmap_2d(&p.tm_w[0], CU_TENSOR_MAP_DATA_TYPE_UINT8, W, rb, nr, rb, 16, kTcBM, CU_TENSOR_MAP_SWIZZLE_NONE);
        if (!r) r = encode_tmap_2d(&p.tm_w[1], CU_TENSOR_MAP_DATA_TYPE_UINT8, W, rb, nr, rb, 32, kTcBM, CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    return r;
}

template <int F, bool DUMP>
static cudaError_t launch_gmmtc_one(const GmmTcParams& p, int grid, cudaStream_t s) {
    static std::atomic<bool> attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(k_gmmtc<F, DUMP>, cudaFuncAttributeMaxDynamicSharedMemorySize, TcSmem<F>::kTotal);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    return launch_pdl(k_gmmtc<F, DUMP>, dim3(grid), dim3(kTcThreads), TcSmem<F>::kTotal, s, p);
}

cudaError_t launch_gmmtc(int fmt, const GmmTcParams& p, int grid, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_gmmtc_one<F_Q8_0, false>(p, grid, s);
    case F_Q4_K: return launch_gmmtc_one<F_Q4_K, false>(p, grid, s);
    case F_MXFP4: return launch_gmmtc_one<F_MXFP4, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_gmmtc_dump(int fmt, const GmmTcParams& p, int grid, cudaStream_t s) {
    switch (fmt) {
    case F_Q8_0: return launch_gmmtc_one<F_Q8_0, true>(p, grid, s);
    case F_Q4_K: return launch_gmmtc_one<F_Q4_K, true>(p, grid, s);
    case F_MXFP4: return launch_gmmtc_one<F_MXFP4, true>(p, grid, s);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace ggq

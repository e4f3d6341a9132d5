// ggq_noalloc.cu -- ggq_mul_mat_vec_noalloc: the decode GEMV for callers that
// must not allocate device memory.
//
// ggq_mul_mat_vec needs a context (whose creation allocates a control block)
// and quantizes X into the context's pool (grown by ggq_reserve).  This entry
// point instead keeps the quantized activations in a fixed array in the
// library's own device data segment, so it needs neither a context nor any
// allocation.  It runs the quantizer and the dp4a streaming GEMV (with the
// pooled call's shared-memory plans: whole rows, row chunks, token groups) at
// every token count; the pooled call takes the tensor-path kernel at 2-8
// tokens where that applies, so the two agree within the fp32 tolerance.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/ggq.h"
#include "ggq_device.cuh"
#include "ggq_internal.h"
#include "ggq_plan.h"

namespace ggq {
cudaError_t launch_stream(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s);
}

using namespace ggq;

namespace {

// Quantized activations of up to 8 tokens x 16384 inputs in either activation
// layout (Q8_K: 8 * 64 * 292 = 149504 bytes; Q8_1: 8 * 512 * 36 = 147456 bytes).
constexpr size_t kNoAllocScratchBytes = 152 * 1024;

// One copy per device that loads the library, kept until the process exits.
// Host code must not use this name as an address: it resolves the device
// address with cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
    bool ready;
    uint8_t* scratch;  // device address of g_noalloc_scratch on this device
    int nsm;
};

NoAllocDevice g_devices[kMaxDevices];
std::mutex g_devices_mu;

int fmt_of_type(int t) {
    switch (t) {
    case GGQ_TYPE_Q4_0: return F_Q4_0;
    case GGQ_TYPE_Q8_0: return F_Q8_0;
    case GGQ_TYPE_Q4_K: return F_Q4_K;
    case GGQ_TYPE_Q5_K: return F_Q5_K;
    case GGQ_TYPE_Q6_K: return F_Q6_K;
    case GGQ_TYPE_MXFP4: return F_MXFP4;
    case GGQ_TYPE_Q2_K: return F_Q2_K;
    case GGQ_TYPE_Q3_K: return F_Q3_K;
    default: return -1;
    }
}

// First call on the current device: check the architecture and resolve the
// array's device address (with this device current).
ggq_status device_setup(NoAllocDevice** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GGQ_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return GGQ_ERR_INVALID_ARG;
    std::lock_guard<std::mutex> lock(g_devices_mu);
    NoAllocDevice& d = g_devices[dev];
    if (!d.ready) {
        int major = 0, minor = 0, nsm = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return GGQ_ERR_CUDA;
        if (major != 10 || minor != 3) return GGQ_ERR_ARCH;
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return GGQ_ERR_CUDA;
        d.scratch = static_cast<uint8_t*>(ptr);
        d.nsm = nsm;
        d.ready = true;
    }
    *out = &d;
    return GGQ_OK;
}

// The streaming GEMV over tokens [0, T) of xq (rows xrow bytes apart), with
// the plan of the pooled call: whole-row stages, row chunks, or the tokens in
// two groups.
ggq_status launch_groups(int f, StreamParams p, const uint8_t* xq, int64_t T, float* Y, int64_t xrow, int nsm,
                         cudaStream_t s) {
    StreamShape sh;
    const bool q81 = f == F_Q4_0;
    const StreamPlan plan = plan_gemv_stream(f, p.rowbytes, static_cast<int>(T), p.K, q81, &sh, &p.chunk_units,
                                             &p.chunk_bytes, &p.row_slot);
    if (plan == StreamPlan::kNone) return GGQ_ERR_SHAPE;
    if (plan == StreamPlan::kSplit) {
        const int64_t T0 = T / 2;
        const ggq_status s0 = launch_groups(f, p, xq, T0, Y, xrow, nsm, s);
        if (s0 != GGQ_OK) return s0;
        return launch_groups(f, p, xq + T0 * xrow, T - T0, Y + T0 * p.N, xrow, nsm, s);
    }
    p.xq = xq;
    p.xrows = static_cast<int>(T);
    p.T = static_cast<int>(T);
    p.Y = Y;
    p.stages = sh.stages;
    p.stage_stride = sh.stride;
    p.x_bytes = sh.x_bytes;
    const int64_t tiles = (p.N + kTileRows - 1) / kTileRows;
    const int grid = static_cast<int>(tiles < nsm ? tiles : nsm);
    const int nt = T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8;
    return launch_stream(KIND_GEMV, f, nt, p, grid, sh.smem, s) == cudaSuccess ? GGQ_OK : GGQ_ERR_CUDA;
}

}  // namespace

extern "C" ggq_status ggq_mul_mat_vec_noalloc(int w, const void* W, int64_t N, int64_t K, const float* X, int64_t T,
                                              float* Y, void* stream) {
    const int f = fmt_of_type(w);
    if (f < 0) return GGQ_ERR_UNSUPPORTED;
    if (!W || !X || !Y) return GGQ_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Y)) & 15)
        return GGQ_ERR_INVALID_ARG;
    const bool q81 = f == F_Q4_0;
    const int64_t ablk = q81 ? 32 : 256;
    if (T < 1 || T > 8 || N < 1 || K < 1 || K % fmt_qk(f) || K % ablk) return GGQ_ERR_SHAPE;
    const int64_t xbytes = T * (q81 ? K / 32 * 36 : K / 256 * 292);
    if (xbytes > static_cast<int64_t>(kNoAllocScratchBytes)) return GGQ_ERR_CAPACITY;

    {  // refused before any launch: token groups shrink down to one token, so one token must fit
        StreamShape sh;
        int cu = 0, cb = 0, rs = 0;
        if (plan_gemv_stream(f, K / fmt_qk(f) * fmt_bytes(f), 1, static_cast<int>(K), q81, &sh, &cu, &cb, &rs) ==
            StreamPlan::kNone)
            return GGQ_ERR_SHAPE;
    }
    NoAllocDevice* d = nullptr;
    ggq_status st = device_setup(&d);
    if (st != GGQ_OK) return st;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (launch_quantize(q81 ? 0 : 1, X, T, K, d->scratch, s) != cudaSuccess) return GGQ_ERR_CUDA;
    StreamParams p{};
    p.W = static_cast<const uint8_t*>(W);
    p.rowbytes = K / fmt_qk(f) * fmt_bytes(f);
    p.N = N;
    p.K = static_cast<int>(K);
    p.err = nullptr;  // bounded-wait timeouts are not reported by this entry point
    return launch_groups(f, p, d->scratch, T, Y, q81 ? K / 32 * 36 : K / 256 * 292, d->nsm, s);
}

// ggq_api.cu -- the C ABI of libggq (include/ggq.h): context, grow-only
// scratch pool, argument checks, launch planning.
//
// Pool discipline follows the review of vllm.cpp PR #523 "grouped +
// non-grouped keep-quant expert GEMM": no per-call cudaMalloc/cudaFree or
// stream synchronisation (both illegal under graph capture), a grow-only pool
// whose old generations are retired rather than freed, per-format availability
// instead of a boolean, and refusals that name the unsupported formats.
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <cstring>
#include <string>
#include <vector>

#include "../../include/ggq.h"
#include "ggq_device.cuh"
#include "ggq_direct.cuh"
#include "ggq_internal.h"
#include "ggq_plan.h"

namespace ggq {
cudaError_t launch_gemv_a(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_gemv_b(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_gemv_c(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_gemv_q80(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_direct_gateup(int fmt, int nt, const DirectParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_direct_down(int fmt, int nt, const DirectParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_direct_downf(int fmt, int nt, const DirectParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_direct_gateup_dump(int fmt, int nt, const DirectParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_direct_down_dump(int fmt, int nt, const DirectParams& p, int grid, int smem, cudaStream_t s);

cudaError_t launch_stream(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s) {
    if (fmt == F_Q4_0 || fmt == F_Q8_0 || fmt == F_MXFP4) return launch_gemv_a(kind, fmt, nt, p, grid, smem, s);
    if (fmt == F_Q2_K || fmt == F_Q3_K) return launch_gemv_c(kind, fmt, nt, p, grid, smem, s);
    return launch_gemv_b(kind, fmt, nt, p, grid, smem, s);
}
}  // namespace ggq

using namespace ggq;

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t v, size_t a = kAlign) { return (v + a - 1) / a * a; }

// Layout of the control block (allocated once at create).
struct Ctrl {
    int err;
    int pad[63];
};

int fmt_of(int t) {
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

// The 2- and 3-bit K-quants run on the dp4a streaming GEMV only (no tensor-path,
// grouped or MoE kernels for them).
bool low_bit_kquant(int f) { return f == F_Q2_K || f == F_Q3_K; }

const char* type_name(int t) {
    switch (t) {
    case GGQ_TYPE_Q4_0: return "Q4_0";
    case GGQ_TYPE_Q8_0: return "Q8_0";
    case GGQ_TYPE_Q8_1: return "Q8_1";
    case GGQ_TYPE_Q4_K: return "Q4_K";
    case GGQ_TYPE_Q5_K: return "Q5_K";
    case GGQ_TYPE_Q6_K: return "Q6_K";
    case GGQ_TYPE_Q8_K: return "Q8_K";
    case GGQ_TYPE_MXFP4: return "MXFP4";
    case GGQ_TYPE_Q2_K: return "Q2_K";
    case GGQ_TYPE_Q3_K: return "Q3_K";
    default: return "unknown";
    }
}

int64_t w_row_bytes(int f, int64_t K) { return K / fmt_qk(f) * fmt_bytes(f); }

size_t gemv_scratch(int64_t T, int64_t K) {
    // quantized X in the wider of the two activation layouts
    const int64_t q81 = K / 32 * 36, q8k = (K + 255) / 256 * 292;
    return align_up(static_cast<size_t>(T) * static_cast<size_t>(q81 > q8k ? q81 : q8k));
}

struct MoeScratch {
    size_t ids, w, h, hq, total;
};

// Direct route (1-4 tokens): routed ids/weights, fp32 h, packed h^ (dumps).
MoeScratch moe_scratch(int64_t T, int64_t H, int64_t I, int64_t k) {
    (void)H;
    MoeScratch m{};
    const size_t P = static_cast<size_t>(T * k);
    size_t off = 0;
    m.ids = off; off += align_up(P * 4);
    m.w = off; off += align_up(P * 4);
    m.h = off; off += align_up(P * static_cast<size_t>(I) * 4);
    m.hq = off; off += align_up(P * (I / 256) * 292);
    m.total = off;
    return m;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Expert-sorted route (5 tokens and up): pitched activation rows for the
// grouped kernel's 16-byte row copies.
struct SortedScratch {
    size_t xq, ids, w, counts, offsets, cursor, ngroups, gexp, goff, gcnt, perm, h, hq, o;
    size_t x16, xbs, xdx, h16, hbs, hdx;  // f16 operands of the grouped f16 GEMM
    size_t u;                              // up outputs of the tcgen05 gate/up GEMM (g goes to h)
    size_t total;
};

// floats per row of the f32 block scales beside the f16 operands
int64_t dx_pitch(int64_t K) { return (K / 256 + 3) / 4 * 4; }

SortedScratch sorted_scratch(int64_t T, int64_t E, int64_t H, int64_t I, int64_t k) {
    SortedScratch m{};
    const size_t P = static_cast<size_t>(T * k);
    const size_t xp = static_cast<size_t>((H / 256 * 292 + 15) / 16 * 16);
    const size_t hp = static_cast<size_t>((I / 256 * 292 + 15) / 16 * 16);
    size_t off = 0;
    auto take = [&](size_t& field, size_t bytes) {
        field = off;
        off += align_up(bytes);
    };
    take(m.xq, static_cast<size_t>(T) * xp);
    take(m.ids, P * 4);
    take(m.w, P * 4);
    take(m.counts, static_cast<size_t>(E) * 4);
    take(m.offsets, static_cast<size_t>(E + 1) * 4);
    take(m.cursor, static_cast<size_t>(E) * 4);
    take(m.ngroups, 4);
    take(m.gexp, static_cast<size_t>(E) * 4);
    take(m.goff, static_cast<size_t>(E) * 4);
    take(m.gcnt, static_cast<size_t>(E) * 4);
    take(m.perm, P * 4);
    take(m.h, P * static_cast<size_t>(I) * 4);
    take(m.hq, P * hp);
    take(m.o, P * static_cast<size_t>(H) * 4);
    take(m.x16, P * static_cast<size_t>(H) * 2);  // one row per (token, expert) pair, expert-sorted
    take(m.xbs, P * static_cast<size_t>(H / 16) * 2);
    take(m.xdx, P * static_cast<size_t>(dx_pitch(H)) * 4);
    take(m.h16, P * static_cast<size_t>(I) * 2);
    take(m.hbs, P * static_cast<size_t>(I / 16) * 2);
    take(m.hdx, P * static_cast<size_t>(dx_pitch(I)) * 4);
    take(m.u, P * static_cast<size_t>(I) * 4);
    m.total = off;
    return m;
}

}  // namespace

struct ggq_ctx {
    int device = 0;
    int nsm = 0;
    uint8_t* pool = nullptr;
    size_t pool_bytes = 0;
    std::vector<void*> retired;
    Ctrl* ctrl = nullptr;
    int static_weights = 0;  // weights never written while calls are in flight
    int direct_max = 32;     // largest token count of the direct MoE route (calls of <= 4 tokens above 4)
    unsigned long long* tel_pairs = nullptr;  // expert-load telemetry (caller's device buffers)
    unsigned long long* tel_calls = nullptr;
    int64_t tel_experts = 0;
    std::string err;
};

namespace {

ggq_status fail(ggq_ctx* c, ggq_status s, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    if (c) c->err = buf;
    return s;
}

ggq_status cuda_fail(ggq_ctx* c, cudaError_t e, const char* what) {
    return fail(c, GGQ_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

ggq_status need_scratch(ggq_ctx* c, size_t bytes) {
    if (bytes <= c->pool_bytes) return GGQ_OK;
    return fail(c, GGQ_ERR_CAPACITY, "call needs %zu scratch bytes but the pool holds %zu: call ggq_reserve first",
                bytes, c->pool_bytes);
}

int pow2_tokens(int64_t T) { return T <= 1 ? 1 : T <= 2 ? 2 : T <= 4 ? 4 : 8; }

// Smallest token count that the decode GEMV sends to the grouped int8
// tensor-core kernel (below it the dp4a streaming kernel is cheaper).
constexpr int kGroupMinTokens = 3;

// Pad a 16-byte-multiple row so that its stride in 32-bit words is 4 mod 32:
// eight rows then land on distinct bank quads for the mma fragment loads.
int bank_stride(int64_t bytes) {
    const int64_t words = bytes / 4;
    const int64_t pad = ((4 - words % 32) % 32 + 32) % 32;
    return static_cast<int>(bytes + 4 * pad);
}

int64_t q8k_pitch(int64_t K) { return (K / 256 * 292 + 15) / 16 * 16; }

// Shared-memory plan of a grouped launch; false if one weight slot and one
// activation slot do not fit.
bool plan_group(GroupParams& p, int nmat, bool resident_x, int* smem) {
    p.wcontig = (p.rowbytes % 16) != 0;
    p.wrow = p.wcontig ? static_cast<int>(p.rowbytes) : bank_stride(p.rowbytes);
    p.wslot = static_cast<int>(align_up(static_cast<size_t>(nmat * kGroupRows * p.wrow + 16), 128));
    p.xcopy = static_cast<int>((p.K / 256 * 292 + 15) / 16 * 16);
    p.xstride = bank_stride(p.xcopy);
    p.xslot = static_cast<int>(align_up(static_cast<size_t>(kGroupCols * p.xstride + 16), 128));
    const int fixed = kGroupConsumerWarps * nmat * 128 * 4 + 32 * 8 + 64;
    if (p.wslot + p.xslot + fixed > kSmemLimit) return false;
    int ws = 4, xs = resident_x ? 1 : 8;
    while (ws > 1 && ws * p.wslot + 2 * p.xslot + fixed > kSmemLimit) --ws;
    if (!resident_x)
        while (xs > 1 && ws * p.wslot + xs * p.xslot + fixed > kSmemLimit) --xs;
    p.wstages = ws;
    p.xstages = xs;
    *smem = ws * p.wslot + xs * p.xslot + fixed;
    return true;
}

// Makes the context's device current for one call and puts the caller's
// device back when the call returns.
struct DeviceScope {
    int prev = -1;
    ~DeviceScope() {
        if (prev >= 0) cudaSetDevice(prev);
    }
};

ggq_status check_ctx(ggq_ctx* c, DeviceScope& scope) {
    if (!c) return GGQ_ERR_INVALID_ARG;
    int cur = -1;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return cuda_fail(c, e, "cudaGetDevice");
    if (cur != c->device) {
        e = cudaSetDevice(c->device);
        if (e != cudaSuccess) return cuda_fail(c, e, "cudaSetDevice");
        scope.prev = cur;
    }
    return GGQ_OK;
}

ggq_status gemv_checks(ggq_ctx* c, int w, const void* W, int64_t N, int64_t K, const void* X, int64_t T,
                       const void* Y, int act = -1) {
    const int f = fmt_of(w);
    if (act >= 0 && act != (f == F_Q4_0 ? GGQ_TYPE_Q8_1 : GGQ_TYPE_Q8_K) &&
        !(act == GGQ_TYPE_Q8_0 && (f == F_Q4_0 || f == F_Q8_0)))
        return fail(c, GGQ_ERR_UNSUPPORTED,
                    "mul_mat_vec: weight type %d (%s) with activation type %d (%s) is not supported; supported: "
                    "Q4_0 x Q8_1, Q4_0 x Q8_0, Q8_0 x Q8_0, and Q8_0, Q2_K, Q3_K, Q4_K, Q5_K, Q6_K, MXFP4 x Q8_K",
                    w, type_name(w), act, type_name(act));
    const bool a80 = act == GGQ_TYPE_Q8_0;
    if (f < 0 || w == GGQ_TYPE_Q8_1 || w == GGQ_TYPE_Q8_K)
        return fail(c, GGQ_ERR_UNSUPPORTED,
                    "mul_mat_vec: weight type %d (%s) is not supported; supported: Q4_0 x Q8_1, and Q8_0, Q2_K, "
                    "Q3_K, Q4_K, Q5_K, Q6_K, MXFP4 x Q8_K",
                    w, type_name(w));
    if (!W || !X || !Y) return fail(c, GGQ_ERR_INVALID_ARG, "mul_mat_vec: null pointer");
    if (!aligned16(W) || !aligned16(X) || !aligned16(Y))
        return fail(c, GGQ_ERR_INVALID_ARG, "mul_mat_vec: pointers must be 16-byte aligned");
    if (T < 1 || T > 8) return fail(c, GGQ_ERR_SHAPE, "mul_mat_vec: T=%lld out of 1..8", static_cast<long long>(T));
    if (N < 1) return fail(c, GGQ_ERR_SHAPE, "mul_mat_vec: N=%lld", static_cast<long long>(N));
    const int64_t ablk = f == F_Q4_0 || a80 ? 32 : 256;
    if (K < 1 || K % fmt_qk(f) || K % ablk)
        return fail(c, GGQ_ERR_SHAPE, "mul_mat_vec: K=%lld must be a multiple of %lld for %s", static_cast<long long>(K),
                    static_cast<long long>(ablk > fmt_qk(f) ? ablk : fmt_qk(f)), type_name(w));
    if (K > (1 << 20)) return fail(c, GGQ_ERR_SHAPE, "mul_mat_vec: K too large");
    {  // token groups shrink down to one token, so the call runs if one token fits: refuse before any launch
        StreamShape sh;
        int cu = 0, cb = 0, rs = 0;
        if (plan_gemv_stream(f, w_row_bytes(f, K), 1, static_cast<int>(K), f == F_Q4_0 || a80, &sh, &cu, &cb, &rs) ==
            StreamPlan::kNone)
            return fail(c, GGQ_ERR_SHAPE, "mul_mat_vec: rows of K=%lld do not fit in shared memory",
                        static_cast<long long>(K));
    }
    return GGQ_OK;
}

// Shared-memory plan of the tensor-path decode GEMV (3-8 tokens); false when
// the shape is not covered (rows not a multiple of 16 bytes, K above 16 chunks
// of 256, Q6_K chunks below 128 inputs, or no room for two stages).
bool plan_mmav(int f, MmavParams& p, int* smem) {
    if (p.rowbytes % 16 != 0 || p.K > 16 * 256 || p.K % 256 != 0) return false;
    int chunk = 64;
    while (p.K / chunk > 16) chunk *= 2;
    if (f == F_Q6_K && chunk < 128) chunk = 128;
    p.chunk = chunk;
    p.nch = p.K / chunk;
    p.wrow = bank_stride(2 * p.rowbytes);  // one stride per pair of rows
    p.stage_stride = static_cast<int>(align_up(static_cast<size_t>(kTileRows / 2 * p.wrow + 16), 128));
    // activation rows in shared memory: the padding (a multiple of 16 bytes, so
    // each row stays one bulk copy) whose stride spreads the mma fragment words
    // of tokens g = 0..7 (word g * stride + t, t = 0..3) over the most banks
    p.xstride = p.xrow;
    if (p.xrow % 16 == 0) {
        int best = 33;
        for (int pad = 0; pad < 128; pad += 16) {
            const int sw = (p.xrow + pad) / 4;
            int hits[32] = {0}, worst = 0;
            for (int g = 0; g < 8; ++g)
                for (int t = 0; t < 4; ++t) worst = std::max(worst, ++hits[(g * sw + t) % 32]);
            if (worst < best) best = worst, p.xstride = p.xrow + pad;
        }
    }
    const int red_bytes = 2 * kConsumerWarps * 130 * 4, x_bytes = p.T * p.xstride;  // partials: [2][16][130] floats
    p.x_bytes = static_cast<int>(align_up(static_cast<size_t>(red_bytes > x_bytes ? red_bytes : x_bytes), 128));
    p.x_bulk = (p.xrow % 16 == 0 && aligned16(p.xq)) ? 1 : 0;
    const int fixed = p.x_bytes + kConsumerWarps * 4 * kMmavCStride * 4 + (2 * kMaxStages + 1) * 8 + 256;
    int stages = (kSmemLimit - fixed) / p.stage_stride;
    if (stages > kMaxStages) stages = kMaxStages;
    if (stages < 2) return false;
    if (stages > kWholeRowStages) stages = kWholeRowStages;
    p.stages = stages;
    *smem = stages * p.stage_stride + fixed;
    return true;
}

// Smallest token count that the decode GEMV sends to the tensor path: three.
// At two tokens the dp4a streaming kernel keeps both tokens' activations in
// registers and measured faster for every format (14336 x 4096 rows, chains of
// launches: Q4_K 8.9 against 10.2 us, Q5_K 10.4 against 12.5 (activations
// staged in shared memory), Q6_K 12.5 against 14.3, Q8_0 11.6 against 12.2).
int mma_min_tokens(int) { return 3; }

ggq_status launch_gemv_kind(ggq_ctx* c, int kind, int w, const void* W, int64_t N, int64_t K, const void* Xq,
                            int64_t T, float* Y, int32_t* coefs, cudaStream_t st, bool a80 = false) {
    const int f = fmt_of(w);
    const bool dump = kind == KIND_DUMP;
    const int ncoef = static_cast<int>(K / fmt_qk(f) * fmt_coefs(f));
    if (!a80 && T >= mma_min_tokens(f) && f != F_Q4_0 && aligned16(Xq)) {
        MmavParams m{};
        m.W = static_cast<const uint8_t*>(W);
        m.rowbytes = w_row_bytes(f, K);
        m.N = N;
        m.K = static_cast<int>(K);
        m.xq = static_cast<const uint8_t*>(Xq);
        m.xrow = static_cast<int>(K / 256 * 292);
        m.T = static_cast<int>(T);
        m.Y = Y;
        m.err = &c->ctrl->err;
        m.early_weights = c->static_weights;
        m.coefs = coefs;
        m.ncoef = ncoef;
        int smem = 0;
        if (plan_mmav(f, m, &smem)) {
            const int64_t tiles = (N + kTileRows - 1) / kTileRows;
            const int grid = static_cast<int>(tiles < c->nsm ? tiles : c->nsm);
            cudaError_t e = cudaSuccess;
            if (dump) {  // superblock coefficients of several warps are added atomically
                e = cudaMemsetAsync(coefs, 0, static_cast<size_t>(T) * N * ncoef * 4, st);
                if (e == cudaSuccess) e = launch_mmav_dump(f, m, grid, smem, st);
            } else {
                e = launch_mmav(f, m, grid, smem, st);
            }
            if (e != cudaSuccess) return cuda_fail(c, e, "mul_mat_vec tensor-path launch");
            return GGQ_OK;
        }
    }
    if (!a80 && T >= kGroupMinTokens && f != F_Q4_0 && !low_bit_kquant(f) && K % 1024 == 0 && aligned16(Xq)) {
        // several activation columns: the int8 tensor-core kernel (Q8_K rows are 16-byte multiples)
        GroupParams g{};
        g.W = static_cast<const uint8_t*>(W);
        g.rowbytes = w_row_bytes(f, K);
        g.N = N;
        g.K = static_cast<int>(K);
        g.T = static_cast<int>(T);
        g.xq = static_cast<const uint8_t*>(Xq);
        g.x_pitch = K / 256 * 292;
        g.Y = Y;
        g.err = &c->ctrl->err;
        g.early_weights = c->static_weights;
        g.coefs[0] = coefs;
        g.ncoef = ncoef;
        int smem = 0;
        if (plan_group(g, 1, true, &smem)) {
            const int64_t tiles = (N + kGroupRows - 1) / kGroupRows;
            const int grid = static_cast<int>(tiles < c->nsm ? tiles : c->nsm);
            cudaError_t e = cudaSuccess;
            if (dump) {  // block dots: the dump variant writes no Y (g.Y is null)
                e = cudaMemsetAsync(coefs, 0, static_cast<size_t>(T) * N * ncoef * 4, st);
                if (e == cudaSuccess) e = launch_group_dump(G_GEMV, f, g, grid, smem, st);
            } else {
                e = launch_group(G_GEMV, f, g, grid, smem, st);
            }
            if (e != cudaSuccess) return cuda_fail(c, e, "mul_mat_vec grouped launch");
            return GGQ_OK;
        }
    }
    StreamParams p{};
    p.W = static_cast<const uint8_t*>(W);
    p.rowbytes = w_row_bytes(f, K);
    p.N = N;
    p.K = static_cast<int>(K);
    p.xq = static_cast<const uint8_t*>(Xq);
    p.xrows = static_cast<int>(T);
    p.T = static_cast<int>(T);
    p.Y = Y;
    p.coefs = coefs;
    p.err = &c->ctrl->err;
    p.early_weights = c->static_weights;
    StreamShape sh;
    const bool a32 = f == F_Q4_0 || a80;  // activation scales per 32 elements
    if (kind == KIND_GEMV) {
        const StreamPlan plan = plan_gemv_stream(f, p.rowbytes, p.xrows, p.K, a32, &sh, &p.chunk_units,
                                                 &p.chunk_bytes, &p.row_slot);
        if (plan == StreamPlan::kSplit) {
            // the tokens as two groups, each streaming the weights once
            const int64_t xrow = a80 ? K / 32 * 34 : f == F_Q4_0 ? K / 32 * 36 : K / 256 * 292;
            const int64_t T0 = T / 2;
            const ggq_status s0 = launch_gemv_kind(c, kind, w, W, N, K, Xq, T0, Y, coefs, st, a80);
            if (s0 != GGQ_OK) return s0;
            return launch_gemv_kind(c, kind, w, W, N, K, static_cast<const uint8_t*>(Xq) + T0 * xrow, T - T0,
                                    Y + T0 * N, coefs, st, a80);
        }
        if (plan == StreamPlan::kNone)
            return fail(c, GGQ_ERR_SHAPE, "mul_mat_vec: K=%lld does not fit in shared memory",
                        static_cast<long long>(K));
    } else if (!plan_stream(kTileRows * p.rowbytes, p.xrows, p.K, a32, &sh)) {
        return fail(c, GGQ_ERR_SHAPE, "block_dots: K=%lld with T=%lld does not fit in shared memory",
                    static_cast<long long>(K), static_cast<long long>(T));
    }
    p.stages = sh.stages;
    p.stage_stride = sh.stride;
    p.x_bytes = sh.x_bytes;
    const int64_t tiles = (N + kTileRows - 1) / kTileRows;
    const int grid = static_cast<int>(tiles < c->nsm ? tiles : c->nsm);
    cudaError_t e = a80 ? launch_gemv_q80(kind, f, pow2_tokens(T), p, grid, sh.smem, st)
                        : launch_stream(kind, f, pow2_tokens(T), p, grid, sh.smem, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "mul_mat_vec launch");
    return GGQ_OK;
}

// One tcgen05 grouped GEMM, dumping its integer core when asked.  Q8_0 and Q4_K
// dump from the launch that computes the outputs.  MXFP4 folds each block's
// power of two into its operand and sums a whole superblock in one accumulator,
// so its integer core (one exact dot per 32-block) comes from a launch of the
// same kernel in its per-block schedule, run first; the folded launch then
// writes the outputs, which are therefore the same with and without the dump.
cudaError_t gmmtc_run(int f, const GmmTcParams& t, bool dump, int grid, cudaStream_t st) {
    if (!dump) return launch_gmmtc(f, t, grid, st);
    cudaError_t e = launch_gmmtc_dump(f, t, grid, st);
    if (e == cudaSuccess && f == F_MXFP4) e = launch_gmmtc(f, t, grid, st);
    return e;
}

// Expert banks that the expert-sorted route runs on the tcgen05 grouped GEMM
// (128-row weight tiles): Q8_0 and MXFP4 gate/up, Q4_K and MXFP4 down.  MXFP4
// goes there once the experts carry at least kMxTcPairs (token, expert) pairs
// on average: each of its k-steps costs a fixed ~0.7 us of role hand-offs
// whatever the column count, and below that load the int8 grouped kernel,
// whose cost scales with the columns, is faster (measured on the 256-expert
// H 4096 / I 2048 layer: 1.95 ms against 3.79 ms at 128 tokens, 4.20 ms against
// 3.86 ms at 512 tokens).
constexpr int64_t kMxTcPairs = 16;
bool tc_format(int f, int64_t P, int64_t E) { return f != F_MXFP4 || P >= kMxTcPairs * E; }
bool tc_gateup(int f, int64_t I, int64_t H, int64_t P, int64_t E) {
    (void)H;
    return (f == F_Q8_0 || f == F_MXFP4) && I % 128 == 0 && tc_format(f, P, E);
}
bool tc_down(int f, int64_t H, int64_t I, int64_t P, int64_t E) {
    (void)I;
    return (f == F_Q4_K || f == F_MXFP4) && H % 128 == 0 && tc_format(f, P, E);
}

// Largest token count of one direct-route launch pair (ds4 PR #656 "Add ROCm
// MXFP4 routed expert kernels", Summary: 2-4 tokens go to direct kernels; 5
// and above use expert-sorted tiles).
constexpr int kDirectMaxTokens = 4;

// Whether T > 4 tokens run as direct-route calls of at most four tokens each
// instead of expert-sorted tiles: up to `limit` tokens (default 32) while the
// pairs number at most twice the experts (few experts shared between the calls).  Measured on
// the 128-expert Q4_K/Q6_K layer (H 2048, I 768) at 5 / 8 / 16 / 32 tokens:
// 57 / 79 / 158 / 316 us against 216 / 298 / 450 / 617 us on sorted tiles;
// on the 256-expert MXFP4 layer (H 4096, I 2048): 170 / 258 / 517 / 1028 us
// against 297 / 438 / 764 / 1195 us, and 1545 against 1489 us at 48 tokens.
bool direct_chunks(int64_t T, int64_t E, int top_k, int limit) { return T <= limit && T * top_k <= 2 * E; }

// Fixed shared memory of a direct-route kernel besides its ring and activations.
constexpr int kDirectFixed = 2 * kMaxStages * 8 + static_cast<int>(sizeof(DirectPlan)) + 256;

// Whether the layer's widths fit the shared-memory plans of the kernels that
// would run it, checked before anything is enqueued: the refusal message, or
// nullptr.  Direct route: 16 gate + 16 up rows of H per stage with x^ of the
// tokens, and 16 down rows of I with h^ of the pairs; expert-sorted route: the
// grouped int8 kernel's whole-row slots where the f16 / tcgen05 kernels (which
// step through K) do not serve the format.
const char* moe_width_refusal(int fg, int fd, int64_t E, int64_t H, int64_t I, int64_t T, int top_k) {
    int smem = 0;
    if (T <= kDirectMaxTokens) {
        StreamShape sh;
        if (!plan_stream(2 * kTileRows * w_row_bytes(fg, H), static_cast<int>(T), static_cast<int>(H), false, &sh,
                         kDirectFixed))
            return "moe_experts: H too wide for shared memory";
        if (!plan_stream(kTileRows * w_row_bytes(fd, I), static_cast<int>(T * top_k), static_cast<int>(I), false,
                         &sh, kDirectFixed))
            return "moe_experts: I too wide for shared memory";
        return nullptr;
    }
    if (!tc_gateup(fg, I, H, T * top_k, E) && !gmm_supported(fg)) {
        GroupParams g{};
        g.rowbytes = w_row_bytes(fg, H);
        g.K = static_cast<int>(H);
        if (!plan_group(g, 2, false, &smem)) return "moe_experts: H too wide for shared memory";
    }
    if (!tc_down(fd, H, I, T * top_k, E) && !gmm_supported(fd)) {
        GroupParams d{};
        d.rowbytes = w_row_bytes(fd, I);
        d.K = static_cast<int>(I);
        if (!plan_group(d, 1, false, &smem)) return "moe_experts: I too wide for shared memory";
    }
    return nullptr;
}

ggq_status moe_sorted(ggq_ctx* c, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I, int top_k,
                      const float* X, const uint8_t* xq_in, const float* logits, const int32_t* ids_in,
                      const float* w_in, int64_t T, float* Y, const ggq_moe_dump* dump, void* stream) {
    const int fg = fmt_of(w->gate_type), fd = fmt_of(w->down_type);
    int32_t* const cg = dump ? dump->coefs_gate : nullptr;  // integer-core dumps (gate and up go together)
    int32_t* const cu = dump ? dump->coefs_up : nullptr;
    int32_t* const cd = dump ? dump->coefs_down : nullptr;
    const int ncg = static_cast<int>(H / fmt_qk(fg) * fmt_coefs(fg)), ncd = static_cast<int>(I / fmt_qk(fd) * fmt_coefs(fd));
    const SortedScratch ms = sorted_scratch(T, E, H, I, top_k);
    ggq_status s = need_scratch(c, ms.total);
    if (s != GGQ_OK) return s;
    if (T * top_k > (int64_t(1) << 30) / std::max<int64_t>(H, I))
        return fail(c, GGQ_ERR_SHAPE, "moe_experts: T*top_k*max(H, I) too large");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint8_t* base = c->pool;
    auto I32 = [&](size_t off) { return reinterpret_cast<int*>(base + off); };
    uint8_t* xq = base + ms.xq;
    const int64_t xrow = H / 256 * 292;
    uint8_t* hq = base + ms.hq;
    float* wts = reinterpret_cast<float*>(base + ms.w);
    float* h = reinterpret_cast<float*>(base + ms.h);
    float* o = reinterpret_cast<float*>(base + ms.o);
    const int64_t xp = q8k_pitch(H), hp = q8k_pitch(I);
    const int P = static_cast<int>(T * top_k);

    cudaError_t e = cudaMemsetAsync(I32(ms.counts), 0, static_cast<size_t>(E) * 4, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: memset");
    if (xq_in) {  // x^ given: its rows at the 16-byte pitch of the grouped kernels' row copies
        e = cudaMemcpy2DAsync(xq, static_cast<size_t>(q8k_pitch(H)), xq_in, static_cast<size_t>(xrow),
                              static_cast<size_t>(xrow), static_cast<size_t>(T), cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: x^ copy");
    }
    e = launch_route_sorted(logits, ids_in, w_in, xq_in ? nullptr : X, static_cast<int>(T), static_cast<int>(E), top_k,
                            static_cast<int>(H), xq, xp, I32(ms.ids), wts, I32(ms.counts), &c->ctrl->err, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: route launch");
    e = launch_group_plan(I32(ms.counts), static_cast<int>(E), I32(ms.offsets), I32(ms.cursor), I32(ms.ngroups),
                          I32(ms.gexp), I32(ms.goff), I32(ms.gcnt), st, c->tel_pairs, c->tel_calls);
    if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: plan launch");
    e = launch_scatter(I32(ms.ids), P, static_cast<int>(E), I32(ms.offsets), I32(ms.cursor), I32(ms.perm), st);
    if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: scatter launch");

    GroupParams g{};
    g.ngroups = I32(ms.ngroups);
    g.group_expert = I32(ms.gexp);
    g.group_off = I32(ms.goff);
    g.group_cnt = I32(ms.gcnt);
    g.perm = I32(ms.perm);
    g.top_k = top_k;
    g.err = &c->ctrl->err;
    // gate/up + SwiGLU -> h
    g.W = static_cast<const uint8_t*>(w->gate);
    g.W2 = static_cast<const uint8_t*>(w->up);
    g.rowbytes = w_row_bytes(fg, H);
    g.N = I;
    g.K = static_cast<int>(H);
    g.xq = xq;
    g.x_pitch = xp;
    g.h = h;
    g.g_dump = dump ? dump->g : nullptr;
    g.u_dump = dump ? dump->u : nullptr;
    // The grouped f16 GEMM (Q8_0, Q4_K) takes the activations as exact f16 rows.
    GmmParams m{};
    m.ngroups = g.ngroups;
    m.group_expert = g.group_expert;
    m.group_off = g.group_off;
    m.group_cnt = g.group_cnt;
    m.perm = g.perm;
    m.err = g.err;
    __half* const x16 = reinterpret_cast<__half*>(base + ms.x16);
    __half* const xbs = reinterpret_cast<__half*>(base + ms.xbs);
    float* const xdx = reinterpret_cast<float*>(base + ms.xdx);
    __half* const h16 = reinterpret_cast<__half*>(base + ms.h16);
    __half* const hbs = reinterpret_cast<__half*>(base + ms.hbs);
    float* const hdx = reinterpret_cast<float*>(base + ms.hdx);
    int smem = 0;
    bool h_dumped = false;  // the SwiGLU quantizer wrote dump->h itself
    const bool tcg = tc_gateup(fg, I, H, P, E);
    if (tcg) {
        // Q8_0 / MXFP4 gate/up on tcgen05: g and u per pair, then h = silu(g) u fused into its quantizer
        e = launch_q8k_to_f16(xq, xp, I32(ms.perm), top_k, P, H, x16, xbs, xdx, dx_pitch(H), st, fg == F_MXFP4);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: x to f16 launch");
        GmmTcParams t{};
        const int r = gmmtc_encode(t, fg, g.W, g.W2, g.rowbytes, E * I, x16, xdx, dx_pitch(H), nullptr, P,
                                   static_cast<int>(H));
        if (r) return fail(c, GGQ_ERR_CUDA, "moe sorted: gate/up tensor maps (CUresult %d)", r);
        t.N = I;
        t.K = static_cast<int>(H);
        t.nmat = 2;
        t.ngroups = g.ngroups;
        t.group_expert = g.group_expert;
        t.group_off = g.group_off;
        t.group_cnt = g.group_cnt;
        t.perm = g.perm;
        t.err = g.err;
        float* const gbuf = dump && dump->g ? dump->g : h;
        float* const ubuf = dump && dump->u ? dump->u : reinterpret_cast<float*>(base + ms.u);
        t.out[0] = gbuf;
        t.out[1] = ubuf;
        t.coefs[0] = cg;
        t.coefs[1] = cu;
        t.ncoef = ncg;
        e = gmmtc_run(fg, t, cg != nullptr, c->nsm, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: gate/up launch");
        e = launch_quantize_silu(gbuf, ubuf, P, I, hq, hp, dump ? dump->h : nullptr, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: SwiGLU quantize launch");
        h_dumped = dump != nullptr;
    } else if (gmm_supported(fg)) {
        e = launch_q8k_to_f16(xq, xp, I32(ms.perm), top_k, P, H, x16, xbs, xdx, dx_pitch(H), st);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: x to f16 launch");
        GmmParams q = m;
        const int r = gmm_encode(q, G_GATEUP, fg, g.W, g.W2, g.rowbytes, E * I, x16, xdx, dx_pitch(H), xbs, P,
                                 static_cast<int>(H));
        if (r) return fail(c, GGQ_ERR_CUDA, "moe sorted: gate/up tensor maps (CUresult %d)", r);
        q.N = I;
        q.K = static_cast<int>(H);
        q.h = h;
        q.g_dump = g.g_dump;
        q.u_dump = g.u_dump;
        q.coefs[0] = cg;
        q.coefs[1] = cu;
        q.ncoef = ncg;
        e = cg ? launch_gmm_dump(G_GATEUP, fg, q, c->nsm, gmm_smem_bytes(), st)
               : launch_gmm(G_GATEUP, fg, q, c->nsm, gmm_smem_bytes(), st);
    } else {
        if (!plan_group(g, 2, false, &smem)) return fail(c, GGQ_ERR_SHAPE, "moe_experts: H too wide for shared memory");
        g.coefs[0] = cg;
        g.coefs[1] = cu;
        g.ncoef = ncg;
        e = cg ? launch_group_dump(G_GATEUP, fg, g, c->nsm, smem, st) : launch_group(G_GATEUP, fg, g, c->nsm, smem, st);
    }
    if (!tcg) {
        if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: gate/up launch");
        // h^ = Q8_K(h)
        e = launch_quantize_pitched(h, P, I, hq, hp, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: quantize h launch");
    }
    // down -> o
    GroupParams d = g;
    d.W = static_cast<const uint8_t*>(w->down);
    d.W2 = nullptr;
    d.rowbytes = w_row_bytes(fd, I);
    d.N = H;
    d.K = static_cast<int>(I);
    d.xq = hq;
    d.x_pitch = hp;
    d.h = nullptr;
    d.g_dump = d.u_dump = nullptr;
    d.o = o;
    d.coefs[0] = d.coefs[1] = cd;
    d.ncoef = ncd;
    if (tc_down(fd, H, I, P, E)) {
        // Q4_K / MXFP4 down on tcgen05
        e = launch_q8k_to_f16(hq, hp, I32(ms.perm), 1, P, I, h16, hbs, hdx, dx_pitch(I), st, fd == F_MXFP4);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: h to f16 launch");
        GmmTcParams t{};
        const int r = gmmtc_encode(t, fd, d.W, nullptr, d.rowbytes, E * H, h16, hdx, dx_pitch(I), hbs, P,
                                   static_cast<int>(I));
        if (r) return fail(c, GGQ_ERR_CUDA, "moe sorted: down tensor maps (CUresult %d)", r);
        t.N = H;
        t.K = static_cast<int>(I);
        t.nmat = 1;
        t.ngroups = g.ngroups;
        t.group_expert = g.group_expert;
        t.group_off = g.group_off;
        t.group_cnt = g.group_cnt;
        t.perm = g.perm;
        t.err = g.err;
        t.out[0] = t.out[1] = o;
        t.coefs[0] = t.coefs[1] = cd;
        t.ncoef = ncd;
        e = gmmtc_run(fd, t, cd != nullptr, c->nsm, st);
    } else if (gmm_supported(fd)) {
        e = launch_q8k_to_f16(hq, hp, I32(ms.perm), 1, P, I, h16, hbs, hdx, dx_pitch(I), st);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: h to f16 launch");
        GmmParams q = m;
        const int r = gmm_encode(q, G_DOWN, fd, d.W, nullptr, d.rowbytes, E * H, h16, hdx, dx_pitch(I), hbs, P,
                                 static_cast<int>(I));
        if (r) return fail(c, GGQ_ERR_CUDA, "moe sorted: down tensor maps (CUresult %d)", r);
        q.N = H;
        q.K = static_cast<int>(I);
        q.o = o;
        q.coefs[0] = q.coefs[1] = cd;
        q.ncoef = ncd;
        e = cd ? launch_gmm_dump(G_DOWN, fd, q, c->nsm, gmm_smem_bytes(), st)
               : launch_gmm(G_DOWN, fd, q, c->nsm, gmm_smem_bytes(), st);
    } else {
        if (!plan_group(d, 1, false, &smem)) return fail(c, GGQ_ERR_SHAPE, "moe_experts: I too wide for shared memory");
        e = cd ? launch_group_dump(G_DOWN, fd, d, c->nsm, smem, st) : launch_group(G_DOWN, fd, d, c->nsm, smem, st);
    }
    if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: down launch");
    e = launch_combine(o, wts, static_cast<int>(T), top_k, H, Y, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "moe sorted: combine launch");
    if (dump) {
        const size_t xb = static_cast<size_t>(H / 256 * 292), hb = static_cast<size_t>(I / 256 * 292);
        if (dump->ids) e = cudaMemcpyAsync(dump->ids, I32(ms.ids), P * 4, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && dump->weights)
            e = cudaMemcpyAsync(dump->weights, wts, P * 4, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && dump->xq)
            e = cudaMemcpy2DAsync(dump->xq, xb, xq, xp, xb, T, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && dump->h && !h_dumped)
            e = cudaMemcpyAsync(dump->h, h, static_cast<size_t>(P) * I * 4, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && dump->hq)
            e = cudaMemcpy2DAsync(dump->hq, hb, hq, hp, hb, P, cudaMemcpyDeviceToDevice, st);
        if (e == cudaSuccess && dump->o)
            e = cudaMemcpyAsync(dump->o, o, static_cast<size_t>(P) * H * 4, cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe dump copy");
    }
    return GGQ_OK;
}

ggq_status moe_direct(ggq_ctx* c, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I, int top_k, int fg,
                      int fd, const float* X, const uint8_t* xq_in, const float* logits, const int32_t* ids,
                      const float* weights, int64_t T, float* Y, const ggq_moe_dump* dump, void* stream,
                      int32_t* ids_out);

ggq_status moe_run(ggq_ctx* c, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I, int top_k, const float* X,
                   const uint8_t* xq_in, const float* logits, const int32_t* ids, const float* weights, int64_t T,
                   float* Y, const ggq_moe_dump* dump, void* stream) {
    if (!w || (!X && !xq_in) || !Y || (!logits && (!ids || !weights)))
        return fail(c, GGQ_ERR_INVALID_ARG, "moe_experts: null pointer");
    if (xq_in && (reinterpret_cast<uintptr_t>(xq_in) & 3))
        return fail(c, GGQ_ERR_INVALID_ARG, "moe_experts_q: Xq must be 4-byte aligned");
    const int fg = fmt_of(w->gate_type), fu = fmt_of(w->up_type), fd = fmt_of(w->down_type);
    for (int t : {w->gate_type, w->up_type, w->down_type}) {
        const int f = fmt_of(t);
        if (f < 0 || f == F_Q4_0 || low_bit_kquant(f))
            return fail(c, GGQ_ERR_UNSUPPORTED,
                        "moe_experts: expert weight type %d (%s) is not supported; supported with Q8_K activations: "
                        "Q8_0, Q4_K, Q5_K, Q6_K, MXFP4",
                        t, type_name(t));
    }
    if (fg != fu)
        return fail(c, GGQ_ERR_UNSUPPORTED, "moe_experts: gate (%s) and up (%s) banks must share one format",
                    type_name(w->gate_type), type_name(w->up_type));
    if (dump && (dump->coefs_gate == nullptr) != (dump->coefs_up == nullptr))
        return fail(c, GGQ_ERR_INVALID_ARG, "moe_experts: coefs_gate and coefs_up are dumped together");
    if (!w->gate || !w->up || !w->down) return fail(c, GGQ_ERR_INVALID_ARG, "moe_experts: null bank");
    if (!aligned16(w->gate) || !aligned16(w->up) || !aligned16(w->down) || (X && !aligned16(X)) || !aligned16(Y))
        return fail(c, GGQ_ERR_INVALID_ARG, "moe_experts: pointers must be 16-byte aligned");
    if (H < 256 || H % 256 || I < 256 || I % 256)
        return fail(c, GGQ_ERR_SHAPE, "moe_experts: H=%lld and I=%lld must be positive multiples of 256",
                    static_cast<long long>(H), static_cast<long long>(I));
    if (top_k < 1 || top_k > 8 || E < top_k || E > 4096)
        return fail(c, GGQ_ERR_SHAPE, "moe_experts: need 1 <= top_k <= 8 and top_k <= E <= 4096");
    if (T < 1) return fail(c, GGQ_ERR_SHAPE, "moe_experts: T=%lld", static_cast<long long>(T));
    // more than four tokens: direct-route calls of four tokens each where they fit and
    // measured faster
    const bool chunked = T > kDirectMaxTokens && direct_chunks(T, E, top_k, c->direct_max) &&
                         moe_width_refusal(fg, fd, E, H, I, kDirectMaxTokens, top_k) == nullptr;
    if (!chunked)
        if (const char* why = moe_width_refusal(fg, fd, E, H, I, T, top_k)) return fail(c, GGQ_ERR_SHAPE, "%s", why);
    if (c->tel_pairs && E > c->tel_experts)
        return fail(c, GGQ_ERR_SHAPE, "moe_experts: E=%lld exceeds the %lld experts of the telemetry buffer",
                    static_cast<long long>(E), static_cast<long long>(c->tel_experts));
    if (T > kDirectMaxTokens && !chunked)
        return moe_sorted(c, w, E, H, I, top_k, X, xq_in, logits, ids, weights, T, Y, dump, stream);
    if (!chunked)
        return moe_direct(c, w, E, H, I, top_k, fg, fd, X, xq_in, logits, ids, weights, T, Y, dump, stream, nullptr);
    // with the expert-load counters on, the launches keep every pair's routed id
    // after the direct route's scratch and one small kernel counts the whole call
    const size_t ids_at = moe_scratch(kDirectMaxTokens, H, I, top_k).total;
    int32_t* ids_all = nullptr;
    if (c->tel_pairs) {
        const ggq_status s = need_scratch(c, ids_at + align_up(static_cast<size_t>(T * top_k) * 4));
        if (s != GGQ_OK) return s;
        ids_all = reinterpret_cast<int32_t*>(c->pool + ids_at);
    }
    const int64_t xrow = H / 256 * 292, ncg = H / fmt_qk(fg) * fmt_coefs(fg), ncd = I / fmt_qk(fd) * fmt_coefs(fd);
    for (int64_t t0 = 0; t0 < T; t0 += kDirectMaxTokens) {
        const int64_t tc = T - t0 < kDirectMaxTokens ? T - t0 : kDirectMaxTokens;
        const int64_t p0 = t0 * top_k;  // first pair of the chunk
        ggq_moe_dump dc{};
        if (dump) {  // the chunk's rows of every dumped array
            const auto at = [](auto* q, int64_t off) { return q ? q + off : q; };
            dc.ids = at(dump->ids, p0);
            dc.weights = at(dump->weights, p0);
            dc.xq = dump->xq ? static_cast<uint8_t*>(dump->xq) + t0 * xrow : nullptr;
            dc.g = at(dump->g, p0 * I);
            dc.u = at(dump->u, p0 * I);
            dc.h = at(dump->h, p0 * I);
            dc.hq = dump->hq ? static_cast<uint8_t*>(dump->hq) + p0 * (I / 256 * 292) : nullptr;
            dc.o = at(dump->o, p0 * H);
            dc.coefs_gate = at(dump->coefs_gate, p0 * I * ncg);
            dc.coefs_up = at(dump->coefs_up, p0 * I * ncg);
            dc.coefs_down = at(dump->coefs_down, p0 * H * ncd);
        }
        const ggq_status s = moe_direct(c, w, E, H, I, top_k, fg, fd, X ? X + t0 * H : nullptr,
                                        xq_in ? xq_in + t0 * xrow : nullptr, logits ? logits + t0 * E : nullptr,
                                        ids ? ids + p0 : nullptr, weights ? weights + p0 : nullptr, tc, Y + t0 * H,
                                        dump ? &dc : nullptr, stream, ids_all ? ids_all + p0 : nullptr);
        if (s != GGQ_OK) return s;
    }
    if (ids_all) {
        cudaError_t e = launch_moe_count(ids_all, static_cast<int>(T * top_k), static_cast<int>(E), c->tel_pairs,
                                         c->tel_calls, static_cast<cudaStream_t>(stream));
        if (e != cudaSuccess) return cuda_fail(c, e, "moe counters launch");
    }
    return GGQ_OK;
}

// The direct route for T <= 4 tokens (arguments checked by moe_run).  ids_out:
// where the routed ids go instead of the scratch (one launch of a several-launch
// call, whose expert-load counters are taken afterwards from all its ids; the
// launches themselves then count nothing), or null.
ggq_status moe_direct(ggq_ctx* c, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I, int top_k, int fg,
                      int fd, const float* X, const uint8_t* xq_in, const float* logits, const int32_t* ids,
                      const float* weights, int64_t T, float* Y, const ggq_moe_dump* dump, void* stream,
                      int32_t* ids_out) {
    const MoeScratch ms = moe_scratch(T, H, I, top_k);
    ggq_status s = need_scratch(c, ms.total);
    if (s != GGQ_OK) return s;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int P = static_cast<int>(T * top_k);
    DirectParams p{};
    p.T = static_cast<int>(T);
    p.E = static_cast<int>(E);
    p.top_k = top_k;
    p.X = X;
    p.xq_in = xq_in;
    p.logits = logits;
    p.ids_in = ids;
    p.w_in = weights;
    p.ids = ids_out ? ids_out : reinterpret_cast<int32_t*>(c->pool + ms.ids);
    p.w = reinterpret_cast<float*>(c->pool + ms.w);
    p.h = reinterpret_cast<float*>(c->pool + ms.h);
    p.xq_dump = dump && !xq_in ? static_cast<uint8_t*>(dump->xq) : nullptr;
    p.hq = c->pool + ms.hq;
    p.early_weights = c->static_weights;
    p.g_dump = dump ? dump->g : nullptr;
    p.u_dump = dump ? dump->u : nullptr;
    p.o_dump = dump ? dump->o : nullptr;
    p.coefs[0] = dump ? dump->coefs_gate : nullptr;
    p.coefs[1] = dump ? dump->coefs_up : nullptr;
    p.ncoef = static_cast<int>(H / fmt_qk(fg) * fmt_coefs(fg));
    p.tel_pairs = ids_out ? nullptr : c->tel_pairs;
    p.tel_calls = ids_out ? nullptr : c->tel_calls;
    p.Y = Y;
    p.err = &c->ctrl->err;
    const int nt = pow2_tokens(T);
    const int direct_fixed = kDirectFixed;
    // gate/up: 16 gate rows + the 16 matching up rows per stage; x^ of the T tokens
    {
        p.W = static_cast<const uint8_t*>(w->gate);
        p.W2 = static_cast<const uint8_t*>(w->up);
        p.rowbytes = w_row_bytes(fg, H);
        p.N = I;
        p.K = static_cast<int>(H);
        StreamShape sh;
        if (!plan_stream(2 * kTileRows * p.rowbytes, static_cast<int>(T), p.K, false, &sh, direct_fixed))
            return fail(c, GGQ_ERR_SHAPE, "moe_experts: H too wide for shared memory");
        p.stages = sh.stages;
        p.stage_stride = sh.stride;
        p.x_bytes = sh.x_bytes;
        cudaError_t e = p.coefs[0] ? launch_direct_gateup_dump(fg, nt, p, c->nsm, sh.smem, st)
                                   : launch_direct_gateup(fg, nt, p, c->nsm, sh.smem, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe gate/up launch");
    }
    // down: 16-row output tile of every selected expert; h^ of the T*k pairs.
    // Fused (no per-pair outputs requested): G experts per stage, the largest G
    // that leaves three stages and at most 256 units per concatenated row
    {
        p.W = static_cast<const uint8_t*>(w->down);
        p.W2 = nullptr;
        p.rowbytes = w_row_bytes(fd, I);
        p.N = H;
        p.K = static_cast<int>(I);
        p.coefs[0] = dump ? dump->coefs_down : nullptr;
        p.coefs[1] = nullptr;
        p.tel_pairs = nullptr;  // counted once, by the gate/up kernel
        p.tel_calls = nullptr;
        p.ncoef = static_cast<int>(I / fmt_qk(fd) * fmt_coefs(fd));
        const bool fused = !(dump && (dump->o || dump->coefs_down));
        StreamShape sh;
        int G = 1;
        if (fused) {
            // one token: its top_k experts are known to be distinct, so G = top_k
            // takes every expert's tile in one stage (one item per CTA: two
            // stages are enough, the second one free for h)
            const int gmax = T == 1 && top_k <= 8 ? top_k : 8;
            for (int g = gmax; g >= 1; --g) {
                if (g * (I / 64) > 256) continue;
                if (plan_stream(g * kTileRows * p.rowbytes, P, p.K, false, &sh, direct_fixed) &&
                    (sh.stages >= 3 || g == 1 || (T == 1 && g == top_k && sh.stages >= 2))) {
                    G = g;
                    break;
                }
            }
        }
        if (!plan_stream(G * kTileRows * p.rowbytes, P, p.K, false, &sh, direct_fixed))
            return fail(c, GGQ_ERR_SHAPE, "moe_experts: I too wide for shared memory");
        p.G = G;
        p.stages = sh.stages;
        p.stage_stride = sh.stride;
        p.x_bytes = sh.x_bytes;
        cudaError_t e = fused         ? launch_direct_downf(fd, nt, p, c->nsm, sh.smem, st)
                        : p.coefs[0] ? launch_direct_down_dump(fd, nt, p, c->nsm, sh.smem, st)
                                     : launch_direct_down(fd, nt, p, c->nsm, sh.smem, st);
        if (e != cudaSuccess) return cuda_fail(c, e, "moe down launch");
    }
    if (dump) {
        struct Cp { void* dst; const void* src; size_t n; } cps[] = {
            {xq_in ? dump->xq : nullptr, xq_in, static_cast<size_t>(T) * (H / 256) * 292},
            {dump->ids, p.ids, static_cast<size_t>(P) * 4},
            {dump->weights, p.w, static_cast<size_t>(P) * 4},
            {dump->h, p.h, static_cast<size_t>(P) * I * 4},
            {dump->hq, p.hq, static_cast<size_t>(P) * (I / 256) * 292},
        };
        for (const Cp& cp : cps)
            if (cp.dst) {
                cudaError_t e = cudaMemcpyAsync(cp.dst, cp.src, cp.n, cudaMemcpyDeviceToDevice, st);
                if (e != cudaSuccess) return cuda_fail(c, e, "moe dump copy");
            }
    }
    return GGQ_OK;
}

}  // namespace

extern "C" {

ggq_status ggq_create(ggq_ctx** out, int device) {
    if (!out) return GGQ_ERR_INVALID_ARG;
    *out = nullptr;
    cudaDeviceProp prop;
    cudaError_t e = cudaGetDeviceProperties(&prop, device);
    if (e != cudaSuccess) return GGQ_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return GGQ_ERR_ARCH;
    DeviceScope scope;
    if (cudaGetDevice(&scope.prev) != cudaSuccess) return GGQ_ERR_CUDA;
    e = cudaSetDevice(device);
    if (e != cudaSuccess) return GGQ_ERR_CUDA;
    ggq_ctx* c = new ggq_ctx();
    c->device = device;
    c->nsm = prop.multiProcessorCount;
    e = cudaMalloc(&c->ctrl, sizeof(Ctrl));
    if (e == cudaSuccess) e = cudaMemset(c->ctrl, 0, sizeof(Ctrl));
    if (e == cudaSuccess) e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        if (c->ctrl) cudaFree(c->ctrl);
        delete c;
        return GGQ_ERR_CUDA;
    }
    *out = c;
    return GGQ_OK;
}

ggq_status ggq_destroy(ggq_ctx* c) {
    if (!c) return GGQ_ERR_INVALID_ARG;
    DeviceScope scope;
    if (check_ctx(c, scope) != GGQ_OK) return GGQ_ERR_CUDA;
    for (void* p : c->retired) cudaFree(p);
    if (c->pool) cudaFree(c->pool);
    if (c->ctrl) cudaFree(c->ctrl);
    delete c;
    return GGQ_OK;
}

const char* ggq_last_error(const ggq_ctx* c) { return c ? c->err.c_str() : "null context"; }

size_t ggq_scratch_bytes(const ggq_ctx* c) { return c ? c->pool_bytes : 0; }

ggq_status ggq_set_static_weights(ggq_ctx* c, int static_weights) {
    if (!c) return GGQ_ERR_INVALID_ARG;
    c->static_weights = static_weights ? 1 : 0;
    return GGQ_OK;
}

ggq_status ggq_set_direct_route_max_tokens(ggq_ctx* c, int max_tokens) {
    if (!c) return GGQ_ERR_INVALID_ARG;
    if (max_tokens < kDirectMaxTokens || max_tokens > 32)
        return fail(c, GGQ_ERR_INVALID_ARG, "set_direct_route_max_tokens: %d is outside [4, 32]", max_tokens);
    c->direct_max = max_tokens;
    return GGQ_OK;
}

ggq_status ggq_reserve(ggq_ctx* c, const ggq_plan* plan, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    if (!plan) return fail(c, GGQ_ERR_INVALID_ARG, "reserve: null plan");
    size_t need = 0;
    const int64_t T = plan->max_tokens > 0 ? plan->max_tokens : 1;
    if (plan->max_k > 0) need = gemv_scratch(T, plan->max_k);
    if (plan->hidden > 0 && plan->inter > 0) {
        const int64_t k = plan->top_k > 0 ? plan->top_k : 8;
        const int64_t E = plan->n_experts > 0 ? plan->n_experts : 4096;
        size_t m = moe_scratch(T < kDirectMaxTokens ? T : kDirectMaxTokens, plan->hidden, plan->inter, k).total;
        if (T > kDirectMaxTokens) {
            m += align_up(static_cast<size_t>(T * k) * 4);  // direct calls of 4 tokens: every routed id kept
            const size_t ms = sorted_scratch(T, E, plan->hidden, plan->inter, k).total;
            if (ms > m) m = ms;
        }
        if (m > need) need = m;
    }
    if (need <= c->pool_bytes) return GGQ_OK;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cs);
    if (e != cudaSuccess) return cuda_fail(c, e, "reserve: cudaStreamIsCapturing");
    if (cs != cudaStreamCaptureStatusNone)
        return fail(c, GGQ_ERR_CAPTURE_ALLOC, "reserve: pool must grow to %zu bytes while the stream is capturing",
                    need);
    void* p = nullptr;
    e = cudaMalloc(&p, need);
    if (e != cudaSuccess) return cuda_fail(c, e, "reserve: cudaMalloc");
    if (c->pool) c->retired.push_back(c->pool);  // work in flight may still use it
    c->pool = static_cast<uint8_t*>(p);
    c->pool_bytes = need;
    return GGQ_OK;
}

int ggq_supported(int w, int act, int op) {
    const int f = fmt_of(w);
    switch (op) {
    case GGQ_OP_QUANTIZE_ACT: return act == GGQ_TYPE_Q8_1 || act == GGQ_TYPE_Q8_K || act == GGQ_TYPE_Q8_0;
    case GGQ_OP_DEQUANT: return f >= 0;
    case GGQ_OP_MUL_MAT_VEC:
        if (f < 0) return 0;
        if (act == GGQ_TYPE_Q8_0) return f == F_Q4_0 || f == F_Q8_0;
        return f == F_Q4_0 ? act == GGQ_TYPE_Q8_1 : act == GGQ_TYPE_Q8_K;
    case GGQ_OP_MOE: return f >= 0 && f != F_Q4_0 && !low_bit_kquant(f) && act == GGQ_TYPE_Q8_K;
    default: return 0;
    }
}

ggq_status ggq_quantize_act(ggq_ctx* c, int act, const float* x, int64_t T, int64_t K, void* out, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    if (act != GGQ_TYPE_Q8_1 && act != GGQ_TYPE_Q8_K && act != GGQ_TYPE_Q8_0)
        return fail(c, GGQ_ERR_UNSUPPORTED, "quantize_act: activation type %d (%s); supported: Q8_1, Q8_0, Q8_K", act,
                    type_name(act));
    const int64_t blk = act == GGQ_TYPE_Q8_K ? 256 : 32;
    if (T < 0 || K < 0 || K % blk)
        return fail(c, GGQ_ERR_SHAPE, "quantize_act: T=%lld, K=%lld (K must be a multiple of %lld)",
                    static_cast<long long>(T), static_cast<long long>(K), static_cast<long long>(blk));
    if (T == 0 || K == 0) return GGQ_OK;  // empty: nothing is read or written
    if (!x || !out) return fail(c, GGQ_ERR_INVALID_ARG, "quantize_act: null pointer");
    if (!aligned16(x) || (reinterpret_cast<uintptr_t>(out) & 3))
        return fail(c, GGQ_ERR_INVALID_ARG, "quantize_act: x must be 16-byte and out 4-byte aligned");
    cudaError_t e = launch_quantize(act == GGQ_TYPE_Q8_1 ? 0 : act == GGQ_TYPE_Q8_K ? 1 : 2, x, T, K,
                                    static_cast<uint8_t*>(out), static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GGQ_OK : cuda_fail(c, e, "quantize_act launch");
}

ggq_status ggq_dequant(ggq_ctx* c, int w, const void* blocks, int64_t rows, int64_t K, float* out, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    const int f = fmt_of(w);
    if (f < 0)
        return fail(c, GGQ_ERR_UNSUPPORTED,
                    "dequant: weight type %d (%s); supported: Q4_0, Q8_0, Q4_K, Q5_K, Q6_K, MXFP4", w, type_name(w));
    if (rows < 0 || K < 0 || K % fmt_qk(f))
        return fail(c, GGQ_ERR_SHAPE, "dequant: rows=%lld, K=%lld (K must be a multiple of %d)",
                    static_cast<long long>(rows), static_cast<long long>(K), fmt_qk(f));
    if (rows == 0 || K == 0) return GGQ_OK;  // empty: nothing is read or written
    if (!blocks || !out) return fail(c, GGQ_ERR_INVALID_ARG, "dequant: null pointer");
    cudaError_t e = launch_dequant(f, static_cast<const uint8_t*>(blocks), rows, K, out,
                                   static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GGQ_OK : cuda_fail(c, e, "dequant launch");
}

ggq_status ggq_mul_mat_vec_q(ggq_ctx* c, int w, const void* W, int64_t N, int64_t K, const void* Xq, int64_t T,
                             float* Y, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    s = gemv_checks(c, w, W, N, K, Xq, T, Y);
    if (s != GGQ_OK) return s;
    return launch_gemv_kind(c, KIND_GEMV, w, W, N, K, Xq, T, Y, nullptr, static_cast<cudaStream_t>(stream));
}

ggq_status ggq_mul_mat_vec(ggq_ctx* c, int w, const void* W, int64_t N, int64_t K, const float* X, int64_t T,
                           float* Y, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    s = gemv_checks(c, w, W, N, K, X, T, Y);
    if (s != GGQ_OK) return s;
    s = need_scratch(c, gemv_scratch(T, K));
    if (s != GGQ_OK) return s;
    const bool q81 = w == GGQ_TYPE_Q4_0;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_quantize(q81 ? 0 : 1, X, T, K, c->pool, st);
    if (e != cudaSuccess) return cuda_fail(c, e, "mul_mat_vec quantize launch");
    return launch_gemv_kind(c, KIND_GEMV, w, W, N, K, c->pool, T, Y, nullptr, st);
}

ggq_status ggq_block_dots(ggq_ctx* c, int w, const void* W, int64_t N, int64_t K, const void* Xq, int64_t T,
                          int32_t* coefs, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    s = gemv_checks(c, w, W, N, K, Xq, T, coefs);
    if (s != GGQ_OK) return s;
    return launch_gemv_kind(c, KIND_DUMP, w, W, N, K, Xq, T, nullptr, coefs, static_cast<cudaStream_t>(stream));
}

ggq_status ggq_mul_mat_vec_qa(ggq_ctx* c, int w, int act, const void* W, int64_t N, int64_t K, const void* Xq,
                              int64_t T, float* Y, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    s = gemv_checks(c, w, W, N, K, Xq, T, Y, act);
    if (s != GGQ_OK) return s;
    return launch_gemv_kind(c, KIND_GEMV, w, W, N, K, Xq, T, Y, nullptr, static_cast<cudaStream_t>(stream),
                            act == GGQ_TYPE_Q8_0);
}

ggq_status ggq_block_dots_qa(ggq_ctx* c, int w, int act, const void* W, int64_t N, int64_t K, const void* Xq,
                             int64_t T, int32_t* coefs, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    s = gemv_checks(c, w, W, N, K, Xq, T, coefs, act);
    if (s != GGQ_OK) return s;
    return launch_gemv_kind(c, KIND_DUMP, w, W, N, K, Xq, T, nullptr, coefs, static_cast<cudaStream_t>(stream),
                            act == GGQ_TYPE_Q8_0);
}

ggq_status ggq_moe_experts(ggq_ctx* c, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I, int top_k,
                           const float* X, const float* router_logits, int64_t T, float* Y, const ggq_moe_dump* dump,
                           void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    if (!router_logits) return fail(c, GGQ_ERR_INVALID_ARG, "moe_experts: null router_logits");
    return moe_run(c, w, E, H, I, top_k, X, nullptr, router_logits, nullptr, nullptr, T, Y, dump, stream);
}

ggq_status ggq_moe_experts_routed(ggq_ctx* c, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I,
                                  int top_k, const float* X, const int32_t* ids, const float* weights, int64_t T,
                                  float* Y, const ggq_moe_dump* dump, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    if (!ids || !weights) return fail(c, GGQ_ERR_INVALID_ARG, "moe_experts_routed: null ids/weights");
    return moe_run(c, w, E, H, I, top_k, X, nullptr, nullptr, ids, weights, T, Y, dump, stream);
}

ggq_status ggq_set_moe_counters(ggq_ctx* c, int64_t* pairs, int64_t n_experts, int64_t* calls) {
    if (!c) return GGQ_ERR_INVALID_ARG;
    if ((pairs == nullptr) != (calls == nullptr))
        return fail(c, GGQ_ERR_INVALID_ARG, "set_moe_counters: pairs and calls are set or cleared together");
    if (pairs && (n_experts < 1 || n_experts > 4096))
        return fail(c, GGQ_ERR_SHAPE, "set_moe_counters: n_experts=%lld out of 1..4096", static_cast<long long>(n_experts));
    if ((reinterpret_cast<uintptr_t>(pairs) | reinterpret_cast<uintptr_t>(calls)) & 7)
        return fail(c, GGQ_ERR_INVALID_ARG, "set_moe_counters: buffers must be 8-byte aligned");
    c->tel_pairs = reinterpret_cast<unsigned long long*>(pairs);
    c->tel_calls = reinterpret_cast<unsigned long long*>(calls);
    c->tel_experts = pairs ? n_experts : 0;
    return GGQ_OK;
}

ggq_status ggq_moe_experts_q(ggq_ctx* c, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I, int top_k,
                             const void* Xq, const float* router_logits, int64_t T, float* Y, const ggq_moe_dump* dump,
                             void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    if (!router_logits || !Xq) return fail(c, GGQ_ERR_INVALID_ARG, "moe_experts_q: null Xq or router_logits");
    return moe_run(c, w, E, H, I, top_k, nullptr, static_cast<const uint8_t*>(Xq), router_logits, nullptr, nullptr, T,
                   Y, dump, stream);
}

ggq_status ggq_sync_status(ggq_ctx* c, void* stream) {
    DeviceScope scope;
    ggq_status s = check_ctx(c, scope);
    if (s != GGQ_OK) return s;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(c, e, "sync_status: stream");
    int word = 0;
    e = cudaMemcpy(&word, &c->ctrl->err, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(c, e, "sync_status: read");
    if (word != 0) {
        cudaMemset(&c->ctrl->err, 0, sizeof(int));
        return fail(c, GGQ_ERR_DEVICE, "device error word %d (%s)", word,
                    word == DEV_ERR_TIMEOUT   ? "a bounded wait ran out"
                    : word == DEV_ERR_BAD_IDS ? "a routed expert id out of range"
                                              : "unknown device error");
    }
    return GGQ_OK;
}

}  // extern "C"

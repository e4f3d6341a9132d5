// ggq_internal.h -- host/device shared declarations inside libggq (not part of the ABI).
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ggq {

// Streaming-kernel geometry: sixteen consumer warps + one producer warp per
// CTA, one weight row per consumer warp per stage (16 rows; gate/up: 8 gate
// rows and the 8 matching up rows).
constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileRows = 16;
constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 232448;  // 227 KB opt-in dynamic shared memory per CTA
constexpr int kMaxDevices = 64;     // device ordinals with per-device launch state
// Depth of the weight rings.  With every SM streaming, a deeper ring adds no
// bandwidth but queueing delay: a launch's first tile then lands later behind
// the other SMs' requests.  Measured on GB300 in chains of 14336 x 4096 GEMVs
// (16-row tiles of 37-70 KB): three whole-row stages beat five or six; row-chunk
// stages (a few KB to tens of KB) keep about kInFlightBytes in flight.
constexpr int kWholeRowStages = 3;
constexpr int kInFlightBytes = 140 * 1024;
// Weight stages streamed before the activations are in (with static weights,
// before the previous kernel has finished): the streaming kernel's whole-row
// rings all but the last (which takes the activation rows), the tensor-path
// GEMV one.

enum Kind : int { KIND_GEMV = 0, KIND_DUMP = 1, KIND_GATEUP = 2, KIND_DOWN = 3, KIND_DOWNF = 4 };

struct StreamParams {
    const uint8_t* W;   // GEMV weight matrix
    int64_t rowbytes;   // bytes of one weight row
    int64_t N;          // rows
    int K;              // input width
    const uint8_t* xq;  // packed activations [T][K/blk]
    int xrows;          // activation rows staged in shared memory
    int T;
    float* Y;           // out [T][N]
    int32_t* coefs;     // block-dot dump [T][N][K/blk*c]
    int* err;           // device error word
    int early_weights;  // 1: stream weights before waiting for the previous kernel
    int stages;
    int stage_stride;   // bytes per ring slot (multiple of 128)
    int x_bytes;        // bytes of the staged-activation region
    int chunk_units;    // GEMV only: 0 = whole rows per stage; else each stage holds
                        // this many 64-weight units of each of the tile's rows
    int chunk_bytes;    // bytes of chunk_units units
    int row_slot;       // bytes between the rows of a chunked stage (a multiple of 16)
};

// Bytes of the structure-of-arrays activation region for `rows` rows of width
// K: padded quants (80 bytes per 64-element unit), scales, per-32 sums, Q8_K
// per-16 sums.
// Offsets of the parts are the running sums, each rounded up to 128 bytes.
__host__ __device__ inline size_t x_up128(size_t v) { return (v + 127) / 128 * 128; }
inline int x_region_bytes(int rows, int K, bool q81) {
    const size_t q = static_cast<size_t>(rows) * (((K + 63) / 64) * 80);  // xq_row_bytes
    const size_t d = static_cast<size_t>(rows) * (K / (q81 ? 32 : 256)) * 4;
    const size_t s32 = static_cast<size_t>(rows) * (K / 32) * 4;
    const size_t bs = q81 ? 0 : static_cast<size_t>(rows) * (K / 16) * 2;
    return static_cast<int>(x_up128(q) + x_up128(d) + x_up128(s32) + x_up128(bs));
}

// Grouped tensor-core kernel geometry (ggq_group.cuh).
constexpr int kGroupConsumerWarps = 8;
constexpr int kGroupThreads = (kGroupConsumerWarps + 1) * 32;
constexpr int kGroupCols = 8;   // activation columns per mma n8 chunk
constexpr int kGroupRows = 16;  // weight rows per item (per matrix)

enum GKind : int { G_GEMV = 0, G_GATEUP = 1, G_DOWN = 2 };

struct GroupParams {
    const uint8_t* W;    // GEMV matrix, gate bank, or down bank
    const uint8_t* W2;   // up bank (gate/up only)
    int64_t rowbytes;    // bytes of one weight row in global
    int64_t N;           // rows per matrix
    int K;               // input width (multiple of 256)
    // groups (MoE): non-empty experts, their column ranges in perm
    const int* ngroups;
    const int* group_expert;
    const int* group_off;
    const int* group_cnt;
    const int* perm;     // pairs sorted by expert
    int top_k;
    int T;               // GEMV: tokens (columns)
    // activations: packed Q8_K rows, x_pitch bytes apart in global
    const uint8_t* xq;
    int64_t x_pitch;
    // outputs
    float* Y;            // GEMV [T][N]
    float* h;            // gate/up [pairs][N]
    float* g_dump;
    float* u_dump;
    float* o;            // down [pairs][N]
    int* err;
    int early_weights;   // 1: stream weights before waiting for the previous kernel (GEMV only)
    int32_t* coefs[2];   // integer-core dump per matrix: [columns or pairs][N][ncoef] (dump launches only)
    int ncoef;           // coefficients per row: K/blk * (2 for Q4_K/Q5_K, else 1)
    // shared-memory plan
    int wstages, wslot, wrow, wcontig;  // weight ring: slots, slot bytes, row stride, one contiguous copy
    int xstages, xslot, xstride, xcopy; // activation ring: slots, slot bytes, row stride, bytes per row copy
};

// Decode GEMV at 2-8 tokens on the int8 tensor path (ggq_mmav.cuh): the
// streaming geometry above, rows copied one by one into bank-padded rows, K
// split into one chunk per consumer warp.
// Floats per (warp, mma column pair) of the tensor-path GEMV's accumulator
// start values in shared memory: 32 used, padded so that the four column pairs
// of a warp fall on distinct banks.
constexpr int kMmavCStride = 34;

struct MmavParams {
    const uint8_t* W;
    int64_t rowbytes;   // bytes of one weight row in global (a multiple of 16)
    int64_t N;
    int K;
    const uint8_t* xq;  // packed Q8_K rows [T][K/256]
    int xrow;           // bytes between activation rows (global)
    int xstride;        // bytes between activation rows in shared memory (padded against bank conflicts)
    int T;
    float* Y;           // [T][N]
    int* err;
    int early_weights;
    int stages;
    int stage_stride;
    int x_bytes;        // shared region: staged activations, then the partials
    int x_bulk;         // 1: the activation rows arrive by one bulk copy (16-byte multiple)
    int wrow;           // stride of a pair of rows in shared memory (padded)
    int chunk;          // inputs per consumer warp (64, 128 or 256)
    int nch;            // chunks (<= 16)
    int32_t* coefs;     // integer-core dump [T][N][ncoef] (dump launches only; zeroed by the caller)
    int ncoef;          // coefficients per row: K/blk * (2 for Q4_K/Q5_K, else 1)
};

// Expert-sorted grouped GEMM on f16 tensor cores (ggq_gmm.cuh): tiles of 64
// weight rows (gate/up: 32 gate + the same 32 up rows) x 128 activation
// columns of one expert; weights decoded once per tile into f16 shared memory,
// activations pre-converted to exact f16 rows in expert-sorted order, every
// operand fetched as 2-D TMA boxes.
constexpr int kGmmBM = 64;
constexpr int kGmmBN = 128;
constexpr int kGmmBK = 64;
constexpr int kGmmThreads = 384;  // 8 consumer warps, 3 decode warps, 1 TMA warp
constexpr int kGmmStages = 6;

struct GmmParams {
    CUtensorMap tm_b;         // f16 activation rows, sorted positions [P][K]: box 64 x 128, 128-byte swizzle
    CUtensorMap tm_dx;        // f32 block scales [P][dx_pitch]: box 4 x 128
    CUtensorMap tm_bs;        // f16 16-group sums [P][K/16]: box 16 x 128
    CUtensorMap tm_w[2][2];   // weight bytes [E*N][rowbytes] of [gate or down, up][Q8_0 span or Q4_K header, Q4_K nibbles]
    int64_t N;                // rows per matrix (I for gate/up, H for down)
    int K;                    // input width (multiple of 256)
    const int* ngroups;
    const int* group_expert;
    const int* group_off;
    const int* group_cnt;
    const int* perm;          // sorted position -> pair
    float* h;                 // gate/up: h [pairs][N]
    float* g_dump;
    float* u_dump;
    float* o;                 // down: o [pairs][N]
    int* err;
    int32_t* coefs[2];        // integer-core dump per matrix [pairs][N][ncoef] (dump launches only)
    int ncoef;                // coefficients per row: K/blk * (2 for Q4_K, else 1)
};

// Launch with the programmatic-dependent-launch attribute (the kernels call
// pdl_wait before touching data of earlier kernels, so this is always safe).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Host launchers (one per kernel family); return the launch error.
cudaError_t launch_stream(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_quantize(int act, const float* x, int64_t T, int64_t K, uint8_t* out, cudaStream_t s);
cudaError_t launch_dequant(int fmt, const uint8_t* blocks, int64_t rows, int64_t K, float* out, cudaStream_t s);
cudaError_t launch_group(int kind, int fmt, const GroupParams& p, int grid, int smem, cudaStream_t s);
// The same kernel also writing its integer core to p.coefs (outputs unchanged).
cudaError_t launch_group_dump(int kind, int fmt, const GroupParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_mmav(int fmt, const MmavParams& p, int grid, int smem, cudaStream_t s);
// The same kernel writing its integer core to p.coefs instead of Y.
cudaError_t launch_mmav_dump(int fmt, const MmavParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_quantize_pitched(const float* x, int64_t rows, int64_t K, uint8_t* out, int64_t pitch,
                                    cudaStream_t s);
cudaError_t launch_route_sorted(const float* logits, const int32_t* ids_in, const float* w_in, const float* X, int T,
                                int E, int k, int H, uint8_t* xq, int64_t x_pitch, int32_t* ids, float* w,
                                int* counts, int* err, cudaStream_t s);
// tel_pairs / tel_calls: optional expert-load telemetry (pairs per expert; calls and distinct experts).
cudaError_t launch_moe_count(const int32_t* ids, int P, int E, unsigned long long* tel_pairs,
                             unsigned long long* tel_calls, cudaStream_t s);
cudaError_t launch_group_plan(const int* counts, int E, int* offsets, int* cursor, int* ngroups, int* group_expert,
                              int* group_off, int* group_cnt, cudaStream_t s, unsigned long long* tel_pairs = nullptr,
                              unsigned long long* tel_calls = nullptr);
cudaError_t launch_scatter(const int32_t* ids, int P, int E, const int* offsets, int* cursor, int* perm,
                           cudaStream_t s);
cudaError_t launch_q8k_to_f16(const uint8_t* q, int64_t pitch, const int* map, int div, int64_t rows, int64_t K,
                              __half* x16, __half* bs16, float* dx, int64_t dx_pitch, cudaStream_t s,
                              bool bf16 = false);
// Tensor maps of one grouped GEMM launch (host encode; 0 or a CUresult).
int gmm_encode(GmmParams& p, int kind, int fmt, const uint8_t* W, const uint8_t* W2, int64_t rowbytes, int64_t wrows,
               const __half* x16, const float* dx, int64_t dx_pitch, const __half* bs16, int64_t P, int K);
cudaError_t launch_gmm(int kind, int fmt, const GmmParams& p, int grid, int smem, cudaStream_t s);
// The same kernel also writing its integer core to p.coefs (outputs unchanged).
cudaError_t launch_gmm_dump(int kind, int fmt, const GmmParams& p, int grid, int smem, cudaStream_t s);
// Row-major 2-D tensor map [dim1][dim0] (rows stride1 bytes apart); 0 or a CUresult.
int encode_tmap_2d(CUtensorMap* m, CUtensorMapDataType type, const void* base, uint64_t dim0, uint64_t dim1,
                   uint64_t stride1, uint32_t box0, uint32_t box1, CUtensorMapSwizzle swz);

// Expert-sorted grouped GEMM on tcgen05 (ggq_gmmtc.cuh), Q8_0 and Q4_K banks: items of 128
// weight rows x 128 activation columns; every matrix of the bank (gate and up
// are separate items) writes its own f32 output rows per pair.
constexpr int kTcThreads = 512;  // 8 epilogue, 6 decode, 1 TMA, 1 MMA warps

struct GmmTcParams {
    CUtensorMap tm_b;     // f16 activation rows, sorted positions [P][K]: box 64 x 128, 128-byte swizzle
    CUtensorMap tm_b32;   // the same rows, box 64 x 32 (items of at most 32 columns)
    CUtensorMap tm_dx;    // f32 block scales [P][dx_pitch]: box 4 x 128
    CUtensorMap tm_bs;    // f16 16-group sums [P][K/16]: box 16 x 128 (Q4_K)
    CUtensorMap tm_w[2];  // weight bytes [E*N][rowbytes]: Q8_0 gate and up (box 80 x 128); Q4_K header (16 x 128) and nibbles (32 x 128)
    int64_t N;            // rows per matrix (multiple of 128)
    int K;                // input width (multiple of 256)
    int nmat;             // matrices per bank (2: gate and up)
    const int* ngroups;
    const int* group_expert;
    const int* group_off;
    const int* group_cnt;
    const int* perm;      // sorted position -> pair
    float* out[2];        // per matrix: [pairs][N]
    int* err;
    int32_t* coefs[2];    // integer-core dump per matrix [pairs][N][ncoef] (dump launches only)
    int ncoef;            // coefficients per row: K/blk * (2 for Q4_K, else 1)
};
int gmmtc_encode(GmmTcParams& p, int fmt, const uint8_t* W, const uint8_t* W2, int64_t rowbytes, int64_t wrows,
                 const __half* x16, const float* dx, int64_t dx_pitch, const __half* bs16, int64_t P, int K);
cudaError_t launch_gmmtc(int fmt, const GmmTcParams& p, int grid, cudaStream_t s);
// The same kernel also writing its integer core to p.coefs (outputs unchanged).
cudaError_t launch_gmmtc_dump(int fmt, const GmmTcParams& p, int grid, cudaStream_t s);
// h = silu(g) * u row by row (optionally written to h_out), quantized to Q8_K rows at out + r * pitch.
cudaError_t launch_quantize_silu(const float* g, const float* u, int64_t rows, int64_t K, uint8_t* out, int64_t pitch,
                                 float* h_out, cudaStream_t s);
int gmm_supported(int fmt);
int gmm_smem_bytes();
cudaError_t launch_combine(const float* o, const float* w, int T, int k, int64_t H, float* Y, cudaStream_t s);

}  // namespace ggq

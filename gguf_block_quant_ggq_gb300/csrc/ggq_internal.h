// ggq_internal.h -- host/device shared declarations inside libggq (not part of the ABI).
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

namespace ggq {

// Streaming-kernel geometry: eight consumer warps + one producer warp per CTA,
// two weight rows per consumer warp per stage (16 rows; gate/up: 8 row pairs).
constexpr int kConsumerWarps = 8;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTileRows = 16;
constexpr int kMaxStages = 8;
constexpr int kSmemLimit = 232448;  // 227 KB opt-in dynamic shared memory per CTA
constexpr int kMaxDevices = 64;     // device ordinals with per-device launch state

// Decode-size MoE plan (T <= 8, so at most 64 (token, slot) pairs).
constexpr int kPlanMaxPairs = 64;
constexpr int kPlanMaxTokens = 8;
struct MoePlan {
    int D;                                  // distinct experts selected
    int err;                                // nonzero: an expert id was out of range
    int expert[kPlanMaxPairs];              // expert id of distinct slot u
    int npairs[kPlanMaxPairs];              // pairs routed to it
    int pair[kPlanMaxPairs][kPlanMaxTokens];   // pair index p = t*k + j
    int token[kPlanMaxPairs][kPlanMaxTokens];  // token of that pair
    float wt[kPlanMaxTokens * 8];           // routing weight of pair p
};

enum Kind : int { KIND_GEMV = 0, KIND_DUMP = 1, KIND_GATEUP = 2, KIND_DOWN = 3 };

struct StreamParams {
    const uint8_t* W;   // weights: GEMV matrix, gate bank, or down bank
    const uint8_t* W2;  // up bank (gate/up only)
    int64_t rowbytes;   // bytes of one weight row
    int64_t N;          // GEMV rows; MoE rows per expert (I for gate/up, H for down)
    int K;              // input width
    const uint8_t* xq;  // packed activations: GEMV [T][K/blk]; gate/up x^ [T][H/256]; down h^ [T*k][I/256]
    int xrows;          // activation rows staged in shared memory
    int T;
    int top_k;
    float* Y;           // GEMV out [T][N]; down: y [T][H]
    int32_t* coefs;     // block-dot dump [T][N][K/blk*c]
    const MoePlan* plan;
    float* h;           // [T*k][I] fp32 (gate/up output)
    float* g_dump;      // optional [T*k][I]
    float* u_dump;      // optional [T*k][I]
    uint8_t* hq;        // [T*k][I/256] Q8_K (gate/up quantizes h into it)
    float* o;           // [T*k][H] down outputs
    int* counters;      // last-CTA counters (self-resetting)
    int* err;           // device error word
    int stages;
    int stage_stride;   // bytes per ring slot (multiple of 128)
    int x_bytes;        // bytes of the staged-activation region
};

// Bytes of the structure-of-arrays activation region for `rows` rows of width K.
inline int x_region_bytes(int rows, int K, bool q81) {
    const size_t q = static_cast<size_t>(rows) * K;
    const size_t d = static_cast<size_t>(rows) * (K / (q81 ? 32 : 256)) * 4;
    const size_t extra = q81 ? static_cast<size_t>(rows) * (K / 32) * 4 : static_cast<size_t>(rows) * (K / 16) * 2;
    auto up = [](size_t v) { return (v + 127) / 128 * 128; };
    return static_cast<int>(up(q) + up(d) + up(extra));
}

// Host launchers (one per kernel family); return the launch error.
cudaError_t launch_stream(int kind, int fmt, int nt, const StreamParams& p, int grid, int smem, cudaStream_t s);
cudaError_t launch_quantize(int act, const float* x, int64_t T, int64_t K, uint8_t* out, cudaStream_t s);
cudaError_t launch_dequant(int fmt, const uint8_t* blocks, int64_t rows, int64_t K, float* out, cudaStream_t s);
cudaError_t launch_moe_route(const float* logits, const int32_t* ids_in, const float* w_in, const float* X, int T,
                             int E, int k, int H, uint8_t* xq, MoePlan* plan, int32_t* ids_out, float* w_out,
                             int* err, cudaStream_t s);

}  // namespace ggq

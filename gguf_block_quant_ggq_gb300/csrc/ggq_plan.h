// ggq_plan.h -- shared-memory plans of the weight-streaming GEMV kernel
// (k_stream), used by the pooled and the allocation-free entry points alike.
#pragma once
#include <stdint.h>

#include "ggq_device.cuh"
#include "ggq_internal.h"

namespace ggq {

// Shared-memory plan of one streaming launch.
struct StreamShape {
    int stages, stride, x_bytes, smem;
};

inline bool plan_stream(int64_t stage_bytes, int xrows, int K, bool q81, StreamShape* s, int extra = 1024) {
    s->stride = static_cast<int>((static_cast<size_t>(stage_bytes) + 16 + 127) / 128 * 128);
    s->x_bytes = x_region_bytes(xrows, K, q81);
    const int fixed = s->x_bytes + 2 * kMaxStages * 8 + extra;
    if (fixed + s->stride > kSmemLimit) return false;
    s->stages = (kSmemLimit - fixed) / s->stride;
    if (s->stages > kMaxStages) s->stages = kMaxStages;
    if (s->stages > kWholeRowStages) s->stages = kWholeRowStages;
    s->smem = s->stages * s->stride + fixed;
    return true;
}

// The row chunk of format f that a chunked stage is a whole number of: it
// starts on a unit (or superblock) boundary and, where the rows are 16-byte
// multiples, is one too (then every chunk is a bulk copy of its own).
// 64-weight units and bytes.
inline void chunk_granule(int f, int64_t rowbytes, int* units, int* bytes) {
    switch (f) {
    case F_Q4_0: *units = 4, *bytes = 144; break;   // 8 blocks of 18 B
    case F_Q8_0: *units = 4, *bytes = 272; break;   // 8 blocks of 34 B
    case F_MXFP4: *units = 8, *bytes = 272; break;  // 16 blocks of 17 B
    case F_Q4_K: *units = 4, *bytes = 144; break;   // one superblock
    case F_Q5_K: *units = 4, *bytes = 176; break;   // one superblock
    case F_Q2_K:                                    // superblocks of 84 B: four are 336 B
        if (rowbytes % 16 == 0) *units = 16, *bytes = 336;
        else *units = 4, *bytes = 84;
        break;
    case F_Q3_K:                                    // superblocks of 110 B: eight are 880 B
        if (rowbytes % 16 == 0) *units = 32, *bytes = 880;
        else *units = 4, *bytes = 110;
        break;
    default:                                        // Q6_K: superblocks of 210 B
        if (rowbytes % 16 == 0) *units = 32, *bytes = 1680;
        else *units = 4, *bytes = 210;
        break;
    }
}

// Plan of the streaming GEMV for rows too long for whole-row stages: the
// activations stay whole in shared memory and each stage holds one chunk of
// every row of a 16-row tile (about six stages in the ring, at least two).
// Rows that are not 16-byte multiples get 16 spare bytes per row slot: their
// chunks land at the same offset modulo 16 as in global memory.  False if two
// stages do not fit.
inline bool plan_stream_chunked(int f, int64_t rowbytes, int xrows, int K, bool q81, StreamShape* s,
                                int* chunk_units, int* chunk_bytes, int* row_slot, bool small_granule = false) {
    int gu = 0, gb = 0;
    chunk_granule(f, rowbytes, &gu, &gb);
    if (small_granule && f == F_Q6_K) gu = 4, gb = 210;  // one superblock: unaligned chunks
    s->x_bytes = x_region_bytes(xrows, K, q81);
    const int fixed = s->x_bytes + 2 * kMaxStages * 8 + 1024;
    const int avail = kSmemLimit - fixed;
    if (avail <= 0) return false;
    // about six stages, but at least 32 units per chunk (one for every lane of
    // a row's warp) while two stages still fit
    const int g_lanes = (32 + gu - 1) / gu;
    int g = avail / 6 / kTileRows / gb;
    if (g < g_lanes) g = g_lanes;
    if (static_cast<int64_t>(g) * gb > rowbytes) g = static_cast<int>((rowbytes + gb - 1) / gb);
    const auto slot_of = [&](int gg) {
        const int cb = gg * gb;
        return (rowbytes % 16 == 0 && cb % 16 == 0) ? cb : (cb + 15) / 16 * 16 + 16;
    };
    const auto stride_of = [&](int gg) {
        return static_cast<int>((static_cast<size_t>(kTileRows) * slot_of(gg) + 16 + 127) / 128 * 128);
    };
    while (g > 1 && avail / stride_of(g) < 2) --g;
    const int cb = g * gb;
    const int slot = slot_of(g);
    s->stride = stride_of(g);
    s->stages = avail / s->stride;
    if (s->stages < 2) {
        if (f == F_Q6_K && !small_granule)
            return plan_stream_chunked(f, rowbytes, xrows, K, q81, s, chunk_units, chunk_bytes, row_slot, true);
        return false;
    }
    if (s->stages > kMaxStages) s->stages = kMaxStages;
    const int cap = kInFlightBytes / s->stride;
    if (s->stages > 2 && s->stages > cap) s->stages = cap > 2 ? cap : 2;
    s->smem = s->stages * s->stride + fixed;
    *chunk_units = g * gu;
    *chunk_bytes = cb;
    *row_slot = slot;
    return true;
}

// The streaming GEMV's plan for T tokens: whole-row stages when two fit; else
// row chunks with at least a unit per lane; when the T tokens' staged
// activations leave no room for that, kSplit: run the tokens as two groups
// (T/2 and T - T/2), each planned the same way.  A single whole-row stage is
// the last resort of one token.
enum class StreamPlan { kNone, kRun, kSplit };

inline StreamPlan plan_gemv_stream(int f, int64_t rowbytes, int T, int K, bool q81, StreamShape* sh,
                                   int* chunk_units, int* chunk_bytes, int* row_slot) {
    *chunk_units = *chunk_bytes = *row_slot = 0;
    const bool whole = plan_stream(kTileRows * rowbytes, T, K, q81, sh);
    if (whole && sh->stages >= 2) return StreamPlan::kRun;
    StreamShape ch;
    int cu = 0, cb = 0, rs = 0;
    const bool chunked = plan_stream_chunked(f, rowbytes, T, K, q81, &ch, &cu, &cb, &rs);
    if (T > 1 && (!chunked || cu < 32)) return StreamPlan::kSplit;
    if (chunked) {
        *sh = ch;
        *chunk_units = cu;
        *chunk_bytes = cb;
        *row_slot = rs;
        return StreamPlan::kRun;
    }
    return whole ? StreamPlan::kRun : StreamPlan::kNone;
}

}  // namespace ggq

// ggq_mmav.cuh -- the decode GEMV at 3-8 tokens on the tensor cores.
//
// y[t][n] = sum over blocks of (weight scale) * (activation scale) * (integer
// block dot), as in the keep-quant matmul of vllm.cpp PR #523 "grouped +
// non-grouped keep-quant expert GEMM" (What changed: DotQ8_0/DotQ4K/DotQ5K/
// DotQ6K superblock dots).  One mma covers 16 rows x 8 token columns:
//   * Q4_K, Q5_K, Q6_K: mma.sync m16n8k16 with f16 operands and f32
//     accumulation.  Weight codes are placed in the mantissa of 1024.0 (one
//     LOP3 per pair of codes) and int8 activations are exact in f16, so every
//     product is exact; C starts at -1024 (Q6_K: -1056) times the activation
//     sum of the block, which leaves the exact integer dot of each sub-block
//     (Q6_K: each 16-group, whose own scale it needs) in D.  Q4_K and Q5_K
//     fold the 6-bit sub-block scale into the operand instead (sc * q is an
//     exact f16 integer) and accumulate in 128-wide (Q4_K) or 64-wide (Q5_K)
//     chains, |partial| <= 128 * 945 * 127 and 64 * 1953 * 127, both below
//     2^24, so every chain holds its exact integer; the chains meet in the f32
//     epilogue.  Block scales are applied in f32; the Q4_K/Q5_K mins term is
//     one more f16 product.  On this part the f16 mma runs at four times the
//     rate of the int8 one.  (Applying the sub-block scale in f32 after
//     per-sub-block mma pairs instead was measured slower.)
//   * Q8_0, MXFP4: mma.sync m16n8k32 on int8 (one 32-block per mma).
//
// Layout on the SM:
//   * one CTA per SM; a producer warp copies each 16-row tile of W into a ring
//     of shared-memory stages, one bulk copy per pair of rows (eight lanes
//     issue the eight copies of a tile at once), pairs padded so that the
//     eight even rows fall on distinct bank quads; mma row g is tile row 2g and
//     mma row g + 8 is tile row 2g + 1, so every fragment load is conflict-free;
//   * sixteen consumer warps split K into sixteen chunks of 64, 128 or 256
//     inputs.  A warp's chunk never changes, so its activation fragments (the
//     mma B operand), activation scales and per-block sums are built once, from
//     the activation rows that one bulk copy brings into shared memory, and
//     kept in registers;
//   * per tile each warp produces a 16 x 8 partial of its chunk; partials meet
//     in a double-buffered shared array behind one barrier per tile.
// Every wait is bounded; on timeout the kernel records an error word, drains
// its copies and returns.
#pragma once
#include "ggq_device.cuh"
#include "ggq_internal.h"

#include <atomic>

namespace ggq {

constexpr int kRedStride = 130;  // floats per warp in the partials buffer

__device__ __forceinline__ void mmav_start_arrive() { asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory"); }
__device__ __forceinline__ void mmav_start_sync() { asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory"); }

__device__ __forceinline__ void mmav_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); }

// Bounded wait that backs off between probes (a few tens of ns), leaving the
// issue slots of a busy SM to the warps that have work.
__device__ __forceinline__ bool mbar_wait_backoff(uint64_t* bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(32);
        if (mbar_test(bar, parity)) return true;
        if (clock64() - t0 > (1ll << 32)) return false;
    }
}

__device__ __forceinline__ void mma_k32_s8(int* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                           uint32_t b1, int c0, int c1) {
    asm(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%10,%11};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "r"(c0), "r"(c1));
}

// The same, accumulating into d (exact int32 sums).
__device__ __forceinline__ void mma_k32_s8_acc(int* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// (a & mask) | c in one LOP3 (mask an immediate, c a register).
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}

// Byte i of w, zero-extended / sign-extended (i a compile-time constant after unrolling).
__device__ __forceinline__ int byte_u(uint32_t w, int i) { return static_cast<int>(prmt(w, 0u, 0x4440u | i)); }
__device__ __forceinline__ int byte_s(uint32_t w, int i) {
    const uint32_t s = 0x8u | static_cast<uint32_t>(i);
    return static_cast<int>(prmt(w, 0u, (s << 12) | (s << 8) | (s << 4) | static_cast<uint32_t>(i)));
}

// m16n8k16 with f16 operands and f32 accumulation.  Used with integer-valued
// operands only (weight codes and int8 activations are exact in f16); every
// product is exact and so is every partial sum below 2^24.
__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Four signed bytes (x0 x1 x2 x3) -> f16 pairs (x0, x2) and (x1, x3):
// 1024 + (x + 128) built in the mantissa, then 1152 subtracted (exact).
__device__ __forceinline__ void s8x4_to_f16(uint32_t w, uint32_t& p02, uint32_t& p13) {
    const uint32_t u = w ^ 0x80808080u;
    const __half2 off = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));  // 1152
    const uint32_t a = prmt(u, 0u, 0x4240u) | 0x64006400u, b = prmt(u, 0u, 0x4341u) | 0x64006400u;
    const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), off);
    const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&b), off);
    p02 = *reinterpret_cast<const uint32_t*>(&ha);
    p13 = *reinterpret_cast<const uint32_t*>(&hb);
}

__device__ __forceinline__ uint32_t f16pair(float a, float b) {
    const __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// One warp's register-resident activations for its chunk.  Thread (g, t) of
// the mma holds the B fragment of token g and the scales and sums of its two
// accumulator columns c0 = 2t, c1 = 2t + 1.
struct MmaX {
    uint32_t b[32];  // int8 path: b[2i], b[2i+1] = sub-block i (Q6_K: b[j] = 16-group j);
                     // f16 path (Q4_K): b[4i + 2s], b[4i + 2s + 1] = sub-block i, 16-step s
    int s[16];       // Q4_K/Q5_K: sum q of sub-block i (s[2i]: c0, s[2i+1]: c1); MXFP4: 12x that;
                     // Q6_K: 16-group sums of c0 (low half) and c1 (high half)
    uint32_t bm[2];  // f16 path: B of the mins product (16-group sums of token g)
    float dx0, dx1;  // Q8_K scale of the chunk's superblock, columns c0 and c1
};

// Build a warp's fragments from the packed Q8_K rows staged in shared memory
// (xs: row c at xs + c * xrow).
template <int F>
__device__ __forceinline__ void mmav_load_x(saddr xs, int xrow, int T, int chunk, int e0, int g, int t, MmaX& X,
                                            float* cs) {
    const int sb = e0 >> 8, off = e0 & 255;
    const int c0 = 2 * t, c1 = 2 * t + 1;
    const saddr rb = xs + static_cast<uint32_t>(g * xrow + 292 * sb);  // B: token g
    const saddr r0 = xs + static_cast<uint32_t>(c0 * xrow + 292 * sb);  // column c0
    const saddr r1 = xs + static_cast<uint32_t>(c1 * xrow + 292 * sb);
    const bool vg = g < T, v0 = c0 < T, v1 = c1 < T;
#pragma unroll
    for (int i = 0; i < 32; ++i) X.b[i] = 0u;
#pragma unroll
    for (int i = 0; i < 16; ++i) X.s[i] = 0;
    X.bm[0] = X.bm[1] = 0u;
    X.dx0 = v0 ? ld_f32(r0) : 0.0f;
    X.dx1 = v1 ? ld_f32(r1) : 0.0f;
    if constexpr (F == F_Q6_K) {
        // f16 fragments of each 16-group (elements 4t, 4t+2 | 4t+1, 4t+3 of the
        // group, as for Q4_K); C = -1056 (groups 0, 1 of a 128-element half: the
        // codes enter as 1024 + code) or -1536 (groups 2, 3: 1024 + 16 code) times
        // the sum of the group's activations, the weights being code - 32
        // the start values of this thread's column pair t are shared by the
        // warp's eight g-lanes: lane (g, t) computes those of groups g and g + 8
        // (all lanes busy; the barrier after this function orders them)
        uint32_t xw[16];
        int bsv[2][2];
#pragma unroll
        for (int j = 0; j < 16; ++j) xw[j] = 16 * j < chunk && vg ? ld_s32(rb + 4 + off + 16 * j + 4 * t) : 0u;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int e = off + 16 * (g + 8 * h);
            const bool in = 16 * (g + 8 * h) < chunk;
            bsv[h][0] = in && v0 ? ld_s16(r0 + 260 + 2 * (e >> 4)) : 0;
            bsv[h][1] = in && v1 ? ld_s16(r1 + 260 + 2 * (e >> 4)) : 0;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j)
            if (16 * j < chunk && vg) s8x4_to_f16(xw[j], X.b[2 * j], X.b[2 * j + 1]);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int j = g + 8 * h;
            if (16 * j < chunk) {
                const float cb = ((off + 16 * j) & 64) ? -1536.0f : -1056.0f;
                *reinterpret_cast<float2*>(cs + 2 * j) =
                    make_float2(cb * static_cast<float>(bsv[h][0]), cb * static_cast<float>(bsv[h][1]));
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (32 * i < chunk) {
                const int e = off + 32 * i;
                uint32_t lo = 0u, hi = 0u;
                if (vg) {
                    lo = ld_s32(rb + 4 + e + 4 * t);
                    hi = ld_s32(rb + 4 + e + 16 + 4 * t);
                }
                if constexpr (F == F_MXFP4) {
                    // the E2M1 lookup yields elements (j, j+16, j+1, j+17 | j+2, j+18, j+3, j+19):
                    // the activation fragment takes the same order
                    X.b[2 * i] = prmt(lo, hi, 0x5140u);
                    X.b[2 * i + 1] = prmt(lo, hi, 0x7362u);
                } else if constexpr (F == F_Q4_K || F == F_Q5_K || F == F_Q3_K) {
                    // f16 fragments; a thread's k slots (2t, 2t+1 | 2t+8, 2t+9) of a
                    // 16-step hold elements (4t, 4t+2 | 4t+1, 4t+3), matching the
                    // weight-side unpack of one 32-bit word
                    s8x4_to_f16(lo, X.b[4 * i], X.b[4 * i + 1]);
                    s8x4_to_f16(hi, X.b[4 * i + 2], X.b[4 * i + 3]);
                } else {
                    X.b[2 * i] = lo;
                    X.b[2 * i + 1] = hi;
                }
                if constexpr (F != F_Q8_0 && F != F_Q2_K && F != F_Q3_K) {
                    const uint32_t w0 = v0 ? ld_s32(r0 + 260 + 2 * (e >> 4)) : 0u;  // bsums 2js, 2js+1
                    const uint32_t w1 = v1 ? ld_s32(r1 + 260 + 2 * (e >> 4)) : 0u;
                    const int s0 = static_cast<int>(static_cast<int16_t>(w0 & 0xFFFFu)) +
                                   static_cast<int>(static_cast<int16_t>(w0 >> 16));
                    const int s1 = static_cast<int>(static_cast<int16_t>(w1 & 0xFFFFu)) +
                                   static_cast<int>(static_cast<int16_t>(w1 >> 16));
                    const int m = F == F_MXFP4 ? 12 : 1;
                    X.s[2 * i] = m * s0;
                    X.s[2 * i + 1] = m * s1;
                }
            }
        }
        if constexpr (F == F_Q4_K || F == F_Q5_K || F == F_Q2_K) {
            // mins product: k slot q <-> 16-group q of the chunk (Q4_K/Q5_K: sub-block q/2)
            if (vg) {
                const int q0 = 2 * t, q1 = 2 * t + 8;  // groups (q0, q0+1) and (q1, q1+1)
                const int ng = chunk >> 4;
                const int a = q0 < ng ? ld_s16(rb + 260 + 2 * ((off >> 4) + q0)) : 0;
                const int b = q0 < ng ? ld_s16(rb + 260 + 2 * ((off >> 4) + q0 + 1)) : 0;
                const int c = q1 < ng ? ld_s16(rb + 260 + 2 * ((off >> 4) + q1)) : 0;
                const int d = q1 < ng ? ld_s16(rb + 260 + 2 * ((off >> 4) + q1 + 1)) : 0;
                X.bm[0] = f16pair(static_cast<float>(a), static_cast<float>(b));
                X.bm[1] = f16pair(static_cast<float>(c), static_cast<float>(d));
            }
        }
    }
}

// Scales (or mins) of sub-blocks js0 .. js0+7 of one Q4_K/Q5_K row as bytes of
// (lo, hi): the 6-bit packed fields of the superblock header words a0..a2.
__device__ __forceinline__ void k4_scale_words(uint32_t a0, uint32_t a1, uint32_t a2, int js0, uint32_t& sl,
                                               uint32_t& sh, uint32_t& ml, uint32_t& mh) {
    const uint32_t sc_lo = a0 & 0x3F3F3F3Fu, m_lo = a1 & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (a2 & 0x0F0F0F0Fu) | ((a0 >> 2) & 0x30303030u);
    const uint32_t m_hi = ((a2 >> 4) & 0x0F0F0F0Fu) | ((a1 >> 2) & 0x30303030u);
    if (js0 == 0) {
        sl = sc_lo, sh = sc_hi, ml = m_lo, mh = m_hi;
    } else if (js0 < 4) {
        sl = __funnelshift_r(sc_lo, sc_hi, 8 * js0), sh = 0u;
        ml = __funnelshift_r(m_lo, m_hi, 8 * js0), mh = 0u;
    } else {
        sl = sc_hi >> (8 * (js0 - 4)), sh = 0u;
        ml = m_hi >> (8 * (js0 - 4)), mh = 0u;
    }
}

// Integer-core dump of one thread's four outputs: coefficient rows of (row r0,
// column c0), (r0, c1), (r1, c0), (r1, c1) in the [T][N][K/blk * c] array
// (null where the output does not exist).  Per-superblock coefficients may be
// split across warps (chunks below 256 inputs) and are added atomically into
// a zeroed array; per-32-block coefficients have one owner and are stored.
struct MmavDump {
    int32_t* q[4];
};

__device__ __forceinline__ void dump_add(int32_t* row, int idx, int v) {
    if (row) atomicAdd(row + idx, v);
}
__device__ __forceinline__ void dump_put(int32_t* row, int idx, int v) {
    if (row) row[idx] = v;
}

// One 32-bit word of a Q6_K superblock at a byte offset that is a multiple of
// 4 from the superblock start; ODD: the superblock itself starts 2 bytes after
// a word boundary, so the word is the middle of two aligned ones.
template <bool ODD>
__device__ __forceinline__ uint32_t q6_word(saddr a) {
    if constexpr (ODD) return prmt(ld_s32(a - 2u), ld_s32(a + 2u), 0x5432u);
    else return ld_s32(a);
}

// Q6_K part of a chunk (one or two 128-element halves of superblock b0 / b1 for
// rows g and g+8).  Element 128h + 32g6 + l: low 4 bits in ql[64h + 32(g6&1) + l]
// (nibble g6>>1), high 2 bits in qh[32h + l] (bits 2g6), scale of 16-group
// (128h + 32g6 + l)/16.  f16 operands without moving any nibble: groups g6 = 0, 1
// read 1024 + code (low nibble, the two high bits placed at bits 4-5), groups
// g6 = 2, 3 read 1024 + 16 code (high nibble in place, the two bits at 8-9;
// 16 code <= 1008, still an exact f16 integer).  The start value C removes 1056
// or 1536 times the group's activation sum, so D is the exact dot of (code - 32)
// and x, times 16 for groups 2 and 3; one m16n8k16 per 16-group (each group has
// its own int8 scale), scaled in f32.
template <bool ODD, bool DUMP>
__device__ __forceinline__ void mmav_q6k(saddr b0, saddr b1, int e0, int chunk, const MmaX& X, saddr cs, int t,
                                         float* acc, const MmavDump& dz) {
    const int h0 = (e0 & 255) >> 7;
    uint32_t sw0[4], sw1[4];  // int8 scales of the chunk's 16-groups, four per word
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        sw0[k] = q6_word<ODD>(b0 + 192u + 4u * k);
        sw1[k] = q6_word<ODD>(b1 + 192u + 4u * k);
    }
    if (h0) {  // second half only: its eight scales are words 2 and 3
        sw0[0] = sw0[2], sw0[1] = sw0[3], sw1[0] = sw1[2], sw1[1] = sw1[3];
    }
    uint32_t Mr = 0x64006400u;
    asm("" : "+r"(Mr));
    float a[4] = {0.0f, 0.0f, 0.0f, 0.0f}, ah[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // groups 0, 1 | 2, 3 (16x)
    int ia[4] = {0, 0, 0, 0};  // dump: sum_j sc_j S_j in int32
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
        if (128 * hh < chunk) {
            const uint32_t h = static_cast<uint32_t>(h0 + hh);
#pragma unroll
            for (int lh = 0; lh < 2; ++lh) {
                const uint32_t l = 16u * lh + 4u * t;
                uint32_t A[4][4];  // [g6][row g even bytes, row g+8 even, row g odd, row g+8 odd]
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    const saddr b = r ? b1 : b0;
                    const uint32_t ql0 = q6_word<ODD>(b + 64u * h + l), ql1 = q6_word<ODD>(b + 64u * h + 32u + l);
                    const uint32_t qh = q6_word<ODD>(b + 128u + 32u * h + l);
                    const uint32_t ql0o = ql0 >> 8, ql1o = ql1 >> 8;  // bytes 1, 3 in the even positions
                    // high bits of g6 = 0 / 2 at 4-5 / 8-9 (<< 4), of g6 = 1 / 3 likewise (<< 2);
                    // the odd bytes' bits are 8 further up (>> 4, >> 6)
                    const uint32_t h4 = qh << 4, h4o = qh >> 4, h2 = qh << 2, h2o = qh >> 6;
                    A[0][r] = and_or<0x00300030u>(h4, and_or<0x000F000Fu>(ql0, Mr));
                    A[0][2 + r] = and_or<0x00300030u>(h4o, and_or<0x000F000Fu>(ql0o, Mr));
                    A[1][r] = and_or<0x00300030u>(h2, and_or<0x000F000Fu>(ql1, Mr));
                    A[1][2 + r] = and_or<0x00300030u>(h2o, and_or<0x000F000Fu>(ql1o, Mr));
                    A[2][r] = and_or<0x03000300u>(h4, and_or<0x00F000F0u>(ql0, Mr));
                    A[2][2 + r] = and_or<0x03000300u>(h4o, and_or<0x00F000F0u>(ql0o, Mr));
                    A[3][r] = and_or<0x03000300u>(h2, and_or<0x00F000F0u>(ql1, Mr));
                    A[3][2 + r] = and_or<0x03000300u>(h2o, and_or<0x00F000F0u>(ql1o, Mr));
                }
#pragma unroll
                for (int g6 = 0; g6 < 4; ++g6) {
                    const int jl = 8 * hh + 2 * g6 + lh;  // 16-group within the chunk
                    const float2 c = ld_f32x2(cs + 8u * jl);
                    float D[4] = {c.x, c.y, c.x, c.y};
                    mma_f16(D, A[g6][0], A[g6][1], A[g6][2], A[g6][3], X.b[2 * jl], X.b[2 * jl + 1]);
                    const int i0 = byte_s(sw0[jl >> 2], jl & 3), i1 = byte_s(sw1[jl >> 2], jl & 3);
                    const float sc0 = static_cast<float>(i0), sc1 = static_cast<float>(i1);
                    float* const dst = g6 < 2 ? a : ah;
                    dst[0] += sc0 * D[0];
                    dst[1] += sc0 * D[1];
                    dst[2] += sc1 * D[2];
                    dst[3] += sc1 * D[3];
                    if constexpr (DUMP) {
                        const int sh = g6 < 2 ? 0 : 4;  // D of groups 2, 3 is 16 times the dot (exact)
                        ia[0] += i0 * (__float2int_rn(D[0]) >> sh);
                        ia[1] += i0 * (__float2int_rn(D[1]) >> sh);
                        ia[2] += i1 * (__float2int_rn(D[2]) >> sh);
                        ia[3] += i1 * (__float2int_rn(D[3]) >> sh);
                    }
                }
            }
        }
    }
    if constexpr (DUMP) {
        const int sb = e0 >> 8;
#pragma unroll
        for (int q = 0; q < 4; ++q) dump_add(dz.q[q], sb, ia[q]);
    }
    const float d0 = ld_h(b0 + 208), d1 = ld_h(b1 + 208);
    acc[0] = fmaf(0.0625f, ah[0], a[0]) * (X.dx0 * d0);
    acc[1] = fmaf(0.0625f, ah[1], a[1]) * (X.dx1 * d0);
    acc[2] = fmaf(0.0625f, ah[2], a[2]) * (X.dx0 * d1);
    acc[3] = fmaf(0.0625f, ah[3], a[3]) * (X.dx1 * d1);
}

// 16 x 8 partial of one chunk: rows (g, g+8) at r0/r1, columns (2t, 2t+1).
template <int F, bool DUMP, int CH>
__device__ __forceinline__ void mmav_chunk(saddr r0, saddr r1, int e0, int chunk_rt, const MmaX& X, saddr cs, int t,
                                           float* acc, const MmavDump& dz) {
    const int chunk = CH > 0 ? CH : chunk_rt;  // inputs of the chunk (compile-time for the common widths)
    const int sb = e0 >> 8;
    if constexpr (F == F_Q4_K || F == F_Q5_K) {
        // f16 operands: a code q placed in the mantissa of 1024.0 reads 1024 + q
        // (low nibble; Q5_K adds its fifth bit at 16) or 1024 + 16q (high nibble
        // masked in place; fifth bit at 256).  One HFMA2 per operand word applies
        // the 6-bit sub-block scale and removes the 1024, leaving 16 q sc 2^-24:
        // the scale enters as the f16 whose bits are the scale byte (sc 2^-24, a
        // subnormal; one PRMT) for high nibbles, shifted up by 4 bits (16 sc
        // 2^-24) for low ones.  16 q sc < 2^15 has at most 11 significant bits,
        // so the operand is exact (subnormal below 2^-14), each mma adds exact
        // products and the chains hold exact multiples of 2^-20; the epilogue's
        // weight scale takes the factor 2^20 back
        constexpr uint32_t SB = F == F_Q4_K ? 144u : 176u;
        constexpr uint32_t QS = F == F_Q4_K ? 16u : 48u;
        const int js0 = CH == 256 ? 0 : (e0 & 255) >> 5;  // 256-input chunks start at a superblock
        const saddr b0 = r0 + SB * sb, b1 = r1 + SB * sb;
        const uint4 h0 = ld_s128(b0), h1 = ld_s128(b1);
        uint32_t s0l, s0h, m0l, m0h, s1l, s1h, m1l, m1h;
        k4_scale_words(h0.y, h0.z, h0.w, js0, s0l, s0h, m0l, m0h);
        k4_scale_words(h1.y, h1.z, h1.w, js0, s1l, s1h, m1l, m1h);
        uint32_t Mr = 0x64006400u;  // the magic exponent in a register: one LOP3 per operand word
        asm("" : "+r"(Mr));
        // (v, v) as f16 for byte idx of w (v <= 63)
        const auto pair = [&](uint32_t w, int idx) -> __half2 {
            const uint32_t u = and_or<0x00FF00FFu>(prmt(w, 0u, 0x4040u | static_cast<uint32_t>(idx) |
                                                                   (static_cast<uint32_t>(idx) << 8)), Mr);
            return __hsub2(*reinterpret_cast<const __half2*>(&u),
                           __halves2half2(__ushort_as_half(0x6400u), __ushort_as_half(0x6400u)));
        };
        // (v 2^-24, v 2^-24) as f16 bits for byte idx of w: the byte itself in each half
        const auto spair = [](uint32_t w, int idx) -> uint32_t {
            return prmt(w, 0u, 0x4040u | static_cast<uint32_t>(idx) | (static_cast<uint32_t>(idx) << 8));
        };
        const auto as_u = [](__half2 h) -> uint32_t { return *reinterpret_cast<const uint32_t*>(&h); };
        const auto fma2 = [&](uint32_t a, __half2 m, __half2 c) -> uint32_t {
            return as_u(__hfma2(*reinterpret_cast<const __half2*>(&a), m, c));
        };
        // mins: sum over sub-blocks of m_j * (sum of the activations of j), one
        // f16 product with k slot q <-> 16-group q (sub-block q/2) of the chunk
        float DM[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_f16(DM, as_u(pair(m0l, t)), as_u(pair(m1l, t)), as_u(pair(m0h, t)), as_u(pair(m1h, t)), X.bm[0],
                X.bm[1]);
        uint32_t qh0a = 0u, qh0b = 0u, qh1a = 0u, qh1b = 0u;
        if constexpr (F == F_Q5_K) {  // high bits of elements 4t.. and 16+4t.., bit js of each byte
            qh0a = ld_s32(b0 + 16 + 4 * t) >> js0;
            qh0b = ld_s32(b0 + 32 + 4 * t) >> js0;
            qh1a = ld_s32(b1 + 16 + 4 * t) >> js0;
            qh1b = ld_s32(b1 + 32 + 4 * t) >> js0;
        }
        const __half2 k1024 = __halves2half2(__ushort_as_half(0xE400u), __ushort_as_half(0xE400u));  // -1024
        // chain ci of i-step i: 64-wide (Q5_K) or 128-wide (Q4_K) runs of the chunk
        constexpr int kChains = F == F_Q5_K ? 4 : 2;
        float Dc[kChains][4];
#pragma unroll
        for (int ci = 0; ci < kChains; ++ci) Dc[ci][0] = Dc[ci][1] = Dc[ci][2] = Dc[ci][3] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; i += 2) {
            float* const D = Dc[F == F_Q5_K ? i / 2 : i / 4];
            if (32 * i < chunk) {
                const uint32_t q = QS + 32u * static_cast<uint32_t>((js0 + i) >> 1) + 4u * t;
                const uint32_t w00 = ld_s32(b0 + q), w01 = ld_s32(b0 + q + 16);  // row g: bytes 4t.. and 16+4t..
                const uint32_t w10 = ld_s32(b1 + q), w11 = ld_s32(b1 + q + 16);  // row g+8
                const uint32_t v00 = w00 >> 8, v01 = w01 >> 8, v10 = w10 >> 8, v11 = w11 >> 8;
                // operand words: index k -> row (k & 1), k slots (k >> 1) & 1, 16-step k >> 2
                uint32_t L[8] = {and_or<0x000F000Fu>(w00, Mr), and_or<0x000F000Fu>(w10, Mr), and_or<0x000F000Fu>(v00, Mr),
                                 and_or<0x000F000Fu>(v10, Mr), and_or<0x000F000Fu>(w01, Mr), and_or<0x000F000Fu>(w11, Mr),
                                 and_or<0x000F000Fu>(v01, Mr), and_or<0x000F000Fu>(v11, Mr)};
                uint32_t H[8] = {and_or<0x00F000F0u>(w00, Mr), and_or<0x00F000F0u>(w10, Mr), and_or<0x00F000F0u>(v00, Mr),
                                 and_or<0x00F000F0u>(v10, Mr), and_or<0x00F000F0u>(w01, Mr), and_or<0x00F000F0u>(w11, Mr),
                                 and_or<0x00F000F0u>(v01, Mr), and_or<0x00F000F0u>(v11, Mr)};
                if constexpr (F == F_Q5_K) {
                    // fifth bit of sub-block js0 + i (low) at bit 4 and of js0 + i + 1 (high) at bit 8
                    // of each half; the qh words were shifted down by js0
                    const uint32_t hq[4] = {qh0a, qh1a, qh0b, qh1b};  // (row g, row g+8) x (step 0, step 1)
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // bytes (0, 2) of the word feed pair (0, 2), bytes (1, 3) pair (1, 3)
                        const uint32_t h02 = hq[k], h13 = hq[k] >> 8;
                        const int a = (k & 1) + 4 * (k >> 1);  // L/H index of (row, step), pair (0, 2)
                        L[a] = and_or<0x00100010u>(i <= 4 ? (h02 << (4 - i)) : (h02 >> (i - 4)), L[a]);
                        L[a + 2] = and_or<0x00100010u>(i <= 4 ? (h13 << (4 - i)) : (h13 >> (i - 4)), L[a + 2]);
                        H[a] = and_or<0x01000100u>(h02 << (7 - i), H[a]);
                        H[a + 2] = and_or<0x01000100u>(h13 << (7 - i), H[a + 2]);
                    }
                }
                // scales of sub-blocks i (low) and i + 1 (high) for rows g, g+8:
                // low: (1024 + q) s - 1024 s with s = 16 sc 2^-24; high: (1024 + 16q) s -
                // 1024 s with s = sc 2^-24; both leave 16 q sc 2^-24
                const uint32_t w0s = i < 4 ? s0l : s0h, w1s = i < 4 ? s1l : s1h;
                const uint32_t ua0 = spair(w0s, i & 3) << 4, ua1 = spair(w1s, i & 3) << 4;
                const uint32_t ub0 = spair(w0s, (i + 1) & 3), ub1 = spair(w1s, (i + 1) & 3);
                const __half2 sa0 = *reinterpret_cast<const __half2*>(&ua0), sa1 = *reinterpret_cast<const __half2*>(&ua1);
                const __half2 sb0 = *reinterpret_cast<const __half2*>(&ub0), sb1 = *reinterpret_cast<const __half2*>(&ub1);
                const __half2 ca0 = __hmul2(sa0, k1024), ca1 = __hmul2(sa1, k1024);
                const __half2 cb0 = __hmul2(sb0, k1024), cb1 = __hmul2(sb1, k1024);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    L[k] = fma2(L[k], (k & 1) ? sa1 : sa0, (k & 1) ? ca1 : ca0);
                    H[k] = fma2(H[k], (k & 1) ? sb1 : sb0, (k & 1) ? cb1 : cb0);
                }
                mma_f16(D, L[0], L[1], L[2], L[3], X.b[4 * i], X.b[4 * i + 1]);
                mma_f16(D, L[4], L[5], L[6], L[7], X.b[4 * i + 2], X.b[4 * i + 3]);
                mma_f16(D, H[0], H[1], H[2], H[3], X.b[4 * i + 4], X.b[4 * i + 5]);
                mma_f16(D, H[4], H[5], H[6], H[7], X.b[4 * i + 6], X.b[4 * i + 7]);
            }
        }
        float D[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            D[q] = Dc[0][q] + Dc[1][q];
            if constexpr (kChains == 4) D[q] += Dc[2][q] + Dc[3][q];
        }
        if constexpr (DUMP) {
            const int sbi = e0 >> 8;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                int a = 0;
#pragma unroll
                for (int ci = 0; ci < kChains; ++ci) a += __float2int_rn(Dc[ci][q] * 1048576.0f);  // exact: 2^20
                dump_add(dz.q[q], 2 * sbi, a);
                dump_add(dz.q[q], 2 * sbi + 1, __float2int_rn(DM[q]));
            }
        }
        // the weight scale d times 2^20 (the operands' 2^-20, exact)
        const float d0 = half_lo(h0.x) * 1048576.0f, dm0 = half_hi(h0.x), d1 = half_lo(h1.x) * 1048576.0f,
                    dm1 = half_hi(h1.x);
        acc[0] = X.dx0 * (d0 * D[0] - dm0 * DM[0]);
        acc[1] = X.dx1 * (d0 * D[1] - dm0 * DM[1]);
        acc[2] = X.dx0 * (d1 * D[2] - dm1 * DM[2]);
        acc[3] = X.dx1 * (d1 * D[3] - dm1 * DM[3]);
    } else if constexpr (F == F_Q2_K) {
        // int8 operands: each byte is a 2-bit code times its 16-group's 4-bit scale
        // (at most 45: one multiply of the masked word by the scale, no carry between
        // bytes), so one m16n8k32 s8 mma per 32 inputs adds sum_j sc_j S_j exactly;
        // the mins sum_j m_j bsum_j is one f16 product with k slot q <-> 16-group q
        // of the chunk (m <= 15 and bsum <= 2032 are exact in f16)
        const saddr b0 = r0 + 84u * sb, b1 = r1 + 84u * sb;
        const int is0 = (e0 & 255) >> 5;  // the chunk's first 32-input step in its superblock
        uint32_t Mr = 0x64006400u;  // the magic exponent in a register
        asm("" : "+r"(Mr));
        // (m of groups gi, gi+1) as an f16 pair, gi even; zero past the superblock
        const auto mpair = [&](saddr blk, int gi) -> uint32_t {
            if (gi >= 16) return 0u;
            const uint32_t w = ld_s32(blk + (gi & ~3));
            const uint32_t k = static_cast<uint32_t>(gi & 3);
            const uint32_t u = and_or<0x000F000Fu>(prmt(w, 0u, 0x4040u | k | ((k + 1) << 8)) >> 4, Mr);
            const __half2 h = __hsub2(*reinterpret_cast<const __half2*>(&u),
                                      __halves2half2(__ushort_as_half(0x6400u), __ushort_as_half(0x6400u)));
            return *reinterpret_cast<const uint32_t*>(&h);
        };
        const int gq = 2 * is0 + 2 * t;  // groups of k slots 2t, 2t+1 (and + 8)
        float DM[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        mma_f16(DM, mpair(b0, gq), mpair(b1, gq), mpair(b0, gq + 8), mpair(b1, gq + 8), X.bm[0], X.bm[1]);
        int A[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (32 * i < chunk) {
                const int is = is0 + i, n = is >> 2, sh = 2 * (is & 3);
                const uint32_t q = 16u + 32u * static_cast<uint32_t>(n) + 4u * t;
                const uint32_t s0 = ld_s32(b0 + ((2 * is) & ~3)), s1 = ld_s32(b1 + ((2 * is) & ~3));
                const int k0 = 8 * ((2 * is) & 3);  // bit offset of group 2is's scale byte
                const uint32_t sc00 = (s0 >> k0) & 15u, sc01 = (s0 >> (k0 + 8)) & 15u;
                const uint32_t sc10 = (s1 >> k0) & 15u, sc11 = (s1 >> (k0 + 8)) & 15u;
                const uint32_t a0 = ((ld_s32(b0 + q) >> sh) & 0x03030303u) * sc00;       // row 2g, group 2is
                const uint32_t a2 = ((ld_s32(b0 + q + 16) >> sh) & 0x03030303u) * sc01;  // row 2g, group 2is+1
                const uint32_t a1 = ((ld_s32(b1 + q) >> sh) & 0x03030303u) * sc10;       // row 2g+1
                const uint32_t a3 = ((ld_s32(b1 + q + 16) >> sh) & 0x03030303u) * sc11;
                mma_k32_s8_acc(A, a0, a1, a2, a3, X.b[2 * i], X.b[2 * i + 1]);
            }
        }
        if constexpr (DUMP) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                dump_add(dz.q[q], 2 * sb, A[q]);
                dump_add(dz.q[q], 2 * sb + 1, __float2int_rn(DM[q]));
            }
        }
        const float d0 = ld_h(b0 + 80), dm0 = ld_h(b0 + 82), d1 = ld_h(b1 + 80), dm1 = ld_h(b1 + 82);
        acc[0] = X.dx0 * (d0 * static_cast<float>(A[0]) - dm0 * DM[0]);
        acc[1] = X.dx1 * (d0 * static_cast<float>(A[1]) - dm0 * DM[1]);
        acc[2] = X.dx0 * (d1 * static_cast<float>(A[2]) - dm1 * DM[2]);
        acc[3] = X.dx1 * (d1 * static_cast<float>(A[3]) - dm1 * DM[3]);
    } else if constexpr (F == F_Q3_K) {
        // f16 operands: the code c = low2 + 4 hbit (0..7) taken as the subnormal f16
        // c 2^-24; one HFMA2 with the 16-group's signed scale s = sc6 - 32 and the
        // addend -4 s 2^-24 leaves q s 2^-24 with q = c - 4 exactly (|q s| <= 128: a
        // subnormal multiple of 2^-24, and the fused operation rounds once, from the
        // exact value).  The scales are in the operands, so one f32 chain per chunk
        // holds sum_j s_j S_j 2^-24 exactly (|sum| < 2^24 units); the epilogue takes
        // the factor 2^24 back.  Element order as for Q4_K: a word's bytes (0, 2)
        // feed k slots (2t, 2t+1), bytes (1, 3) slots (2t+8, 2t+9)
        const uint32_t sbo = 110u * static_cast<uint32_t>(sb);  // 2 bytes off a word at odd sb
        const saddr b0 = r0 + sbo, b1 = r1 + sbo;
        const int is0 = CH == 256 ? 0 : (e0 & 255) >> 5;  // 256-input chunks start at a superblock
        // the lane's qs words of both 128-element halves n: every 32-input step of
        // a half reads the same bytes at another shift.  [n][r], r as in w[] below
        uint32_t W[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            const uint32_t q = 32u + 32u * static_cast<uint32_t>(n) + 4u * t;
            ld_words_any<1>(b0 + q, W[n]);
            ld_words_any<1>(b0 + q + 16, W[n] + 1);
            ld_words_any<1>(b1 + q, W[n] + 2);
            ld_words_any<1>(b1 + q + 16, W[n] + 3);
        }
        uint32_t hm[4];  // hmask bytes 4t.. (groups 2is) and 16+4t.. (2is+1), rows 2g and 2g+1
        ld_words_any<1>(b0 + 4 * t, hm);
        ld_words_any<1>(b0 + 16 + 4 * t, hm + 1);
        ld_words_any<1>(b1 + 4 * t, hm + 2);
        ld_words_any<1>(b1 + 16 + 4 * t, hm + 3);
        uint32_t sw0[3], sw1[3];  // the 12 packed scale bytes of each row
        ld_words_any<3>(b0 + 96, sw0);
        ld_words_any<3>(b1 + 96, sw1);
        // unsigned 6-bit scales of groups 4v .. 4v+3, one per byte
        const auto sc6w = [](const uint32_t* w, int v) -> uint32_t {
            return ((v < 2 ? w[v & 1] : w[v & 1] >> 4) & 0x0F0F0F0Fu) | (((w[2] >> (2 * v)) & 0x03030303u) << 4);
        };
        // (s, s) as f16 for byte idx of a scale word: 1024 + sc6 in the mantissa, minus 1056
        const auto spair = [](uint32_t w, int idx) -> __half2 {
            const uint32_t u = (prmt(w, 0u, 0x4040u | static_cast<uint32_t>(idx) | (static_cast<uint32_t>(idx) << 8)) &
                                0x00FF00FFu) | 0x64006400u;
            return __hsub2(*reinterpret_cast<const __half2*>(&u),
                           __halves2half2(__ushort_as_half(0x6420u), __ushort_as_half(0x6420u)));
        };
        const __half2 m4 = __halves2half2(__ushort_as_half(0x8004u), __ushort_as_half(0x8004u));  // -4 2^-24
        const auto op = [](uint32_t cbits, __half2 sc, __half2 c4) -> uint32_t {
            const __half2 r = __hfma2(*reinterpret_cast<const __half2*>(&cbits), sc, c4);
            return *reinterpret_cast<const uint32_t*>(&r);
        };
        float D[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (32 * i < chunk) {
                const int is = is0 + i, j = is & 3, sh = 2 * j, hb = 4 * (is >> 2) + j;
                // (row 2g, group 2is), (2g, 2is+1), (2g+1, 2is), (2g+1, 2is+1)
                uint32_t w[4];
#pragma unroll
                for (int r = 0; r < 4; ++r) w[r] = (is >> 2) ? W[1][r] : W[0][r];
                const int v = is >> 1, k = 2 * (is & 1);  // groups 2is, 2is+1: bytes k, k+1 of word v
                const uint32_t s0w = sc6w(sw0, v), s1w = sc6w(sw1, v);
                const __half2 sa0 = spair(s0w, k), sb0 = spair(s0w, k + 1);
                const __half2 sa1 = spair(s1w, k), sb1 = spair(s1w, k + 1);
                const __half2 ca0 = __hmul2(sa0, m4), cb0 = __hmul2(sb0, m4);
                const __half2 ca1 = __hmul2(sa1, m4), cb1 = __hmul2(sb1, m4);
                uint32_t L[8];
#pragma unroll
                for (int r = 0; r < 4; ++r) {  // r: (row, group) as in w[]
                    const uint32_t lo = ((w[r] >> sh) & 0x00030003u) | (((hm[r] >> hb) & 0x00010001u) << 2);
                    const uint32_t hi = ((w[r] >> (sh + 8)) & 0x00030003u) | (((hm[r] >> (hb + 8)) & 0x00010001u) << 2);
                    const __half2 sc = r == 0 ? sa0 : r == 1 ? sb0 : r == 2 ? sa1 : sb1;
                    const __half2 c4 = r == 0 ? ca0 : r == 1 ? cb0 : r == 2 ? ca1 : cb1;
                    // operand index: row (r >> 1), k slots (lo: 0, hi: 1), 16-step (group r & 1)
                    L[(r >> 1) + 4 * (r & 1)] = op(lo, sc, c4);
                    L[(r >> 1) + 2 + 4 * (r & 1)] = op(hi, sc, c4);
                }
                mma_f16(D, L[0], L[1], L[2], L[3], X.b[4 * i], X.b[4 * i + 1]);
                mma_f16(D, L[4], L[5], L[6], L[7], X.b[4 * i + 2], X.b[4 * i + 3]);
            }
        }
        if constexpr (DUMP) {
#pragma unroll
            for (int q = 0; q < 4; ++q) dump_add(dz.q[q], sb, __float2int_rn(D[q] * 16777216.0f));  // exact: 2^24
        }
        const float d0 = ld_h(b0 + 108) * 16777216.0f, d1 = ld_h(b1 + 108) * 16777216.0f;
        acc[0] = X.dx0 * (d0 * D[0]);
        acc[1] = X.dx1 * (d0 * D[1]);
        acc[2] = X.dx0 * (d1 * D[2]);
        acc[3] = X.dx1 * (d1 * D[3]);
    } else if constexpr (F == F_Q6_K) {
        // superblocks are 210 bytes: at an odd index they start 2 bytes off a word
        const uint32_t sbo = 210u * static_cast<uint32_t>(sb);
        if ((r0 + sbo) & 2u)
            mmav_q6k<true, DUMP>(r0 + sbo, r1 + sbo, e0, chunk, X, cs, t, acc, dz);
        else
            mmav_q6k<false, DUMP>(r0 + sbo, r1 + sbo, e0, chunk, X, cs, t, acc, dz);
    } else {  // Q8_0 and MXFP4: one scale per 32-block
        const int blk0 = e0 >> 5;  // even: chunks start at multiples of 64
        acc[0] = acc[1] = acc[2] = acc[3] = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (32 * i < chunk) {
                const int blk = blk0 + i;
                uint32_t a0, a1, a2, a3;
                float w0, w1;
                int c0 = 0, c1 = 0;
                if constexpr (F == F_Q8_0) {
                    const saddr p0 = r0 + 34u * blk, p1 = r1 + 34u * blk;
                    if (i & 1) {  // odd block: quants start on a 4-byte boundary
                        a0 = ld_s32(p0 + 2 + 4 * t);
                        a2 = ld_s32(p0 + 18 + 4 * t);
                        a1 = ld_s32(p1 + 2 + 4 * t);
                        a3 = ld_s32(p1 + 18 + 4 * t);
                    } else {  // even block: two aligned words, take the middle
                        a0 = prmt(ld_s32(p0 + 4 * t), ld_s32(p0 + 4 + 4 * t), 0x5432u);
                        a2 = prmt(ld_s32(p0 + 16 + 4 * t), ld_s32(p0 + 20 + 4 * t), 0x5432u);
                        a1 = prmt(ld_s32(p1 + 4 * t), ld_s32(p1 + 4 + 4 * t), 0x5432u);
                        a3 = prmt(ld_s32(p1 + 16 + 4 * t), ld_s32(p1 + 20 + 4 * t), 0x5432u);
                    }
                    w0 = ld_h(p0);
                    w1 = ld_h(p1);
                } else {
                    const saddr p0 = r0 + 17u * blk, p1 = r1 + 17u * blk;
                    uint32_t q0, q1;
                    ld_words_any<1>(p0 + 1 + 4 * t, &q0);
                    ld_words_any<1>(p1 + 1 + 4 * t, &q1);
                    a0 = mx_lookup(q0 & 0xFFFFu);
                    a2 = mx_lookup(q0 >> 16);
                    a1 = mx_lookup(q1 & 0xFFFFu);
                    a3 = mx_lookup(q1 >> 16);
                    w0 = e8m0_half_scale(ld_u8(p0));
                    w1 = e8m0_half_scale(ld_u8(p1));
                    c0 = -X.s[2 * i];  // the tables hold 2*value + 12
                    c1 = -X.s[2 * i + 1];
                }
                int D[4];
                mma_k32_s8(D, a0, a1, a2, a3, X.b[2 * i], X.b[2 * i + 1], c0, c1);
                if constexpr (DUMP) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) dump_put(dz.q[q], blk, D[q]);
                }
                acc[0] += static_cast<float>(D[0]) * (w0 * X.dx0);
                acc[1] += static_cast<float>(D[1]) * (w0 * X.dx1);
                acc[2] += static_cast<float>(D[2]) * (w1 * X.dx0);
                acc[3] += static_cast<float>(D[3]) * (w1 * X.dx1);
            }
        }
    }
}

template <int F, bool DUMP, int CH>
__global__ void __launch_bounds__(kThreads, 1) k_gemv_mma(const MmavParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();

    // ---- shared memory: ring | activations, later the partials [2][16 rows x 8 columns][16 warps]
    //      | f16-path C values | barriers
    uint8_t* ring = smem;
    uint8_t* xreg = smem + static_cast<size_t>(p.stages) * p.stage_stride;
    float* red = reinterpret_cast<float*>(xreg);
    float* creg = reinterpret_cast<float*>(xreg + p.x_bytes);  // [16 warps][4][kMmavCStride]
    uint64_t* full = reinterpret_cast<uint64_t*>(creg + kConsumerWarps * 4 * kMmavCStride);
    uint64_t* empty = full + kMaxStages;
    uint64_t* xbar = empty + kMaxStages;

    const int nitems = static_cast<int>((p.N + kTileRows - 1) / kTileRows);
    if (static_cast<int>(blockIdx.x) >= nitems) return;  // whole CTA idle (uniform)
    if (warp == kConsumerWarps) {
        // ================= producer warp: initialises the barriers and releases the
        // consumers (start barrier, no wait); lane 0 waits, lanes 0..7 copy the row pairs
        if (lane == 0) {
            for (int s = 0; s < p.stages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kConsumerWarps);
            }
            mbar_init(xbar, 1);
            fence_barrier_init();
        }
        __syncwarp();
        mmav_start_arrive();
        const uint64_t pol = policy_evict_first();
        if (!p.early_weights) pdl_wait();  // the previous kernel may still be writing the weights
        int j = 0, s = 0;
        uint32_t ph = 0u;  // ring slot and phase of tile j
        bool ok = true;
        for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++j) {
            const int64_t r0 = static_cast<int64_t>(item) * kTileRows;
            const int nr = static_cast<int>(p.N - r0 < kTileRows ? p.N - r0 : kTileRows);
            if (lane == 0) {
                // with static weights, the stages after the first once the activations are in
                // (their bulk copies' barrier; without it, once the previous kernel has finished):
                // measured faster than streaming all but the last stage first
                if (p.early_weights && j == 1) {
                    if (p.x_bulk) ok = mbar_wait(xbar, 0u);
                    else pdl_wait();
                }
                ok = ok && mbar_wait(&empty[s], ph ^ 1u);
                if (ok) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(nr * p.rowbytes));
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) set_error(p.err, DEV_ERR_TIMEOUT);
                break;
            }
            const int pr = 2 * lane;
            if (pr < nr) {
                const int rows = nr - pr < 2 ? nr - pr : 2;
                bulk_g2s(ring + static_cast<size_t>(s) * p.stage_stride + static_cast<size_t>(lane) * p.wrow,
                         p.W + (r0 + pr) * p.rowbytes, static_cast<uint32_t>(rows * p.rowbytes), &full[s], pol);
            }
            if (++s == p.stages) {
                s = 0;
                ph ^= 1u;
            }
        }
        if (lane == 0) {
            for (int q = (j > p.stages ? j - p.stages : 0); q < j; ++q) {
                if (!mbar_wait(&full[q % p.stages], static_cast<uint32_t>(q / p.stages) & 1u)) {
                    set_error(p.err, DEV_ERR_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ================= consumers
    mmav_start_sync();  // barriers initialised
    pdl_wait();  // activations come from the previous kernel; outputs are written after it finished
    // activation row r -> xreg + r * xstride (the padded stride puts the eight
    // rows' fragment words on distinct banks)
    bool xok = true;
    if (p.x_bulk) {
        if (warp == 0) {  // lane r copies row r, after lane 0 has announced the bytes
            if (lane == 0) mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(p.T * p.xrow));
            __syncwarp();
            if (lane < p.T)
                bulk_g2s(xreg + static_cast<size_t>(lane) * p.xstride, p.xq + static_cast<size_t>(lane) * p.xrow,
                         static_cast<uint32_t>(p.xrow), xbar, policy_evict_last());
        }
        xok = mbar_wait(xbar, 0u);
        if (!xok) set_error(p.err, DEV_ERR_TIMEOUT);
    } else {
        const int wr = p.xrow / 4;
        for (int i = tid; i < p.T * wr; i += kConsumerWarps * 32) {
            const int r = i / wr, w = i - r * wr;
            reinterpret_cast<uint32_t*>(xreg + static_cast<size_t>(r) * p.xstride)[w] =
                __ldg(reinterpret_cast<const uint32_t*>(p.xq + static_cast<size_t>(r) * p.xrow) + w);
        }
        mmav_sync();
    }
    const int g = lane >> 2, t = lane & 3;
    const bool active = warp < p.nch;
    const int e0 = warp * p.chunk;
    MmaX X;
    float* cs = creg + (warp * 4 + t) * kMmavCStride;
    mmav_load_x<F>(smem_addr(xreg), p.xstride, active ? p.T : 0, p.chunk, e0, g, t, X, cs);
    mmav_sync();  // the region now holds partials
    const saddr ring_s = smem_addr(ring);
    int j = 0, s = 0;
    uint32_t ph = 0u;  // ring slot and phase of tile j
    for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++j) {
        const bool ready = xok && __all_sync(0xffffffffu, mbar_wait_backoff(&full[s], ph));
        if (!ready) set_error(p.err, DEV_ERR_TIMEOUT);
        float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (ready && active) {
            const saddr r0 = ring_s + static_cast<uint32_t>(s * p.stage_stride + g * p.wrow);  // tile row 2g
            MmavDump dz{};
            if constexpr (DUMP) {
                // this thread's outputs: tile rows 2g, 2g + 1 and columns 2t, 2t + 1
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int64_t row = static_cast<int64_t>(item) * kTileRows + 2 * g + (q >> 1);
                    const int col = 2 * t + (q & 1);
                    dz.q[q] = row < p.N && col < p.T ? p.coefs + (static_cast<int64_t>(col) * p.N + row) * p.ncoef
                                                     : nullptr;
                }
            }
            mmav_chunk<F, DUMP, CH>(r0, r0 + static_cast<uint32_t>(p.rowbytes), e0, p.chunk, X, smem_addr(cs), t, acc,
                                    dz);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[s]);
        if (++s == p.stages) {
            s = 0;
            ph ^= 1u;
        }
        // partials of this tile -> buffer j & 1, laid out [warp][tile row x 8 + column]
        // with a warp stride of kRedStride floats (2 mod 32: the reads below hit 32
        // distinct banks); one barrier per tile (a warp writes buffer j & 1 again only
        // after the next tile's barrier, which the readers of this tile reach after reading)
        float* rb = red + (j & 1) * (kRedStride * kConsumerWarps);
        float* rw = rb + warp * kRedStride;
        *reinterpret_cast<float2*>(rw + (2 * g) * 8 + 2 * t) = make_float2(acc[0], acc[1]);
        *reinterpret_cast<float2*>(rw + (2 * g + 1) * 8 + 2 * t) = make_float2(acc[2], acc[3]);
        mmav_sync();
        {
            // output o = tid / 4 (tile row o / 8, column o % 8): four threads sum four warps each
            const int o = tid >> 2, q = tid & 3;
            const float* rr = rb + (4 * q) * kRedStride + o;
            float v = (rr[0] + rr[kRedStride]) + (rr[2 * kRedStride] + rr[3 * kRedStride]);
            v += __shfl_xor_sync(0xffffffffu, v, 1);
            v += __shfl_xor_sync(0xffffffffu, v, 2);
            const int row = o >> 3, col = o & 7;
            const int64_t grow = static_cast<int64_t>(item) * kTileRows + row;
            if (!DUMP && q == 0 && col < p.T && grow < p.N && ready) p.Y[static_cast<int64_t>(col) * p.N + grow] = v;
        }
    }
}

template <int F, bool DUMP, int CH>
cudaError_t launch_mmav_ch(const MmavParams& p, int grid, int smem, cudaStream_t s) {
    static std::atomic<bool> attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(k_gemv_mma<F, DUMP, CH>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    return launch_pdl(k_gemv_mma<F, DUMP, CH>, dim3(grid), dim3(kThreads), smem, s, p);
}

// Chunks of 256 inputs (K = 4096: the decode widths of the 14336 x 4096 GEMV)
// run a variant with the chunk width fixed at compile time; others take it
// at run time.
template <int F, bool DUMP>
cudaError_t launch_mmav_one(const MmavParams& p, int grid, int smem, cudaStream_t s) {
    return p.chunk == 256 ? launch_mmav_ch<F, DUMP, 256>(p, grid, smem, s) : launch_mmav_ch<F, DUMP, 0>(p, grid, smem, s);
}

}  // namespace ggq

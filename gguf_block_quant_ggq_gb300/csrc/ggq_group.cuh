// ggq_group.cuh -- the grouped int8 tensor-core kernel: decode GEMV at 3-8
// tokens, and the expert-sorted MoE route (5 tokens and up, prefill).
//
// GB300 has no tcgen05 kind::i8 path (ptxas rejects it for sm_103a), and the
// legacy mma.sync s8 path runs at the int8 CUDA-core rate; it is still the
// right engine once an expert (or a GEMV) has several activation columns,
// because one mma.sync.m16n8k32 covers 16 rows x 8 columns x 32 inputs in one
// instruction where dp4a needs 32 -- the dp4a kernels run out of issue slots
// first.  All arithmetic stays exact: int8 x int8 products accumulate in
// int32, and the block scales are applied per block in the epilogue.
//
// Work item = (group, 16-row tile).  A group is one weight matrix (one expert)
// with its list of activation columns (tokens, or (token, slot) pairs sorted
// by expert: the expert-sorted tiles of ds4 PR #656 "Add ROCm MXFP4 routed
// expert kernels", Correctness).  The producer warp copies the item's weight
// rows (gate and up rows together for the gate/up stage) into a weight ring,
// then the item's activation rows eight at a time into an activation ring.
// Eight consumer warps split K by 256-element superblocks, each computing an
// m16 x n8 partial per chunk with mma.sync; partials meet in shared memory
// and the epilogue writes y (GEMV), h = silu(g)*u (gate/up) or o (down).
#pragma once
#include "ggq_device.cuh"
#include "ggq_internal.h"

#include <atomic>

namespace ggq {

__device__ __forceinline__ void group_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kGroupConsumerWarps * 32) : "memory");
}

__device__ __forceinline__ void mma_s8_k32(int* d, const uint32_t* a, uint32_t b0, uint32_t b1, const int* c) {
    asm volatile(
        "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]));
}

__device__ __forceinline__ void mma_s8_k16(int* d, uint32_t a0, uint32_t a1, uint32_t b0, const int* c) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5}, {%6}, {%7,%8,%9,%10};"
        : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
        : "r"(a0), "r"(a1), "r"(b0), "r"(c[0]), "r"(c[1]), "r"(c[2]), "r"(c[3]));
}

// Activation rows of a chunk in shared memory: packed Q8_K blocks, row stride
// xstride.  Thread (g, tig) of an mma reads token g for B and the tokens of
// its accumulator columns c0 = 2 tig, c1 = 2 tig + 1 for scales and sums.
struct GX {
    saddr base;
    int xstride;
    int ncols;
};

__device__ __forceinline__ saddr gx_row(const GX& x, int c) { return x.base + static_cast<uint32_t>(c * x.xstride); }

// B fragment words of one 32-element sub-block (elements e0 + 4 tig and
// e0 + 16 + 4 tig of token g), zero for an absent column.
__device__ __forceinline__ void gx_b32(const GX& x, int g, int tig, int sb, int s, uint32_t& b0, uint32_t& b1) {
    if (g < x.ncols) {
        const saddr a = gx_row(x, g) + 292u * sb + 4u + 32u * s + 4u * tig;
        b0 = ld_s32(a);
        b1 = ld_s32(a + 16);
    } else {
        b0 = b1 = 0u;
    }
}

__device__ __forceinline__ float gx_d(const GX& x, int c, int sb) {
    return c < x.ncols ? ld_f32(gx_row(x, c) + 292u * sb) : 0.0f;
}

// Sum of the quants of 32-block s (0..7) of superblock sb of column c.
__device__ __forceinline__ int gx_s32(const GX& x, int c, int sb, int s) {
    if (c >= x.ncols) return 0;
    const uint32_t v = ld_s32(gx_row(x, c) + 292u * sb + 260u + 4u * s);
    return static_cast<int>(static_cast<int16_t>(v & 0xFFFFu)) + static_cast<int>(static_cast<int16_t>(v >> 16));
}

// Accumulate superblock sb of rows g and g+8 (row addresses r0, r1) against
// the chunk's columns into acc[4] = (row g, c0), (row g, c1), (row g+8, c0),
// (row g+8, c1).  With DUMP, dq[] are the coefficient rows of those four
// outputs (null: no output) and receive the integer core of the superblock:
// A and B (Q4_K/Q5_K), A (Q6_K) or the eight 32-block dots (Q8_0, MXFP4).
template <int F, bool DUMP>
__device__ __forceinline__ void group_superblock(saddr r0, saddr r1, int sb, const GX& x, int g, int tig,
                                                 float* acc, int32_t* const* dq) {
    const int c0 = 2 * tig, c1 = 2 * tig + 1;
    const int zero[4] = {0, 0, 0, 0};
    if constexpr (F == F_Q4_K || F == F_Q5_K) {
        constexpr uint32_t SB = F == F_Q4_K ? 144u : 176u;
        constexpr uint32_t QS = F == F_Q4_K ? 16u : 48u;
        const saddr b0r = r0 + SB * sb, b1r = r1 + SB * sb;
        const uint4 h0 = ld_s128(b0r), h1 = ld_s128(b1r);
        // scales and mins of all eight sub-blocks, four per word, per row
        const uint32_t sc0_lo = h0.y & 0x3F3F3F3Fu, m0_lo = h0.z & 0x3F3F3F3Fu;
        const uint32_t sc0_hi = (h0.w & 0x0F0F0F0Fu) | ((h0.y >> 2) & 0x30303030u);
        const uint32_t m0_hi = ((h0.w >> 4) & 0x0F0F0F0Fu) | ((h0.z >> 2) & 0x30303030u);
        const uint32_t sc1_lo = h1.y & 0x3F3F3F3Fu, m1_lo = h1.z & 0x3F3F3F3Fu;
        const uint32_t sc1_hi = (h1.w & 0x0F0F0F0Fu) | ((h1.y >> 2) & 0x30303030u);
        const uint32_t m1_hi = ((h1.w >> 4) & 0x0F0F0F0Fu) | ((h1.z >> 2) & 0x30303030u);
        uint32_t qh0a = 0, qh0b = 0, qh1a = 0, qh1b = 0;
        if constexpr (F == F_Q5_K) {
            qh0a = ld_s32(b0r + 16 + 4 * tig);
            qh0b = ld_s32(b0r + 32 + 4 * tig);
            qh1a = ld_s32(b1r + 16 + 4 * tig);
            qh1b = ld_s32(b1r + 32 + 4 * tig);
        }
        int iA[4] = {0, 0, 0, 0}, iB[4] = {0, 0, 0, 0};
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const saddr q0 = b0r + QS + 32u * cc + 4u * tig, q1 = b1r + QS + 32u * cc + 4u * tig;
            const uint32_t qa0 = ld_s32(q0), qb0 = ld_s32(q0 + 16), qa1 = ld_s32(q1), qb1 = ld_s32(q1 + 16);
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                const int s = 2 * cc + hb;
                uint32_t a[4] = {(qa0 >> (4 * hb)) & 0x0F0F0F0Fu, (qa1 >> (4 * hb)) & 0x0F0F0F0Fu,
                                 (qb0 >> (4 * hb)) & 0x0F0F0F0Fu, (qb1 >> (4 * hb)) & 0x0F0F0F0Fu};
                if constexpr (F == F_Q5_K) {
                    a[0] |= ((qh0a >> s) & 0x01010101u) << 4;
                    a[1] |= ((qh1a >> s) & 0x01010101u) << 4;
                    a[2] |= ((qh0b >> s) & 0x01010101u) << 4;
                    a[3] |= ((qh1b >> s) & 0x01010101u) << 4;
                }
                uint32_t bb0, bb1;
                gx_b32(x, g, tig, sb, s, bb0, bb1);
                int d[4];
                mma_s8_k32(d, a, bb0, bb1, zero);
                const uint32_t w0 = s < 4 ? sc0_lo : sc0_hi, w1 = s < 4 ? sc1_lo : sc1_hi;
                const int sc0 = (w0 >> (8 * (s & 3))) & 0xFF, sc1 = (w1 >> (8 * (s & 3))) & 0xFF;
                iA[0] += sc0 * d[0];
                iA[1] += sc0 * d[1];
                iA[2] += sc1 * d[2];
                iA[3] += sc1 * d[3];
                const uint32_t v0 = s < 4 ? m0_lo : m0_hi, v1 = s < 4 ? m1_lo : m1_hi;
                const int mm0 = (v0 >> (8 * (s & 3))) & 0xFF, mm1 = (v1 >> (8 * (s & 3))) & 0xFF;
                const int sa = gx_s32(x, c0, sb, s), sbb = gx_s32(x, c1, sb, s);
                iB[0] += mm0 * sa;
                iB[1] += mm0 * sbb;
                iB[2] += mm1 * sa;
                iB[3] += mm1 * sbb;
            }
        }
        if constexpr (DUMP) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (dq[q]) {
                    dq[q][2 * sb] = iA[q];
                    dq[q][2 * sb + 1] = iB[q];
                }
        }
        const float d0 = half_lo(h0.x), dm0 = half_hi(h0.x), d1 = half_lo(h1.x), dm1 = half_hi(h1.x);
        const float x0 = gx_d(x, c0, sb), x1 = gx_d(x, c1, sb);
        acc[0] += x0 * (d0 * static_cast<float>(iA[0]) - dm0 * static_cast<float>(iB[0]));
        acc[1] += x1 * (d0 * static_cast<float>(iA[1]) - dm0 * static_cast<float>(iB[1]));
        acc[2] += x0 * (d1 * static_cast<float>(iA[2]) - dm1 * static_cast<float>(iB[2]));
        acc[3] += x1 * (d1 * static_cast<float>(iA[3]) - dm1 * static_cast<float>(iB[3]));
    } else if constexpr (F == F_Q6_K) {
        const saddr b0r = r0 + 210u * sb, b1r = r1 + 210u * sb;
        uint32_t scw0[4], scw1[4];  // int8 scales of the 16 groups, four per word
        ld_words_any<4>(b0r + 192, scw0);
        ld_words_any<4>(b1r + 192, scw1);
        int iA[4] = {0, 0, 0, 0};
#pragma unroll
        for (int h = 0; h < 2; ++h) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                const uint32_t l0 = 16u * hf + 4u * tig;
                uint32_t qla0, qlb0, qh0, qla1, qlb1, qh1;
                ld_words_any<1>(b0r + 64 * h + l0, &qla0);
                ld_words_any<1>(b0r + 64 * h + 32 + l0, &qlb0);
                ld_words_any<1>(b0r + 128 + 32 * h + l0, &qh0);
                ld_words_any<1>(b1r + 64 * h + l0, &qla1);
                ld_words_any<1>(b1r + 64 * h + 32 + l0, &qlb1);
                ld_words_any<1>(b1r + 128 + 32 * h + l0, &qh1);
#pragma unroll
                for (int g6 = 0; g6 < 4; ++g6) {
                    const int j = 8 * h + 2 * g6 + hf;  // 16-element group index
                    const uint32_t l0w = (g6 & 1) ? qlb0 : qla0, l1w = (g6 & 1) ? qlb1 : qla1;
                    const uint32_t a0 = ((l0w >> (4 * (g6 >> 1))) & 0x0F0F0F0Fu) | (((qh0 >> (2 * g6)) & 0x03030303u) << 4);
                    const uint32_t a1 = ((l1w >> (4 * (g6 >> 1))) & 0x0F0F0F0Fu) | (((qh1 >> (2 * g6)) & 0x03030303u) << 4);
                    uint32_t bj = 0u;
                    if (g < x.ncols) bj = ld_s32(gx_row(x, g) + 292u * sb + 4u + 16u * j + 4u * tig);
                    // C = -32 * (sum of the 16 quants) of each column: the codes are stored unsigned
                    int cinit[4];
                    const int bsa = c0 < x.ncols ? ld_s16(gx_row(x, c0) + 292u * sb + 260u + 2u * j) : 0;
                    const int bsb = c1 < x.ncols ? ld_s16(gx_row(x, c1) + 292u * sb + 260u + 2u * j) : 0;
                    cinit[0] = cinit[2] = -32 * bsa;
                    cinit[1] = cinit[3] = -32 * bsb;
                    int d[4];
                    mma_s8_k16(d, a0, a1, bj, cinit);
                    const int s0 = static_cast<int>(static_cast<int8_t>((scw0[j >> 2] >> (8 * (j & 3))) & 0xFF));
                    const int s1 = static_cast<int>(static_cast<int8_t>((scw1[j >> 2] >> (8 * (j & 3))) & 0xFF));
                    iA[0] += s0 * d[0];
                    iA[1] += s0 * d[1];
                    iA[2] += s1 * d[2];
                    iA[3] += s1 * d[3];
                }
            }
        }
        if constexpr (DUMP) {
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (dq[q]) dq[q][sb] = iA[q];
        }
        const float d0 = ld_h(b0r + 208), d1 = ld_h(b1r + 208);
        const float x0 = gx_d(x, c0, sb), x1 = gx_d(x, c1, sb);
        acc[0] += static_cast<float>(iA[0]) * (x0 * d0);
        acc[1] += static_cast<float>(iA[1]) * (x1 * d0);
        acc[2] += static_cast<float>(iA[2]) * (x0 * d1);
        acc[3] += static_cast<float>(iA[3]) * (x1 * d1);
    } else {  // Q8_0, MXFP4: eight 32-blocks, one scale each
        const float x0 = gx_d(x, c0, sb), x1 = gx_d(x, c1, sb);
        if constexpr (F == F_MXFP4 && !DUMP) {
            if (x.ncols == 1) {
                // one column (an expert that carries one pair): dp4a instead of an mma
                // that would fill one of its eight columns.  Lane (g, tig) takes the
                // fragment's codes (rows g, g + 8; elements 4 tig .. + 3 and 16 + 4 tig
                // .. + 3) as doubled magnitudes of the positive and, with selector bit
                // 3 flipped, of the negative codes, in the lookup's element order, and
                // the column's activations in the same order; the four lanes of a row
                // add their parts, so each block's integer and its scale product are
                // those of the mma path
                uint32_t tl = MX_MAG_LO, th = MX_MAG_HI;
                asm("" : "+r"(tl), "+r"(th));
                const saddr xr = gx_row(x, 0) + 292u * sb + 4u + 4u * tig;
#pragma unroll
                for (int s = 0; s < 8; ++s) {
                    const int blk = 8 * sb + s;
                    const saddr p0 = r0 + 17u * blk, p1 = r1 + 17u * blk;
                    uint32_t q0, q1;
                    ld_words_any<1>(p0 + 1 + 4 * tig, &q0);
                    ld_words_any<1>(p1 + 1 + 4 * tig, &q1);
                    const uint32_t xlo = ld_s32(xr + 32u * s), xhi = ld_s32(xr + 32u * s + 16u);
                    const int u0 = static_cast<int>(prmt(xlo, xhi, 0x5140u)), u1 = static_cast<int>(prmt(xlo, xhi, 0x7362u));
                    const uint32_t f0 = q0 ^ 0x88888888u, f1 = q1 ^ 0x88888888u;
                    int P0 = __dp4a(static_cast<int>(prmt(tl, th, q0)), u0, 0);
                    P0 = __dp4a(static_cast<int>(prmt(tl, th, q0 >> 16)), u1, P0);
                    int N0 = __dp4a(static_cast<int>(prmt(tl, th, f0)), u0, 0);
                    N0 = __dp4a(static_cast<int>(prmt(tl, th, f0 >> 16)), u1, N0);
                    int P1 = __dp4a(static_cast<int>(prmt(tl, th, q1)), u0, 0);
                    P1 = __dp4a(static_cast<int>(prmt(tl, th, q1 >> 16)), u1, P1);
                    int N1 = __dp4a(static_cast<int>(prmt(tl, th, f1)), u0, 0);
                    N1 = __dp4a(static_cast<int>(prmt(tl, th, f1 >> 16)), u1, N1);
                    int d0 = P0 - N0, d1 = P1 - N1;
                    d0 += __shfl_xor_sync(0xffffffffu, d0, 1);
                    d1 += __shfl_xor_sync(0xffffffffu, d1, 1);
                    d0 += __shfl_xor_sync(0xffffffffu, d0, 2);
                    d1 += __shfl_xor_sync(0xffffffffu, d1, 2);
                    const float w0 = e8m0_half_scale(ld_u8(p0)), w1 = e8m0_half_scale(ld_u8(p1));
                    acc[0] += static_cast<float>(d0) * (w0 * x0);  // column 0: lanes with tig 0
                    acc[2] += static_cast<float>(d1) * (w1 * x0);
                }
                return;
            }
        }
#pragma unroll
        for (int s = 0; s < 8; ++s) {
            const int blk = 8 * sb + s;
            uint32_t a[4];
            float w0, w1;
            int cinit[4] = {0, 0, 0, 0};
            if constexpr (F == F_Q8_0) {
                const saddr p0 = r0 + 34u * blk, p1 = r1 + 34u * blk;
                ld_words_any<1>(p0 + 2 + 4 * tig, &a[0]);
                ld_words_any<1>(p1 + 2 + 4 * tig, &a[1]);
                ld_words_any<1>(p0 + 18 + 4 * tig, &a[2]);
                ld_words_any<1>(p1 + 18 + 4 * tig, &a[3]);
                w0 = ld_h(p0);
                w1 = ld_h(p1);
            } else {
                const saddr p0 = r0 + 17u * blk, p1 = r1 + 17u * blk;
                uint32_t q0, q1;
                ld_words_any<1>(p0 + 1 + 4 * tig, &q0);
                ld_words_any<1>(p1 + 1 + 4 * tig, &q1);
                // lookup order is (j, j+16, j+1, j+17) / (j+2, j+18, j+3, j+19): split it
                const uint32_t L0 = mx_lookup(q0 & 0xFFFFu), H0 = mx_lookup(q0 >> 16);
                const uint32_t L1 = mx_lookup(q1 & 0xFFFFu), H1 = mx_lookup(q1 >> 16);
                a[0] = prmt(L0, H0, 0x6420u);
                a[2] = prmt(L0, H0, 0x7531u);
                a[1] = prmt(L1, H1, 0x6420u);
                a[3] = prmt(L1, H1, 0x7531u);
                w0 = e8m0_half_scale(ld_u8(p0));
                w1 = e8m0_half_scale(ld_u8(p1));
                // the tables hold 2*value + 12: remove 12 * (sum of the block's quants)
                const int sa = gx_s32(x, c0, sb, s), sbb = gx_s32(x, c1, sb, s);
                cinit[0] = cinit[2] = -12 * sa;
                cinit[1] = cinit[3] = -12 * sbb;
            }
            uint32_t bb0, bb1;
            gx_b32(x, g, tig, sb, s, bb0, bb1);
            int d[4];
            mma_s8_k32(d, a, bb0, bb1, cinit);
            if constexpr (DUMP) {
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (dq[q]) dq[q][blk] = d[q];
            }
            acc[0] += static_cast<float>(d[0]) * (w0 * x0);
            acc[1] += static_cast<float>(d[1]) * (w0 * x1);
            acc[2] += static_cast<float>(d[2]) * (w1 * x0);
            acc[3] += static_cast<float>(d[3]) * (w1 * x1);
        }
    }
}

template <int KIND, int F, bool DUMP>
__global__ void __launch_bounds__(kGroupThreads, 1) k_group(const GroupParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr int NMAT = KIND == G_GATEUP ? 2 : 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- layout: weight ring | activation ring | reduction | barriers
    uint8_t* wring = smem;
    uint8_t* xring = wring + static_cast<size_t>(p.wstages) * p.wslot;
    float* red = reinterpret_cast<float*>(xring + static_cast<size_t>(p.xstages) * p.xslot);  // [8][NMAT][16][8]
    uint64_t* wfull = reinterpret_cast<uint64_t*>(red + kGroupConsumerWarps * NMAT * 128);
    uint64_t* wempty = wfull + 4;
    uint64_t* xfull = wempty + 4;
    uint64_t* xempty = xfull + 8;
    int* s_abort = reinterpret_cast<int*>(xempty + 8);

    pdl_launch_dependents();
    if (KIND != G_GEMV) pdl_wait();  // the grouping comes from the previous kernels
    const int ngroups = KIND == G_GEMV ? 1 : *p.ngroups;
    const int tiles = static_cast<int>(p.N / kGroupRows);  // N % 16 == 0 except the GEMV tail
    const int tiles_all = KIND == G_GEMV ? static_cast<int>((p.N + kGroupRows - 1) / kGroupRows) : tiles;
    const int nitems = ngroups * tiles_all;
    if (static_cast<int>(blockIdx.x) >= nitems) return;

    if (tid == 0) {
        for (int s = 0; s < p.wstages; ++s) {
            mbar_init(&wfull[s], 1);
            mbar_init(&wempty[s], kGroupConsumerWarps);
        }
        for (int s = 0; s < p.xstages; ++s) {
            mbar_init(&xfull[s], 1);
            mbar_init(&xempty[s], kGroupConsumerWarps);
        }
        *s_abort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    // item -> (group, tile); group -> (expert, column offset, column count)
    auto item_group = [&](int item, int& gi, int& tile) {
        gi = item / tiles_all;
        tile = item - gi * tiles_all;
    };
    auto group_cols = [&](int gi, int& e, int& off, int& cnt) {
        if constexpr (KIND == G_GEMV) {
            e = 0;
            off = 0;
            cnt = p.T;
        } else {
            e = p.group_expert[gi];
            off = p.group_off[gi];
            cnt = p.group_cnt[gi];
        }
    };
    auto col_row = [&](int pos) -> int64_t {  // activation row of sorted column pos
        if constexpr (KIND == G_GEMV) return pos;
        const int pair = p.perm[pos];
        return KIND == G_GATEUP ? pair / p.top_k : pair;
    };

    if (warp == kGroupConsumerWarps) {
        // ================= producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            if (KIND == G_GEMV && !p.early_weights) pdl_wait();
            int wj = 0, xj = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++wj) {
                int gi, tile, e, off, cnt;
                item_group(item, gi, tile);
                group_cols(gi, e, off, cnt);
                // weights
                {
                    const int s = wj % p.wstages;
                    if (!mbar_wait(&wempty[s], (static_cast<uint32_t>(wj / p.wstages) & 1u) ^ 1u)) {
                        set_error(p.err, DEV_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const int64_t r0 = static_cast<int64_t>(tile) * kGroupRows;
                    const int nr = static_cast<int>(p.N - r0 < kGroupRows ? p.N - r0 : kGroupRows);
                    uint8_t* dst = wring + static_cast<size_t>(s) * p.wslot;
                    uint32_t total = 0;
                    // ragged tail (GEMV only): plain copy of the bytes past the last 16-byte multiple
                    for (int m = 0; m < NMAT; ++m) {
                        const uint8_t* src = (m == 0 ? p.W : p.W2) + (static_cast<int64_t>(e) * p.N + r0) * p.rowbytes;
                        if (p.wcontig) {
                            const uint32_t bytes = static_cast<uint32_t>(nr * p.rowbytes), bulk = bytes & ~15u;
                            for (uint32_t b = bulk; b < bytes; ++b) dst[m * kGroupRows * p.wrow + b] = __ldg(src + b);
                            total += bulk;
                        } else {
                            total += static_cast<uint32_t>(nr * p.rowbytes);
                        }
                    }
                    mbar_arrive_expect_tx(&wfull[s], total);
                    for (int m = 0; m < NMAT; ++m) {
                        const uint8_t* src = (m == 0 ? p.W : p.W2) + (static_cast<int64_t>(e) * p.N + r0) * p.rowbytes;
                        uint8_t* d = dst + m * kGroupRows * p.wrow;
                        if (p.wcontig) {
                            const uint32_t bulk = static_cast<uint32_t>(nr * p.rowbytes) & ~15u;
                            if (bulk) bulk_g2s(d, src, bulk, &wfull[s], pol);
                        } else {
                            for (int r = 0; r < nr; ++r)
                                bulk_g2s(d + r * p.wrow, src + r * p.rowbytes, static_cast<uint32_t>(p.rowbytes),
                                         &wfull[s], pol);
                        }
                    }
                }
                // activation chunks (the GEMV's single chunk is loaded once and kept)
                const int nchunks = KIND == G_GEMV ? (wj == 0 ? 1 : 0) : (cnt + kGroupCols - 1) / kGroupCols;
                if (KIND == G_GEMV && wj == 0 && p.early_weights) pdl_wait();  // x^ comes from the previous kernel
                for (int ch = 0; ch < nchunks; ++ch, ++xj) {
                    const int s = xj % p.xstages;
                    if (!mbar_wait(&xempty[s], (static_cast<uint32_t>(xj / p.xstages) & 1u) ^ 1u)) {
                        set_error(p.err, DEV_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    const int nc = cnt - ch * kGroupCols < kGroupCols ? cnt - ch * kGroupCols : kGroupCols;
                    mbar_arrive_expect_tx(&xfull[s], static_cast<uint32_t>(nc * p.xcopy));
                    uint8_t* dst = xring + static_cast<size_t>(s) * p.xslot;
                    for (int c = 0; c < nc; ++c)
                        bulk_g2s(dst + c * p.xstride, p.xq + col_row(off + ch * kGroupCols + c) * p.x_pitch,
                                 static_cast<uint32_t>(p.xcopy), &xfull[s], policy_evict_last());
                }
            }
            // never leave copies in flight
            for (int q = (wj > p.wstages ? wj - p.wstages : 0); q < wj; ++q)
                if (!mbar_wait(&wfull[q % p.wstages], static_cast<uint32_t>(q / p.wstages) & 1u)) break;
            for (int q = (xj > p.xstages ? xj - p.xstages : 0); q < xj; ++q)
                if (!mbar_wait(&xfull[q % p.xstages], static_cast<uint32_t>(q / p.xstages) & 1u)) break;
        }
        return;
    }

    // ================= consumers (256 threads)
    if (KIND == G_GEMV) pdl_wait();  // outputs are written after the previous kernel finished
    const int g = lane >> 2, tig = lane & 3;
    const int nsb = p.K >> 8;
    const saddr wring_s = smem_addr(wring), xring_s = smem_addr(xring);
    int wj = 0, xj = 0;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++wj) {
        int gi, tile, e, off, cnt;
        item_group(item, gi, tile);
        group_cols(gi, e, off, cnt);
        const int ws = wj % p.wstages;
        const bool wready = __all_sync(0xffffffffu, mbar_wait(&wfull[ws], static_cast<uint32_t>(wj / p.wstages) & 1u));
        if (!wready) *s_abort = 1;
        const saddr wslot = wring_s + static_cast<uint32_t>(ws * p.wslot);
        const int nchunks = (cnt + kGroupCols - 1) / kGroupCols;
        const int64_t r0 = static_cast<int64_t>(tile) * kGroupRows;
        for (int ch = 0; ch < nchunks; ++ch) {
            // GEMV: chunk 0 stays resident in slot 0 for every item
            const int xs = KIND == G_GEMV ? 0 : xj % p.xstages;
            const uint32_t xph = KIND == G_GEMV ? 0u : static_cast<uint32_t>(xj / p.xstages) & 1u;
            const bool xready = __all_sync(0xffffffffu, mbar_wait(&xfull[xs], xph));
            if (!xready) *s_abort = 1;
            GX x;
            x.base = xring_s + static_cast<uint32_t>(xs * p.xslot);
            x.xstride = p.xstride;
            x.ncols = cnt - ch * kGroupCols < kGroupCols ? cnt - ch * kGroupCols : kGroupCols;
            float acc[NMAT][4];
#pragma unroll
            for (int m = 0; m < NMAT; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.0f;
            if (wready && xready) {
                // dump: coefficient rows of this thread's outputs (rows g, g + 8; columns 2 tig, 2 tig + 1)
                int32_t* dq[NMAT][4] = {};
                if constexpr (DUMP) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int col = 2 * tig + (q & 1);
                        const int64_t row = r0 + g + 8 * (q >> 1);
                        if (col < x.ncols && row < p.N) {
                            const int pos = off + ch * kGroupCols + col;
                            const int64_t oc = KIND == G_GEMV ? pos : p.perm[pos];
#pragma unroll
                            for (int m = 0; m < NMAT; ++m) dq[m][q] = p.coefs[m] + (oc * p.N + row) * p.ncoef;
                        }
                    }
                }
                for (int sb = warp; sb < nsb; sb += kGroupConsumerWarps) {
#pragma unroll
                    for (int m = 0; m < NMAT; ++m) {
                        const saddr rb = wslot + static_cast<uint32_t>(m * kGroupRows * p.wrow);
                        group_superblock<F, DUMP>(rb + static_cast<uint32_t>(g * p.wrow),
                                                  rb + static_cast<uint32_t>((g + 8) * p.wrow), sb, x, g, tig, acc[m],
                                                  dq[m]);
                    }
                }
            }
            __syncwarp();
            if (KIND != G_GEMV && lane == 0) mbar_arrive(&xempty[xs]);
            if (KIND != G_GEMV) ++xj;
            // partials -> shared, reduced over the eight warps
#pragma unroll
            for (int m = 0; m < NMAT; ++m) {
                float* rw = red + (warp * NMAT + m) * 128;
                rw[g * 8 + 2 * tig] = acc[m][0];
                rw[g * 8 + 2 * tig + 1] = acc[m][1];
                rw[(g + 8) * 8 + 2 * tig] = acc[m][2];
                rw[(g + 8) * 8 + 2 * tig + 1] = acc[m][3];
            }
            group_sync();
            const int ctid = tid;
            if (ctid < 128) {
                const int row = ctid >> 3, col = ctid & 7;
                float v[NMAT];
#pragma unroll
                for (int m = 0; m < NMAT; ++m) {
                    float sum = 0.0f;
#pragma unroll
                    for (int w = 0; w < kGroupConsumerWarps; ++w) sum += red[(w * NMAT + m) * 128 + ctid];
                    v[m] = sum;
                }
                const int64_t grow = r0 + row;
                if (col < x.ncols && grow < p.N && wready && xready) {
                    const int pos = off + ch * kGroupCols + col;
                    if constexpr (KIND == G_GEMV) {
                        if (!DUMP || p.Y) p.Y[static_cast<int64_t>(pos) * p.N + grow] = v[0];
                    } else if constexpr (KIND == G_GATEUP) {
                        const int pair = p.perm[pos];
                        const float hval = __fmul_rn(__fdiv_rn(v[0], 1.0f + expf(-v[0])), v[NMAT - 1]);
                        const int64_t o = static_cast<int64_t>(pair) * p.N + grow;
                        p.h[o] = hval;
                        if (p.g_dump) p.g_dump[o] = v[0];
                        if (p.u_dump) p.u_dump[o] = v[NMAT - 1];
                    } else {
                        p.o[static_cast<int64_t>(p.perm[pos]) * p.N + grow] = v[0];
                    }
                }
            }
            group_sync();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&wempty[ws]);
        if (*s_abort) {  // read after the last group_sync of the item: the same for all warps
            set_error(p.err, DEV_ERR_TIMEOUT);
            break;
        }
    }
}

template <int KIND, int F, bool DUMP>
cudaError_t launch_group_one(const GroupParams& p, int grid, int smem, cudaStream_t s) {
    static std::atomic<bool> attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(k_group<KIND, F, DUMP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    return launch_pdl(k_group<KIND, F, DUMP>, dim3(grid), dim3(kGroupThreads), smem, s, p);
}

}  // namespace ggq

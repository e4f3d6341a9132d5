// ggq_gmm.cuh -- the expert-sorted grouped GEMM on f16 tensor cores: gate/up
// (+ SwiGLU) and down of the MoE layer once experts carry many columns
// (prefill).
//
// Same arithmetic as the keep-quant expert GEMM of vllm.cpp PR #523
// "grouped + non-grouped keep-quant expert GEMM" (What changed: the keep-quant
// matmul grouped over expert_ids, DotQ8_0/DotQ4K superblock dots): per block,
// (weight scale) * (activation scale) * (integer dot).  Here the integer dots
// run on mma.sync m16n8k16 with f16 operands holding integers: int8
// activations are exact in f16 (pre-converted once), Q8_0 codes are exact, and
// Q4_K codes enter already multiplied by their 6-bit sub-block scale
// (sc * q <= 945, exact).  Every product is exact; Q8_0 partials are taken per
// 32-block (|dot| < 2^19, exact) and scaled in f32 registers; Q4_K partials
// accumulate over a 256-superblock (possible rounding beyond 2^24, relative
// 2^-24) and take d, dmin and the activation scale at its end, the mins term
// being one more f16 product of the 6-bit mins with the activations' exact
// 16-group sums.
//
// Tiling: a work item is (expert, 64 weight rows, 128 columns); gate/up items
// take 32 gate rows and the same 32 up rows, interleaved by 16 so that every
// warp holds a gate value and its up value in the same fragment slot and forms
// SwiGLU in registers.  The activation operand is laid out in expert-sorted
// order (one f16 row per (token, expert) pair, gathered when it is converted),
// so an item's columns are consecutive rows and every operand of a 64-wide
// k-step is a 2-D TMA box:
//   * activations: 128 rows x 128 bytes, 128-byte swizzle (conflict-free
//     ldmatrix);
//   * weights: the k-step's raw bytes of 16 or 64 rows (Q8_0: the 80-byte
//     16-aligned span holding its two blocks; Q4_K: the 16-byte header and
//     the 32 nibble bytes), zero-filled past the row end;
//   * at a superblock's end: the activation scales and 16-group sums.
// Warp roles:
//   * one elected producer thread issues the TMA boxes of a k-step into a
//     6-stage ring (completion counted on one mbarrier per stage), four k-steps
//     ahead of the decode, across item boundaries;
//   * 4 producer warps decode the weight bytes of a k-step once into an f16
//     tile (double-buffered) that the consumer warps share;
//   * 8 consumer warps (2 x 4, 32 x 32 each) read fragments with ldmatrix and
//     run the mma, applying the block scales in registers.
// Decode and mma meet at hardware named barriers (tile full / tile free, one
// pair per f16 buffer); only the stage mbarriers are polled, with a bound: a
// wait that gives up sets the error word and the CTA runs to its end without
// further waits.
#pragma once
#include "ggq_device.cuh"
#include "ggq_internal.h"

namespace ggq {

constexpr int kGmmLd = kGmmBK + 8;  // halves per row of the decoded weight tile (16-byte pad: ldmatrix rows on distinct banks)
constexpr int kGmmRaw = 80;         // Q8_0 raw bytes per row per stage
constexpr int kGmmMaxGroups = 4096;
constexpr int kGmmConsumers = 256;  // threads
constexpr int kGmmProducers = 128;
constexpr int kGmmAhead = kGmmStages - 2;  // k-steps in flight beyond the one being decoded
constexpr int kGmmIssuers = 4;             // producer warps whose lane 0 issues TMA boxes
// named barrier ids (0 is __syncthreads)
constexpr int kBarAFull = 2, kBarAEmpty = 4;
static_assert(kGmmConsumers + kGmmProducers == kGmmThreads, "warp roles");

struct GmmSmem {
    static constexpr int kB16 = kGmmBN * kGmmBK * 2;        // 16384, 1024-aligned (swizzle atom)
    static constexpr int kRaw = kGmmBM * kGmmRaw;           // 5120 (Q4_K: headers 64 x 16, then nibbles 64 x 32)
    static constexpr int kDX = kGmmBN * 4 * 4;              // 2048: 4 superblock scales per column
    static constexpr int kBS = kGmmBN * 16 * 2;             // 4096: 16 group sums per column
    static constexpr int kStage = kB16 + kRaw + kDX + kBS;  // 27648 = 27 KB
    static constexpr int kA16 = kGmmBM * kGmmLd * 2;        // 9216
    static constexpr int kPrefix = (kGmmMaxGroups + 1) * 4;
    static constexpr int oA16 = kGmmStages * kStage;
    static constexpr int oPrefix = oA16 + 2 * kA16;
    static constexpr int oBars = (oPrefix + kPrefix + 7) / 8 * 8;
    static constexpr int kTotal = oBars + kGmmStages * 8 + 1024;  // + alignment slack of the dynamic base
};
static_assert(GmmSmem::kStage % 1024 == 0, "swizzled activation tiles stay 1024-aligned");
static_assert(GmmSmem::kTotal <= kSmemLimit, "grouped GEMM shared memory");

__device__ __forceinline__ void named_sync(int id, int n) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory"); }
__device__ __forceinline__ void named_arrive(int id, int n) { asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory"); }

// 2-D tiled TMA load of one box at element coordinates (x, y).
__device__ __forceinline__ void tma_2d(saddr dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(saddr a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}

__device__ __forceinline__ void gmm_mma(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// the same with a zero accumulator
__device__ __forceinline__ void gmm_mma_z(float* d, const uint32_t* a, uint32_t b0, uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1), "f"(0.0f));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }
__device__ __forceinline__ __half2 h2c(unsigned short bits) {
    return __halves2half2(__ushort_as_half(bits), __ushort_as_half(bits));
}

// 6-bit scales (sl: sub-blocks 0..3, sh: 4..7) and mins (ml, mh), one per
// byte, from the 12 packed scale bytes a0..a2 of a Q4_K superblock header.
__device__ __forceinline__ void k4_words(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t& sl, uint32_t& sh,
                                         uint32_t& ml, uint32_t& mh) {
    sl = a0 & 0x3F3F3F3Fu;
    ml = a1 & 0x3F3F3F3Fu;
    sh = (a2 & 0x0F0F0F0Fu) | ((a0 >> 2) & 0x30303030u);
    mh = ((a2 >> 4) & 0x0F0F0F0Fu) | ((a1 >> 2) & 0x30303030u);
}

// (v, v) as f16 for byte idx (runtime) of w (v <= 255)
__device__ __forceinline__ __half2 byte_pair(uint32_t w, int idx) {
    const uint32_t sel = 0x4040u | static_cast<uint32_t>(idx) | (static_cast<uint32_t>(idx) << 8);
    return __hsub2(u2h(prmt(w, 0u, sel) | 0x64006400u), h2c(0x6400u));
}

// One work item: expert e, m tile mt, columns [n0, n0 + ncols) of group gi.
struct GmmItem {
    int gi, mt, n0, ncols;
    int64_t e;
};

__device__ __forceinline__ GmmItem gmm_item(const GmmParams& p, const int* s_pref, int ngroups, int item) {
    int lo = 0, hi = ngroups - 1;  // last group with s_pref[g] <= item
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pref[mid] <= item) lo = mid; else hi = mid - 1;
    }
    GmmItem r;
    r.gi = lo;
    const int cnt = p.group_cnt[lo];
    const int ntl = (cnt + kGmmBN - 1) / kGmmBN;
    const int local = item - s_pref[lo];
    r.mt = local / ntl;
    r.n0 = (local - r.mt * ntl) * kGmmBN;
    r.ncols = min(cnt - r.n0, kGmmBN);
    r.e = p.group_expert[lo];
    return r;
}

template <int KIND, int F>
__global__ void __launch_bounds__(kGmmThreads, 1) k_gmm(const __grid_constant__ GmmParams p) {
    static_assert(F == F_Q8_0 || F == F_Q4_K, "grouped f16 GEMM formats");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* const smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();

    uint8_t* const a16 = smem + GmmSmem::oA16;
    int* const s_pref = reinterpret_cast<int*>(smem + GmmSmem::oPrefix);
    uint64_t* const full = reinterpret_cast<uint64_t*>(smem + GmmSmem::oBars);
    const auto B16 = [&](int s) { return smem + s * GmmSmem::kStage; };
    const auto RAW = [&](int s) { return smem + s * GmmSmem::kStage + GmmSmem::kB16; };
    const auto DXS = [&](int s) { return smem + s * GmmSmem::kStage + GmmSmem::kB16 + GmmSmem::kRaw; };
    const auto BSS = [&](int s) { return smem + s * GmmSmem::kStage + GmmSmem::kB16 + GmmSmem::kRaw + GmmSmem::kDX; };
    if (tid == 0) {
        for (int s = 0; s < kGmmStages; ++s) mbar_init(&full[s], 1);
        fence_barrier_init();
    }
    pdl_wait();  // groups, permutation and activations come from the previous kernels

    // ---- item table: per group, mtiles x ceil(cols / 128) items
    const int ngroups = *p.ngroups;
    constexpr int mrows = KIND == G_GATEUP ? kGmmBM / 2 : kGmmBM;  // distinct rows of one matrix per item
    const int mtiles = static_cast<int>(p.N / mrows);
    if (warp == 0) {  // exclusive prefix over the groups: lane l owns a contiguous run
        const int per = (ngroups + 31) >> 5, b0 = lane * per, b1 = min(b0 + per, ngroups);
        int own = 0;
        for (int gi = b0; gi < b1; ++gi) own += mtiles * ((p.group_cnt[gi] + kGmmBN - 1) / kGmmBN);
        int incl = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        int acc = incl - own;
        for (int gi = b0; gi < b1; ++gi) {
            s_pref[gi] = acc;
            acc += mtiles * ((p.group_cnt[gi] + kGmmBN - 1) / kGmmBN);
        }
        if (lane == 31) s_pref[ngroups] = incl;
    }
    __syncthreads();
    const int nitems = s_pref[ngroups];
    const int nk = p.K / kGmmBK;
    const int my_items = static_cast<int>(blockIdx.x) < nitems
                             ? (nitems - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
    const int total = my_items * nk;  // k-steps of this CTA
    constexpr uint32_t M = 0x64006400u;
    constexpr uint32_t kRawBytes = F == F_Q8_0 ? kGmmBM * kGmmRaw : kGmmBM * 48;

    if (tid >= kGmmConsumers) {
        // ================================================================ producers
        const int pt = tid - kGmmConsumers;
        GmmItem cur{};
        // TMA boxes of k-step c into its ring slot (nothing past the end).  Box j of the list
        // (0 activations, 1..kRawBoxes weights, then scales and group sums at a superblock's
        // end) is issued by lane 0 of producer warp j % kGmmIssuers: a TMA instruction keeps its
        // thread for a while, so the boxes of a k-step leave from several threads.
        constexpr int kRawBoxes = (KIND == G_GATEUP ? 4 : 1) * (F == F_Q8_0 ? 1 : 2);
        const auto issue = [&](int c) {
            const int role = pt >> 5;
            if ((pt & 31) != 0 || role >= kGmmIssuers || c >= total) return;
            const int it = c / nk, kt = c - it * nk, s = c % kGmmStages;
            if (kt == 0) cur = gmm_item(p, s_pref, ngroups, static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x));
            const bool sb_end = (kt & 3) == 3;
            if (role == 0) {
                uint32_t bytes = GmmSmem::kB16 + kRawBytes;
                if (sb_end) bytes += GmmSmem::kDX + (F == F_Q4_K ? GmmSmem::kBS : 0);
                mbar_arrive_expect_tx(&full[s], bytes);
            }
            const int y0 = p.group_off[cur.gi] + cur.n0;  // first sorted activation row of the item
            const saddr raw = smem_addr(RAW(s));
#pragma unroll
            for (int j = 0; j < kRawBoxes + 3; ++j) {
                if (j % kGmmIssuers != role) continue;
                if (j == 0) {
                    tma_2d(smem_addr(B16(s)), &p.tm_b, kt * kGmmBK, y0, &full[s]);
                } else if (j <= kRawBoxes) {
                    // gate/up: boxes of 16 rows alternate gate, up, gate, up
                    constexpr int parts = F == F_Q8_0 ? 1 : 2, nbox = kRawBoxes / parts, rows = kGmmBM / nbox;
                    const int k = (j - 1) / parts, part = (j - 1) % parts;
                    const int m = KIND == G_GATEUP ? (k & 1) : 0;
                    const int row = static_cast<int>(cur.e * p.N) + cur.mt * mrows + (KIND == G_GATEUP ? (k >> 1) * 16 : 0);
                    if constexpr (F == F_Q8_0) {
                        tma_2d(raw + static_cast<uint32_t>(k * rows * kGmmRaw), &p.tm_w[m][0], (68 * kt) & ~15, row, &full[s]);
                    } else if (part == 0) {
                        tma_2d(raw + static_cast<uint32_t>(k * rows * 16), &p.tm_w[m][0], (kt >> 2) * 144, row, &full[s]);
                    } else {
                        tma_2d(raw + static_cast<uint32_t>(kGmmBM * 16 + k * rows * 32), &p.tm_w[m][1],
                               (kt >> 2) * 144 + 16 + 32 * (kt & 3), row, &full[s]);
                    }
                } else if (j == kRawBoxes + 1) {
                    if (sb_end) tma_2d(smem_addr(DXS(s)), &p.tm_dx, (kt >> 2) & ~3, y0, &full[s]);
                } else if (F == F_Q4_K && sb_end) {
                    tma_2d(smem_addr(BSS(s)), &p.tm_bs, (kt >> 2) * 16, y0, &full[s]);
                }
            }
        };
        if (pt == 0) {  // descriptors into the TMA unit's cache before the first copies
            for (const CUtensorMap* m : {&p.tm_b, &p.tm_dx, &p.tm_bs, &p.tm_w[0][0], &p.tm_w[0][1], &p.tm_w[1][0], &p.tm_w[1][1]})
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
        }
        for (int c = 0; c < kGmmAhead; ++c) issue(c);
        bool live = true;  // false once a stage wait gave up: no further waits
        for (int d = 0; d < total; ++d) {
            // ---- decode k-step d into the f16 tile d & 1
            const int s = d % kGmmStages, b = d & 1, kt = d % nk;
            if (d >= 2) named_sync(kBarAEmpty + b, kGmmThreads);  // consumers are done with k-step d-2 (tile b, its ring slot)
            if (live && !mbar_wait(&full[s], (d / kGmmStages) & 1)) {
                set_error(p.err, DEV_ERR_TIMEOUT);
                live = false;
            }
            const uint8_t* raw = RAW(s);
            uint8_t* const at = a16 + b * GmmSmem::kA16;
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int r = (pt >> 3) + 16 * h, ge = pt & 7;
                uint32_t o4[4];
                if constexpr (F == F_Q8_0) {
                    const int o0 = (68 * kt) & 15;
                    const saddr src = smem_addr(raw) + static_cast<uint32_t>(r * kGmmRaw + o0 + 34 * (ge >> 2) + 2 + 8 * (ge & 3));
                    uint32_t w[2];
                    ld_words_any<2>(src, w);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint32_t u = w[k] ^ 0x80808080u;  // code + 128 per byte; 1152 = 1024 + 128
                        o4[2 * k] = h2u(__hsub2(u2h(prmt(u, 0u, 0x4140u) | M), h2c(0x6480u)));
                        o4[2 * k + 1] = h2u(__hsub2(u2h(prmt(u, 0u, 0x4342u) | M), h2c(0x6480u)));
                    }
                } else {
                    const uint4 hd = ld_s128(smem_addr(raw) + static_cast<uint32_t>(r * 16));
                    uint32_t sl, sh, ml, mh;
                    k4_words(hd.y, hd.z, hd.w, sl, sh, ml, mh);
                    const int js = 2 * (kt & 3) + (ge >> 2);  // sub-block of this group of 8
                    const __half2 sc = byte_pair(js < 4 ? sl : sh, js & 3);
                    const saddr qa = smem_addr(raw) + static_cast<uint32_t>(kGmmBM * 16 + r * 32 + 8 * (ge & 3));
                    const uint32_t qw[2] = {ld_s32(qa), ld_s32(qa + 4)};
                    if (ge < 4) {  // low nibbles: (1024 + n) sc - 1024 sc
                        const __half2 cc = __hmul2(sc, h2c(0xE400u));
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            o4[2 * k] = h2u(__hfma2(u2h((prmt(qw[k], 0u, 0x4140u) & 0x000F000Fu) | M), sc, cc));
                            o4[2 * k + 1] = h2u(__hfma2(u2h((prmt(qw[k], 0u, 0x4342u) & 0x000F000Fu) | M), sc, cc));
                        }
                    } else {  // high nibbles masked in place: (1024 + 16 n) sc/16 - 64 sc
                        const __half2 s16 = __hmul2(sc, h2c(0x2C00u));
                        const __half2 cc = __hmul2(sc, h2c(0xD400u));
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            o4[2 * k] = h2u(__hfma2(u2h((prmt(qw[k], 0u, 0x4140u) & 0x00F000F0u) | M), s16, cc));
                            o4[2 * k + 1] = h2u(__hfma2(u2h((prmt(qw[k], 0u, 0x4342u) & 0x00F000F0u) | M), s16, cc));
                        }
                    }
                }
                *reinterpret_cast<uint4*>(at + (r * kGmmLd + 8 * ge) * 2) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
            named_arrive(kBarAFull + b, kGmmThreads);
            issue(d + kGmmAhead);  // into the ring slot of k-step d-2
        }
        return;
    }

    // ==================================================================== consumers
    const int wm = warp & 1, wn = warp >> 1;  // 2 x 4 warps, 32 x 32 each
    const int g = lane >> 2, t = lane & 3;
    bool live = true;
    for (int it = 0; it < my_items; ++it) {
        const GmmItem cur = gmm_item(p, s_pref, ngroups, static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x));
        int pc[4][2];  // output pair of each column this thread stores (-1: none)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int col = wn * 32 + 8 * j + 2 * t + cc;
                pc[j][cc] = col < cur.ncols ? p.perm[p.group_off[cur.gi] + cur.n0 + col] : -1;
            }
        float acc[2][4][4], D[2][4][4], T[2][4][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][j][q] = 0.0f;
        for (int kt = 0; kt < nk; ++kt) {
            const int c = it * nk + kt, s = c % kGmmStages, b = c & 1;
            named_sync(kBarAFull + b, kGmmThreads);
            // the producers saw this stage land; observe it here too (already complete)
            if (live && !mbar_wait(&full[s], (c / kGmmStages) & 1)) {
                set_error(p.err, DEV_ERR_TIMEOUT);
                live = false;
            }
            const saddr a_base = smem_addr(a16 + b * GmmSmem::kA16), b_base = smem_addr(B16(s));
            const saddr raw = smem_addr(RAW(s));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t af[2][4], bf[4][2];
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    ldmatrix_x4(a_base + static_cast<uint32_t>(((wm * 32 + 16 * i + (lane & 15)) * kGmmLd + kk * 16 + (lane >> 4) * 8) * 2),
                                af[i][0], af[i][1], af[i][2], af[i][3]);
                // activation tile: row = column of the item, 16-byte chunk index xor (row & 7)
                const int chunk = kk * 2 + ((lane >> 3) & 1);
#pragma unroll
                for (int jp = 0; jp < 2; ++jp)
                    ldmatrix_x4(b_base + static_cast<uint32_t>((wn * 32 + 16 * jp + (lane & 7) + ((lane >> 4) << 3)) * 128 +
                                                               ((chunk ^ (lane & 7)) << 4)),
                                bf[2 * jp][0], bf[2 * jp][1], bf[2 * jp + 1][0], bf[2 * jp + 1][1]);
                // a fresh accumulator at the start of a 32-block (Q8_0) or of a superblock (Q4_K)
                const bool fresh = F == F_Q8_0 ? (kk & 1) == 0 : (kk == 0 && (kt & 3) == 0);
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        if (fresh) gmm_mma_z(D[i][j], af[i], bf[j][0], bf[j][1]);
                        else gmm_mma(D[i][j], af[i], bf[j][0], bf[j][1]);
                    }
                if constexpr (F == F_Q8_0) {
                    if (kk & 1) {  // end of a 32-block: T (+)= D * d_w; the activation scale waits for the superblock
                        const int blk = kk >> 1, o0 = (68 * kt) & 15;
                        float dw[2][2];
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh)
                                dw[i][hh] = ld_h(raw + static_cast<uint32_t>((wm * 32 + 16 * i + g + 8 * hh) * kGmmRaw + o0 + 34 * blk));
                        const bool first = blk == 0 && (kt & 3) == 0;
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int j = 0; j < 4; ++j)
#pragma unroll
                                for (int q = 0; q < 4; ++q)
                                    T[i][j][q] = first ? D[i][j][q] * dw[i][q >> 1] : fmaf(D[i][j][q], dw[i][q >> 1], T[i][j][q]);
                    }
                }
            }
            if ((kt & 3) == 3) {  // end of a superblock: activation scale (and Q4_K: d, mins)
                const saddr dxs = smem_addr(DXS(s)) + 4u * ((kt >> 2) & 3);
                float dv[4][2];
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) dv[j][cc] = ld_f32(dxs + 16u * (wn * 32 + 8 * j + 2 * t + cc));
                if constexpr (F == F_Q8_0) {
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[i][j][q] = fmaf(T[i][j][q], dv[j][q & 1], acc[i][j][q]);
                } else {
                    float dd[2][2], dm[2][2];
                    uint32_t amin[2][4];  // [m tile] A fragment of the mins: k slot q <-> 16-group q (sub-block q / 2)
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const uint4 hd = ld_s128(raw + static_cast<uint32_t>((wm * 32 + 16 * i + g + 8 * hh) * 16));
                            dd[i][hh] = half_lo(hd.x);
                            dm[i][hh] = half_hi(hd.x);
                            uint32_t sl, sh, ml, mh;
                            k4_words(hd.y, hd.z, hd.w, sl, sh, ml, mh);
                            amin[i][hh] = h2u(byte_pair(ml, t));      // k 2t, 2t+1: sub-block t
                            amin[i][2 + hh] = h2u(byte_pair(mh, t));  // k 2t+8, 2t+9: sub-block 4+t
                        }
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[i][j][q] = fmaf(D[i][j][q], dd[i][q >> 1] * dv[j][q & 1], acc[i][j][q]);
                    const saddr bss = smem_addr(BSS(s));
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int col = wn * 32 + 8 * j + g;
                        const uint32_t b0 = ld_s32(bss + static_cast<uint32_t>((col * 16 + 2 * t) * 2));
                        const uint32_t b1 = ld_s32(bss + static_cast<uint32_t>((col * 16 + 2 * t + 8) * 2));
#pragma unroll
                        for (int i = 0; i < 2; ++i) gmm_mma_z(D[i][j], amin[i], b0, b1);
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[i][j][q] = fmaf(-D[i][j][q], dm[i][q >> 1] * dv[j][q & 1], acc[i][j][q]);
                }
            }
            if (c + 2 < total) named_arrive(kBarAEmpty + b, kGmmThreads);
        }
        // ---- epilogue
        if constexpr (KIND == G_GATEUP) {
            // m tile 0 of the warp holds gate rows, m tile 1 the up rows of the same outputs
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int r = wm * 16 + g + 8 * (q >> 1);
                    const int pair = pc[j][q & 1];
                    if (pair >= 0) {
                        const float gv = acc[0][j][q], uv = acc[1][j][q];
                        const int64_t o = static_cast<int64_t>(pair) * p.N + static_cast<int64_t>(cur.mt) * 32 + r;
                        p.h[o] = __fmul_rn(__fdiv_rn(gv, 1.0f + expf(-gv)), uv);
                        if (p.g_dump) p.g_dump[o] = gv;
                        if (p.u_dump) p.u_dump[o] = uv;
                    }
                }
        } else {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = wm * 32 + 16 * i + g + 8 * (q >> 1);
                        const int pair = pc[j][q & 1];
                        if (pair >= 0) p.o[static_cast<int64_t>(pair) * p.N + static_cast<int64_t>(cur.mt) * kGmmBM + r] = acc[i][j][q];
                    }
        }
    }
}

template <int KIND, int F>
cudaError_t launch_gmm_one(const GmmParams& p, int grid, int smem, cudaStream_t s) {
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(k_gmm<KIND, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    return launch_pdl(k_gmm<KIND, F>, dim3(grid), dim3(kGmmThreads), smem, s, p);
}

}  // namespace ggq

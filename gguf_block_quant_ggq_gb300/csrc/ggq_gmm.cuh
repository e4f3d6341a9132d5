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
// accumulate in two 128-wide chains per 256-superblock (|partial| <= 128 * 945
// * 127 < 2^24: each chain holds its exact integer) and take d, dmin and the
// activation scale at the superblock's end, the mins term being one more f16
// product of the 6-bit mins with the activations' exact 16-group sums.
//
// Tiling: a work item is (expert, 64 weight rows, 128 columns); gate/up items
// take 32 gate rows and the same 32 up rows (one weight box each), and the
// decode interleaves them by 16 in the f16 tile so that every warp holds a gate
// value and its up value in the same fragment slot and forms SwiGLU in
// registers.  The activation operand is laid out in expert-sorted
// order (one f16 row per (token, expert) pair, gathered when it is converted),
// so an item's columns are consecutive rows and every operand of a 64-wide
// k-step is a 2-D TMA box:
//   * activations: 128 rows x 128 bytes, 128-byte swizzle (conflict-free
//     ldmatrix);
//   * weights: the k-step's raw bytes of 32 or 64 rows (Q8_0: the 80-byte
//     16-aligned span holding its two blocks; Q4_K: the 16-byte header and
//     the 32 nibble bytes), zero-filled past the row end;
//   * at a superblock's end: the activation scales and 16-group sums.
// Warp roles:
//   * one thread of the last producer warp issues the TMA boxes of each k-step
//     into a 6-stage ring (completion counted on one mbarrier per stage, slot
//     release on another, arrived by the consumer warps), as far ahead as the
//     ring allows, across item boundaries: a box instruction holds its thread
//     for several hundred cycles, so this thread does nothing else;
//   * 3 producer warps decode the weight bytes of a k-step once into an f16
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

#include <atomic>

namespace ggq {

constexpr int kGmmLd = kGmmBK + 8;  // halves per row of the decoded weight tile (16-byte pad: ldmatrix rows on distinct banks)
constexpr int kGmmRaw = 80;         // Q8_0 raw bytes per row per stage
constexpr int kGmmMaxGroups = 4096;
constexpr int kGmmConsumers = 256;  // threads
constexpr int kGmmProducers = 128;
constexpr int kGmmDecoders = 96;           // producer threads that decode (the last producer warp issues TMA)
constexpr int kGmmSync = kGmmConsumers + kGmmDecoders;  // threads on the tile full / free barriers
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
    static constexpr int kTotal = oBars + 2 * kGmmStages * 8 + 1024;  // + alignment slack of the dynamic base
};
static_assert(GmmSmem::kStage % 1024 == 0, "swizzled activation tiles stay 1024-aligned");
static_assert(GmmSmem::kTotal <= kSmemLimit, "grouped GEMM shared memory");

// Bounded wait that suspends between probes (try_wait) instead of spinning: for
// the TMA thread, which runs ahead and should leave issue slots to the others.
__device__ __forceinline__ bool mbar_wait_sleep(uint64_t* bar, uint32_t parity) {
    const long long t0 = clock64();
    for (;;) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
        if (clock64() - t0 > (1ll << 32)) return false;
    }
}

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

// Raw weight rows hold gate rows 0..31 then up rows 0..31 of a gate/up item; the
// f16 tile row of raw row r swaps bits 4 and 5 of r (gate 16, up 16, gate 16,
// up 16).  The map is its own inverse.
template <int KIND>
__device__ __forceinline__ int tile_row(int r) {
    if constexpr (KIND == G_GATEUP) return (r & ~48) | ((r & 16) << 1) | ((r & 32) >> 1);
    else return r;
}

// One work item: expert e, m tile mt, columns [n0, n0 + ncols) of group gi.
struct GmmItem {
    int gi, mt, n0, ncols;
    int y0;     // first sorted activation row of the item
    int wrow;   // first weight row of the item in its bank (e * N + mt * rows per matrix)
    int64_t e;
};

template <int KIND>
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
    r.y0 = p.group_off[lo] + r.n0;
    r.wrow = static_cast<int>(r.e * p.N) + r.mt * (KIND == G_GATEUP ? kGmmBM / 2 : kGmmBM);
    return r;
}

// Integer-core dump of a consumer warp's 32 x 32 tile: coefficient idx of each
// of its outputs gets D (plus E when given: the second half-superblock chain),
// each an exact integer held in f32.  Gate/up: m tile i of the warp is matrix i
// (gate, up); down: both m tiles are rows of the one matrix.
template <int KIND>
__device__ __forceinline__ void dump_tile(const GmmParams& p, const float (&D)[2][4][4], const int (&pc)[4][2], int mt,
                                          int wm, int g, int idx, const float (*E)[4][4] = nullptr) {
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int pair = pc[j][q & 1];
                if (pair < 0) continue;
                int v = __float2int_rn(D[i][j][q]);
                if (E) v += __float2int_rn(E[i][j][q]);
                const int m = KIND == G_GATEUP ? i : 0;
                const int64_t row = KIND == G_GATEUP ? static_cast<int64_t>(mt) * 32 + wm * 16 + g + 8 * (q >> 1)
                                                     : static_cast<int64_t>(mt) * kGmmBM + wm * 32 + 16 * i + g + 8 * (q >> 1);
                p.coefs[m][(static_cast<int64_t>(pair) * p.N + row) * p.ncoef + idx] = v;
            }
}

template <int KIND, int F, bool DUMP>
__global__ void __launch_bounds__(kGmmThreads, 1) k_gmm(const __grid_constant__ GmmParams p) {
    static_assert(F == F_Q8_0 || F == F_Q4_K, "grouped f16 GEMM formats");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* const smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();

    uint8_t* const a16 = smem + GmmSmem::oA16;
    int* const s_pref = reinterpret_cast<int*>(smem + GmmSmem::oPrefix);
    uint64_t* const full = reinterpret_cast<uint64_t*>(smem + GmmSmem::oBars);
    uint64_t* const empty = full + kGmmStages;
    const auto B16 = [&](int s) { return smem + s * GmmSmem::kStage; };
    const auto RAW = [&](int s) { return smem + s * GmmSmem::kStage + GmmSmem::kB16; };
    const auto DXS = [&](int s) { return smem + s * GmmSmem::kStage + GmmSmem::kB16 + GmmSmem::kRaw; };
    const auto BSS = [&](int s) { return smem + s * GmmSmem::kStage + GmmSmem::kB16 + GmmSmem::kRaw + GmmSmem::kDX; };
    if (tid == 0) {
        for (int s = 0; s < kGmmStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kGmmConsumers / 32);
        }
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
    constexpr uint32_t kRawBytes = F == F_Q8_0 ? kGmmBM * kGmmRaw : kGmmBM * 48;

    if (tid >= kGmmConsumers) {
        // ================================================================ producers
        const int pt = tid - kGmmConsumers;
        if (pt >= kGmmDecoders) {
            // ---------------------------------------------------------- TMA issue
            if (pt != kGmmDecoders) return;
            for (const CUtensorMap* m : {&p.tm_b, &p.tm_dx, &p.tm_bs, &p.tm_w[0][0], &p.tm_w[0][1], &p.tm_w[1][0], &p.tm_w[1][1]})
                asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
            GmmItem cur{};
            for (int c = 0; c < total; ++c) {
                const int it = c / nk, kt = c - it * nk, s = c % kGmmStages;
                if (kt == 0) cur = gmm_item<KIND>(p, s_pref, ngroups, static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x));
                // the slot's previous k-step (c - kGmmStages) is done: decoded and consumed
                if (c >= kGmmStages && !mbar_wait_sleep(&empty[s], ((c / kGmmStages) - 1) & 1)) {
                    set_error(p.err, DEV_ERR_TIMEOUT);
                    return;
                }
                const bool sb_end = (kt & 3) == 3;
                uint32_t bytes = GmmSmem::kB16 + kRawBytes;
                if (sb_end) bytes += GmmSmem::kDX + (F == F_Q4_K ? GmmSmem::kBS : 0);
                mbar_arrive_expect_tx(&full[s], bytes);
                tma_2d(smem_addr(B16(s)), &p.tm_b, kt * kGmmBK, cur.y0, &full[s]);
                const saddr raw = smem_addr(RAW(s));
#pragma unroll
                for (int k = 0; k < (KIND == G_GATEUP ? 2 : 1); ++k) {
                    // gate/up: a box of 32 gate rows, then a box of the same 32 up rows
                    constexpr int rows = KIND == G_GATEUP ? kGmmBM / 2 : kGmmBM;
                    if constexpr (F == F_Q8_0) {
                        tma_2d(raw + static_cast<uint32_t>(k * rows * kGmmRaw), &p.tm_w[k][0], (68 * kt) & ~15, cur.wrow, &full[s]);
                    } else {
                        tma_2d(raw + static_cast<uint32_t>(k * rows * 16), &p.tm_w[k][0], (kt >> 2) * 144, cur.wrow, &full[s]);
                        tma_2d(raw + static_cast<uint32_t>(kGmmBM * 16 + k * rows * 32), &p.tm_w[k][1],
                               (kt >> 2) * 144 + 16 + 32 * (kt & 3), cur.wrow, &full[s]);
                    }
                }
                if (sb_end) {
                    tma_2d(smem_addr(DXS(s)), &p.tm_dx, (kt >> 2) & ~3, cur.y0, &full[s]);
                    if constexpr (F == F_Q4_K) tma_2d(smem_addr(BSS(s)), &p.tm_bs, (kt >> 2) * 16, cur.y0, &full[s]);
                }
            }
            return;
        }
        // -------------------------------------------------------------- decode
        bool live = true;  // false once a stage wait gave up: no further waits
        for (int d = 0; d < total; ++d) {
            // ---- decode k-step d into the f16 tile d & 1
            const int s = d % kGmmStages, b = d & 1, kt = d % nk;
            if (d >= 2) named_sync(kBarAEmpty + b, kGmmSync);  // consumers are done with k-step d-2 (tile b)
            if (live && !mbar_wait(&full[s], (d / kGmmStages) & 1)) {
                set_error(p.err, DEV_ERR_TIMEOUT);
                live = false;
            }
            const saddr raw = smem_addr(RAW(s));
            uint8_t* const at = a16 + b * GmmSmem::kA16;
            // 256 units of 16 outputs per k-step, up to kUnits per thread; all shared-memory
            // reads of the thread's units first, then the conversions (independent chains)
            constexpr int kUnits = (kGmmBM * 4 + kGmmDecoders - 1) / kGmmDecoders;
            if constexpr (F == F_Q8_0) {
                // unit: 16 codes of one row (half of a 32-block): row u >> 2, block (u >> 1) & 1, half u & 1
                const int o0 = (68 * kt) & 15;
                uint32_t w[kUnits][4];
#pragma unroll
                for (int h = 0; h < kUnits; ++h) {
                    const int u = pt + kGmmDecoders * h;
                    if (u < kGmmBM * 4)
                        ld_words_any<4>(raw + static_cast<uint32_t>((u >> 2) * kGmmRaw + o0 + 34 * ((u >> 1) & 1) + 2 + 16 * (u & 1)), w[h]);
                }
#pragma unroll
                for (int h = 0; h < kUnits; ++h) {
                    const int u = pt + kGmmDecoders * h;
                    if (u >= kGmmBM * 4) break;
                    uint32_t o8[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // code + 128 per byte (xor), as 1024 + (code + 128) (prmt with 0x64 high bytes), minus 1152
                        const uint32_t v = w[h][k] ^ 0x80808080u;
                        o8[2 * k] = h2u(__hsub2(u2h(prmt(v, 0x64646464u, 0x4140u)), h2c(0x6480u)));
                        o8[2 * k + 1] = h2u(__hsub2(u2h(prmt(v, 0x64646464u, 0x4342u)), h2c(0x6480u)));
                    }
                    uint8_t* const dst = at + (tile_row<KIND>(u >> 2) * kGmmLd + 16 * (u & 3)) * 2;
                    *reinterpret_cast<uint4*>(dst) = make_uint4(o8[0], o8[1], o8[2], o8[3]);
                    *reinterpret_cast<uint4*>(dst + 16) = make_uint4(o8[4], o8[5], o8[6], o8[7]);
                }
            } else {
                // unit: 8 nibble bytes of one row, group u & 3: low nibbles are outputs 8 (u & 3) .. +7
                // (sub-block 2 (kt & 3)), high nibbles outputs 32 + 8 (u & 3) .. +7 (the next sub-block)
                uint4 hd[kUnits];
                uint32_t qw[kUnits][2];
#pragma unroll
                for (int h = 0; h < kUnits; ++h) {
                    const int u = pt + kGmmDecoders * h;
                    if (u < kGmmBM * 4) {
                        hd[h] = ld_s128(raw + static_cast<uint32_t>((u >> 2) * 16));
                        const saddr qa = raw + static_cast<uint32_t>(kGmmBM * 16 + (u >> 2) * 32 + 8 * (u & 3));
                        qw[h][0] = ld_s32(qa);
                        qw[h][1] = ld_s32(qa + 4);
                    }
                }
                const int cc = kt & 3;
#pragma unroll
                for (int h = 0; h < kUnits; ++h) {
                    const int u = pt + kGmmDecoders * h;
                    if (u >= kGmmBM * 4) break;
                    // 6-bit scales of sub-blocks 2 cc (low nibbles) and 2 cc + 1 (high nibbles)
                    const uint32_t sw = cc < 2 ? (hd[h].y & 0x3F3F3F3Fu)
                                               : ((hd[h].w & 0x0F0F0F0Fu) | ((hd[h].y >> 2) & 0x30303030u));
                    const __half2 slo = byte_pair(sw, 2 * (cc & 1)), shi = byte_pair(sw, 2 * (cc & 1) + 1);
                    const __half2 clo = __hmul2(slo, h2c(0xE400u));                      // -1024 sc
                    const __half2 s16 = __hmul2(shi, h2c(0x2C00u)), chi = __hmul2(shi, h2c(0xD400u));  // sc / 16, -64 sc
                    uint32_t lo[4], hi[4];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint32_t x0 = prmt(qw[h][k], 0x64646464u, 0x4140u), x1 = prmt(qw[h][k], 0x64646464u, 0x4342u);
                        // low nibble: (1024 + n) sc - 1024 sc; high nibble in place: (1024 + 16 n) sc/16 - 64 sc
                        lo[2 * k] = h2u(__hfma2(u2h(x0 & 0xFF0FFF0Fu), slo, clo));
                        lo[2 * k + 1] = h2u(__hfma2(u2h(x1 & 0xFF0FFF0Fu), slo, clo));
                        hi[2 * k] = h2u(__hfma2(u2h(x0 & 0xFFF0FFF0u), s16, chi));
                        hi[2 * k + 1] = h2u(__hfma2(u2h(x1 & 0xFFF0FFF0u), s16, chi));
                    }
                    uint8_t* const dst = at + (tile_row<KIND>(u >> 2) * kGmmLd + 8 * (u & 3)) * 2;
                    *reinterpret_cast<uint4*>(dst) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<uint4*>(dst + 64) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                }
            }
            named_arrive(kBarAFull + b, kGmmSync);
        }
        return;
    }

    // ==================================================================== consumers
    const int wm = warp & 1, wn = warp >> 1;  // 2 x 4 warps, 32 x 32 each
    const int g = lane >> 2, t = lane & 3;
    bool live = true;
    for (int it = 0; it < my_items; ++it) {
        const GmmItem cur = gmm_item<KIND>(p, s_pref, ngroups, static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x));
        int pc[4][2];  // output pair of each column this thread stores (-1: none)
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
                const int col = wn * 32 + 8 * j + 2 * t + cc;
                pc[j][cc] = col < cur.ncols ? p.perm[cur.y0 + col] : -1;
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
            named_sync(kBarAFull + b, kGmmSync);
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
                // a fresh accumulator at the start of a 32-block (Q8_0) or of a 128-wide half
                // superblock (Q4_K: first half in D, second half in T)
                const bool fresh = F == F_Q8_0 ? (kk & 1) == 0 : (kk == 0 && (kt & 1) == 0);
                const bool second = F == F_Q4_K && ((kt >> 1) & 1);
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        float* const acc_c = second ? T[i][j] : D[i][j];
                        if (fresh) gmm_mma_z(acc_c, af[i], bf[j][0], bf[j][1]);
                        else gmm_mma(acc_c, af[i], bf[j][0], bf[j][1]);
                    }
                if constexpr (F == F_Q8_0) {
                    if (kk & 1) {  // end of a 32-block: T (+)= D * d_w; the activation scale waits for the superblock
                        const int blk = kk >> 1, o0 = (68 * kt) & 15;
                        float dw[2][2];
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh)
                                dw[i][hh] = ld_h(raw + static_cast<uint32_t>(tile_row<KIND>(wm * 32 + 16 * i + g + 8 * hh) * kGmmRaw + o0 + 34 * blk));
                        const bool first = blk == 0 && (kt & 3) == 0;
                        if constexpr (DUMP) dump_tile<KIND>(p, D, pc, cur.mt, wm, g, 2 * kt + blk);
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
                            const uint4 hd = ld_s128(raw + static_cast<uint32_t>(tile_row<KIND>(wm * 32 + 16 * i + g + 8 * hh) * 16));
                            dd[i][hh] = half_lo(hd.x);
                            dm[i][hh] = half_hi(hd.x);
                            uint32_t sl, sh, ml, mh;
                            k4_words(hd.y, hd.z, hd.w, sl, sh, ml, mh);
                            amin[i][hh] = h2u(byte_pair(ml, t));      // k 2t, 2t+1: sub-block t
                            amin[i][2 + hh] = h2u(byte_pair(mh, t));  // k 2t+8, 2t+9: sub-block 4+t
                        }
                    if constexpr (DUMP) dump_tile<KIND>(p, D, pc, cur.mt, wm, g, 2 * (kt >> 2), T);
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                D[i][j][q] += T[i][j][q];  // the two exact half-superblock chains
                                acc[i][j][q] = fmaf(D[i][j][q], dd[i][q >> 1] * dv[j][q & 1], acc[i][j][q]);
                            }
                    const saddr bss = smem_addr(BSS(s));
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int col = wn * 32 + 8 * j + g;
                        const uint32_t b0 = ld_s32(bss + static_cast<uint32_t>((col * 16 + 2 * t) * 2));
                        const uint32_t b1 = ld_s32(bss + static_cast<uint32_t>((col * 16 + 2 * t + 8) * 2));
#pragma unroll
                        for (int i = 0; i < 2; ++i) gmm_mma_z(D[i][j], amin[i], b0, b1);
                    }
                    if constexpr (DUMP) dump_tile<KIND>(p, D, pc, cur.mt, wm, g, 2 * (kt >> 2) + 1);
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int q = 0; q < 4; ++q) acc[i][j][q] = fmaf(-D[i][j][q], dm[i][q >> 1] * dv[j][q & 1], acc[i][j][q]);
                }
            }
            if (c + 2 < total) named_arrive(kBarAEmpty + b, kGmmSync);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);  // the ring slot may take k-step c + kGmmStages
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

template <int KIND, int F, bool DUMP>
cudaError_t launch_gmm_one(const GmmParams& p, int grid, int smem, cudaStream_t s) {
    static std::atomic<bool> attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(k_gmm<KIND, F, DUMP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    return launch_pdl(k_gmm<KIND, F, DUMP>, dim3(grid), dim3(kGmmThreads), smem, s, p);
}

}  // namespace ggq

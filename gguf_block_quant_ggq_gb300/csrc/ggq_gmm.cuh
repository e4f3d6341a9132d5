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
// take 32 gate rows and the same 32 up rows so that SwiGLU is formed in the
// CTA.  Eight warps (2 x 4), 32 x 32 each.  A k-step of 64: all threads copy
// the activation tile (f16) and the raw weight bytes with cp.async into a
// 4-stage ring, then decode the weight tile once into an f16 tile that the
// four column warps share; fragments come from ldmatrix.
#pragma once
#include "ggq_device.cuh"
#include "ggq_internal.h"

namespace ggq {

constexpr int kGmmLd = kGmmBK + 8;   // halves per row of the f16 operand tiles (16-byte pad: ldmatrix rows on distinct banks)
constexpr int kGmmRaw = 80;          // raw weight bytes per row per stage
constexpr int kGmmBsLd = 24;         // halves per column of the 16-group sums
constexpr int kGmmMaxGroups = 4096;

struct GmmSmem {
    static constexpr int kB16 = kGmmBN * kGmmLd * 2;           // 18432
    static constexpr int kRaw = kGmmBM * kGmmRaw;              // 5120
    static constexpr int kDX = kGmmBN * 4;                     // 512
    static constexpr int kBS = kGmmBN * kGmmBsLd * 2;          // 6144
    static constexpr int kStage = kB16 + kRaw + kDX + kBS;     // 30208
    static constexpr int kA16 = kGmmBM * kGmmLd * 2;           // 9216
    static constexpr int kMeta = 2 * kGmmBN * 4;               // column pairs and activation rows
    static constexpr int kPrefix = (kGmmMaxGroups + 1) * 4;
    static constexpr int kTotal = kGmmStages * kStage + kA16 + kMeta + kPrefix;
};

__device__ __forceinline__ void cp_async16(saddr dst, const void* src, int bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async4(saddr dst, const void* src, int bytes) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(dst), "l"(src), "r"(bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldmatrix_x4(saddr a, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(a));
}

__device__ __forceinline__ void gmm_mma(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                        uint32_t b1) {
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t h2u(__half2 h) { return *reinterpret_cast<const uint32_t*>(&h); }
__device__ __forceinline__ __half2 u2h(uint32_t u) { return *reinterpret_cast<const __half2*>(&u); }

// 6-bit scales (or mins) of the eight sub-blocks of a Q4_K superblock header:
// bytes 0..3 of lo and hi.
__device__ __forceinline__ void k4_words(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t& sl, uint32_t& sh,
                                         uint32_t& ml, uint32_t& mh) {
    sl = a0 & 0x3F3F3F3Fu;
    ml = a1 & 0x3F3F3F3Fu;
    sh = (a2 & 0x0F0F0F0Fu) | ((a0 >> 2) & 0x30303030u);
    mh = ((a2 >> 4) & 0x0F0F0F0Fu) | ((a1 >> 2) & 0x30303030u);
}

// (v, v) as f16 for the byte idx (runtime) of w (v <= 63)
__device__ __forceinline__ __half2 byte_pair(uint32_t w, int idx) {
    const uint32_t sel = 0x4040u | static_cast<uint32_t>(idx) | (static_cast<uint32_t>(idx) << 8);
    const uint32_t u = (prmt(w, 0u, sel) & 0x00FF00FFu) | 0x64006400u;
    return __hsub2(u2h(u), __halves2half2(__ushort_as_half(0x6400u), __ushort_as_half(0x6400u)));
}

template <int KIND, int F>
__global__ void __launch_bounds__(kGmmThreads, 1) k_gmm(const GmmParams p) {
    static_assert(F == F_Q8_0 || F == F_Q4_K, "grouped f16 GEMM formats");
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int wm = warp & 1, wn = warp >> 1;  // 2 x 4 warps, 32 x 32 each
    const int g = lane >> 2, t = lane & 3;
    pdl_launch_dependents();
    pdl_wait();  // groups, permutation and activations come from the previous kernels

    uint8_t* stage0 = smem;
    uint8_t* a16 = smem + kGmmStages * GmmSmem::kStage;
    int* s_pair = reinterpret_cast<int*>(a16 + GmmSmem::kA16);
    int* s_brow = s_pair + kGmmBN;
    int* s_pref = s_brow + kGmmBN;
    const auto B16 = [&](int s) { return stage0 + s * GmmSmem::kStage; };
    const auto RAW = [&](int s) { return stage0 + s * GmmSmem::kStage + GmmSmem::kB16; };
    const auto DXS = [&](int s) { return reinterpret_cast<float*>(stage0 + s * GmmSmem::kStage + GmmSmem::kB16 + GmmSmem::kRaw); };
    const auto BSS = [&](int s) { return stage0 + s * GmmSmem::kStage + GmmSmem::kB16 + GmmSmem::kRaw + GmmSmem::kDX; };

    // ---- item table: per group, (rows / 64 or 32) x ceil(cols / 128) items
    const int ngroups = *p.ngroups;
    const int mrows = KIND == G_GATEUP ? kGmmBM / 2 : kGmmBM;  // distinct weight rows per item
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
    constexpr uint32_t M = 0x64006400u;

    for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
        // group of the item: last gi with s_pref[gi] <= item
        int lo = 0, hi = ngroups - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (s_pref[mid] <= item) lo = mid; else hi = mid - 1;
        }
        const int gi = lo;
        const int cnt = p.group_cnt[gi];
        const int ntl = (cnt + kGmmBN - 1) / kGmmBN;
        const int local = item - s_pref[gi];
        const int mt = local / ntl, nt = local - mt * ntl;
        const int64_t e = p.group_expert[gi];
        const int n0 = nt * kGmmBN;
        const int ncols = cnt - n0 < kGmmBN ? cnt - n0 : kGmmBN;
        if (tid < kGmmBN) {
            const int pair = tid < ncols ? p.perm[p.group_off[gi] + n0 + tid] : -1;
            s_pair[tid] = pair;
            s_brow[tid] = pair < 0 ? -1 : (KIND == G_GATEUP ? pair / p.top_k : pair);
        }
        __syncthreads();

        // bank row of A-tile row r
        const auto arow = [&](int r) -> const uint8_t* {
            if constexpr (KIND == G_GATEUP)
                return (r < kGmmBM / 2 ? p.W : p.W2) + (e * p.N + static_cast<int64_t>(mt) * (kGmmBM / 2) + (r & 31)) * p.rowbytes;
            else
                return p.W + (e * p.N + static_cast<int64_t>(mt) * kGmmBM + r) * p.rowbytes;
        };
        const auto load_stage = [&](int s, int kt) {
            // activation tile: 128 columns x 64 halves
            for (int i = tid; i < kGmmBN * 8; i += kGmmThreads) {
                const int c = i >> 3, q = i & 7;
                const int br = s_brow[c];
                const __half* src = br >= 0 ? p.x16 + static_cast<int64_t>(br) * p.K + kt * kGmmBK + 8 * q : p.x16;
                cp_async16(smem_addr(B16(s)) + static_cast<uint32_t>((c * kGmmLd + 8 * q) * 2), src, br >= 0 ? 16 : 0);
            }
            // activation scale of the stage's superblock, and (Q4_K) its 16-group sums
            if (tid < kGmmBN) {
                const int br = s_brow[tid];
                const float* src = br >= 0 ? p.dx + static_cast<int64_t>(br) * p.dx_pitch + (kt * kGmmBK >> 8) : p.dx;
                cp_async4(smem_addr(DXS(s)) + 4u * tid, src, br >= 0 ? 4 : 0);
            }
            if constexpr (F == F_Q4_K) {
                if ((kt & 3) == 3) {  // the superblock's last stage applies the mins
                const int c = tid >> 1, q = tid & 1;  // 256 threads: 128 columns x 2 chunks
                const int br = s_brow[c];
                const __half* src = br >= 0 ? p.bs16 + static_cast<int64_t>(br) * (p.K / 16) + (kt * kGmmBK >> 8) * 16 + 8 * q : p.bs16;
                cp_async16(smem_addr(BSS(s)) + static_cast<uint32_t>((c * kGmmBsLd + 8 * q) * 2), src, br >= 0 ? 16 : 0);
                }
            }
            // raw weight bytes of the 64 rows
            if constexpr (F == F_Q8_0) {
                // blocks 2kt, 2kt+1: bytes [68 kt, 68 kt + 68) of the row, from the 16-byte boundary below
                const int a = (68 * kt) & ~15;
                for (int i = tid; i < kGmmBM * 5; i += kGmmThreads) {
                    const int r = i / 5, q = i - r * 5;
                    const int64_t o = a + 16 * q;
                    const int64_t left = p.rowbytes - o;
                    const int bytes = left >= 16 ? 16 : (left > 0 ? static_cast<int>(left) : 0);
                    cp_async16(smem_addr(RAW(s)) + static_cast<uint32_t>(r * kGmmRaw + 16 * q), arow(r) + (bytes ? o : 0), bytes);
                }
            } else {
                // header (16 B) and the 32 bytes of nibbles of this 64-element slice
                const int sb = kt >> 2, cc = kt & 3;
                for (int i = tid; i < kGmmBM * 3; i += kGmmThreads) {
                    const int r = i / 3, q = i - r * 3;
                    const int64_t o = static_cast<int64_t>(sb) * 144 + (q == 0 ? 0 : 16 + 32 * cc + 16 * (q - 1));
                    cp_async16(smem_addr(RAW(s)) + static_cast<uint32_t>(r * kGmmRaw + 16 * q), arow(r) + o, 16);
                }
            }
        };

        float acc[2][4][4], D[2][4][4];
#pragma unroll
        for (int i = 0; i < 2; ++i)
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[i][j][q] = D[i][j][q] = 0.0f;

#pragma unroll
        for (int s = 0; s < kGmmStages - 1; ++s) {
            if (s < nk) load_stage(s, s);
            cp_async_commit();
        }
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % kGmmStages;
            cp_async_wait<kGmmStages - 2>();
            __syncthreads();  // stage kt landed; every warp is done with the previous A tile and stage kt-1
            if (kt + kGmmStages - 1 < nk) load_stage((kt + kGmmStages - 1) % kGmmStages, kt + kGmmStages - 1);
            cp_async_commit();

            // ---- decode the weight tile into f16: thread -> (row, 8-element group)
            const uint8_t* raw = RAW(s);
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int idx = tid + h * kGmmThreads;
                const int r = idx >> 3, ge = idx & 7;
                uint32_t o4[4];
                if constexpr (F == F_Q8_0) {
                    const int o0 = (68 * kt) & 15;
                    const saddr src = smem_addr(raw) + static_cast<uint32_t>(r * kGmmRaw + o0 + 34 * (ge >> 2) + 2 + 8 * (ge & 3));
                    uint32_t w[2];
                    ld_words_any<2>(src, w);
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint32_t u = w[k] ^ 0x80808080u;
                        const __half2 off = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));
                        o4[2 * k] = h2u(__hsub2(u2h(prmt(u, 0u, 0x4140u) | M), off));
                        o4[2 * k + 1] = h2u(__hsub2(u2h(prmt(u, 0u, 0x4342u) | M), off));
                    }
                } else {
                    const uint4 hd = *reinterpret_cast<const uint4*>(raw + r * kGmmRaw);
                    uint32_t sl, sh, ml, mh;
                    k4_words(hd.y, hd.z, hd.w, sl, sh, ml, mh);
                    const int js = 2 * (kt & 3) + (ge >> 2);  // sub-block of this group
                    const __half2 sc = byte_pair(js < 4 ? sl : sh, js & 3);
                    const uint2 qw = *reinterpret_cast<const uint2*>(raw + r * kGmmRaw + 16 + 8 * (ge & 3));
                    if (ge < 4) {  // low nibbles: (1024 + n) sc - 1024 sc
                        const __half2 c = __hmul2(sc, __halves2half2(__ushort_as_half(0xE400u), __ushort_as_half(0xE400u)));
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const uint32_t w = k ? qw.y : qw.x;
                            o4[2 * k] = h2u(__hfma2(u2h((prmt(w, 0u, 0x4140u) & 0x000F000Fu) | M), sc, c));
                            o4[2 * k + 1] = h2u(__hfma2(u2h((prmt(w, 0u, 0x4342u) & 0x000F000Fu) | M), sc, c));
                        }
                    } else {  // high nibbles masked in place: (1024 + 16 n) sc/16 - 64 sc
                        const __half2 s16 = __hmul2(sc, __halves2half2(__ushort_as_half(0x2C00u), __ushort_as_half(0x2C00u)));
                        const __half2 c = __hmul2(sc, __halves2half2(__ushort_as_half(0xD400u), __ushort_as_half(0xD400u)));
#pragma unroll
                        for (int k = 0; k < 2; ++k) {
                            const uint32_t w = k ? qw.y : qw.x;
                            o4[2 * k] = h2u(__hfma2(u2h((prmt(w, 0u, 0x4140u) & 0x00F000F0u) | M), s16, c));
                            o4[2 * k + 1] = h2u(__hfma2(u2h((prmt(w, 0u, 0x4342u) & 0x00F000F0u) | M), s16, c));
                        }
                    }
                }
                *reinterpret_cast<uint4*>(a16 + (r * kGmmLd + 8 * ge) * 2) = make_uint4(o4[0], o4[1], o4[2], o4[3]);
            }
            __syncthreads();

            // ---- tensor cores: 4 k16 steps
            const saddr a_base = smem_addr(a16), b_base = smem_addr(B16(s));
            const float* dxs = DXS(s);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                uint32_t af[2][4], bf[4][2];
#pragma unroll
                for (int i = 0; i < 2; ++i)
                    ldmatrix_x4(a_base + static_cast<uint32_t>(((wm * 32 + 16 * i + (lane & 15)) * kGmmLd + kk * 16 + (lane >> 4) * 8) * 2),
                                af[i][0], af[i][1], af[i][2], af[i][3]);
#pragma unroll
                for (int jp = 0; jp < 2; ++jp)
                    ldmatrix_x4(b_base + static_cast<uint32_t>(((wn * 32 + 16 * jp + (lane & 7) + ((lane >> 4) << 3)) * kGmmLd + kk * 16 +
                                                                ((lane >> 3) & 1) * 8) * 2),
                                bf[2 * jp][0], bf[2 * jp][1], bf[2 * jp + 1][0], bf[2 * jp + 1][1]);
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j) gmm_mma(D[i][j], af[i][0], af[i][1], af[i][2], af[i][3], bf[j][0], bf[j][1]);
                if constexpr (F == F_Q8_0) {
                    if (kk & 1) {  // end of a 32-block: acc += D * d_w * d_x
                        const int blk = kk >> 1, o0 = (68 * kt) & 15;
                        float dw[2][2], dv[4][2];
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int hh = 0; hh < 2; ++hh)
                                dw[i][hh] = ld_h(smem_addr(raw) + static_cast<uint32_t>((wm * 32 + 16 * i + g + 8 * hh) * kGmmRaw + o0 + 34 * blk));
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int c = 0; c < 2; ++c) dv[j][c] = dxs[wn * 32 + 8 * j + 2 * t + c];
#pragma unroll
                        for (int i = 0; i < 2; ++i)
#pragma unroll
                            for (int j = 0; j < 4; ++j)
#pragma unroll
                                for (int q = 0; q < 4; ++q) {
                                    acc[i][j][q] += D[i][j][q] * (dw[i][q >> 1] * dv[j][q & 1]);
                                    D[i][j][q] = 0.0f;
                                }
                    }
                }
            }
            if constexpr (F == F_Q4_K) {
                if ((kt & 3) == 3) {  // end of a superblock: d, mins, activation scale
                    float dd[2][2], dm[2][2], dv[4][2];
                    uint32_t amin[2][2][2];  // [m tile][row g, g+8][sub-block t, t+4] as (m, m)
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int hh = 0; hh < 2; ++hh) {
                            const uint4 hd = *reinterpret_cast<const uint4*>(raw + (wm * 32 + 16 * i + g + 8 * hh) * kGmmRaw);
                            dd[i][hh] = half_lo(hd.x);
                            dm[i][hh] = half_hi(hd.x);
                            uint32_t sl, sh, ml, mh;
                            k4_words(hd.y, hd.z, hd.w, sl, sh, ml, mh);
                            amin[i][hh][0] = h2u(byte_pair(ml, t));
                            amin[i][hh][1] = h2u(byte_pair(mh, t));
                        }
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int c = 0; c < 2; ++c) dv[j][c] = dxs[wn * 32 + 8 * j + 2 * t + c];
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                acc[i][j][q] += D[i][j][q] * (dd[i][q >> 1] * dv[j][q & 1]);
                                D[i][j][q] = 0.0f;
                            }
                    // mins: k slot q <-> 16-group q (sub-block q / 2) against the exact group sums
                    const uint8_t* bss = BSS(s);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int col = wn * 32 + 8 * j + g;
                        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(bss + (col * kGmmBsLd + 2 * t) * 2);
                        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(bss + (col * kGmmBsLd + 2 * t + 8) * 2);
#pragma unroll
                        for (int i = 0; i < 2; ++i)
                            gmm_mma(D[i][j], amin[i][0][0], amin[i][1][0], amin[i][0][1], amin[i][1][1], b0, b1);
                    }
#pragma unroll
                    for (int i = 0; i < 2; ++i)
#pragma unroll
                        for (int j = 0; j < 4; ++j)
#pragma unroll
                            for (int q = 0; q < 4; ++q) {
                                acc[i][j][q] -= D[i][j][q] * (dm[i][q >> 1] * dv[j][q & 1]);
                                D[i][j][q] = 0.0f;
                            }
                }
            }
        }
        cp_async_wait<0>();
        __syncthreads();  // every warp is out of the k loop; the stage area is free

        // ---- epilogue
        if constexpr (KIND == G_GATEUP) {
            float* ex = reinterpret_cast<float*>(stage0);  // up values [32][kGmmBN + 4]
            if (wm == 1) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            ex[(16 * i + g + 8 * (q >> 1)) * (kGmmBN + 4) + wn * 32 + 8 * j + 2 * t + (q & 1)] = acc[i][j][q];
            }
            __syncthreads();
            if (wm == 0) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
#pragma unroll
                    for (int j = 0; j < 4; ++j)
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const int r = 16 * i + g + 8 * (q >> 1), c = wn * 32 + 8 * j + 2 * t + (q & 1);
                            const int pair = s_pair[c];
                            if (pair >= 0) {
                                const float gv = acc[i][j][q], uv = ex[r * (kGmmBN + 4) + c];
                                const int64_t o = static_cast<int64_t>(pair) * p.N + static_cast<int64_t>(mt) * 32 + r;
                                p.h[o] = __fmul_rn(__fdiv_rn(gv, 1.0f + expf(-gv)), uv);
                                if (p.g_dump) p.g_dump[o] = gv;
                                if (p.u_dump) p.u_dump[o] = uv;
                            }
                        }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 2; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j)
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int r = wm * 32 + 16 * i + g + 8 * (q >> 1), c = wn * 32 + 8 * j + 2 * t + (q & 1);
                        const int pair = s_pair[c];
                        if (pair >= 0) p.o[static_cast<int64_t>(pair) * p.N + static_cast<int64_t>(mt) * kGmmBM + r] = acc[i][j][q];
                    }
        }
        __syncthreads();  // the tile's metadata and the stage area are reused by the next item
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

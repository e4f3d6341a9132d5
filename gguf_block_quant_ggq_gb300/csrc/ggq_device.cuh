// ggq_device.cuh -- device building blocks of libggq (sm_103a).
//
//  * PTX wrappers: mbarrier (bounded waits only), 1-D bulk async copy
//    (cp.async.bulk, the TMA engine's linear mode) global -> shared.
//  * Per-format decoders of one 64-weight "unit" of a row into sixteen int8x4
//    words plus its integer scale fields, and the int8 dp4a integer core.
//  * The activation quantizer (bit-exact IEEE fp32 sequence).
//  * A warp "transpose reduction" that sums V per-lane partials in V-1 shuffles.
//
// Block layouts are the GGUF ones; the keep-quant integer core follows
// vllm.cpp PR #523 "grouped + non-grouped keep-quant expert GEMM" (What changed:
// DotQ8_0/DotQ4K/DotQ5K/DotQ6K superblocks with dp4a) and ds4 PR #656 "Add ROCm
// MXFP4 routed expert kernels" (Summary: MXFP4 nibbles unpacked with register
// permutations).  Here the permutation is one PRMT table lookup per four codes.
#pragma once
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace ggq {

enum Fmt : int { F_Q4_0 = 0, F_Q8_0 = 1, F_Q4_K = 2, F_Q5_K = 3, F_Q6_K = 4, F_MXFP4 = 5, F_Q2_K = 6, F_Q3_K = 7, F_COUNT = 8 };

__host__ __device__ constexpr int fmt_qk(int f) {
    return (f == F_Q4_K || f == F_Q5_K || f == F_Q6_K || f == F_Q2_K || f == F_Q3_K) ? 256 : 32;
}
__host__ __device__ constexpr int fmt_bytes(int f) {
    return f == F_Q4_0 ? 18 : f == F_Q8_0 ? 34 : f == F_Q4_K ? 144 : f == F_Q5_K ? 176 : f == F_Q6_K ? 210
         : f == F_Q2_K ? 84 : f == F_Q3_K ? 110 : 17;
}
// int32 coefficients per weight block in the debug dump (see ggq_block_dots).
__host__ __device__ constexpr int fmt_coefs(int f) { return (f == F_Q4_K || f == F_Q5_K || f == F_Q2_K) ? 2 : 1; }
__host__ __device__ constexpr bool fmt_q81(int f) { return f == F_Q4_0; }

// Device error word values (a bounded wait ran out; a routed expert id out of range).
enum : int { DEV_OK = 0, DEV_ERR_TIMEOUT = 1, DEV_ERR_BAD_IDS = 2 };

// ---------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Orders this thread's earlier generic shared-memory accesses before its later
// async-proxy ones (bulk copies into the same bytes).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Non-blocking probe of a phase (test_wait never suspends the thread; the
// blocking try_wait form sleeps for a fixed time slice when the phase is not
// yet complete, which quantizes short kernels to multiples of that slice).
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, polling.  Bounded:
// gives up after ~2^32 SM cycles (about 2 s at 2 GHz) and returns false.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    while (!mbar_test(bar, parity)) {
        if (clock64() - t0 > (1ll << 32)) return false;
    }
    return true;
}

// Linear bulk copy global -> this CTA's shared memory; completion is counted
// on `bar` in bytes.  dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                         uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// L2 policy for data read exactly once (weights): evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// L2 policy for data every CTA reads (activation rows): evict last.
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Byte permute with the sign-replicate selector mode (bit 3 of a selector nibble).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// Programmatic dependent launch.  Every kernel lets the next kernel in the
// stream start launching as soon as all of its CTAs are running, and waits for
// the previous kernel (completion and memory) before it reads anything that
// kernel may have produced or writes any output.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void set_error(int* err, int code) {
    if (err) atomicCAS(err, DEV_OK, code);
}

// ---------------------------------------------------------------- shared-memory loads

// Hot-path reads of shared memory go through explicit ld.shared on 32-bit
// shared-window addresses: integer arithmetic on generic pointers (needed for
// unaligned block layouts) would otherwise turn them into generic loads.
using saddr = uint32_t;

__device__ __forceinline__ uint32_t ld_s32(saddr a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint4 ld_s128(saddr a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}
__device__ __forceinline__ int ld_s8(saddr a) {
    int v;
    asm volatile("ld.shared.s8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ uint32_t ld_u8(saddr a) {
    uint32_t v;
    asm volatile("ld.shared.u8 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ int ld_s16(saddr a) {
    int v;
    asm volatile("ld.shared.s16 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ float ld_f32(saddr a) { return __uint_as_float(ld_s32(a)); }
__device__ __forceinline__ float2 ld_f32x2(saddr a) {
    uint32_t x, y;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(x), "=r"(y) : "r"(a));
    return make_float2(__uint_as_float(x), __uint_as_float(y));
}
__device__ __forceinline__ float ld_h(saddr a) {
    uint32_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=r"(v) : "r"(a));
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v)));
}

// N consecutive little-endian 32-bit words starting at any byte address of
// shared memory (reads up to 4 bytes past the end: buffers are padded).
template <int N>
__device__ __forceinline__ void ld_words_any(saddr a, uint32_t* out) {
    const saddr base = a & ~3u;
    const uint32_t sh = (a & 3u) * 8u;
    uint32_t w[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) w[i] = ld_s32(base + 4u * i);
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

// ---------------------------------------------------------------- activations in shared memory

// Quantized activations, one row per "slot", structure-of-arrays in shared
// memory.  Quants are stored with 16 bytes of padding after every 64, so the
// 64-element runs that consecutive lanes read fall on distinct bank groups.
// Row stride: 80 bytes per (possibly partial) 64-element unit, a multiple of 16.
__host__ __device__ constexpr int xq_row_bytes(int K) { return ((K + 63) >> 6) * 80; }
__device__ __forceinline__ int xq_addr(int e) { return e + ((e >> 6) << 4); }

struct XS {
    saddr q;    // int8 [rows][xq_row_bytes(K)] padded quants
    saddr d;    // f32 [rows][K/ablk] scales (ablk = 32 for Q8_1, 256 for Q8_K)
    saddr s32;  // i32 [rows][K/32] sum of the quants of each 32-block
    saddr bs;   // i16 [rows][K/16] Q8_K sums of 16 (Q8_K only)
    int K;
};

// ---------------------------------------------------------------- weight units

// 64 weights of one row, as four groups of 16: w[4g .. 4g+3] are int8x4 words
// that pair with the activations x[xo[g] .. xo[g]+15].
struct Unit {
    uint32_t w[16];
    int xo[4];
    int sc[4];     // integer scale per group (K-quants)
    int mn[4];     // mins: Q4_K/Q5_K per sub-block (mn[0], mn[1]), Q2_K per group
    float da, db;  // K-quants: d and dmin (Q6_K: d); 32-block formats: scale of block 0 and block 1
};

// E2M1 code -> doubled value + 12, as PRMT tables (codes 0..7 and 8..15).
constexpr uint32_t MX_POS_LO = 0x0F0E0D0Cu, MX_POS_HI = 0x18141210u;  // 12,13,14,15 | 16,18,20,24
constexpr uint32_t MX_NEG_LO = 0x090A0B0Cu, MX_NEG_HI = 0x00040608u;  // 12,11,10,9  | 8,6,4,0

// Four E2M1 codes (the 16-bit selector's nibbles) -> four bytes (2*value + 12).
// Selector bit 3 set makes PRMT replicate the selected byte's sign bit, which
// is 0 in both tables: each table answers for its half of the codes only.
__device__ __forceinline__ uint32_t mx_lookup(uint32_t sel) {
    return prmt(MX_POS_LO, MX_POS_HI, sel) | prmt(MX_NEG_LO, MX_NEG_HI, sel ^ 0x8888u);
}

// Doubled E2M1 magnitudes by the code's low three bits: 0, 1, 2, 3 | 4, 6, 8, 12.
// With these tables a selector nibble whose bit 3 is set (a negative code) reads
// 0 (the replicated sign bit of a byte below 128), so one PRMT of the codes
// yields the positive codes' magnitudes and one of the codes with bit 3 flipped
// the negative codes' magnitudes, four codes each (selector bits 0-15).
constexpr uint32_t MX_MAG_LO = 0x03020100u, MX_MAG_HI = 0x0C080604u;

__device__ __forceinline__ float e8m0_half_scale(uint32_t e) {
    // 2^(e-128): the doubled E2M1 codes carry the other factor of two.
    if (e >= 2u && e < 255u) return __int_as_float(static_cast<int>((e - 1u) << 23));
    if (e == 1u) return __int_as_float(1 << 22);
    if (e == 0u) return __int_as_float(1 << 21);
    return __int_as_float(0x7fc00000);
}

__device__ __forceinline__ float half_lo(uint32_t v) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
}
__device__ __forceinline__ float half_hi(uint32_t v) { return half_lo(v >> 16); }

// Number of 64-weight units in a row of K weights (32-block formats may end
// with a half unit: its second block is absent and contributes nothing).
__host__ __device__ constexpr int units_per_row(int K) { return (K + 63) >> 6; }

// Decode unit u (weights 64u .. 64u+63 in the order below) of a row.
template <int F>
__device__ __forceinline__ void load_unit(saddr row, int u, int nblk32, Unit& un) {
    if constexpr (F == F_Q4_0) {
        // two blocks of 18 B: fp16 d, 16 B nibbles (element j low, j+16 high nibble of byte j)
        const saddr b = row + 36u * u;
        const bool two = 2 * u + 1 < nblk32;
        uint32_t q0[4], q1[4];
        ld_words_any<4>(b + 2, q0);
        un.da = ld_h(b);
        if (two) {
            ld_words_any<4>(b + 20, q1);
            un.db = ld_h(b + 18);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) q1[k] = 0u;  // absent block: zero words, zero scale
            un.db = 0.0f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            un.w[k] = q0[k] & 0x0F0F0F0Fu;
            un.w[4 + k] = (q0[k] >> 4) & 0x0F0F0F0Fu;
            un.w[8 + k] = q1[k] & 0x0F0F0F0Fu;
            un.w[12 + k] = (q1[k] >> 4) & 0x0F0F0F0Fu;
        }
    } else if constexpr (F == F_Q8_0) {
        const saddr b = row + 68u * u;
        const bool two = 2 * u + 1 < nblk32;
        ld_words_any<8>(b + 2, un.w);
        un.da = ld_h(b);
        if (two) {
            ld_words_any<8>(b + 36, un.w + 8);
            un.db = ld_h(b + 34);
        } else {
#pragma unroll
            for (int k = 8; k < 16; ++k) un.w[k] = 0u;
            un.db = 0.0f;
        }
    } else if constexpr (F == F_MXFP4) {
        // element j (0..15) = low nibble of byte j, element j+16 = high nibble.
        // The lookup keeps PRMT's nibble order (j, j+16, j+1, j+17, ...); the
        // activations are stored in the same interleaved order.
        const saddr b = row + 34u * u;
        const bool two = 2 * u + 1 < nblk32;
        uint32_t q0[4], q1[4];
        ld_words_any<4>(b + 1, q0);
        un.da = e8m0_half_scale(ld_u8(b));
        if (two) {
            ld_words_any<4>(b + 18, q1);
            un.db = e8m0_half_scale(ld_u8(b + 17));
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) q1[k] = 0u;
            un.db = 0.0f;
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            un.w[2 * k] = mx_lookup(q0[k] & 0xFFFFu);
            un.w[2 * k + 1] = mx_lookup(q0[k] >> 16);
            un.w[8 + 2 * k] = mx_lookup(q1[k] & 0xFFFFu);
            un.w[8 + 2 * k + 1] = mx_lookup(q1[k] >> 16);
        }
    } else if constexpr (F == F_Q4_K || F == F_Q5_K) {
        // unit = sub-blocks 2cc (low nibbles of qs chunk cc) and 2cc+1 (high nibbles)
        const int sb = u >> 2, cc = u & 3;
        const saddr b = row + (F == F_Q4_K ? 144u : 176u) * sb;
        const uint4 hd = ld_s128(b);
        const saddr qsp = b + (F == F_Q4_K ? 16u : 48u) + 32u * cc;
        const uint4 qa = ld_s128(qsp), qb = ld_s128(qsp + 16);
        un.da = half_lo(hd.x);
        un.db = half_hi(hd.x);
        // all eight 6-bit scales (sc) and mins (m), four per word
        const uint32_t a0 = hd.y, a1 = hd.z, a2 = hd.w;
        const uint32_t sc_lo = a0 & 0x3F3F3F3Fu, m_lo = a1 & 0x3F3F3F3Fu;
        const uint32_t sc_hi = (a2 & 0x0F0F0F0Fu) | ((a0 >> 2) & 0x30303030u);
        const uint32_t m_hi = ((a2 >> 4) & 0x0F0F0F0Fu) | ((a1 >> 2) & 0x30303030u);
        const uint32_t scw = cc < 2 ? sc_lo : sc_hi, mw = cc < 2 ? m_lo : m_hi;
        const int sh = 16 * (cc & 1);
        const int s0 = (scw >> sh) & 0xFF, s1 = (scw >> (sh + 8)) & 0xFF;
        un.sc[0] = un.sc[1] = s0;
        un.sc[2] = un.sc[3] = s1;
        un.mn[0] = (mw >> sh) & 0xFF;
        un.mn[1] = (mw >> (sh + 8)) & 0xFF;
        const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        if constexpr (F == F_Q4_K) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                un.w[k] = q[k] & 0x0F0F0F0Fu;
                un.w[8 + k] = (q[k] >> 4) & 0x0F0F0F0Fu;
            }
        } else {
            const uint4 ha = ld_s128(b + 16), hb = ld_s128(b + 32);
            const uint32_t hq[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                un.w[k] = (q[k] & 0x0F0F0F0Fu) | (((hq[k] >> (2 * cc)) & 0x01010101u) << 4);
                un.w[8 + k] = ((q[k] >> 4) & 0x0F0F0F0Fu) | (((hq[k] >> (2 * cc + 1)) & 0x01010101u) << 4);
            }
        }
    } else if constexpr (F == F_Q2_K || F == F_Q3_K) {
        // element 128n + 32j + l: bits 2j, 2j+1 of qs[32n + l] (Q3_K: bit 4n + j of hmask[l]
        // adds 4 to the stored code, which is q + 4).  Unit v = u&3 is elements 64v .. 64v+63:
        // n = v>>1, j0 = 2(v&1); w[0..7] take shift j0 (groups 4v, 4v+1), w[8..15] shift j0+1.
        const int sb = u >> 2, v = u & 3, n = v >> 1, j0 = 2 * (v & 1);
        const saddr b = row + static_cast<uint32_t>(fmt_bytes(F)) * sb;
        uint32_t q[8];
        ld_words_any<8>(b + (F == F_Q2_K ? 16 : 32) + 32 * n, q);
        if constexpr (F == F_Q2_K) {
            const uint32_t s4 = ld_s32(b + 4 * v);  // scales[4v .. 4v+3]: low nibble scale, high nibble min
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                un.sc[g] = (s4 >> (8 * g)) & 15;
                un.mn[g] = (s4 >> (8 * g + 4)) & 15;
            }
            un.da = ld_h(b + 80);
            un.db = ld_h(b + 82);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                un.w[k] = (q[k] >> (2 * j0)) & 0x03030303u;
                un.w[8 + k] = (q[k] >> (2 * j0 + 2)) & 0x03030303u;
            }
        } else {
            uint32_t hm[8], sw[2];
            ld_words_any<8>(b, hm);
            ld_words_any<1>(b + 96 + 4 * (v & 1), sw);      // low nibbles of groups 4v .. 4v+3
            ld_words_any<1>(b + 104, sw + 1);               // their high two bits
            const uint32_t sc6 = ((v < 2 ? sw[0] : sw[0] >> 4) & 0x0F0F0F0Fu) | (((sw[1] >> (2 * v)) & 0x03030303u) << 4);
#pragma unroll
            for (int g = 0; g < 4; ++g) un.sc[g] = static_cast<int>((sc6 >> (8 * g)) & 0xFFu) - 32;
            un.da = ld_h(b + 108);
            const int hb = 4 * n + j0;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                un.w[k] = ((q[k] >> (2 * j0)) & 0x03030303u) | (((hm[k] >> hb) & 0x01010101u) << 2);
                un.w[8 + k] = ((q[k] >> (2 * j0 + 2)) & 0x03030303u) | (((hm[k] >> (hb + 1)) & 0x01010101u) << 2);
            }
        }
    } else {  // F_Q6_K
        // element 128h + 32g + l: ql[64h + 32(g&1) + l] nibble g>>1, qh[32h + l] bits 2g..2g+1,
        // scale index (128h + 32g + l)/16.  Unit v = u&3: h = v>>1, g1 = v&1; w[0..7] are
        // group g1 (low nibbles), w[8..15] group g1+2 (high nibbles).
        const int sb = u >> 2, v = u & 3, h = v >> 1, g1 = v & 1;
        const saddr b = row + 210u * sb;
        uint32_t ql[8], qh[8];
        ld_words_any<8>(b + 64 * h + 32 * g1, ql);
        ld_words_any<8>(b + 128 + 32 * h, qh);
        const int j0 = 8 * h + 2 * g1;
        un.sc[0] = ld_s8(b + 192 + j0);
        un.sc[1] = ld_s8(b + 192 + j0 + 1);
        un.sc[2] = ld_s8(b + 192 + j0 + 4);
        un.sc[3] = ld_s8(b + 192 + j0 + 5);
        un.da = ld_h(b + 208);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            un.w[k] = (ql[k] & 0x0F0F0F0Fu) | (((qh[k] >> (2 * g1)) & 0x03030303u) << 4);
            un.w[8 + k] = ((ql[k] >> 4) & 0x0F0F0F0Fu) | (((qh[k] >> (2 * g1 + 4)) & 0x03030303u) << 4);
        }
    }
}

// x^ element offsets of the unit's four groups.
template <int F>
__device__ __forceinline__ void unit_offsets(int u, int* xo) {
    if constexpr (F == F_Q6_K) {
        const int sb = u >> 2, v = u & 3;
        const int base = 256 * sb + 128 * (v >> 1) + 32 * (v & 1);
        xo[0] = base;
        xo[1] = base + 16;
        xo[2] = base + 64;
        xo[3] = base + 80;
    } else {
#pragma unroll
        for (int g = 0; g < 4; ++g) xo[g] = 64 * u + 16 * g;
    }
}

// Integer core of one unit against activation row r: per-group dp4a sums, then
// the format's integer coefficients (A, and B for Q4_K/Q5_K mins; for 32-block
// formats A0/A1 are the two blocks).
template <int F>
__device__ __forceinline__ void unit_ints(const Unit& un, const int* xo, const XS& xs, int r, int u, int& A0,
                                          int& A1) {
    const saddr xq = xs.q + static_cast<uint32_t>(r * xq_row_bytes(xs.K));
    int S[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint4 x = ld_s128(xq + xq_addr(xo[g]));
        int a = __dp4a(static_cast<int>(un.w[4 * g]), static_cast<int>(x.x), 0);
        a = __dp4a(static_cast<int>(un.w[4 * g + 1]), static_cast<int>(x.y), a);
        a = __dp4a(static_cast<int>(un.w[4 * g + 2]), static_cast<int>(x.z), a);
        S[g] = __dp4a(static_cast<int>(un.w[4 * g + 3]), static_cast<int>(x.w), a);
    }
    const saddr s32 = xs.s32 + 4u * static_cast<uint32_t>(r * (xs.K >> 5));
    if constexpr (F == F_Q4_0) {
        A0 = S[0] + S[1] - 8 * static_cast<int>(ld_s32(s32 + 8 * u));  // sum (nib - 8) q
        A1 = S[2] + S[3] - 8 * (2 * u + 1 < (xs.K >> 5) ? static_cast<int>(ld_s32(s32 + 8 * u + 4)) : 0);
    } else if constexpr (F == F_Q8_0) {
        A0 = S[0] + S[1];
        A1 = S[2] + S[3];
    } else if constexpr (F == F_MXFP4) {
        A0 = S[0] + S[1] - 12 * static_cast<int>(ld_s32(s32 + 8 * u));  // tables hold 2*value + 12
        A1 = S[2] + S[3] - 12 * (2 * u + 1 < (xs.K >> 5) ? static_cast<int>(ld_s32(s32 + 8 * u + 4)) : 0);
    } else if constexpr (F == F_Q4_K || F == F_Q5_K) {
        A0 = un.sc[0] * (S[0] + S[1]) + un.sc[2] * (S[2] + S[3]);
        A1 = un.mn[0] * static_cast<int>(ld_s32(s32 + 8 * u)) + un.mn[1] * static_cast<int>(ld_s32(s32 + 8 * u + 4));
    } else if constexpr (F == F_Q2_K) {  // per group of 16: scale * S, min * sum(q)
        const saddr bs = xs.bs + 2u * static_cast<uint32_t>(r * (xs.K >> 4));
        A0 = un.sc[0] * S[0] + un.sc[1] * S[1] + un.sc[2] * S[2] + un.sc[3] * S[3];
        A1 = un.mn[0] * ld_s16(bs + 2 * (xo[0] >> 4)) + un.mn[1] * ld_s16(bs + 2 * (xo[1] >> 4)) +
             un.mn[2] * ld_s16(bs + 2 * (xo[2] >> 4)) + un.mn[3] * ld_s16(bs + 2 * (xo[3] >> 4));
    } else if constexpr (F == F_Q3_K) {  // codes stored as q + 4: subtract 4 * sum(q) per group of 16
        const saddr bs = xs.bs + 2u * static_cast<uint32_t>(r * (xs.K >> 4));
        A0 = un.sc[0] * (S[0] - 4 * ld_s16(bs + 2 * (xo[0] >> 4))) + un.sc[1] * (S[1] - 4 * ld_s16(bs + 2 * (xo[1] >> 4))) +
             un.sc[2] * (S[2] - 4 * ld_s16(bs + 2 * (xo[2] >> 4))) + un.sc[3] * (S[3] - 4 * ld_s16(bs + 2 * (xo[3] >> 4)));
        A1 = 0;
    } else {  // Q6_K: 6-bit codes stored unsigned; subtract 32 * sum(q) per group of 16
        const saddr bs = xs.bs + 2u * static_cast<uint32_t>(r * (xs.K >> 4));
        A0 = un.sc[0] * (S[0] - 32 * ld_s16(bs + 2 * (xo[0] >> 4))) + un.sc[1] * (S[1] - 32 * ld_s16(bs + 2 * (xo[1] >> 4))) +
             un.sc[2] * (S[2] - 32 * ld_s16(bs + 2 * (xo[2] >> 4))) + un.sc[3] * (S[3] - 32 * ld_s16(bs + 2 * (xo[3] >> 4)));
        A1 = 0;
    }
}

// Scale epilogue of unit u: fp32 contribution of (A0, A1).
template <int F, bool A32 = (F == F_Q4_0)>
__device__ __forceinline__ float unit_value(const Unit& un, const XS& xs, int r, int u, int A0, int A1) {
    if constexpr (F == F_Q4_0 || (F == F_Q8_0 && A32)) {  // one activation scale per 32 elements
        const saddr d = xs.d + 4u * static_cast<uint32_t>(r * (xs.K >> 5));
        const float d1 = 2 * u + 1 < (xs.K >> 5) ? ld_f32(d + 8 * u + 4) : 0.0f;
        return static_cast<float>(A0) * (un.da * ld_f32(d + 8 * u)) + static_cast<float>(A1) * (un.db * d1);
    } else if constexpr (F == F_Q8_0 || F == F_MXFP4) {
        const float dx = ld_f32(xs.d + 4u * static_cast<uint32_t>(r * (xs.K >> 8) + (u >> 2)));
        return dx * (static_cast<float>(A0) * un.da + static_cast<float>(A1) * un.db);
    } else if constexpr (F == F_Q6_K || F == F_Q3_K) {
        const float dx = ld_f32(xs.d + 4u * static_cast<uint32_t>(r * (xs.K >> 8) + (u >> 2)));
        return static_cast<float>(A0) * (dx * un.da);
    } else {  // Q4_K, Q5_K, Q2_K: d * A - dmin * B
        const float dx = ld_f32(xs.d + 4u * static_cast<uint32_t>(r * (xs.K >> 8) + (u >> 2)));
        return dx * (un.da * static_cast<float>(A0) - un.db * static_cast<float>(A1));
    }
}

// ---------------------------------------------------------------- one token, activations in registers

// dp4a with unsigned bytes in a and signed bytes in b.
__device__ __forceinline__ int dp4a_us(uint32_t a, uint32_t b, int c) {
    int d;
    asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

// A single token's activations for one 64-weight unit, loaded once per kernel
// and kept in registers: the lane that owns unit u reads the same 64 quants for
// every row.  x[4g..4g+3] pair with weight group g (the unit's group order);
// c[] are the integer offsets of the format's epilogue (Q4_0: 8 * sum q per
// block, MXFP4: 12 * sum q per block, Q4_K/Q5_K: sum q per sub-block for the
// mins, Q6_K: 32 * sum q per group of 16); d0/d1 the activation scales.
struct XUnit {
    uint32_t x[16];
    int c[4];
    float d0, d1;
};

template <int F, bool A32 = (F == F_Q4_0)>
__device__ __forceinline__ void load_xunit(const XS& xs, int u, XUnit& xu) {
    const int nb32 = xs.K >> 5;
    int xo[4];
    unit_offsets<F>(u, xo);
#pragma unroll
    for (int g = 0; g < 4; ++g) {
        const uint4 v = ld_s128(xs.q + xq_addr(xo[g]));
        xu.x[4 * g] = v.x;
        xu.x[4 * g + 1] = v.y;
        xu.x[4 * g + 2] = v.z;
        xu.x[4 * g + 3] = v.w;
    }
    const bool two = 2 * u + 1 < nb32;
    const int s0 = static_cast<int>(ld_s32(xs.s32 + 8u * u));
    const int s1 = two ? static_cast<int>(ld_s32(xs.s32 + 8u * u + 4)) : 0;
    xu.c[0] = xu.c[1] = xu.c[2] = xu.c[3] = 0;
    if constexpr (F == F_Q4_0 || (F == F_Q8_0 && A32)) {  // per-32 activation scales
        xu.d0 = ld_f32(xs.d + 8u * u);
        xu.d1 = two ? ld_f32(xs.d + 8u * u + 4) : 0.0f;
        if constexpr (F == F_Q4_0) {
            xu.c[0] = 8 * s0;
            xu.c[1] = 8 * s1;
        }
    } else {
        xu.d0 = ld_f32(xs.d + 4u * static_cast<uint32_t>(u >> 2));
        xu.d1 = 0.0f;
        if constexpr (F == F_MXFP4) {
            xu.c[0] = 12 * s0;
            xu.c[1] = 12 * s1;
        } else if constexpr (F == F_Q4_K || F == F_Q5_K) {
            xu.c[0] = s0;
            xu.c[1] = s1;
        } else if constexpr (F == F_Q6_K || F == F_Q3_K || F == F_Q2_K) {
            constexpr int off = F == F_Q6_K ? 32 : F == F_Q3_K ? 4 : 1;  // Q2_K: the sums for the mins
#pragma unroll
            for (int g = 0; g < 4; ++g) xu.c[g] = off * ld_s16(xs.bs + 2u * static_cast<uint32_t>(xo[g] >> 4));
        }
    }
}

// fp32 contributions of unit u of a row (shared memory) against NX tokens'
// register-resident activations xu[0..NX-1]: the weights are loaded and masked
// once, each token takes its own dp4a chains and epilogue (per token the same
// integers and operation order whatever NX).  High nibbles are masked in place
// (16x their value, as unsigned bytes) and the exact factor 16 is shifted out
// of the integer sum, which saves a shift per weight word.
template <int F, bool A32, int NX>
__device__ __forceinline__ void unit_dot_rxn(saddr row, int u, int nb32, const XUnit* xu, float* out) {
    if constexpr (F == F_Q4_0) {
        const saddr b = row + 36u * u;
        const bool two = 2 * u + 1 < nb32;
        uint32_t q0[4], q1[4];
        ld_words_any<4>(b + 2, q0);
        const float da = ld_h(b);
        float db = 0.0f;
        if (two) {
            ld_words_any<4>(b + 20, q1);
            db = ld_h(b + 18);
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) q1[k] = 0u;
        }
        int l0[NX], h0[NX], l1[NX], h1[NX];
#pragma unroll
        for (int i = 0; i < NX; ++i) l0[i] = h0[i] = l1[i] = h1[i] = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t wl0 = q0[k] & 0x0F0F0F0Fu, wh0 = q0[k] & 0xF0F0F0F0u;
            const uint32_t wl1 = q1[k] & 0x0F0F0F0Fu, wh1 = q1[k] & 0xF0F0F0F0u;
#pragma unroll
            for (int i = 0; i < NX; ++i) {
                l0[i] = __dp4a(static_cast<int>(wl0), static_cast<int>(xu[i].x[k]), l0[i]);
                h0[i] = dp4a_us(wh0, xu[i].x[4 + k], h0[i]);
                l1[i] = __dp4a(static_cast<int>(wl1), static_cast<int>(xu[i].x[8 + k]), l1[i]);
                h1[i] = dp4a_us(wh1, xu[i].x[12 + k], h1[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < NX; ++i) {
            const int A0 = l0[i] + (h0[i] >> 4) - xu[i].c[0];
            const int A1 = l1[i] + (h1[i] >> 4) - xu[i].c[1];
            out[i] = static_cast<float>(A0) * (da * xu[i].d0) + static_cast<float>(A1) * (db * xu[i].d1);
        }
    } else if constexpr (F == F_Q8_0) {
        const saddr b = row + 68u * u;
        const bool two = 2 * u + 1 < nb32;
        uint32_t w[16];
        ld_words_any<8>(b + 2, w);
        const float da = ld_h(b);
        float db = 0.0f;
        if (two) {
            ld_words_any<8>(b + 36, w + 8);
            db = ld_h(b + 34);
        } else {
#pragma unroll
            for (int k = 8; k < 16; ++k) w[k] = 0u;
        }
        int S0[NX], S1[NX];
#pragma unroll
        for (int i = 0; i < NX; ++i) S0[i] = S1[i] = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
#pragma unroll
            for (int i = 0; i < NX; ++i) {
                S0[i] = __dp4a(static_cast<int>(w[k]), static_cast<int>(xu[i].x[k]), S0[i]);
                S1[i] = __dp4a(static_cast<int>(w[8 + k]), static_cast<int>(xu[i].x[8 + k]), S1[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < NX; ++i) {
            if constexpr (A32) out[i] = static_cast<float>(S0[i]) * (da * xu[i].d0) + static_cast<float>(S1[i]) * (db * xu[i].d1);
            else out[i] = xu[i].d0 * (static_cast<float>(S0[i]) * da + static_cast<float>(S1[i]) * db);
        }
    } else if constexpr (F == F_MXFP4) {
        const saddr b = row + 34u * u;
        const bool two = 2 * u + 1 < nb32;
        uint32_t q0[4], q1[4];
        ld_words_any<4>(b + 1, q0);
        const float da = e8m0_half_scale(ld_u8(b));
        float db = 0.0f;
        if (two) {
            ld_words_any<4>(b + 18, q1);
            db = e8m0_half_scale(ld_u8(b + 17));
        } else {
#pragma unroll
            for (int k = 0; k < 4; ++k) q1[k] = 0u;
        }
        // positive and negative codes' magnitudes in dp4a chains of their own:
        // S = P - N is the exact integer sum of (2 value) x of each block
        uint32_t tl = MX_MAG_LO, th = MX_MAG_HI;
        asm("" : "+r"(tl), "+r"(th));  // the two table words stay in registers
        int P0[NX], N0[NX], P1[NX], N1[NX];
#pragma unroll
        for (int i = 0; i < NX; ++i) P0[i] = N0[i] = P1[i] = N1[i] = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t f0 = q0[k] ^ 0x88888888u, f1 = q1[k] ^ 0x88888888u;
            const int pa0 = static_cast<int>(prmt(tl, th, q0[k])), pa1 = static_cast<int>(prmt(tl, th, q0[k] >> 16));
            const int na0 = static_cast<int>(prmt(tl, th, f0)), na1 = static_cast<int>(prmt(tl, th, f0 >> 16));
            const int pb0 = static_cast<int>(prmt(tl, th, q1[k])), pb1 = static_cast<int>(prmt(tl, th, q1[k] >> 16));
            const int nb0 = static_cast<int>(prmt(tl, th, f1)), nb1 = static_cast<int>(prmt(tl, th, f1 >> 16));
#pragma unroll
            for (int i = 0; i < NX; ++i) {
                P0[i] = __dp4a(pa0, static_cast<int>(xu[i].x[2 * k]), P0[i]);
                P0[i] = __dp4a(pa1, static_cast<int>(xu[i].x[2 * k + 1]), P0[i]);
                N0[i] = __dp4a(na0, static_cast<int>(xu[i].x[2 * k]), N0[i]);
                N0[i] = __dp4a(na1, static_cast<int>(xu[i].x[2 * k + 1]), N0[i]);
                P1[i] = __dp4a(pb0, static_cast<int>(xu[i].x[8 + 2 * k]), P1[i]);
                P1[i] = __dp4a(pb1, static_cast<int>(xu[i].x[8 + 2 * k + 1]), P1[i]);
                N1[i] = __dp4a(nb0, static_cast<int>(xu[i].x[8 + 2 * k]), N1[i]);
                N1[i] = __dp4a(nb1, static_cast<int>(xu[i].x[8 + 2 * k + 1]), N1[i]);
            }
        }
#pragma unroll
        for (int i = 0; i < NX; ++i)
            out[i] = xu[i].d0 * (static_cast<float>(P0[i] - N0[i]) * da + static_cast<float>(P1[i] - N1[i]) * db);
    } else if constexpr (F == F_Q4_K || F == F_Q5_K) {
        const int sb = u >> 2, cc = u & 3;
        const saddr b = row + (F == F_Q4_K ? 144u : 176u) * sb;
        const uint4 hd = ld_s128(b);
        const saddr qsp = b + (F == F_Q4_K ? 16u : 48u) + 32u * cc;
        const uint4 qa = ld_s128(qsp), qb = ld_s128(qsp + 16);
        const float da = half_lo(hd.x), dm = half_hi(hd.x);
        const uint32_t a0 = hd.y, a1 = hd.z, a2 = hd.w;
        const uint32_t scw = cc < 2 ? (a0 & 0x3F3F3F3Fu) : ((a2 & 0x0F0F0F0Fu) | ((a0 >> 2) & 0x30303030u));
        const uint32_t mw = cc < 2 ? (a1 & 0x3F3F3F3Fu) : (((a2 >> 4) & 0x0F0F0F0Fu) | ((a1 >> 2) & 0x30303030u));
        const int sh = 16 * (cc & 1);
        const int s0 = (scw >> sh) & 0xFF, s1 = (scw >> (sh + 8)) & 0xFF;
        const int m0 = (mw >> sh) & 0xFF, m1 = (mw >> (sh + 8)) & 0xFF;
        const uint32_t q[8] = {qa.x, qa.y, qa.z, qa.w, qb.x, qb.y, qb.z, qb.w};
        int lo[NX], hi[NX];
#pragma unroll
        for (int i = 0; i < NX; ++i) lo[i] = hi[i] = 0;
        if constexpr (F == F_Q4_K) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t wl = q[k] & 0x0F0F0F0Fu, wh = q[k] & 0xF0F0F0F0u;
#pragma unroll
                for (int i = 0; i < NX; ++i) {
                    lo[i] = __dp4a(static_cast<int>(wl), static_cast<int>(xu[i].x[k]), lo[i]);
                    hi[i] = dp4a_us(wh, xu[i].x[8 + k], hi[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < NX; ++i) hi[i] >>= 4;
        } else {
            const uint4 ha = ld_s128(b + 16), hb = ld_s128(b + 32);
            const uint32_t hq[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint32_t h = hq[k] >> (2 * cc);
                const int wl = static_cast<int>((q[k] & 0x0F0F0F0Fu) | ((h << 4) & 0x10101010u));
                const int wh = static_cast<int>(((q[k] >> 4) & 0x0F0F0F0Fu) | ((h << 3) & 0x10101010u));
#pragma unroll
                for (int i = 0; i < NX; ++i) {
                    lo[i] = __dp4a(wl, static_cast<int>(xu[i].x[k]), lo[i]);
                    hi[i] = __dp4a(wh, static_cast<int>(xu[i].x[8 + k]), hi[i]);
                }
            }
        }
#pragma unroll
        for (int i = 0; i < NX; ++i) {
            const int A0 = s0 * lo[i] + s1 * hi[i];
            const int A1 = m0 * xu[i].c[0] + m1 * xu[i].c[1];
            out[i] = xu[i].d0 * (da * static_cast<float>(A0) - dm * static_cast<float>(A1));
        }
    } else if constexpr (F == F_Q2_K) {  // (element layout as in load_unit)
        // each 2-bit field is masked in place (4^j times its value, as unsigned
        // bytes) and the exact factor is shifted out of the group's integer sum
        const int sb = u >> 2, v = u & 3, n = v >> 1, j0 = 2 * (v & 1);
        const saddr b = row + 84u * sb;
        uint32_t q[8];
        ld_words_any<8>(b + 16 + 32 * n, q);
        const uint32_t s4 = ld_s32(b + 4 * v);
        const uint32_t m0 = 0x03030303u << (2 * j0), m1 = m0 << 2;
        int S[NX][4];
#pragma unroll
        for (int i = 0; i < NX; ++i) S[i][0] = S[i][1] = S[i][2] = S[i][3] = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t w0 = q[k] & m0, w1 = q[k] & m1;
#pragma unroll
            for (int i = 0; i < NX; ++i) {
                S[i][k >> 2] = dp4a_us(w0, xu[i].x[k], S[i][k >> 2]);
                S[i][2 + (k >> 2)] = dp4a_us(w1, xu[i].x[8 + k], S[i][2 + (k >> 2)]);
            }
        }
        const float dq = ld_h(b + 80), dmin = ld_h(b + 82);
#pragma unroll
        for (int i = 0; i < NX; ++i) {
            int A0 = 0, A1 = 0;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                A0 += static_cast<int>((s4 >> (8 * g)) & 15u) * (S[i][g] >> (2 * j0 + 2 * (g >> 1)));
                A1 += static_cast<int>((s4 >> (8 * g + 4)) & 15u) * xu[i].c[g];
            }
            out[i] = xu[i].d0 * (dq * static_cast<float>(A0) - dmin * static_cast<float>(A1));
        }
    } else if constexpr (F == F_Q3_K) {  // (element layout as in load_unit)
        // the two low bits masked in place (4^j times their value) and the high bit
        // in place (2^hb times it), each in a dp4a of its own; the exact factors are
        // shifted out of each group's sums: S' = S_low / 4^j + 4 S_high / 2^hb is the
        // sum of (q + 4) x, and c[] holds 4 * sum(x) per group
        const int sb = u >> 2, v = u & 3, n = v >> 1, j0 = 2 * (v & 1);
        const saddr b = row + 110u * sb;
        uint32_t q[8], hm[8], sw[2];
        ld_words_any<8>(b + 32 + 32 * n, q);
        ld_words_any<8>(b, hm);
        ld_words_any<1>(b + 96 + 4 * (v & 1), sw);
        ld_words_any<1>(b + 104, sw + 1);
        const uint32_t sc6 = ((v < 2 ? sw[0] : sw[0] >> 4) & 0x0F0F0F0Fu) | (((sw[1] >> (2 * v)) & 0x03030303u) << 4);
        const int hb = 4 * n + j0;
        const uint32_t m0 = 0x03030303u << (2 * j0), m1 = m0 << 2;
        const uint32_t h0 = 0x01010101u << hb, h1 = h0 << 1;
        int L[NX][4], H[NX][4];
#pragma unroll
        for (int i = 0; i < NX; ++i)
#pragma unroll
            for (int g = 0; g < 4; ++g) L[i][g] = H[i][g] = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t wl0 = q[k] & m0, wl1 = q[k] & m1, wh0 = hm[k] & h0, wh1 = hm[k] & h1;
#pragma unroll
            for (int i = 0; i < NX; ++i) {
                L[i][k >> 2] = dp4a_us(wl0, xu[i].x[k], L[i][k >> 2]);
                L[i][2 + (k >> 2)] = dp4a_us(wl1, xu[i].x[8 + k], L[i][2 + (k >> 2)]);
                H[i][k >> 2] = dp4a_us(wh0, xu[i].x[k], H[i][k >> 2]);
                H[i][2 + (k >> 2)] = dp4a_us(wh1, xu[i].x[8 + k], H[i][2 + (k >> 2)]);
            }
        }
        const float dq = ld_h(b + 108);
#pragma unroll
        for (int i = 0; i < NX; ++i) {
            int A0 = 0;
#pragma unroll
            for (int g = 0; g < 4; ++g) {
                const int Sg = (L[i][g] >> (2 * j0 + 2 * (g >> 1))) + 4 * (H[i][g] >> (hb + (g >> 1)));
                A0 += (static_cast<int>((sc6 >> (8 * g)) & 0xFFu) - 32) * (Sg - xu[i].c[g]);
            }
            out[i] = static_cast<float>(A0) * (xu[i].d0 * dq);
        }
    } else {  // F_Q6_K (element layout as in load_unit)
        const int sb = u >> 2, v = u & 3, h = v >> 1, g1 = v & 1;
        const saddr b = row + 210u * sb;
        uint32_t ql[8], qh[8];
        ld_words_any<8>(b + 64 * h + 32 * g1, ql);
        ld_words_any<8>(b + 128 + 32 * h, qh);
        const int j0 = 8 * h + 2 * g1;
        const int sc0 = ld_s8(b + 192 + j0), sc1 = ld_s8(b + 192 + j0 + 1);
        const int sc2 = ld_s8(b + 192 + j0 + 4), sc3 = ld_s8(b + 192 + j0 + 5);
        const float da = ld_h(b + 208);
        // nibbles and high bit pairs masked in place, each in a dp4a of its own (high
        // nibbles 16x, high pairs 4^g1 and 4^(g1+2) times their value); the exact
        // factors are shifted out of each group's sums
        const uint32_t m0 = 0x03030303u << (2 * g1), m1 = m0 << 4;
        int N[NX][4], P[NX][4];
#pragma unroll
        for (int i = 0; i < NX; ++i)
#pragma unroll
            for (int g = 0; g < 4; ++g) N[i][g] = P[i][g] = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint32_t wl = ql[k] & 0x0F0F0F0Fu, wh = ql[k] & 0xF0F0F0F0u, p0 = qh[k] & m0, p1 = qh[k] & m1;
#pragma unroll
            for (int i = 0; i < NX; ++i) {
                N[i][k >> 2] = __dp4a(static_cast<int>(wl), static_cast<int>(xu[i].x[k]), N[i][k >> 2]);
                N[i][2 + (k >> 2)] = dp4a_us(wh, xu[i].x[8 + k], N[i][2 + (k >> 2)]);
                P[i][k >> 2] = dp4a_us(p0, xu[i].x[k], P[i][k >> 2]);
                P[i][2 + (k >> 2)] = dp4a_us(p1, xu[i].x[8 + k], P[i][2 + (k >> 2)]);
            }
        }
#pragma unroll
        for (int i = 0; i < NX; ++i) {
            int S[4];
#pragma unroll
            for (int g = 0; g < 4; ++g)
                S[g] = (g < 2 ? N[i][g] : N[i][g] >> 4) + 16 * (P[i][g] >> (2 * g1 + (g < 2 ? 0 : 4)));
            const int A0 = sc0 * (S[0] - xu[i].c[0]) + sc1 * (S[1] - xu[i].c[1]) + sc2 * (S[2] - xu[i].c[2]) +
                           sc3 * (S[3] - xu[i].c[3]);
            out[i] = static_cast<float>(A0) * (xu[i].d0 * da);
        }
    }
}

// fp32 contribution of unit u of a row against one token's register-resident activations.
template <int F, bool A32 = (F == F_Q4_0)>
__device__ __forceinline__ float unit_dot_rx(saddr row, int u, int nb32, const XUnit& xu) {
    float out[1];
    unit_dot_rxn<F, A32, 1>(row, u, nb32, &xu, out);
    return out[0];
}

// ---------------------------------------------------------------- reductions

// Sum each of V = 2^L per-lane values across the warp.  Afterwards lane l holds
// the total of value index (l >> (5 - L)) in v[0].  Costs V - 1 + (5 - L) shuffles.
template <int L>
__device__ __forceinline__ float warp_transpose_reduce(float* v, int lane) {
    constexpr int V = 1 << L;
#pragma unroll
    for (int step = 0; step < L; ++step) {
        const int s = 16 >> step;
        const int n = V >> step;
        const bool upper = (lane & s) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float send = upper ? v[i] : v[i + n / 2];
            const float keep = upper ? v[i + n / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, s);
        }
    }
    float r = v[0];
#pragma unroll
    for (int s = 16 >> L; s >= 1; s >>= 1) r += __shfl_xor_sync(0xffffffffu, r, s);
    return r;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, s));
    return v;
}

__device__ __forceinline__ int warp_sum_i(int v) {
#pragma unroll
    for (int s = 16; s >= 1; s >>= 1) v += __shfl_xor_sync(0xffffffffu, v, s);
    return v;
}

// ---------------------------------------------------------------- activation quantizer

// One int8 quant of the fixed IEEE fp32 sequence q = clamp(roundf(x * (1/d))).
__device__ __forceinline__ int quant_one(float x, float id) {
    float r = roundf(__fmul_rn(x, id));
    r = fminf(fmaxf(r, -127.0f), 127.0f);
    return static_cast<int>(r);
}

__device__ __forceinline__ float quant_scale(float amax, float* id) {
    const float d = __fdiv_rn(amax, 127.0f);
    *id = d != 0.0f ? __fdiv_rn(1.0f, d) : 0.0f;
    return d;
}

// One warp quantizes one 256-element block to Q8_K (292 bytes at dst, 4-byte
// aligned).  src is read with __ldcg (L2) so data written by other CTAs of the
// same kernel is seen after their fence.
__device__ __forceinline__ void warp_quant_q8k_regs(const float (&x)[8], uint8_t* dst, int lane);

__device__ __forceinline__ void warp_quant_q8k(const float* src, uint8_t* dst, int lane) {
    float x[8];
    const float4 a = __ldcg(reinterpret_cast<const float4*>(src) + 2 * lane);
    const float4 b = __ldcg(reinterpret_cast<const float4*>(src) + 2 * lane + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    warp_quant_q8k_regs(x, dst, lane);
}

// The same with the block's values already in registers (lane l holds elements 8 l .. 8 l + 7).
__device__ __forceinline__ void warp_quant_q8k_regs(const float (&x)[8], uint8_t* dst, int lane) {
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(x[i]));
    const float amax = warp_max(m);
    float id;
    const float d = quant_scale(amax, &id);
    int q[8], s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q[i] = quant_one(x[i], id);
        s += q[i];
    }
    uint32_t w0 = (q[0] & 0xFF) | ((q[1] & 0xFF) << 8) | ((q[2] & 0xFF) << 16) | (static_cast<uint32_t>(q[3] & 0xFF) << 24);
    uint32_t w1 = (q[4] & 0xFF) | ((q[5] & 0xFF) << 8) | ((q[6] & 0xFF) << 16) | (static_cast<uint32_t>(q[7] & 0xFF) << 24);
    uint32_t* dq = reinterpret_cast<uint32_t*>(dst + 4 + 8 * lane);
    dq[0] = w0;
    dq[1] = w1;
    s += __shfl_xor_sync(0xffffffffu, s, 1);  // 16-element group = lanes 2g, 2g+1
    if ((lane & 1) == 0) reinterpret_cast<int16_t*>(dst + 260)[lane >> 1] = static_cast<int16_t>(s);
    if (lane == 0) *reinterpret_cast<float*>(dst) = d;
}

// One warp quantizes one 32-element block to Q8_1 (36 bytes at dst, 4-aligned).
__device__ __forceinline__ void warp_quant_q8_1(const float* src, uint8_t* dst, int lane) {
    const float x = src[lane];
    const float amax = warp_max(fabsf(x));
    float id;
    const float d = quant_scale(amax, &id);
    const int q = quant_one(x, id);
    const int s = warp_sum_i(q);
    dst[4 + lane] = static_cast<uint8_t>(q & 0xFF);
    if (lane == 0) {
        const __half hd = __float2half_rn(d);
        const __half hs = __float2half_rn(__fmul_rn(d, static_cast<float>(s)));
        reinterpret_cast<__half*>(dst)[0] = hd;
        reinterpret_cast<__half*>(dst)[1] = hs;
    }
}

// One warp quantizes one 32-element block to a Q8_0 activation block (34
// bytes at dst, 2-byte aligned): fp16 d, then the 32 quants -- the Q8_0
// weight layout, with the Q8_1 quantizer's arithmetic.
__device__ __forceinline__ void warp_quant_q8_0(const float* src, uint8_t* dst, int lane) {
    const float x = src[lane];
    const float amax = warp_max(fabsf(x));
    float id;
    const float d = quant_scale(amax, &id);
    const int q = quant_one(x, id);
    dst[2 + lane] = static_cast<uint8_t>(q & 0xFF);
    if (lane == 0) reinterpret_cast<__half*>(dst)[0] = __float2half_rn(d);
}

}  // namespace ggq
// ggq_device.cuh -- device building blocks of libggq (sm_103a).
//
//  * PTX wrappers: mbarrier (bounded waits only), 1-D bulk async copy
//    (cp.async.bulk, the TMA engine's linear mode) global -> shared.
//  * Per-format decoders of one 32-weight "chunk" into eight int8x4 words plus
//    its integer scale fields, and the int8 dp4a integer core per token.
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

enum Fmt : int { F_Q4_0 = 0, F_Q8_0 = 1, F_Q4_K = 2, F_Q5_K = 3, F_Q6_K = 4, F_MXFP4 = 5, F_COUNT = 6 };

__host__ __device__ constexpr int fmt_qk(int f) { return (f == F_Q4_K || f == F_Q5_K || f == F_Q6_K) ? 256 : 32; }
__host__ __device__ constexpr int fmt_bytes(int f) {
    return f == F_Q4_0 ? 18 : f == F_Q8_0 ? 34 : f == F_Q4_K ? 144 : f == F_Q5_K ? 176 : f == F_Q6_K ? 210 : 17;
}
// int32 coefficients per weight block in the debug dump (see ggq_block_dots).
__host__ __device__ constexpr int fmt_coefs(int f) { return (f == F_Q4_K || f == F_Q5_K) ? 2 : 1; }
__host__ __device__ constexpr bool fmt_q81(int f) { return f == F_Q4_0; }

// Device error word values.
enum : int { DEV_OK = 0, DEV_ERR_TIMEOUT = 1 };

// ---------------------------------------------------------------- PTX

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

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

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Bounded: gives up
// after ~2^32 SM cycles (about 2 s at 2 GHz) and returns false.
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

// Byte permute with the sign-replicate selector mode (bit 3 of a selector nibble).
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

__device__ __forceinline__ void set_error(int* err, int code) {
    if (err) atomicCAS(err, DEV_OK, code);
}

// ---------------------------------------------------------------- loads

__device__ __forceinline__ uint4 ld128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }
__device__ __forceinline__ float ldh(const uint8_t* p) { return __half2float(*reinterpret_cast<const __half*>(p)); }

// N consecutive little-endian 32-bit words starting at any byte address of
// shared memory (reads up to 4 bytes past the end: buffers are padded).
template <int N>
__device__ __forceinline__ void ld_words_any(const uint8_t* p, uint32_t* out) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    const uint32_t* base = reinterpret_cast<const uint32_t*>(a & ~uintptr_t(3));
    const uint32_t sh = static_cast<uint32_t>(a & 3) * 8u;
    uint32_t w[N + 1];
#pragma unroll
    for (int i = 0; i <= N; ++i) w[i] = base[i];
#pragma unroll
    for (int i = 0; i < N; ++i) out[i] = __funnelshift_r(w[i], w[i + 1], sh);
}

// ---------------------------------------------------------------- activations in shared memory

// Quantized activations, one row per "slot", structure-of-arrays in shared
// memory so that every 16-element group is one aligned 128-bit load.
struct XS {
    const int8_t* q;     // [rows][K]
    const float* d;      // [rows][K/ablk]  (ablk = 32 for Q8_1, 256 for Q8_K)
    const int16_t* bs;   // [rows][K/16]    Q8_K only
    const int32_t* qs32; // [rows][K/32]    Q8_1 only: sum of the 32 quants
    int K;
};

// ---------------------------------------------------------------- weight chunks

// 32 weights of one row: eight int8x4 words w[0..3] (16 weights that pair with
// activations x[xo0 .. xo0+15]) and w[4..7] (pair with x[xo1 .. xo1+15]), plus
// the block's scale fields.
struct Chunk {
    uint32_t w[8];
    int s0, s1, m0, m1;
    float da, db;
    int xo0, xo1;
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

__device__ __forceinline__ float e8m0_half_scale(uint32_t e) {
    // 2^(e-128): the doubled E2M1 codes carry the other factor of two.
    if (e >= 2u && e < 255u) return __int_as_float(static_cast<int>((e - 1u) << 23));
    if (e == 1u) return __int_as_float(1 << 22);
    if (e == 0u) return __int_as_float(1 << 21);
    return __int_as_float(0x7fc00000);
}

// Decode chunk c (weights 32c .. 32c+31 in the chunk order below) of a row.
template <int F>
__device__ __forceinline__ void load_chunk(const uint8_t* row, int c, Chunk& ch) {
    if constexpr (F == F_Q4_0) {
        const uint8_t* b = row + 18 * c;
        uint32_t q[4];
        ld_words_any<4>(b + 2, q);
        ch.da = ldh(b);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            ch.w[k] = q[k] & 0x0F0F0F0Fu;
            ch.w[4 + k] = (q[k] >> 4) & 0x0F0F0F0Fu;
        }
        ch.xo0 = 32 * c;
        ch.xo1 = 32 * c + 16;
    } else if constexpr (F == F_Q8_0) {
        const uint8_t* b = row + 34 * c;
        ld_words_any<8>(b + 2, ch.w);
        ch.da = ldh(b);
        ch.xo0 = 32 * c;
        ch.xo1 = 32 * c + 16;
    } else if constexpr (F == F_MXFP4) {
        // element j (0..15) = low nibble of byte j, element j+16 = high nibble.
        // The lookup keeps PRMT's nibble order (j, j+16, j+1, j+17, ...); the
        // activations are stored in the same interleaved order.
        const uint8_t* b = row + 17 * c;
        uint32_t q[4];
        ld_words_any<4>(b + 1, q);
        ch.da = e8m0_half_scale(b[0]);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            ch.w[2 * k] = mx_lookup(q[k] & 0xFFFFu);
            ch.w[2 * k + 1] = mx_lookup(q[k] >> 16);
        }
        ch.xo0 = 32 * c;
        ch.xo1 = 32 * c + 16;
    } else if constexpr (F == F_Q4_K || F == F_Q5_K) {
        const int sb = c >> 3, p = c & 7, cc = p >> 1, hf = p & 1;
        const uint8_t* b = row + (F == F_Q4_K ? 144 : 176) * sb;
        const uint4 hd = ld128(b);
        const uint4 qv = ld128(b + (F == F_Q4_K ? 16 : 48) + 32 * cc + 16 * hf);
        ch.da = __half2float(__ushort_as_half(static_cast<unsigned short>(hd.x & 0xFFFFu)));
        ch.db = __half2float(__ushort_as_half(static_cast<unsigned short>(hd.x >> 16)));
        // all eight 6-bit scales (sc) and mins (m), four per word
        const uint32_t a0 = hd.y, a1 = hd.z, a2 = hd.w;
        const uint32_t sc_lo = a0 & 0x3F3F3F3Fu, m_lo = a1 & 0x3F3F3F3Fu;
        const uint32_t sc_hi = (a2 & 0x0F0F0F0Fu) | ((a0 >> 2) & 0x30303030u);
        const uint32_t m_hi = ((a2 >> 4) & 0x0F0F0F0Fu) | ((a1 >> 2) & 0x30303030u);
        const uint32_t scw = cc < 2 ? sc_lo : sc_hi, mw = cc < 2 ? m_lo : m_hi;
        const int sh = 16 * (cc & 1);
        ch.s0 = (scw >> sh) & 0xFF;
        ch.s1 = (scw >> (sh + 8)) & 0xFF;
        ch.m0 = (mw >> sh) & 0xFF;
        ch.m1 = (mw >> (sh + 8)) & 0xFF;
        const uint32_t q[4] = {qv.x, qv.y, qv.z, qv.w};
        if constexpr (F == F_Q4_K) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                ch.w[k] = q[k] & 0x0F0F0F0Fu;
                ch.w[4 + k] = (q[k] >> 4) & 0x0F0F0F0Fu;
            }
        } else {
            const uint4 hv = ld128(b + 16 + 16 * hf);
            const uint32_t h[4] = {hv.x, hv.y, hv.z, hv.w};
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                ch.w[k] = (q[k] & 0x0F0F0F0Fu) | (((h[k] >> (2 * cc)) & 0x01010101u) << 4);
                ch.w[4 + k] = ((q[k] >> 4) & 0x0F0F0F0Fu) | (((h[k] >> (2 * cc + 1)) & 0x01010101u) << 4);
            }
        }
        ch.xo0 = 256 * sb + 64 * cc + 16 * hf;
        ch.xo1 = ch.xo0 + 32;
    } else {  // F_Q6_K
        // element 128h + 32g + l: ql[64h + 32(g&1) + l] nibble g>>1, qh[32h + l] bits 2g..2g+1,
        // scale index (128h + 32g + l)/16.  Chunk p: h = p>>2, g1 = (p>>1)&1, half = p&1;
        // w[0..3] are group g1 (low nibbles), w[4..7] group g1+2 (high nibbles).
        const int sb = c >> 3, p = c & 7, h = p >> 2, g1 = (p >> 1) & 1, hf = p & 1;
        const uint8_t* b = row + 210 * sb;
        uint32_t ql[4], qh[4];
        ld_words_any<4>(b + 64 * h + 32 * g1 + 16 * hf, ql);
        ld_words_any<4>(b + 128 + 32 * h + 16 * hf, qh);
        const int j0 = 8 * h + 2 * g1 + hf;
        ch.s0 = static_cast<int8_t>(b[192 + j0]);
        ch.s1 = static_cast<int8_t>(b[192 + j0 + 4]);
        ch.da = ldh(b + 208);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            ch.w[k] = (ql[k] & 0x0F0F0F0Fu) | (((qh[k] >> (2 * g1)) & 0x03030303u) << 4);
            ch.w[4 + k] = ((ql[k] >> 4) & 0x0F0F0F0Fu) | (((qh[k] >> (2 * g1 + 4)) & 0x03030303u) << 4);
        }
        ch.xo0 = 256 * sb + 128 * h + 32 * g1 + 16 * hf;
        ch.xo1 = ch.xo0 + 64;
    }
}

// Integer core of one chunk against activation row `r`: the coefficients A
// (and B for Q4_K/Q5_K) whose scale epilogue gives the chunk's contribution.
template <int F>
__device__ __forceinline__ void chunk_ints(const Chunk& ch, const XS& xs, int r, int c, int& A, int& B) {
    const int8_t* xq = xs.q + static_cast<size_t>(r) * xs.K;
    const uint4 x0 = *reinterpret_cast<const uint4*>(xq + ch.xo0);
    const uint4 x1 = *reinterpret_cast<const uint4*>(xq + ch.xo1);
    int S0 = __dp4a(static_cast<int>(ch.w[0]), static_cast<int>(x0.x), 0);
    S0 = __dp4a(static_cast<int>(ch.w[1]), static_cast<int>(x0.y), S0);
    S0 = __dp4a(static_cast<int>(ch.w[2]), static_cast<int>(x0.z), S0);
    S0 = __dp4a(static_cast<int>(ch.w[3]), static_cast<int>(x0.w), S0);
    int S1 = __dp4a(static_cast<int>(ch.w[4]), static_cast<int>(x1.x), 0);
    S1 = __dp4a(static_cast<int>(ch.w[5]), static_cast<int>(x1.y), S1);
    S1 = __dp4a(static_cast<int>(ch.w[6]), static_cast<int>(x1.z), S1);
    S1 = __dp4a(static_cast<int>(ch.w[7]), static_cast<int>(x1.w), S1);
    B = 0;
    if constexpr (F == F_Q4_0) {
        A = S0 + S1 - 8 * xs.qs32[r * (xs.K >> 5) + c];  // sum (nib - 8) q
    } else if constexpr (F == F_Q8_0) {
        A = S0 + S1;
    } else if constexpr (F == F_MXFP4) {
        const int16_t* bs = xs.bs + r * (xs.K >> 4);
        A = S0 + S1 - 12 * (bs[2 * c] + bs[2 * c + 1]);  // tables hold 2*value + 12
    } else if constexpr (F == F_Q4_K || F == F_Q5_K) {
        const int16_t* bs = xs.bs + r * (xs.K >> 4);
        A = ch.s0 * S0 + ch.s1 * S1;
        B = ch.m0 * bs[ch.xo0 >> 4] + ch.m1 * bs[ch.xo1 >> 4];
    } else {  // Q6_K: 6-bit codes are stored unsigned; subtract 32 * sum(q) per group
        const int16_t* bs = xs.bs + r * (xs.K >> 4);
        A = ch.s0 * (S0 - 32 * bs[ch.xo0 >> 4]) + ch.s1 * (S1 - 32 * bs[ch.xo1 >> 4]);
    }
}

// Scale epilogue of chunk c: fp32 contribution of (A, B).
template <int F>
__device__ __forceinline__ float chunk_value(const Chunk& ch, const XS& xs, int r, int c, int A, int B) {
    if constexpr (F == F_Q4_0) {
        return static_cast<float>(A) * (ch.da * xs.d[r * (xs.K >> 5) + c]);
    } else if constexpr (F == F_Q8_0 || F == F_MXFP4 || F == F_Q6_K) {
        return static_cast<float>(A) * (ch.da * xs.d[r * (xs.K >> 8) + (c >> 3)]);
    } else {
        const float dx = xs.d[r * (xs.K >> 8) + (c >> 3)];
        return dx * (ch.da * static_cast<float>(A) - ch.db * static_cast<float>(B));
    }
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
__device__ __forceinline__ void warp_quant_q8k(const float* src, uint8_t* dst, int lane) {
    float x[8];
    const float4 a = __ldcg(reinterpret_cast<const float4*>(src) + 2 * lane);
    const float4 b = __ldcg(reinterpret_cast<const float4*>(src) + 2 * lane + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
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

}  // namespace ggq

// ggq_gmmtc.cuh -- the expert-sorted grouped GEMM on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory) for Q8_0, Q4_K and MXFP4
// expert banks.
//
// Same arithmetic as the keep-quant expert GEMM of vllm.cpp PR #523
// "grouped + non-grouped keep-quant expert GEMM" (What changed: DotQ8_0 /
// DotQ4K block dots grouped over expert_ids): per weight block, (weight scale)
// * (activation scale) * (integer dot).  The integer dots run as tcgen05.mma
// kind::f16 with f16 operands that hold integers exactly:
//   * Q8_0: the int8 codes; each 32-block gets its own tensor-memory accumulator
//     (|dot| < 2^19: exact in f32), so the weight block scale, which differs per
//     row and block, is applied by the epilogue warps;
//   * Q4_K: the codes already multiplied by their 6-bit sub-block scale
//     (sc * q <= 945); one accumulator per 128-wide half superblock (|partial|
//     <= 128 * 945 * 127 < 2^24: exact), and the mins term sum_j m_j * (16-group
//     sums of x) is one more K = 16 MMA of the mins against the activations'
//     exact group sums; the epilogue adds D d d_x after the first half and
//     (D d - Dmin dmin) d_x after the second;
//   * MXFP4 (ds4 PR #656 "Add ROCm MXFP4 routed expert kernels", Summary:
//     MXFP4 x Q8_K gate/up and down): bf16 operands.  A doubled E2M1 code
//     (2v <= 12, 4 significant bits) times its block's E8M0 power of two is
//     exact in bf16 for every scale whose products fit in f32, and so is an
//     int8 activation; the power of two is folded into the decoded weight,
//     every product is exact, and one accumulator spans a whole superblock
//     (one drain and one d_x per 256 inputs, as Q4_K).  The f32 sums inside a
//     superblock then round at 2^-24 relative when the block exponents differ;
//     to dump the integer core, the same kernel keeps the codes unscaled and
//     one accumulator per 32-block (the Q8_0 schedule), whose dots are exact.
//
// Work item: (expert, matrix, 128 weight rows, 128 activation columns).  The
// activation operand is f16 rows in expert-sorted order (one per (token,
// expert) pair), so an item's columns are 128 consecutive rows.  Per 64-wide
// k-step:
//   * TMA (one elected lane of warp 14): the activation tile (128 rows x 128
//     bytes, 128-byte swizzle = the UMMA K-major SW128 layout), the raw Q8_0
//     bytes of the 128 weight rows (the 80-byte 16-aligned span holding the
//     k-step's two blocks) and, at a superblock's end, the activation scales;
//     4-stage ring, completion on one mbarrier per stage;
//   * decode (warps 8-13; MXFP4: 4-13): raw codes -> f16 (bf16) weight tile in
//     the same SW128 K-major layout (4-5 buffers), then fence.proxy.async so the
//     tensor core sees the generic-proxy stores;
//   * MMA (one elected lane of warp 15): two K=16 MMAs per 32-block into one of
//     two 128-column tensor-memory accumulators, tcgen05.commit to the
//     accumulator's mbarrier (the thread's only commits: a tcgen05 instruction
//     costs its issuing thread ~90 cycles); the epilogue, having seen a k-step's
//     last accumulator land (every earlier MMA has then completed), releases the
//     k-step's weight tile and ring slot;
//   * epilogue (warps 0-7, MXFP4: 0-3; warp w owns TMEM lanes 32 (w & 3) .. +31
//     = tile rows and 64 (MXFP4: all 128) columns): tcgen05.ld of each block accumulator,
//     T += D * d_w (d_w: this thread's row), and at the superblock's end
//     acc += T * d_x (d_x: per column) in a third tensor-memory region; at the
//     item's end acc goes to the output rows (one f32 row per pair: lanes write
//     consecutive rows, 128-byte segments).
// Gate and up are separate items (SwiGLU is fused into the quantizer of h).
// Every wait is bounded: a wait that gives up sets the error word and the
// shared abort flag, and every role leaves its loop.
#pragma once
#include <cuda_bf16.h>

#include "ggq_device.cuh"
#include "ggq_internal.h"

namespace ggq {

constexpr int kTcBM = 128, kTcBN = 128, kTcBK = 64;
constexpr int kTcTmaWarp = 14, kTcMmaWarp = 15;
constexpr int kTcRaw = 80;  // raw bytes per weight row per k-step (Q8_0: the 16-aligned span of two 34-byte blocks)
constexpr int kTcRawMx = 48;  // MXFP4: the 16-aligned span of two 17-byte blocks (34 bytes at an even offset < 16)
constexpr int kTcMaxGroups = 4096;

// Warp roles per format: epilogue warps 0 .. kEpi/32 - 1, decode warps up to 13,
// then the TMA and MMA warps.  MXFP4 drains once per superblock and decodes
// the most per weight (a table lookup per code), so it trades epilogue warps
// for decode warps: eight of them (one 32-block per thread and k-step), none
// on the MMA warp's SMSP (warps 7 and 11 stay idle), whose single issuing
// thread otherwise waits for issue slots at every step of its loop.
template <int F, bool DUMP = false>
struct TcRoles {
    static constexpr bool kMx = F == F_MXFP4 && !DUMP;
    static constexpr int kEpi = kMx ? 128 : 256;                   // epilogue threads
    static constexpr int kDec = kMx ? 256 : kTcThreads - 64 - kEpi;  // decode threads
    static constexpr int kEpiCols = kTcBN * 128 / kEpi;            // accumulator columns per epilogue warp (64 or 128)
    // decode ordinal of a warp (its threads are dt = 32 * ordinal + lane), or -1
    __device__ static int dec_ord(int warp) {
        if (kMx) return warp == 7 || warp == 11 ? -1 : warp - 4 - (warp > 7) - (warp > 11);
        return warp - kEpi / 32;
    }
};
static_assert(kTcThreads == TcRoles<F_Q8_0>::kEpi + TcRoles<F_Q8_0>::kDec + 64, "warp roles");
static_assert(TcRoles<F_MXFP4>::kEpi + TcRoles<F_MXFP4>::kDec + 2 * 32 + 64 == kTcThreads, "MXFP4 warp roles");

// Shared-memory layout per format: the TMA ring, then the decoded weight tiles
// (Q8_0: 5, Q4_K: 4 plus the two mins-term tiles), the item table, the barriers.
// More weight tiles decouple the decode from the MMA's completion.
template <int F>
struct TcSmem {
    // TMA ring depth and decoded weight tiles: a stage is released only once its
    // k-step's MMAs have completed, so the ring must cover the weight fetch, the
    // decode and the MMA of several k-steps; Q4_K also holds the mins operands
    static constexpr int kStages = F == F_MXFP4 ? 6 : F == F_Q8_0 ? 5 : 4;
    static constexpr int kABufs = F == F_Q4_K ? 4 : 3;
    static constexpr int kB = kTcBN * kTcBK * 2;     // 16384, SW128 K-major
    static constexpr int kRawRow = F == F_MXFP4 ? kTcRawMx : kTcRaw;  // raw bytes per weight row per k-step
    static constexpr int kRaw = kTcBM * kRawRow;     // 10240
    static constexpr int kDX = kTcBN * 16;           // 2048: 4 superblock scales per column
    static constexpr int kStage = kB + kRaw + kDX;   // 28672 (28 KB: activation tiles stay 1024-aligned)
    static constexpr int kA = kTcBM * kTcBK * 2;     // 16384, SW128 K-major
    static constexpr int oA = kStages * kStage;
    static constexpr int oMin = oA + kABufs * kA;    // Q4_K mins-term operands: two SW128 tiles
    static constexpr int oPrefix = oMin + (F == F_Q4_K ? 2 * kA : 0);
    static constexpr int kPrefix = (kTcMaxGroups + 1) * 4;
    static constexpr int oBars = (oPrefix + kPrefix + 7) / 8 * 8;
    static constexpr int kBars = (2 * kStages + 2 * kABufs + 6) * 8 + 16;
    static constexpr int kTotal = oBars + kBars + 1024;  // + alignment slack of the dynamic base
};
static_assert(TcSmem<F_Q8_0>::kStage % 1024 == 0 && TcSmem<F_Q8_0>::oA % 1024 == 0, "SW128 tiles need 1024-byte alignment");
static_assert(TcSmem<F_MXFP4>::kStage % 1024 == 0 && TcSmem<F_MXFP4>::oA % 1024 == 0, "SW128 tiles need 1024-byte alignment");
static_assert(TcSmem<F_Q8_0>::kTotal <= kSmemLimit && TcSmem<F_Q4_K>::kTotal <= kSmemLimit &&
                  TcSmem<F_MXFP4>::kTotal <= kSmemLimit,
              "tcgen05 grouped GEMM shared memory");

// tensor-memory columns: two block accumulators, then the item accumulator
constexpr uint32_t kTmemCols = 512;

// UMMA shared-memory descriptor of a K-major tile with 128-byte swizzle: rows of
// 128 bytes, 8-row groups 1024 bytes apart (descriptor version 1).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFF) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) | (static_cast<uint64_t>(2) << 61);
}
// instruction descriptor: f32 accumulate, f16 (bf16: both operands bf16) A and
// B, both K-major, M = 128, N = n
__host__ __device__ constexpr uint32_t tc_idesc(uint32_t n, bool bf16 = false) {
    return (1u << 4) | (bf16 ? (1u << 7) | (1u << 10) : 0u) | ((n >> 3) << 17) |
           ((static_cast<uint32_t>(kTcBM) >> 4) << 24);
}
// Items with at most this many columns load a 32-row activation box and run N = 32
// MMAs (decode-sized token counts spread over many experts).
constexpr int kTcNarrow = 32;

__device__ __forceinline__ void tc_mma(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
__device__ __forceinline__ void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive tensor-memory columns of this thread's lane
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
          "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
          "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float* v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])), "r"(__float_as_uint(v[3])),
        "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])), "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])),
        "r"(__float_as_uint(v[8])), "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
        : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// (d0, d1) = (a0, a1) * b + (c0, c1) as one packed f32x2 FMA (round to nearest,
// each lane exactly an fmaf): half the issue slots of two FFMAs.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c0, float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %4};\n\tmov.b64 rc, {%5, %6};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b), "f"(c0), "f"(c1));
}

// (d0, d1) = (a0, a1) * (b0, b1) + (c0, c1), packed
__device__ __forceinline__ void ffma2p(float& d0, float& d1, float a0, float a1, float b0, float b1, float c0, float c1) {
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\tmov.b64 ra, {%2, %3};\n\tmov.b64 rb, {%4, %5};\n\tmov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\tmov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d0), "=f"(d1)
        : "f"(a0), "f"(a1), "f"(b0), "f"(b1), "f"(c0), "f"(c1));
}

__device__ __forceinline__ void tc_tma_2d(saddr dst, const CUtensorMap* map, int x, int y, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

// (v, v) as f16 for byte idx (runtime) of w (v <= 255)
__device__ __forceinline__ __half2 tc_byte_pair(uint32_t w, int idx) {
    const uint32_t sel = 0x4040u | static_cast<uint32_t>(idx) | (static_cast<uint32_t>(idx) << 8);
    const uint32_t u = prmt(w, 0u, sel) | 0x64006400u;
    return __hsub2(*reinterpret_cast<const __half2*>(&u), __halves2half2(__ushort_as_half(0x6400u), __ushort_as_half(0x6400u)));
}

// One work item: matrix m of expert e, m tile mt (128 rows), columns [n0, n0 + ncols) of group gi.
struct TcItem {
    int m, mt, ncols, y0;  // y0: first sorted activation row
    int wrow;              // first weight row in the bank (e * N + mt * 128)
};

__device__ __forceinline__ TcItem tc_item(const GmmTcParams& p, const int* s_pref, int ngroups, int mtiles, int item) {
    int lo = 0, hi = ngroups - 1;  // last group with s_pref[g] <= item
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_pref[mid] <= item) lo = mid; else hi = mid - 1;
    }
    const int cnt = p.group_cnt[lo];
    const int ntl = (cnt + kTcBN - 1) / kTcBN;
    const int local = item - s_pref[lo];
    const int mta = local / ntl, nt = local - mta * ntl;  // mta over nmat * mtiles
    TcItem r;
    r.m = mta / mtiles;
    r.mt = mta - r.m * mtiles;
    const int n0 = nt * kTcBN;
    r.ncols = min(cnt - n0, kTcBN);
    r.y0 = p.group_off[lo] + n0;
    r.wrow = static_cast<int>(static_cast<int64_t>(p.group_expert[lo]) * p.N) + r.mt * kTcBM;
    return r;
}

// Bounded wait by a whole warp (every lane polls); the result is the same in
// every lane, so loops leave together.  On failure flags the CTA (abort) and
// the error word.
// Bounded wait that sleeps a little between probes: for the roles that wait
// long (the epilogue between drains, the TMA warp for a free slot), so that
// they leave the issue slots of their SMSP to the roles with work (the single
// MMA thread shares one with an epilogue warp).
__device__ __forceinline__ bool mbar_wait_nap(uint64_t* bar, uint32_t parity) {
    if (mbar_test(bar, parity)) return true;
    const long long t0 = clock64();
    for (;;) {
        __nanosleep(64);
        if (mbar_test(bar, parity)) return true;
        if (clock64() - t0 > (1ll << 32)) return false;
    }
}

__device__ __forceinline__ bool tc_wait(uint64_t* bar, uint32_t parity, volatile int* abort, int* err, bool nap = false) {
    bool ok = !*abort && (nap ? mbar_wait_nap(bar, parity) : mbar_wait(bar, parity));
    ok = __all_sync(0xFFFFFFFFu, ok);
    if (!ok) {
        *abort = 1;
        set_error(err, DEV_ERR_TIMEOUT);
    }
    return ok;
}

// The same wait by one thread (the MMA role runs on one lane).
__device__ __forceinline__ bool tc_wait1(uint64_t* bar, uint32_t parity, volatile int* abort, int* err) {
    const bool ok = !*abort && mbar_wait(bar, parity);
    if (!ok) {
        *abort = 1;
        set_error(err, DEV_ERR_TIMEOUT);
    }
    return ok;
}

// Position of k-step c in the rings, advanced without divisions (a role's
// loop bookkeeping is on its critical path): TMA slot s and the phase of its
// current use, decoded tile a and its phase, k-step kt of item it.
struct TcPos {
    int s = 0, a = 0, kt = 0, it = 0;
    uint32_t fph = 0u, aph = 0u;
    __device__ __forceinline__ void next(int stages, int abufs, int nk) {
        if (++s == stages) s = 0, fph ^= 1u;
        if (++a == abufs) a = 0, aph ^= 1u;
        if (++kt == nk) kt = 0, ++it;
    }
};

// Integer-core dump of 32 accumulator columns of this thread's row: the exact
// integer each holds goes to coefficient idx of the column's pair (added to
// what is there with `add`: the second half of a Q4_K superblock).
__device__ __forceinline__ void tc_dump32(const GmmTcParams& p, const TcItem& cur, int r, int col0, const float* v,
                                          int idx, bool add) {
    const int64_t row = static_cast<int64_t>(cur.mt) * kTcBM + r;
    for (int j = 0; j < 32; ++j) {
        const int col = col0 + j;
        if (col >= cur.ncols) break;
        int32_t* const q = p.coefs[cur.m] + (static_cast<int64_t>(p.perm[cur.y0 + col]) * p.N + row) * p.ncoef + idx;
        const int iv = __float2int_rn(v[j]);
        *q = add ? *q + iv : iv;
    }
}

// The bf16 pair (2^(e-128), 2^(e-128)) for an E8M0 byte e: the power of two by
// which the doubled E2M1 codes are scaled (bf16 holds it for every e below 255,
// as a subnormal for e = 0, 1; e = 255 is NaN).
__device__ __forceinline__ uint32_t tc_e8m0_bf16x2(uint32_t e) {
    const uint32_t b = e == 255u ? 0x7FC0u : e >= 2u ? (e - 1u) << 7 : (e == 1u ? 0x40u : 0x20u);  // 255: NaN
    return b | (b << 16);
}

// MXFP4 decode of one 32-block of one row into its 64-byte span of a SW128 bf16
// tile row (chunks 4 blk .. 4 blk + 3, XOR-swizzled by the row): the doubled
// E2M1 codes come from the PRMT lookup as 2v + 12 (ordered j, j+16, j+1, j+17),
// are placed as 128 + (2v + 12) in bf16 (exponent 2^7, exact), and become
// 2v * s with s = 2^(e-128) (production; exact in bf16 for every E8M0 value
// whose products fit) or s = 1 (integer-core dump: the exact doubled codes).
__device__ __forceinline__ void tc_mx_block(uint8_t* at, int r, int blk, const uint32_t* q, uint32_t s2) {
    const uint32_t k43 = 0x43434343u;
    const __nv_bfloat162 k140 = __halves2bfloat162(__ushort_as_bfloat16(0x430Cu), __ushort_as_bfloat16(0x430Cu));
    const __nv_bfloat162 sv = *reinterpret_cast<const __nv_bfloat162*>(&s2);
    const auto conv = [&](uint32_t x) -> uint32_t {
        const __nv_bfloat162 v = __hmul2(__hsub2(*reinterpret_cast<const __nv_bfloat162*>(&x), k140), sv);
        return *reinterpret_cast<const uint32_t*>(&v);
    };
    uint32_t lo[8], hi[8];  // elements 0..15 and 16..31 as bf16 pairs
#pragma unroll
    for (int w = 0; w < 4; ++w) {
        const uint32_t L = mx_lookup(q[w] & 0xFFFFu), H = mx_lookup(q[w] >> 16);  // (4w, 4w+16, 4w+1, 4w+17), (+2 ..)
        lo[2 * w] = conv(prmt(L, k43, 0x4240u));
        lo[2 * w + 1] = conv(prmt(H, k43, 0x4240u));
        hi[2 * w] = conv(prmt(L, k43, 0x4341u));
        hi[2 * w + 1] = conv(prmt(H, k43, 0x4341u));
    }
    uint8_t* const row = at + r * 128;
    const int c0 = 4 * blk;
    *reinterpret_cast<uint4*>(row + (((c0 + 0) ^ (r & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    *reinterpret_cast<uint4*>(row + (((c0 + 2) ^ (r & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(row + (((c0 + 3) ^ (r & 7)) << 4)) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
}

template <int F, bool DUMP>
__global__ void __launch_bounds__(kTcThreads, 1) k_gmmtc(const __grid_constant__ GmmTcParams p) {
    static_assert(F == F_Q8_0 || F == F_Q4_K || F == F_MXFP4, "tcgen05 grouped GEMM: Q8_0, Q4_K and MXFP4 banks");
    constexpr bool MX = F == F_MXFP4;
    // PB: one accumulator and one weight scale per 32-block, applied by the
    // epilogue (Q8_0; MXFP4 when dumping the integer core).  Otherwise one
    // accumulator per half superblock (Q4_K) or superblock (MXFP4, whose
    // power-of-two block scales are folded into the bf16 operand).
    constexpr bool PB = F == F_Q8_0 || (MX && DUMP);
    constexpr int kTcEpi = TcRoles<F, DUMP>::kEpi, kTcDec = TcRoles<F, DUMP>::kDec;
    constexpr int kEpiCols = TcRoles<F, DUMP>::kEpiCols, kEpiChunks = kEpiCols / 32;
    constexpr int kRawRow = TcSmem<F>::kRawRow;
    // tensor-memory columns: block, half-superblock or superblock accumulators
    // 0..255, Q4_K mins term 256..383, item accumulator
    // per-block schedule: three block accumulators (0..383), so the MMA runs a block
    // further ahead of the epilogue's drains
    constexpr int kTB = PB ? 3 : 2;
    constexpr uint32_t kAcc = F == F_Q4_K || PB ? 384u : 256u, kDmin = 256u;
    using SM = TcSmem<F>;
    constexpr int kTcABufs = SM::kABufs, kTcStages = SM::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* const smem = smem_raw + ((1024 - (smem_addr(smem_raw) & 1023)) & 1023);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();

    int* const s_pref = reinterpret_cast<int*>(smem + SM::oPrefix);
    uint64_t* const full = reinterpret_cast<uint64_t*>(smem + SM::oBars);
    uint64_t* const empty = full + kTcStages;
    uint64_t* const afull = empty + kTcStages;
    uint64_t* const aempty = afull + kTcABufs;
    uint64_t* const tfull = aempty + kTcABufs;
    uint64_t* const tempty = tfull + 3;
    uint32_t* const tslot = reinterpret_cast<uint32_t*>(tempty + 3);
    volatile int* const abort = reinterpret_cast<volatile int*>(tslot + 1);
    const auto B16 = [&](int s) { return smem + s * SM::kStage; };
    const auto RAW = [&](int s) { return smem + s * SM::kStage + SM::kB; };
    const auto DXS = [&](int s) { return smem + s * SM::kStage + SM::kB + SM::kRaw; };
    const auto ATILE = [&](int a) { return smem + SM::oA + a * SM::kA; };
    uint8_t* const min_a = smem + SM::oMin;              // Q4_K: 6-bit mins per 16-group, SW128 rows
    uint8_t* const min_b = smem + SM::oMin + SM::kA;  // Q4_K: activation 16-group sums, SW128 rows

    if (tid == 0) {
        for (int s = 0; s < kTcStages; ++s) {
            mbar_init(&full[s], 1);
            // PB: decode and epilogue threads (the epilogue has seen the k-step's MMAs complete);
            // otherwise the MMA's commit, decode and epilogue threads
            mbar_init(&empty[s], kTcDec + kTcEpi + (PB ? 0 : 1));
        }
        for (int a = 0; a < kTcABufs; ++a) {
            mbar_init(&afull[a], kTcDec);
            mbar_init(&aempty[a], PB ? kTcEpi : 1);
        }
        for (int d = 0; d < kTB; ++d) {
            mbar_init(&tfull[d], 1);
            mbar_init(&tempty[d], kTcEpi);
        }
        *abort = 0;
        fence_barrier_init();
    }
    if (warp == kTcMmaWarp) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(tslot)),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    pdl_wait();  // groups, permutation and activations come from the previous kernels

    // ---- item table: per group, nmat * mtiles * ceil(cols / 128) items
    const int ngroups = *p.ngroups;
    const int mtiles = static_cast<int>(p.N / kTcBM);
    if (warp == 0) {
        const int per = (ngroups + 31) >> 5, b0 = lane * per, b1 = min(b0 + per, ngroups);
        int own = 0;
        for (int gi = b0; gi < b1; ++gi) own += p.nmat * mtiles * ((p.group_cnt[gi] + kTcBN - 1) / kTcBN);
        int incl = own;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        int acc = incl - own;
        for (int gi = b0; gi < b1; ++gi) {
            s_pref[gi] = acc;
            acc += p.nmat * mtiles * ((p.group_cnt[gi] + kTcBN - 1) / kTcBN);
        }
        if (lane == 31) s_pref[ngroups] = incl;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    const int nitems = s_pref[ngroups];
    const int nk = p.K / kTcBK;
    const int my_items = static_cast<int>(blockIdx.x) < nitems
                             ? (nitems - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                             : 0;
    const int total = my_items * nk;
    const auto item_of = [&](int it) {
        return tc_item(p, s_pref, ngroups, mtiles, static_cast<int>(blockIdx.x) + it * static_cast<int>(gridDim.x));
    };
    // raw bytes per k-step: Q8_0 the 80-byte spans, MXFP4 the 48-byte spans; Q4_K
    // headers [128][16], nibbles [128][32], then at a superblock's end the
    // activation 16-group sums [128][32]
    constexpr uint32_t kRawTx = F == F_Q4_K ? kTcBM * 48 : SM::kRaw;
    constexpr int kQsOff = kTcBM * 16, kBsOff = kTcBM * 48;

    if (warp == kTcTmaWarp) {
        // ================================================================ TMA
        TcItem cur{};
        TcPos q;
        for (int c = 0; c < total; ++c, q.next(kTcStages, kTcABufs, nk)) {
            const int kt = q.kt, s = q.s;
            if (kt == 0) cur = item_of(q.it);
            if (c >= kTcStages && !tc_wait(&empty[s], q.fph ^ 1u, abort, p.err, true)) break;
            if (lane == 0) {
                const bool sb_end = (kt & 3) == 3;
                const bool dx_load = F == F_Q4_K ? (kt & 1) == 1 : sb_end;  // Q4_K: at each half superblock's end
                const bool narrow = cur.ncols <= kTcNarrow;  // 32 activation rows suffice
                mbar_arrive_expect_tx(&full[s], (narrow ? kTcNarrow * 128 : SM::kB) + kRawTx + (dx_load ? SM::kDX : 0) +
                                                    (sb_end && F == F_Q4_K ? kTcBN * 32 : 0));
                tc_tma_2d(smem_addr(B16(s)), narrow ? &p.tm_b32 : &p.tm_b, kt * kTcBK, cur.y0, &full[s]);
                if constexpr (F == F_Q8_0) {
                    tc_tma_2d(smem_addr(RAW(s)), &p.tm_w[cur.m], (68 * kt) & ~15, cur.wrow, &full[s]);
                } else if constexpr (MX) {
                    tc_tma_2d(smem_addr(RAW(s)), &p.tm_w[cur.m], (34 * kt) & ~15, cur.wrow, &full[s]);
                } else {
                    const int x = (kt >> 2) * 144;
                    tc_tma_2d(smem_addr(RAW(s)), &p.tm_w[0], x, cur.wrow, &full[s]);
                    tc_tma_2d(smem_addr(RAW(s)) + kQsOff, &p.tm_w[1], x + 16 + 32 * (kt & 3), cur.wrow, &full[s]);
                }
                if (dx_load) tc_tma_2d(smem_addr(DXS(s)), &p.tm_dx, (kt >> 2) & ~3, cur.y0, &full[s]);
                if (F == F_Q4_K && sb_end) tc_tma_2d(smem_addr(RAW(s)) + kBsOff, &p.tm_bs, (kt >> 2) * 16, cur.y0, &full[s]);
            }
            __syncwarp();
        }
    } else if (warp == kTcMmaWarp) {
        // ================================================================ MMA (one lane)
        if (lane == 0) {
            uint32_t idesc = tc_idesc(kTcBN, MX);
            TcPos q;
            int tb = 0;           // per-block schedule: accumulator of the next block
            uint32_t tph = 0u;    // and the phase of its use
            for (int c = 0; c < total; ++c, q.next(kTcStages, kTcABufs, nk)) {
                const int s = q.s, a = q.a, kt = q.kt;
                if (kt == 0) idesc = tc_idesc(item_of(q.it).ncols <= kTcNarrow ? kTcNarrow : kTcBN, MX);
                if (!tc_wait1(&full[s], q.fph, abort, p.err)) break;
                if (!tc_wait1(&afull[a], q.aph, abort, p.err)) break;
                tc_fence_after();
                // descriptors are linear in the start address (16-byte units): K steps add 2 per 32 bytes
                const uint64_t adesc = umma_desc_sw128(smem_addr(ATILE(a))), bdesc = umma_desc_sw128(smem_addr(B16(s)));
                bool ok = true;
                if constexpr (PB) {
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const int gb = 2 * c + b;
                        if (gb >= kTB && !tc_wait1(&tempty[tb], tph ^ 1u, abort, p.err)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 2; ++kk) {
                            const uint64_t koff = static_cast<uint64_t>((2 * b + kk) * 2);
                            tc_mma(tmem + static_cast<uint32_t>(tb * kTcBN), adesc + koff, bdesc + koff, idesc,
                                   static_cast<uint32_t>(kk));
                        }
                        tc_commit(&tfull[tb]);
                        if (++tb == kTB) tb = 0, tph ^= 1u;
                    }
                } else {
                    // one accumulator per span of SP k-steps (Q4_K: a half superblock, buffer 0
                    // taking the first halves, buffer 1 the second halves and, beside it, the mins
                    // term; MXFP4: a superblock).  nk is a multiple of 4, so c and kt agree on
                    // (c & 3).  For Q4_K, waiting for buffer 1's previous drain also frees the
                    // single mins region (the epilogue reads both together).
                    constexpr int SH = MX ? 2 : 1, SP = 1 << SH;
                    const int hsi = c >> SH, db = hsi & 1;
                    const bool first = (kt & (SP - 1)) == 0, last = (kt & (SP - 1)) == SP - 1;
                    if (first && hsi >= 2 && !tc_wait1(&tempty[db], ((hsi >> 1) - 1) & 1, abort, p.err)) ok = false;
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            tc_mma(tmem + static_cast<uint32_t>(db * kTcBN), adesc + static_cast<uint64_t>(2 * kk),
                                   bdesc + static_cast<uint64_t>(2 * kk), idesc, static_cast<uint32_t>(!first || kk != 0));
                        if (F == F_Q4_K && (kt & 3) == 3)
                            tc_mma(tmem + kDmin, umma_desc_sw128(smem_addr(min_a)), umma_desc_sw128(smem_addr(min_b)), idesc,
                                   0u);
                        if (last) tc_commit(&tfull[db]);
                        tc_commit(&aempty[a]);
                        tc_commit(&empty[s]);
                    }
                }
                if (!ok) break;
            }
        }
        __syncwarp();
    } else if (warp >= kTcEpi / 32) {
        // ================================================================ decode
        const int ord = TcRoles<F, DUMP>::dec_ord(warp);
        if (ord < 0) goto idle;  // no role (MXFP4: the warps on the MMA warp's SMSP)
        const int dt = 32 * ord + lane;
        constexpr int kUnits = (kTcBM * 4 + kTcDec - 1) / kTcDec;  // 16-output units of the 128 x 64 tile
        TcPos q;
        for (int c = 0; c < total; ++c, q.next(kTcStages, kTcABufs, nk)) {
            const int s = q.s, a = q.a, kt = q.kt;
            if (!tc_wait(&full[s], q.fph, abort, p.err)) break;
            if (c >= kTcABufs && !tc_wait(&aempty[a], q.aph ^ 1u, abort, p.err)) break;
            const saddr raw = smem_addr(RAW(s));
            uint8_t* const at = ATILE(a);
            if constexpr (MX) {
                // unit: one 32-block of one row (row u >> 1, block u & 1): its E8M0 byte and 16 nibble bytes
                const int o0 = (34 * kt) & 15;
                for (int u = dt; u < 2 * kTcBM; u += kTcDec) {
                    const int r = u >> 1, blk = u & 1;
                    const saddr b = raw + static_cast<uint32_t>(r * kRawRow + o0 + 17 * blk);
                    uint32_t q[4];
                    ld_words_any<4>(b + 1, q);
                    const uint32_t s2 = DUMP ? 0x3F803F80u : tc_e8m0_bf16x2(ld_u8(b));
                    tc_mx_block(at, r, blk, q, s2);
                }
            } else if constexpr (F == F_Q8_0) {
                const int o0 = (68 * kt) & 15;
                uint32_t w[kUnits][4];
#pragma unroll
                for (int h = 0; h < kUnits; ++h) {
                    const int u = dt + kTcDec * h;  // row u >> 2, block (u >> 1) & 1, half u & 1
                    if (u < kTcBM * 4)
                        ld_words_any<4>(raw + static_cast<uint32_t>((u >> 2) * kRawRow + o0 + 34 * ((u >> 1) & 1) + 2 + 16 * (u & 1)), w[h]);
                }
#pragma unroll
                for (int h = 0; h < kUnits; ++h) {
                    const int u = dt + kTcDec * h;
                    if (u >= kTcBM * 4) break;
                    uint32_t o8[8];
#pragma unroll
                    for (int k = 0; k < 4; ++k) {
                        // code + 128 per byte (xor), as 1024 + (code + 128) (prmt with 0x64 high bytes), minus 1152
                        const uint32_t v = w[h][k] ^ 0x80808080u;
                        const __half2 o = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));
                        const uint32_t x0 = prmt(v, 0x64646464u, 0x4140u), x1 = prmt(v, 0x64646464u, 0x4342u);
                        const __half2 h0 = __hsub2(*reinterpret_cast<const __half2*>(&x0), o);
                        const __half2 h1 = __hsub2(*reinterpret_cast<const __half2*>(&x1), o);
                        o8[2 * k] = *reinterpret_cast<const uint32_t*>(&h0);
                        o8[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&h1);
                    }
                    // 16 outputs = 16-byte chunks 2 (u & 3) and 2 (u & 3) + 1 of row u >> 2, XOR-swizzled by row
                    const int r = u >> 2, c0 = 2 * (u & 3);
                    *reinterpret_cast<uint4*>(at + r * 128 + ((c0 ^ (r & 7)) << 4)) = make_uint4(o8[0], o8[1], o8[2], o8[3]);
                    *reinterpret_cast<uint4*>(at + r * 128 + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(o8[4], o8[5], o8[6], o8[7]);
                }
            } else {
                // unit: 8 nibble bytes of row u >> 2, group u & 3: low nibbles are outputs 8 (u & 3) .. +7
                // (sub-block 2 (kt & 3)), high nibbles outputs 32 + 8 (u & 3) .. +7 (the next sub-block),
                // each already multiplied by its 6-bit scale (sc * q <= 945: exact)
                uint4 hd[kUnits];
                uint32_t qw[kUnits][2];
#pragma unroll
                for (int h = 0; h < kUnits; ++h) {
                    const int u = dt + kTcDec * h;
                    if (u < kTcBM * 4) {
                        hd[h] = ld_s128(raw + static_cast<uint32_t>((u >> 2) * 16));
                        const saddr qa = raw + static_cast<uint32_t>(kQsOff + (u >> 2) * 32 + 8 * (u & 3));
                        qw[h][0] = ld_s32(qa);
                        qw[h][1] = ld_s32(qa + 4);
                    }
                }
                const int cc = kt & 3;
#pragma unroll
                for (int h = 0; h < kUnits; ++h) {
                    const int u = dt + kTcDec * h;
                    if (u >= kTcBM * 4) break;
                    const uint32_t sw = cc < 2 ? (hd[h].y & 0x3F3F3F3Fu) : ((hd[h].w & 0x0F0F0F0Fu) | ((hd[h].y >> 2) & 0x30303030u));
                    const __half2 slo = tc_byte_pair(sw, 2 * (cc & 1)), shi = tc_byte_pair(sw, 2 * (cc & 1) + 1);
                    const __half2 clo = __hmul2(slo, __halves2half2(__ushort_as_half(0xE400u), __ushort_as_half(0xE400u)));
                    const __half2 s16 = __hmul2(shi, __halves2half2(__ushort_as_half(0x2C00u), __ushort_as_half(0x2C00u)));
                    const __half2 chi = __hmul2(shi, __halves2half2(__ushort_as_half(0xD400u), __ushort_as_half(0xD400u)));
                    uint32_t lo[4], hi[4];
#pragma unroll
                    for (int k = 0; k < 2; ++k) {
                        const uint32_t x0 = prmt(qw[h][k], 0x64646464u, 0x4140u), x1 = prmt(qw[h][k], 0x64646464u, 0x4342u);
                        // low nibble: (1024 + n) sc - 1024 sc; high nibble in place: (1024 + 16 n) sc/16 - 64 sc
                        const uint32_t l0 = x0 & 0xFF0FFF0Fu, l1 = x1 & 0xFF0FFF0Fu, h0 = x0 & 0xFFF0FFF0u, h1 = x1 & 0xFFF0FFF0u;
                        const __half2 a0 = __hfma2(*reinterpret_cast<const __half2*>(&l0), slo, clo);
                        const __half2 a1 = __hfma2(*reinterpret_cast<const __half2*>(&l1), slo, clo);
                        const __half2 b0 = __hfma2(*reinterpret_cast<const __half2*>(&h0), s16, chi);
                        const __half2 b1 = __hfma2(*reinterpret_cast<const __half2*>(&h1), s16, chi);
                        lo[2 * k] = *reinterpret_cast<const uint32_t*>(&a0);
                        lo[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&a1);
                        hi[2 * k] = *reinterpret_cast<const uint32_t*>(&b0);
                        hi[2 * k + 1] = *reinterpret_cast<const uint32_t*>(&b1);
                    }
                    const int r = u >> 2, g = u & 3;
                    *reinterpret_cast<uint4*>(at + r * 128 + ((g ^ (r & 7)) << 4)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
                    *reinterpret_cast<uint4*>(at + r * 128 + (((4 + g) ^ (r & 7)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
                }
                if (cc == 3) {
                    // the mins term operands: A row r = the 16-group mins (m_j twice, j = 0..7), B row c =
                    // the 16-group activation sums; only the first 32 bytes (K = 16) of each SW128 row
                    for (int i = dt; i < 2 * kTcBM; i += kTcDec) {
                        const int r = i >> 1, ch = i & 1;
                        const uint4 h4 = ld_s128(raw + static_cast<uint32_t>(r * 16));
                        const uint32_t mw = ch == 0 ? (h4.z & 0x3F3F3F3Fu) : (((h4.w >> 4) & 0x0F0F0F0Fu) | ((h4.z >> 2) & 0x30303030u));
                        uint32_t m4[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            const __half2 mk = tc_byte_pair(mw, k);
                            m4[k] = *reinterpret_cast<const uint32_t*>(&mk);
                        }
                        *reinterpret_cast<uint4*>(min_a + r * 128 + ((ch ^ (r & 7)) << 4)) = make_uint4(m4[0], m4[1], m4[2], m4[3]);
                        const uint4 b4 = ld_s128(raw + static_cast<uint32_t>(kBsOff + r * 32 + 16 * ch));
                        *reinterpret_cast<uint4*>(min_b + r * 128 + ((ch ^ (r & 7)) << 4)) = b4;
                    }
                }
            }
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // generic stores -> tensor-core reads
            mbar_arrive(&afull[a]);
            mbar_arrive(&empty[s]);
        }
    } else {
        // ================================================================ epilogue
        // warp w: tensor-memory lanes 32 (w & 3) .. +31 (tile rows) and kEpiCols columns
        const int q = warp & 3, col0 = kEpiCols * (warp >> 2), r = 32 * q + lane;
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * q) << 16);
        float T[PB ? kEpiCols : 1];
        bool live = true;
        TcPos pos;
        int tb = 0;          // per-block schedule: accumulator of the next block
        uint32_t tph = 0u;   // and the phase of its use
        for (int it = 0; it < my_items && live; ++it) {
            const TcItem cur = item_of(it);
            // column chunks h2 of this warp that hold accumulators (narrow items: the first 32 columns)
            const int ncol_acc = cur.ncols <= kTcNarrow ? kTcNarrow : kTcBN;
            bool act[kEpiChunks];
#pragma unroll
            for (int h2 = 0; h2 < kEpiChunks; ++h2) act[h2] = col0 + 32 * h2 < ncol_acc;
            for (int kt = 0; kt < nk && live; ++kt) {
                const int c = it * nk + kt, s = pos.s;
                const saddr raw = smem_addr(RAW(s));
                if constexpr (PB) {
                    const int o0 = MX ? (34 * kt) & 15 : (68 * kt) & 15;
#pragma unroll
                    for (int b = 0; b < 2; ++b) {
                        const int db = tb;
                        if (!tc_wait(&tfull[db], tph, abort, p.err, true)) { live = false; break; }
                        if (++tb == kTB) tb = 0, tph ^= 1u;
                        tc_fence_after();
                        const saddr wb = raw + static_cast<uint32_t>(r * kRawRow + o0 + (MX ? 17 : 34) * b);
                        const float dw = MX ? e8m0_half_scale(ld_u8(wb)) : ld_h(wb);
                        const bool first = b == 0 && (kt & 3) == 0;
#pragma unroll
                        for (int h2 = 0; h2 < kEpiChunks; ++h2) {
                            if (!act[h2]) continue;
                            float v[32];
                            tmem_ld32(lane_base + static_cast<uint32_t>(db * kTcBN + col0 + 32 * h2), v);
                            if constexpr (DUMP) tc_dump32(p, cur, r, col0 + 32 * h2, v, 2 * kt + b, false);
#pragma unroll
                            for (int j = 0; j < 32; j += 2) {
                                float* const t = T + 32 * h2 + j;
                                ffma2(t[0], t[1], v[j], v[j + 1], dw, first ? 0.0f : t[0], first ? 0.0f : t[1]);
                            }
                        }
                        tc_fence_before();
                        mbar_arrive(&tempty[db]);
                        if (b == 1) mbar_arrive(&aempty[pos.a]);  // every MMA of the k-step has completed
                    }
                    if (!live) break;
                    if ((kt & 3) == 3) {  // superblock end: acc += T * d_x (per column)
                        const saddr dxs = smem_addr(DXS(s)) + 4u * ((kt >> 2) & 3);
#pragma unroll
                        for (int h2 = 0; h2 < kEpiChunks; ++h2) {
                            if (!act[h2]) continue;
                            float a[32];
                            const uint32_t ta = lane_base + kAcc + static_cast<uint32_t>(col0 + 32 * h2);
                            if (kt == 3) {
#pragma unroll
                                for (int j = 0; j < 32; ++j) a[j] = 0.0f;
                            } else {
                                tmem_ld32(ta, a);
                            }
#pragma unroll
                            for (int j = 0; j < 32; j += 2)
                                ffma2p(a[j], a[j + 1], T[32 * h2 + j], T[32 * h2 + j + 1], ld_f32(dxs + 16u * (col0 + 32 * h2 + j)),
                                       ld_f32(dxs + 16u * (col0 + 32 * h2 + j + 1)), a[j], a[j + 1]);
                            tmem_st32(ta, a);
                        }
                    }
                } else if (MX ? (kt & 3) == 3 : (kt & 1) == 1) {
                    // MXFP4: superblock end, acc += D d_x (the block scales are in the operands);
                    // Q4_K: half-superblock end, acc += D d d_x (first half) or (D d - Dmin dmin) d_x (second)
                    const int hsi = c >> (MX ? 2 : 1), db = hsi & 1;
                    const bool second = (kt & 3) == 3;
                    if (!tc_wait(&tfull[db], (hsi >> 1) & 1, abort, p.err, true)) { live = false; break; }
                    tc_fence_after();
                    float dd = 1.0f, dm = 0.0f;
                    if constexpr (!MX) {
                        const uint32_t dh = ld_s32(raw + static_cast<uint32_t>(r * 16));  // d, dmin of this row
                        dd = half_lo(dh), dm = half_hi(dh);
                    }
                    const saddr dxs = smem_addr(DXS(s)) + 4u * ((kt >> 2) & 3);
#pragma unroll
                    for (int h2 = 0; h2 < kEpiChunks; ++h2) {
                        if (!act[h2]) continue;
                        float v[32], m[32], a[32];
                        tmem_ld32(lane_base + static_cast<uint32_t>(db * kTcBN + col0 + 32 * h2), v);
                        if (!MX && second) {
                            tmem_ld32(lane_base + kDmin + static_cast<uint32_t>(col0 + 32 * h2), m);
                        } else {
#pragma unroll
                            for (int j = 0; j < 32; ++j) m[j] = 0.0f;
                        }
                        if constexpr (DUMP && !MX) {
                            tc_dump32(p, cur, r, col0 + 32 * h2, v, 2 * (kt >> 2), second);
                            if (second) tc_dump32(p, cur, r, col0 + 32 * h2, m, 2 * (kt >> 2) + 1, false);
                        }
                        const uint32_t ta = lane_base + kAcc + static_cast<uint32_t>(col0 + 32 * h2);
                        if (kt == (MX ? 3 : 1)) {
#pragma unroll
                            for (int j = 0; j < 32; ++j) a[j] = 0.0f;
                        } else {
                            tmem_ld32(ta, a);
                        }
#pragma unroll
                        for (int j = 0; j < 32; j += 2) {
                            float w0, w1;  // D d - Dmin dmin (MXFP4: D)
                            ffma2(w0, w1, v[j], v[j + 1], dd, -m[j] * dm, -m[j + 1] * dm);
                            ffma2p(a[j], a[j + 1], w0, w1, ld_f32(dxs + 16u * (col0 + 32 * h2 + j)),
                                   ld_f32(dxs + 16u * (col0 + 32 * h2 + j + 1)), a[j], a[j + 1]);
                        }
                        tmem_st32(ta, a);
                    }
                    tc_fence_before();
                    mbar_arrive(&tempty[db]);
                }
                mbar_arrive(&empty[s]);
                pos.next(kTcStages, kTcABufs, nk);
            }
            if (!live) break;
            // item end: this thread's row of the item's columns
            float* const out = p.out[cur.m];
            const int64_t row = static_cast<int64_t>(cur.mt) * kTcBM + r;
#pragma unroll
            for (int h2 = 0; h2 < kEpiChunks; ++h2) {
                if (!act[h2]) continue;
                float a[32];
                tmem_ld32(lane_base + kAcc + static_cast<uint32_t>(col0 + 32 * h2), a);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int col = col0 + 32 * h2 + j;
                    if (col < cur.ncols) out[static_cast<int64_t>(p.perm[cur.y0 + col]) * p.N + row] = a[j];
                }
            }
        }
    }
idle:
    tc_fence_before();
    __syncthreads();
    if (warp == kTcMmaWarp) {
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
}

}  // namespace ggq

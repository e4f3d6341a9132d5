// ggq_stream.cuh -- the weight-streaming kernel behind the decode GEMV at 1-2
// tokens and the block-dot dump; its consumer (row_accumulate) also serves the
// direct tiny-batch MoE route (ggq_direct.cuh).
//
// HBM-bound design for sm_103a:
//   * one CTA per SM (persistent: items blockIdx.x, +gridDim.x, ...);
//   * a producer warp streams each item's weight rows (a contiguous byte range
//     per matrix: rows are stored back to back) into a ring of shared-memory
//     stages with cp.async.bulk, completion counted on an mbarrier in bytes, so
//     tens of KB per SM are in flight without tying up registers;
//   * sixteen consumer warps take one row each per stage; each lane decodes
//     64-weight units of its row (nibbles and 6-bit scales unpacked in
//     registers, the scale decode paid once per 64 weights) and runs the int8
//     dp4a integer core against the quantized activations, staged once per
//     CTA into shared memory (structure of arrays, padded against bank
//     conflicts);
//   * per-lane fp32 partials of (row, token) are summed with one transpose
//     reduction per stage;
//   * rows too long for two whole 16-row stages stream in row chunks (one
//     chunk of each of the tile's rows per stage, a row's partials kept in
//     registers across its chunks and reduced once per tile).
// Every wait is bounded; on timeout the kernel records an error word, drains
// its own copies and returns.
#pragma once
#include <atomic>
#include "ggq_device.cuh"
#include "ggq_internal.h"

namespace ggq {

// Start barrier between the producer warp (arrives once the mbarriers are
// initialised, without waiting) and the consumer warps (wait for it).
__device__ __forceinline__ void start_arrive() { asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory"); }
__device__ __forceinline__ void start_sync() { asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory"); }

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); }

// Shared-memory activation region (layout of x_region_bytes).
struct XRegion {
    int8_t* q;
    float* d;
    int32_t* s32;
    int16_t* bs;
};

__device__ __forceinline__ XRegion x_region(uint8_t* base, int rows, int K, bool q81) {
    XRegion r;
    const size_t qb = x_up128(static_cast<size_t>(rows) * xq_row_bytes(K));
    const size_t db = x_up128(static_cast<size_t>(rows) * (K / (q81 ? 32 : 256)) * 4);
    const size_t sb = x_up128(static_cast<size_t>(rows) * (K / 32) * 4);
    r.q = reinterpret_cast<int8_t*>(base);
    r.d = reinterpret_cast<float*>(base + qb);
    r.s32 = reinterpret_cast<int32_t*>(base + qb + db);
    r.bs = reinterpret_cast<int16_t*>(base + qb + db + sb);
    return r;
}

// Stage packed activation rows (Q8_K: 292-byte blocks, rows `pitch` bytes
// apart (0: packed); Q8_1: 36-byte blocks) from global into the
// structure-of-arrays region.  PERM stores each 32-block's quants in the
// interleaved order (0,16,1,17,...) that the MXFP4 lookup produces.  The Q8_1
// per-32 sums must be zero on entry (they are accumulated with atomics).
// Q8_K work unit: one 32-element quant group (8 words) or the scale and the
// sixteen sums of a block (9 words); two units per thread per round, all their
// loads in flight together.  G: src is in global memory (read through L2), else
// a raw copy of the rows already in shared memory.
template <bool G>
__device__ __forceinline__ uint32_t ld_act(const uint32_t* a) {
    if constexpr (G) return __ldcg(a);
    else return *a;
}
template <bool Q81, bool PERM, bool G = true>
__device__ void stage_acts(const uint8_t* __restrict__ src, int rows, int K, const XRegion& x, int tid, int nthr,
                           int pitch = 0) {
    const int rb = xq_row_bytes(K);
    if constexpr (!Q81) {
        const int nbr = K >> 8;
        const int units = rows * nbr * 9;
        if (pitch == 0) pitch = nbr * 292;
        for (int u0 = tid; u0 < units; u0 += 2 * nthr) {
            uint32_t w[2][9];
            int blk[2], part[2], row[2], cb[2];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int u = u0 + h * nthr;
                blk[h] = u / 9;
                part[h] = u - blk[h] * 9;
                row[h] = blk[h] / nbr;
                cb[h] = blk[h] - row[h] * nbr;
                if (u < units) {
                    const uint32_t* bp = reinterpret_cast<const uint32_t*>(src + static_cast<size_t>(row[h]) * pitch +
                                                                           static_cast<size_t>(cb[h]) * 292);
                    if (part[h] < 8) {
#pragma unroll
                        for (int i = 0; i < 8; ++i) w[h][i] = ld_act<G>(bp + 1 + 8 * part[h] + i);
                        w[h][8] = 0u;
                    } else {
                        w[h][0] = ld_act<G>(bp);
#pragma unroll
                        for (int i = 0; i < 8; ++i) w[h][1 + i] = ld_act<G>(bp + 65 + i);
                    }
                }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (u0 + h * nthr >= units) break;
                const int b = blk[h];
                if (part[h] < 8) {
                    const uint32_t* v = w[h];
                    uint4 lo, hi;
                    if constexpr (PERM) {  // (j, j+16, j+1, j+17) per output word
                        lo = make_uint4(prmt(v[0], v[4], 0x5140u), prmt(v[0], v[4], 0x7362u), prmt(v[1], v[5], 0x5140u),
                                        prmt(v[1], v[5], 0x7362u));
                        hi = make_uint4(prmt(v[2], v[6], 0x5140u), prmt(v[2], v[6], 0x7362u), prmt(v[3], v[7], 0x5140u),
                                        prmt(v[3], v[7], 0x7362u));
                    } else {
                        lo = make_uint4(v[0], v[1], v[2], v[3]);
                        hi = make_uint4(v[4], v[5], v[6], v[7]);
                    }
                    // a 32-group lies inside one padded 64-element unit: 32 contiguous bytes, 16-aligned
                    int8_t* dq = x.q + static_cast<size_t>(row[h]) * rb + xq_addr(256 * cb[h] + 32 * part[h]);
                    reinterpret_cast<uint4*>(dq)[0] = lo;
                    reinterpret_cast<uint4*>(dq)[1] = hi;
                } else {
                    x.d[b] = __uint_as_float(w[h][0]);
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        const uint32_t v = w[h][1 + j];  // bsums 2j, 2j+1
                        reinterpret_cast<uint32_t*>(x.bs + static_cast<size_t>(b) * 16)[j] = v;
                        x.s32[static_cast<size_t>(b) * 8 + j] = static_cast<int>(static_cast<int16_t>(v & 0xFFFFu)) +
                                                               static_cast<int>(static_cast<int16_t>(v >> 16));
                    }
                }
            }
        }
    } else {
        const int nbr = K >> 5;
        const int nb = rows * nbr;
        const int words = nb * 9;
        for (int i = tid; i < words; i += nthr) {
            const int b = i / 9, w = i - b * 9;
            const uint32_t v = ld_act<G>(reinterpret_cast<const uint32_t*>(src + static_cast<size_t>(b) * 36) + w);
            if (w == 0) {
                x.d[b] = half_lo(v);
            } else {
                const int row = b / nbr, cb = b - row * nbr;
                *reinterpret_cast<uint32_t*>(x.q + static_cast<size_t>(row) * rb + xq_addr(32 * cb + 4 * (w - 1))) = v;
                atomicAdd(&x.s32[b], __dp4a(static_cast<int>(v), 0x01010101, 0));
            }
        }
    }
}

// Stage packed Q8_0 activation rows (34-byte blocks: fp16 d, 32 quants) into
// the per-32 structure-of-arrays region (the layout Q8_1 rows are staged in):
// one thread per block, its 17 halfwords loaded together (G: from global).
template <bool G = true>
__device__ inline void stage_acts_q8_0(const uint8_t* __restrict__ src, int rows, int K, const XRegion& x, int tid, int nthr) {
    const int rb = xq_row_bytes(K), nbr = K >> 5;
    for (int b = tid; b < rows * nbr; b += nthr) {
        const uint16_t* h = reinterpret_cast<const uint16_t*>(src + static_cast<size_t>(b) * 34);
        uint32_t hw[17];
#pragma unroll
        for (int i = 0; i < 17; ++i) hw[i] = G ? __ldg(h + i) : h[i];
        uint32_t w[8];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            w[i] = hw[1 + 2 * i] | (hw[2 + 2 * i] << 16);
            sum += __dp4a(static_cast<int>(w[i]), 0x01010101, 0);
        }
        const int row = b / nbr, cb = b - row * nbr;
        uint4* dq = reinterpret_cast<uint4*>(x.q + static_cast<size_t>(row) * rb + xq_addr(32 * cb));
        dq[0] = make_uint4(w[0], w[1], w[2], w[3]);
        dq[1] = make_uint4(w[4], w[5], w[6], w[7]);
        x.d[b] = __half2float(__ushort_as_half(static_cast<unsigned short>(hw[0])));
        x.s32[b] = sum;
    }
}

// Accumulate one row against the activation rows xr[0..nslots) into acc[].
// For 1-2 slots two units per lane are kept in flight (units u and u+32) so
// that their load, decode and dp4a chains overlap.  With ue >= 0 only units
// [u0, ue) are taken; `row` is then the address the row's start would have,
// so that unit u still sits at its offset in the row.
template <int F, int NT, bool A32 = (F == F_Q4_0)>
__device__ __forceinline__ void row_accumulate(saddr row, const XS& xs, const int* xr, int nslots,
                                               float* acc, int lane, int u0 = 0, int ue = -1) {
    const int nu = ue < 0 ? units_per_row(xs.K) : ue, nb32 = xs.K >> 5;
    int u = u0 + lane;
    // two units in flight for 1-2 slots; at 4+ slots the slot loop supplies the
    // independent work and a second unit would only spill (17 warps cap a
    // thread at 96 registers)
    for (; NT <= 2 && u + 32 < nu; u += 64) {
        Unit ua, ub;
        load_unit<F>(row, u, nb32, ua);
        load_unit<F>(row, u + 32, nb32, ub);
        int xa[4], xb[4];
        unit_offsets<F>(u, xa);
        unit_offsets<F>(u + 32, xb);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if (j < nslots) {
                int A0, A1, B0, B1;
                unit_ints<F>(ua, xa, xs, xr[j], u, A0, A1);
                unit_ints<F>(ub, xb, xs, xr[j], u + 32, B0, B1);
                acc[j] += unit_value<F, A32>(ua, xs, xr[j], u, A0, A1) + unit_value<F, A32>(ub, xs, xr[j], u + 32, B0, B1);
            }
        }
    }
    for (; u < nu; u += 32) {
        Unit un;
        load_unit<F>(row, u, nb32, un);
        int xo[4];
        unit_offsets<F>(u, xo);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if (j < nslots) {
                int A0, A1;
                unit_ints<F>(un, xo, xs, xr[j], u, A0, A1);
                acc[j] += unit_value<F, A32>(un, xs, xr[j], u, A0, A1);
            }
        }
    }
}

// Integer coefficients of one row for the dump: out[j][row_index][...].
template <int F, int NT>
__device__ __forceinline__ void row_coefs(saddr row, const XS& xs, int nslots, int64_t row_index,
                                          int64_t N, int32_t* out, int lane) {
    const int nu = units_per_row(xs.K), nb32 = xs.K >> 5;
    const int ncoef = (xs.K / fmt_qk(F)) * fmt_coefs(F);
    for (int u0 = 0; u0 < nu; u0 += 32) {
        const int u = u0 + lane;
        const bool valid = u < nu;
        Unit un;
        int xo[4];
        if (valid) {
            load_unit<F>(row, u, nb32, un);
            unit_offsets<F>(u, xo);
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if (j < nslots) {
                int A0 = 0, A1 = 0;
                if (valid) unit_ints<F>(un, xo, xs, j, u, A0, A1);
                int32_t* o = out + (static_cast<int64_t>(j) * N + row_index) * ncoef;
                if constexpr (fmt_qk(F) == 32) {
                    if (valid) {
                        o[2 * u] = A0;
                        if (2 * u + 1 < nb32) o[2 * u + 1] = A1;
                    }
                } else {
                    // the four units of a superblock sit on four consecutive lanes
                    A0 += __shfl_xor_sync(0xffffffffu, A0, 1);
                    A1 += __shfl_xor_sync(0xffffffffu, A1, 1);
                    A0 += __shfl_xor_sync(0xffffffffu, A0, 2);
                    A1 += __shfl_xor_sync(0xffffffffu, A1, 2);
                    if (valid && (u & 3) == 0) {
                        if constexpr (fmt_coefs(F) == 2) {
                            o[2 * (u >> 2)] = A0;
                            o[2 * (u >> 2) + 1] = A1;
                        } else {
                            o[u >> 2] = A0;
                        }
                    }
                }
            }
        }
    }
}

// Integer coefficients of one staged row against one activation row (xrow)
// into out[0 .. K/blk * c): the dp4a integer core of row_accumulate, for the
// dumps of the kernels that use it.  Kept out of line so that the hot loops
// do not carry its registers.
template <int F>
__device__ __noinline__ void row_coefs_one(saddr row, const XS& xs, int xrow, int32_t* out, int lane) {
    const int nu = units_per_row(xs.K), nb32 = xs.K >> 5;
    for (int u0 = 0; u0 < nu; u0 += 32) {
        const int u = u0 + lane;
        const bool valid = u < nu;
        Unit un;
        int xo[4];
        int A0 = 0, A1 = 0;
        if (valid) {
            load_unit<F>(row, u, nb32, un);
            unit_offsets<F>(u, xo);
            unit_ints<F>(un, xo, xs, xrow, u, A0, A1);
        }
        if constexpr (fmt_qk(F) == 32) {
            if (valid) {
                out[2 * u] = A0;
                if (2 * u + 1 < nb32) out[2 * u + 1] = A1;
            }
        } else {
            // the four units of a superblock sit on four consecutive lanes
            A0 += __shfl_xor_sync(0xffffffffu, A0, 1);
            A1 += __shfl_xor_sync(0xffffffffu, A1, 1);
            A0 += __shfl_xor_sync(0xffffffffu, A0, 2);
            A1 += __shfl_xor_sync(0xffffffffu, A1, 2);
            if (valid && (u & 3) == 0) {
                if constexpr (fmt_coefs(F) == 2) {
                    out[2 * (u >> 2)] = A0;
                    out[2 * (u >> 2) + 1] = A1;
                } else {
                    out[u >> 2] = A0;
                }
            }
        }
    }
}

// AK: the activation blocks -- 0: the format's own pairing (Q8_1 for Q4_0, Q8_K
// otherwise); 1: Q8_0 activation blocks (with Q4_0 or Q8_0 weights).  CH: the
// GEMV streams row chunks (p.chunk_units > 0), else whole rows.  The two are
// separate instances: with both schedules in one kernel the row-chunk one ran
// 1.4 us slower per launch on the 4096 x 14336 Q8_0 shape.
template <int KIND, int F, int NT, int AK = 0, bool CH = false>
__global__ void __launch_bounds__(kThreads, 1) k_stream(const StreamParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr bool Q81 = fmt_q81(F) || AK == 1;  // per-32 activation scales
    constexpr int LV = NT == 1 ? 0 : NT == 2 ? 1 : NT == 4 ? 2 : 3;  // log2(NT)
    constexpr int SH = 5 - LV;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    pdl_launch_dependents();

    // ---- shared memory layout: ring | activations | barriers | misc
    uint8_t* ring = smem;
    uint8_t* xreg = smem + static_cast<size_t>(p.stages) * p.stage_stride;
    const int K = p.K;
    const XRegion xr_ = x_region(xreg, p.xrows, K, Q81);
    uint64_t* full = reinterpret_cast<uint64_t*>(xreg + p.x_bytes);
    uint64_t* empty = full + kMaxStages;
    uint64_t* xready = empty + kMaxStages;  // the consumers hold their activations
    uint64_t* xbar = xready + 1;            // the raw activation rows have landed
    int* s_flag = reinterpret_cast<int*>(xbar + 1);  // [1] abort

    // Whole-row rings: the packed activation rows come in by one bulk copy into
    // the ring's last stage when they fit there (every CTA reads the same few
    // KB, and word loads from 152 SMs queue on those few L2 lines: ~1.8 us for
    // one token), and the producer fills that stage only once the consumers
    // hold their activations (xready).  Row-chunk rings (small stages, about
    // six of them) measured slower that way: there the activations are read
    // directly and every stage streams at once.
    const int xtot = p.xrows * (AK == 1 ? (K >> 5) * 34 : Q81 ? (K >> 5) * 36 : (K >> 8) * 292);
    const bool xb = !CH && p.stages >= 2 && xtot <= p.stage_stride && xtot % 16 == 0 &&
                    (reinterpret_cast<uintptr_t>(p.xq) & 15) == 0;

    // ---- work items: 16-row tiles
    const int nitems = static_cast<int>((p.N + kTileRows - 1) / kTileRows);
    if (static_cast<int>(blockIdx.x) >= nitems) return;  // whole CTA idle (uniform)

    if (warp == kConsumerWarps) {
        // ================= producer: initialise the barriers, release the
        // consumers (start barrier, no wait), then stream
        if (lane == 0) {
            for (int s = 0; s < p.stages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kConsumerWarps);
            }
            mbar_init(xready, 1);
            mbar_init(xbar, 1);
            s_flag[0] = 0;
            s_flag[1] = 0;
            fence_barrier_init();
        }
        __syncwarp();
        start_arrive();
        if constexpr (KIND == KIND_GEMV && CH) {
            // rows too long for whole-row stages: stage j = (tile, chunk kc); lane i
            // brings row i's chunk.  A row slot holds global byte x at slot + (x -
            // x0), x0 the chunk start rounded down to 16 bytes: the 16-byte-aligned
            // middle of the chunk is one bulk copy, the ragged ends (rows that are
            // not 16-byte multiples only) are copied byte by byte
            const uint64_t pol = policy_evict_first();
            if (!p.early_weights) pdl_wait();
            const int nkc = (units_per_row(K) + p.chunk_units - 1) / p.chunk_units;
            int j = 0;
            bool ok = true;
            for (int item = blockIdx.x; ok && item < nitems; item += gridDim.x) {
                const int64_t r0 = static_cast<int64_t>(item) * kTileRows;
                const int nr = static_cast<int>(p.N - r0 < kTileRows ? p.N - r0 : kTileRows);
                for (int kc = 0; kc < nkc; ++kc, ++j) {
                    const int s = j % p.stages;
                    if (xb && j == p.stages - 1) {  // the last stage once the activations are in
                        if (lane == 0) ok = mbar_wait(xready, 0u);
                        ok = __shfl_sync(0xffffffffu, ok, 0);
                        if (!ok) {
                            if (lane == 0) set_error(p.err, DEV_ERR_TIMEOUT);
                            break;
                        }
                    }
                    const int64_t off = static_cast<int64_t>(kc) * p.chunk_bytes;
                    const int64_t cb = p.rowbytes - off < p.chunk_bytes ? p.rowbytes - off : p.chunk_bytes;
                    if (lane == 0) ok = mbar_wait(&empty[s], (static_cast<uint32_t>(j / p.stages) & 1u) ^ 1u);
                    ok = __shfl_sync(0xffffffffu, ok, 0);
                    if (!ok) {
                        if (lane == 0) set_error(p.err, DEV_ERR_TIMEOUT);
                        break;
                    }
                    uint32_t bulk = 0u;
                    if (lane < nr) {
                        const uint8_t* src = p.W + (r0 + lane) * p.rowbytes + off;
                        const uintptr_t x0 = reinterpret_cast<uintptr_t>(src) & ~static_cast<uintptr_t>(15);
                        const uintptr_t a0 = (reinterpret_cast<uintptr_t>(src) + 15) & ~static_cast<uintptr_t>(15);
                        const uintptr_t a1 = (reinterpret_cast<uintptr_t>(src) + cb) & ~static_cast<uintptr_t>(15);
                        uint8_t* slot = ring + static_cast<size_t>(s) * p.stage_stride + static_cast<size_t>(lane) * p.row_slot;
                        const uint8_t* end = src + cb;
                        const uint8_t* mid0 = a1 > a0 ? reinterpret_cast<const uint8_t*>(a0) : end;
                        const uint8_t* mid1 = a1 > a0 ? reinterpret_cast<const uint8_t*>(a1) : end;
                        for (const uint8_t* q = src; q < mid0; ++q) slot[q - reinterpret_cast<const uint8_t*>(x0)] = __ldg(q);
                        for (const uint8_t* q = mid1; q < end; ++q) slot[q - reinterpret_cast<const uint8_t*>(x0)] = __ldg(q);
                        // this lane's byte stores (now and in earlier passes over the slot)
                        // before the bulk copies that may later land on the same bytes
                        if (mid0 != src || mid1 != end) fence_proxy_async_smem();
                        if (a1 > a0) {
                            bulk = static_cast<uint32_t>(a1 - a0);
                            bulk_g2s(slot + (a0 - x0), reinterpret_cast<const uint8_t*>(a0), bulk, &full[s], pol);
                        }
                    }
                    // the byte stores above happen before lane 0's arrive (release)
                    const uint32_t total = __reduce_add_sync(0xffffffffu, bulk);
                    __syncwarp();
                    if (lane == 0) mbar_arrive_expect_tx(&full[s], total);
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
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            if (!p.early_weights) pdl_wait();  // the previous kernel may still be writing the weights
            int j = 0;
            for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++j) {
                const int s = j % p.stages;
                const uint32_t ph = static_cast<uint32_t>(j / p.stages) & 1u;
                if (xb && j == p.stages - 1 && !mbar_wait(xready, 0u)) {  // the last stage once the activations are in
                    set_error(p.err, DEV_ERR_TIMEOUT);
                    break;
                }
                if (!mbar_wait(&empty[s], ph ^ 1u)) {
                    set_error(p.err, DEV_ERR_TIMEOUT);
                    break;
                }
                const uint8_t* src[2];
                uint32_t bytes[2];
                int ncopy = 1;
                if constexpr (KIND == KIND_GEMV || KIND == KIND_DUMP) {
                    const int64_t r0 = static_cast<int64_t>(item) * kTileRows;
                    const int64_t nr = p.N - r0 < kTileRows ? p.N - r0 : kTileRows;
                    src[0] = p.W + r0 * p.rowbytes;
                    bytes[0] = static_cast<uint32_t>(nr * p.rowbytes);
                }
                uint8_t* dst = ring + static_cast<size_t>(s) * p.stage_stride;
                uint32_t total = 0;
                uint32_t off = 0;
                for (int c = 0; c < ncopy; ++c) {
                    const uint32_t bulk = bytes[c] & ~15u;
                    for (uint32_t b = bulk; b < bytes[c]; ++b) dst[off + b] = __ldg(src[c] + b);  // ragged tail
                    total += bulk;
                    off += bytes[c];
                }
                mbar_arrive_expect_tx(&full[s], total);
                off = 0;
                for (int c = 0; c < ncopy; ++c) {
                    const uint32_t bulk = bytes[c] & ~15u;
                    if (bulk) bulk_g2s(dst + off, src[c], bulk, &full[s], pol);
                    off += bytes[c];
                }
            }
            // never leave copies in flight: wait for the last issued phase of every stage
            for (int q = (j > p.stages ? j - p.stages : 0); q < j; ++q) {
                if (!mbar_wait(&full[q % p.stages], static_cast<uint32_t>(q / p.stages) & 1u)) {
                    set_error(p.err, DEV_ERR_TIMEOUT);
                    break;
                }
            }
        }
        return;
    }

    // ================= consumers (512 threads)
    const int ctid = tid;
    if constexpr (Q81) {  // per-32 sums are accumulated with atomics
        for (int i = tid; i < p.xrows * (K >> 5); i += kConsumerWarps * 32) xr_.s32[i] = 0;
    }
    start_sync();  // barriers initialised, sums zeroed
    pdl_wait();  // activations come from the previous kernel; outputs are written after it finished
    const uint8_t* xsrc = p.xq;
    if (xb) {
        uint8_t* const raw = ring + static_cast<size_t>(p.stages - 1) * p.stage_stride;
        if (tid == 0) {
            mbar_arrive_expect_tx(xbar, static_cast<uint32_t>(xtot));
            bulk_g2s(raw, p.xq, static_cast<uint32_t>(xtot), xbar, policy_evict_last());
        }
        if (!mbar_wait(xbar, 0u)) set_error(p.err, DEV_ERR_TIMEOUT);
        xsrc = raw;
    }
    if constexpr (AK == 1) {
        if (xb) stage_acts_q8_0<false>(xsrc, p.xrows, K, xr_, ctid, kConsumerWarps * 32);
        else stage_acts_q8_0<true>(xsrc, p.xrows, K, xr_, ctid, kConsumerWarps * 32);
    } else {
        if (xb) stage_acts<Q81, F == F_MXFP4, false>(xsrc, p.xrows, K, xr_, ctid, kConsumerWarps * 32);
        else stage_acts<Q81, F == F_MXFP4, true>(xsrc, p.xrows, K, xr_, ctid, kConsumerWarps * 32);
    }
    consumer_sync();
    if (tid == 0) mbar_arrive(xready);  // the producer may now stream the remaining weight stages
    XS xs;
    xs.q = smem_addr(xr_.q);
    xs.d = smem_addr(xr_.d);
    xs.s32 = smem_addr(xr_.s32);
    xs.bs = smem_addr(xr_.bs);
    xs.K = K;
    const saddr ring_s = smem_addr(ring);

    if constexpr (KIND == KIND_GEMV && NT == 1) {
        const int nu = units_per_row(K), nb32 = K >> 5;
        if (!CH && nu <= 64) {
            // One token, K <= 4096: lane l owns units l and l + 32 of every row,
            // so its activations stay in registers for the whole kernel.
            XUnit xa, xb;
            const bool va = lane < nu, vb = lane + 32 < nu;
            if (va) load_xunit<F, Q81>(xs, lane, xa);
            if (vb) load_xunit<F, Q81>(xs, lane + 32, xb);
            int j = 0;
            for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++j) {
                const int s = j % p.stages;
                const uint32_t ph = static_cast<uint32_t>(j / p.stages) & 1u;
                const bool ready = __all_sync(0xffffffffu, mbar_wait(&full[s], ph));  // warp-uniform
                if (!ready) set_error(p.err, DEV_ERR_TIMEOUT);
                const int64_t r = static_cast<int64_t>(item) * kTileRows + warp;
                if (ready && r < p.N) {
                    const saddr row = ring_s + static_cast<uint32_t>(s * p.stage_stride + warp * p.rowbytes);
                    float acc;
                    if (nu > 32) {
                        const float a = unit_dot_rx<F, Q81>(row, lane, nb32, xa);
                        const float b = vb ? unit_dot_rx<F, Q81>(row, lane + 32, nb32, xb) : 0.0f;
                        acc = a + b;
                    } else {
                        acc = va ? unit_dot_rx<F, Q81>(row, lane, nb32, xa) : 0.0f;
                    }
                    const float v = warp_transpose_reduce<0>(&acc, lane);
                    if (lane == 0) p.Y[r] = v;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            return;
        }
    }

    if constexpr (KIND == KIND_GEMV && NT == 2) {
        const int nu = units_per_row(K), nb32 = K >> 5;
        if (!CH && nu <= 64 && p.T == 2) {
            // Two tokens, K <= 4096: a lane holds both tokens' activations of one
            // unit for the whole kernel and loads and masks each weight word once
            // for both.  Up to 32 units a warp takes row w of the tile, unit = lane;
            // above, warps 2i and 2i + 1 take rows 2i and 2i + 1, units lane and
            // lane + 32, and the odd warp's four sums (row, token) reach the even
            // warp through shared memory: two buffers by tile parity, one 64-thread
            // named barrier per warp pair.
            const bool split = nu > 32;
            const int hh = split ? (warp & 1) : 0;
            const int uu = lane + 32 * hh;
            const bool vu = uu < nu;
            XUnit x2[2];
            if (vu) {
                load_xunit<F, Q81>(xs, uu, x2[0]);
                XS x1 = xs;
                x1.q = xs.q + static_cast<uint32_t>(xq_row_bytes(K));
                x1.d = xs.d + 4u * static_cast<uint32_t>(K / (Q81 ? 32 : 256));
                x1.s32 = xs.s32 + 4u * static_cast<uint32_t>(K >> 5);
                x1.bs = xs.bs + 2u * static_cast<uint32_t>(K >> 4);
                load_xunit<F, Q81>(x1, uu, x2[1]);
            }
            consumer_sync();  // every warp holds its activations: the region now carries the partials
            float* const red = reinterpret_cast<float*>(xr_.q);  // [2][8 pairs][4]
            int j = 0;
            for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++j) {
                const int s = j % p.stages;
                const uint32_t ph = static_cast<uint32_t>(j / p.stages) & 1u;
                const bool ready = __all_sync(0xffffffffu, mbar_wait(&full[s], ph));  // warp-uniform
                if (!ready) set_error(p.err, DEV_ERR_TIMEOUT);
                const saddr stage = ring_s + static_cast<uint32_t>(s * p.stage_stride);
                const int64_t r0 = static_cast<int64_t>(item) * kTileRows;
                if (split) {
                    // rows 2i, 2i + 1 of the tile: acc = {row 2i tok 0, row 2i tok 1, row 2i+1 tok 0, row 2i+1 tok 1}
                    const int i2 = warp & ~1;
                    float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                    if (ready && vu) {
                        if (r0 + i2 < p.N) unit_dot_rxn<F, Q81, 2>(stage + static_cast<uint32_t>(i2 * p.rowbytes), uu, nb32, x2, acc);
                        if (r0 + i2 + 1 < p.N)
                            unit_dot_rxn<F, Q81, 2>(stage + static_cast<uint32_t>((i2 + 1) * p.rowbytes), uu, nb32, x2, acc + 2);
                    }
                    float v = warp_transpose_reduce<2>(acc, lane);  // lane >> 3 = 2 row + token
                    float* const slot = red + 32 * (j & 1) + 4 * (warp >> 1) + (lane >> 3);
                    if (hh == 1 && (lane & 7) == 0) *slot = v;
                    asm volatile("bar.sync %0, 64;" ::"r"(3 + (warp >> 1)) : "memory");
                    if (hh == 0 && (lane & 7) == 0) {
                        v += *slot;
                        const int64_t r = r0 + i2 + (lane >> 4);
                        if (ready && r < p.N) p.Y[((lane >> 3) & 1) * p.N + r] = v;
                    }
                } else {
                    const int64_t r = r0 + warp;
                    float acc[2] = {0.0f, 0.0f};
                    if (ready && r < p.N && vu) unit_dot_rxn<F, Q81, 2>(stage + static_cast<uint32_t>(warp * p.rowbytes), uu, nb32, x2, acc);
                    const float v = warp_transpose_reduce<1>(acc, lane);  // lane >> 4 = token
                    if (ready && r < p.N && (lane & 15) == 0) p.Y[(lane >> 4) * p.N + r] = v;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
            }
            return;
        }
    }

    if constexpr (KIND == KIND_GEMV) {
        if constexpr (CH) {
            // chunked rows: the warp's row sums its chunks in acc[] and is reduced once per tile
            const int nu = units_per_row(K);
            const int nkc = (nu + p.chunk_units - 1) / p.chunk_units;
            int xr[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) xr[t] = t;
            int j = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
                const int64_t r = static_cast<int64_t>(item) * kTileRows + warp;
                float acc[NT];
#pragma unroll
                for (int i = 0; i < NT; ++i) acc[i] = 0.0f;
                for (int kc = 0; kc < nkc; ++kc, ++j) {
                    const int s = j % p.stages;
                    const uint32_t ph = static_cast<uint32_t>(j / p.stages) & 1u;
                    if (!__all_sync(0xffffffffu, mbar_wait(&full[s], ph))) {  // warp-uniform
                        set_error(p.err, DEV_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    if (r < p.N) {
                        const int u0 = kc * p.chunk_units;
                        const int ue = u0 + p.chunk_units < nu ? u0 + p.chunk_units : nu;
                        // the row's start, as if the whole row were staged: unit u keeps its
                        // offset (the slot starts at the chunk's global address rounded down to 16)
                        const uint32_t lead = static_cast<uint32_t>((r * p.rowbytes + static_cast<int64_t>(kc) * p.chunk_bytes) & 15);
                        const saddr row = ring_s + static_cast<uint32_t>(s * p.stage_stride + warp * p.row_slot) + lead -
                                          static_cast<uint32_t>(kc) * static_cast<uint32_t>(p.chunk_bytes);
                        row_accumulate<F, NT, Q81>(row, xs, xr, p.T, acc, lane, u0, ue);
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                }
                const float v = warp_transpose_reduce<LV>(acc, lane);
                const int t = lane >> SH;
                if (ok && r < p.N && (lane & ((1 << SH) - 1)) == 0 && t < p.T) p.Y[t * p.N + r] = v;
                if (!ok) break;
            }
            return;
        }
    }

    int j = 0;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++j) {
        const int s = j % p.stages;
        const uint32_t ph = static_cast<uint32_t>(j / p.stages) & 1u;
        const bool ready = __all_sync(0xffffffffu, mbar_wait(&full[s], ph));  // warp-uniform
        if (!ready) {
            set_error(p.err, DEV_ERR_TIMEOUT);
            s_flag[1] = 1;
        }
        const saddr stage = ring_s + static_cast<uint32_t>(s * p.stage_stride);

        {
            const int64_t r = static_cast<int64_t>(item) * kTileRows + warp;
            int xr[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) xr[t] = t;
            if (ready && r < p.N) {
                if constexpr (KIND == KIND_GEMV) {
                    float acc[NT];
#pragma unroll
                    for (int i = 0; i < NT; ++i) acc[i] = 0.0f;
                    row_accumulate<F, NT, Q81>(stage + static_cast<uint32_t>(warp * p.rowbytes), xs, xr, p.T, acc, lane);
                    const float v = warp_transpose_reduce<LV>(acc, lane);
                    const int t = lane >> SH;
                    if ((lane & ((1 << SH) - 1)) == 0 && t < p.T) p.Y[t * p.N + r] = v;
                } else {
                    row_coefs<F, NT>(stage + static_cast<uint32_t>(warp * p.rowbytes), xs, p.T, r, p.N, p.coefs, lane);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }
}

template <int KIND, int F, int NT, int AK = 0, bool CH = false>
cudaError_t launch_one(const StreamParams& p, int grid, int smem, cudaStream_t s) {
    // The dynamic shared-memory limit is a per-device function attribute: set it
    // on the first launch of each instantiation on each device (before capture).
    static std::atomic<bool> attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(k_stream<KIND, F, NT, AK, CH>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    return launch_pdl(k_stream<KIND, F, NT, AK, CH>, dim3(grid), dim3(kThreads), smem, s, p);
}

template <int KIND, int F, int AK, bool CH>
cudaError_t launch_nt_ch(int nt, const StreamParams& p, int grid, int smem, cudaStream_t s) {
    switch (nt) {
    case 1: return launch_one<KIND, F, 1, AK, CH>(p, grid, smem, s);
    case 2: return launch_one<KIND, F, 2, AK, CH>(p, grid, smem, s);
    case 4: return launch_one<KIND, F, 4, AK, CH>(p, grid, smem, s);
    default: return launch_one<KIND, F, 8, AK, CH>(p, grid, smem, s);
    }
}

// The GEMV instance for nt tokens and the plan's schedule (row chunks or whole rows).
template <int KIND, int F, int AK = 0>
cudaError_t launch_nt(int nt, const StreamParams& p, int grid, int smem, cudaStream_t s) {
    if constexpr (KIND == KIND_GEMV)
        if (p.chunk_units > 0) return launch_nt_ch<KIND, F, AK, true>(nt, p, grid, smem, s);
    return launch_nt_ch<KIND, F, AK, false>(nt, p, grid, smem, s);
}

}  // namespace ggq

// ggq_stream.cuh -- the weight-streaming kernel behind the decode GEMV, the
// block-dot dump and the decode-size MoE gate/up and down stages.
//
// HBM-bound design for sm_103a:
//   * one CTA per SM (persistent: items blockIdx.x, +gridDim.x, ...);
//   * a producer warp streams each item's weight rows (a contiguous byte range
//     per matrix: rows are stored back to back) into a ring of shared-memory
//     stages with cp.async.bulk, completion counted on an mbarrier in bytes, so
//     several tens of KB per SM are in flight without tying up registers;
//   * eight consumer warps take two rows each per stage; lanes stride over the
//     rows' 32-weight chunks, unpack nibbles / 6-bit scales in registers and
//     run the int8 dp4a integer core against the quantized activations, which
//     were staged once per CTA into shared memory (structure of arrays);
//   * per-lane fp32 partials of (row, token) are summed with one transpose
//     reduction per stage.
// Every wait is bounded; on timeout the kernel records an error word, drains
// its own copies and returns.
#pragma once
#include "ggq_device.cuh"
#include "ggq_internal.h"

namespace ggq {

__device__ __forceinline__ void consumer_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); }

// Stage packed activation blocks (Q8_K: 292 B, or Q8_1: 36 B) from global into
// the structure-of-arrays region.  PERM stores each 32-block's quants in the
// interleaved order (0,16,1,17,...) that the MXFP4 lookup produces.
template <bool Q81, bool PERM>
__device__ void stage_acts(const uint8_t* __restrict__ src, int rows, int K, int8_t* q, float* d, int16_t* bs,
                           int32_t* qs32, int tid, int nthr) {
    if constexpr (!Q81) {
        const int nb = rows * (K >> 8);
        const int words = nb * 73;
        for (int i = tid; i < words; i += nthr) {
            const int b = i / 73, w = i - b * 73;
            const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(src + static_cast<size_t>(b) * 292) + w);
            if (w == 0) {
                d[b] = __uint_as_float(v);
            } else if (w <= 64) {
                int8_t* dq = q + static_cast<size_t>(b) * 256;
                const int e = 4 * (w - 1);
                if constexpr (!PERM) {
                    *reinterpret_cast<uint32_t*>(dq + e) = v;
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        const int el = e + j, r = el & 31;
                        dq[(el & ~31) + 2 * (r & 15) + (r >> 4)] = static_cast<int8_t>((v >> (8 * j)) & 0xFF);
                    }
                }
            } else {
                reinterpret_cast<uint32_t*>(bs + static_cast<size_t>(b) * 16)[w - 65] = v;
            }
        }
    } else {
        const int nb = rows * (K >> 5);
        const int words = nb * 9;
        for (int i = tid; i < words; i += nthr) {
            const int b = i / 9, w = i - b * 9;
            const uint32_t v = __ldg(reinterpret_cast<const uint32_t*>(src + static_cast<size_t>(b) * 36) + w);
            if (w == 0) {
                d[b] = __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xFFFFu)));
            } else {
                reinterpret_cast<uint32_t*>(q + static_cast<size_t>(b) * 32)[w - 1] = v;
                int s = __dp4a(static_cast<int>(v), 0x01010101, 0);
                atomicAdd(&qs32[b], s);
            }
        }
    }
}

template <int F, int NT>
__device__ __forceinline__ void row_accumulate(const uint8_t* row, const XS& xs, const int* xr, int nslots,
                                               float* acc, int lane) {
    const int nc = xs.K >> 5;
    for (int c = lane; c < nc; c += 32) {
        Chunk ch;
        load_chunk<F>(row, c, ch);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if (j < nslots) {
                int A, B;
                chunk_ints<F>(ch, xs, xr[j], c, A, B);
                acc[j] += chunk_value<F>(ch, xs, xr[j], c, A, B);
            }
        }
    }
}

// Integer coefficients of one row for the dump.
template <int F, int NT>
__device__ __forceinline__ void row_coefs(const uint8_t* row, const XS& xs, int nslots, int64_t row_index,
                                          int64_t N, int32_t* out, int lane) {
    const int nc = xs.K >> 5;
    const int ncoef = (xs.K / fmt_qk(F)) * fmt_coefs(F);
    for (int c0 = 0; c0 < nc; c0 += 32) {
        const int c = c0 + lane;
        const bool valid = c < nc;
        Chunk ch;
        if (valid) load_chunk<F>(row, c, ch);
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if (j < nslots) {
                int A = 0, B = 0;
                if (valid) chunk_ints<F>(ch, xs, j, c, A, B);
                int32_t* o = out + (static_cast<int64_t>(j) * N + row_index) * ncoef;
                if constexpr (fmt_qk(F) == 32) {
                    if (valid) o[c] = A;
                } else {
                    // the 8 chunks of a superblock sit on 8 consecutive lanes
#pragma unroll
                    for (int s = 1; s < 8; s <<= 1) {
                        A += __shfl_xor_sync(0xffffffffu, A, s);
                        B += __shfl_xor_sync(0xffffffffu, B, s);
                    }
                    if (valid && (c & 7) == 0) {
                        if constexpr (fmt_coefs(F) == 2) {
                            o[2 * (c >> 3)] = A;
                            o[2 * (c >> 3) + 1] = B;
                        } else {
                            o[c >> 3] = A;
                        }
                    }
                }
            }
        }
    }
}

template <int KIND, int F, int NT>
__global__ void __launch_bounds__(kThreads, 1) k_stream(const StreamParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr bool Q81 = fmt_q81(F);
    constexpr int LV = NT == 1 ? 1 : NT == 2 ? 2 : NT == 4 ? 3 : 4;  // log2(2 * NT)
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    // ---- shared memory layout: ring | activations | barriers | misc
    uint8_t* ring = smem;
    uint8_t* xreg = smem + static_cast<size_t>(p.stages) * p.stage_stride;
    const int K = p.K;
    const size_t qbytes = (static_cast<size_t>(p.xrows) * K + 127) / 128 * 128;
    const size_t dbytes = (static_cast<size_t>(p.xrows) * (K / (Q81 ? 32 : 256)) * 4 + 127) / 128 * 128;
    int8_t* xs_q = reinterpret_cast<int8_t*>(xreg);
    float* xs_d = reinterpret_cast<float*>(xreg + qbytes);
    int16_t* xs_bs = reinterpret_cast<int16_t*>(xreg + qbytes + dbytes);
    int32_t* xs_s32 = reinterpret_cast<int32_t*>(xreg + qbytes + dbytes);
    uint64_t* full = reinterpret_cast<uint64_t*>(xreg + p.x_bytes);
    uint64_t* empty = full + kMaxStages;
    int* s_flag = reinterpret_cast<int*>(empty + kMaxStages);  // [0] last-CTA flag, [1] abort

    // ---- work items
    int nitems;
    int D = 0;
    if constexpr (KIND == KIND_GEMV || KIND == KIND_DUMP) {
        nitems = static_cast<int>((p.N + kTileRows - 1) / kTileRows);
    } else if constexpr (KIND == KIND_GATEUP) {
        D = p.plan->D;
        nitems = D * static_cast<int>(p.N / (kTileRows / 2));
    } else {
        D = p.plan->D;
        nitems = D * static_cast<int>(p.N / kTileRows);
    }

    if (static_cast<int>(blockIdx.x) >= nitems) return;  // whole CTA idle (uniform)

    if (tid == 0) {
        for (int s = 0; s < p.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        s_flag[0] = 0;
        s_flag[1] = 0;
        fence_barrier_init();
    }
    if constexpr (Q81) {
        for (int i = tid; i < p.xrows * (K >> 5); i += kThreads) xs_s32[i] = 0;
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ================= producer
        if (lane == 0) {
            const uint64_t pol = policy_evict_first();
            int j = 0;
            bool ok = true;
            for (int item = blockIdx.x; item < nitems && ok; item += gridDim.x, ++j) {
                const int s = j % p.stages;
                const uint32_t ph = static_cast<uint32_t>(j / p.stages) & 1u;
                if (!mbar_wait(&empty[s], ph ^ 1u)) {
                    set_error(p.err, DEV_ERR_TIMEOUT);
                    ok = false;
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
                } else if constexpr (KIND == KIND_GATEUP) {
                    const int nt = static_cast<int>(p.N / (kTileRows / 2));
                    const int u = item / nt, tile = item - u * nt;
                    const int64_t e = p.plan->expert[u];
                    const int64_t off = (e * p.N + static_cast<int64_t>(tile) * (kTileRows / 2)) * p.rowbytes;
                    src[0] = p.W + off;
                    src[1] = p.W2 + off;
                    bytes[0] = bytes[1] = static_cast<uint32_t>((kTileRows / 2) * p.rowbytes);
                    ncopy = 2;
                } else {
                    const int u = item % D, tile = item / D;
                    const int64_t e = p.plan->expert[u];
                    src[0] = p.W + (e * p.N + static_cast<int64_t>(tile) * kTileRows) * p.rowbytes;
                    bytes[0] = static_cast<uint32_t>(kTileRows * p.rowbytes);
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

    // ================= consumers (256 threads)
    const int ctid = tid;
    stage_acts<Q81, F == F_MXFP4>(p.xq, p.xrows, K, xs_q, xs_d, xs_bs, xs_s32, ctid, kConsumerWarps * 32);
    consumer_sync();
    XS xs;
    xs.q = xs_q;
    xs.d = xs_d;
    xs.bs = xs_bs;
    xs.qs32 = xs_s32;
    xs.K = K;

    int j = 0;
    for (int item = blockIdx.x; item < nitems; item += gridDim.x, ++j) {
        const int s = j % p.stages;
        const uint32_t ph = static_cast<uint32_t>(j / p.stages) & 1u;
        const bool ready = __all_sync(0xffffffffu, mbar_wait(&full[s], ph));  // warp-uniform
        if (!ready) {
            set_error(p.err, DEV_ERR_TIMEOUT);
            s_flag[1] = 1;
        }
        const uint8_t* stage = ring + static_cast<size_t>(s) * p.stage_stride;

        if constexpr (KIND == KIND_GEMV || KIND == KIND_DUMP) {
            const int64_t r0 = static_cast<int64_t>(item) * kTileRows;
            int xr[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) xr[t] = t;
            if (ready) {
                if constexpr (KIND == KIND_GEMV) {
                    float acc[2 * NT];
#pragma unroll
                    for (int i = 0; i < 2 * NT; ++i) acc[i] = 0.0f;
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        const int64_t r = r0 + 2 * warp + g;
                        if (r < p.N)
                            row_accumulate<F, NT>(stage + (2 * warp + g) * p.rowbytes, xs, xr, p.T, acc + g * NT,
                                                  lane);
                    }
                    const float v = warp_transpose_reduce<LV>(acc, lane);
                    const int idx = lane >> (5 - LV);  // = g * NT + t
                    const int g = idx / NT, t = idx - g * NT;
                    const int64_t r = r0 + 2 * warp + g;
                    if ((lane & ((1 << (5 - LV)) - 1)) == 0 && t < p.T && r < p.N) p.Y[t * p.N + r] = v;
                } else {
#pragma unroll
                    for (int g = 0; g < 2; ++g) {
                        const int64_t r = r0 + 2 * warp + g;
                        if (r < p.N)
                            row_coefs<F, NT>(stage + (2 * warp + g) * p.rowbytes, xs, p.T, r, p.N, p.coefs, lane);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        } else if constexpr (KIND == KIND_GATEUP) {
            const int nt = static_cast<int>(p.N / (kTileRows / 2));
            const int u = item / nt, tile = item - u * nt;
            const int np = p.plan->npairs[u];
            int xr[NT], pr[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                xr[t] = t < np ? p.plan->token[u][t] : 0;
                pr[t] = t < np ? p.plan->pair[u][t] : 0;
            }
            const int64_t row = static_cast<int64_t>(tile) * (kTileRows / 2) + warp;
            if (ready) {
                float acc[2 * NT];
#pragma unroll
                for (int i = 0; i < 2 * NT; ++i) acc[i] = 0.0f;
                row_accumulate<F, NT>(stage + warp * p.rowbytes, xs, xr, np, acc, lane);                       // gate
                row_accumulate<F, NT>(stage + (kTileRows / 2 + warp) * p.rowbytes, xs, xr, np, acc + NT, lane);  // up
                const float v = warp_transpose_reduce<LV>(acc, lane);
                const int sh = 5 - LV;
                const float uval = __shfl_down_sync(0xffffffffu, v, NT << sh);
                const int idx = lane >> sh;
                if ((lane & ((1 << sh) - 1)) == 0 && idx < NT && idx < np) {
                    const float gval = v;
                    const float hval = __fmul_rn(__fdiv_rn(gval, 1.0f + expf(-gval)), uval);
                    const int64_t o = static_cast<int64_t>(pr[idx]) * p.N + row;
                    p.h[o] = hval;
                    if (p.g_dump) p.g_dump[o] = gval;
                    if (p.u_dump) p.u_dump[o] = uval;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            // last CTA to finish a 256-row block of this expert quantizes h there
            __threadfence();
            consumer_sync();
            const int nblk = static_cast<int>(p.N >> 8);
            const int blk = static_cast<int>((static_cast<int64_t>(tile) * (kTileRows / 2)) >> 8);
            if (ctid == 0) {
                const int old = atomicAdd(&p.counters[u * nblk + blk], 1);
                s_flag[0] = (old == 256 / (kTileRows / 2) - 1);
            }
            consumer_sync();
            if (s_flag[0]) {
                __threadfence();
                for (int q = warp; q < np; q += kConsumerWarps) {
                    const int pp = p.plan->pair[u][q];
                    warp_quant_q8k(p.h + static_cast<int64_t>(pp) * p.N + 256 * blk,
                                   p.hq + (static_cast<int64_t>(pp) * nblk + blk) * 292, lane);
                }
                if (ctid == 0) p.counters[u * nblk + blk] = 0;
            }
            if (s_flag[1]) break;
        } else {  // KIND_DOWN
            const int u = item % D, tile = item / D;
            const int np = p.plan->npairs[u];
            int xr[NT];
#pragma unroll
            for (int t = 0; t < NT; ++t) xr[t] = t < np ? p.plan->pair[u][t] : 0;
            if (ready) {
                float acc[2 * NT];
#pragma unroll
                for (int i = 0; i < 2 * NT; ++i) acc[i] = 0.0f;
#pragma unroll
                for (int g = 0; g < 2; ++g)
                    row_accumulate<F, NT>(stage + (2 * warp + g) * p.rowbytes, xs, xr, np, acc + g * NT, lane);
                const float v = warp_transpose_reduce<LV>(acc, lane);
                const int sh = 5 - LV;
                const int idx = lane >> sh;
                const int g = idx / NT, t = idx - g * NT;
                if ((lane & ((1 << sh) - 1)) == 0 && t < np) {
                    const int64_t r = static_cast<int64_t>(tile) * kTileRows + 2 * warp + g;
                    p.o[static_cast<int64_t>(xr[t]) * p.N + r] = v;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            // last of the D experts of this row tile combines y = sum_j w_j o_j
            __threadfence();
            consumer_sync();
            if (ctid == 0) {
                const int old = atomicAdd(&p.counters[tile], 1);
                s_flag[0] = (old == D - 1);
            }
            consumer_sync();
            if (s_flag[0]) {
                __threadfence();
                for (int i = ctid; i < kTileRows * p.T; i += kConsumerWarps * 32) {
                    const int t = i / kTileRows;
                    const int64_t r = static_cast<int64_t>(tile) * kTileRows + (i - t * kTileRows);
                    float acc = 0.0f;
                    for (int q = 0; q < p.top_k; ++q) {
                        const int pp = t * p.top_k + q;
                        acc += p.plan->wt[pp] * __ldcg(&p.o[static_cast<int64_t>(pp) * p.N + r]);
                    }
                    p.Y[static_cast<int64_t>(t) * p.N + r] = acc;
                }
                if (ctid == 0) p.counters[tile] = 0;
            }
            if (s_flag[1]) break;
        }
    }
}

template <int KIND, int F, int NT>
cudaError_t launch_one(const StreamParams& p, int grid, int smem, cudaStream_t s) {
    // The dynamic shared-memory limit is a per-device function attribute: set it
    // on the first launch of each instantiation on each device (before capture).
    static bool attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        e = cudaFuncSetAttribute(k_stream<KIND, F, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    k_stream<KIND, F, NT><<<grid, kThreads, smem, s>>>(p);
    return cudaGetLastError();
}

template <int KIND, int F>
cudaError_t launch_nt(int nt, const StreamParams& p, int grid, int smem, cudaStream_t s) {
    switch (nt) {
    case 1: return launch_one<KIND, F, 1>(p, grid, smem, s);
    case 2: return launch_one<KIND, F, 2>(p, grid, smem, s);
    case 4: return launch_one<KIND, F, 4>(p, grid, smem, s);
    default: return launch_one<KIND, F, 8>(p, grid, smem, s);
    }
}

}  // namespace ggq

// ggq_misc.cu -- activation quantizer, dequantizer and the decode-size MoE
// router / planner.
//
// Quantizer: the fixed IEEE fp32 sequence d = amax/127, q = round-half-away(x *
// (1/d)) clamped to +-127 (Q8_1 and Q8_K activation blocks; vllm.cpp PR #523
// "grouped + non-grouped keep-quant expert GEMM", What changed: activation
// quantizers).  Dequantizer: the GGUF element formulas (FreeToken PR #136
// "enable native GGUF kernels on ROCm", Summary: Q4_0 dequantization).
// Router: softmax top-k with renormalisation; ids are chosen by logit, ties to
// the lower expert index.  Also the expert-sorted route's grouping kernels.
#include "ggq_device.cuh"
#include "ggq_internal.h"

namespace ggq {

// ---------------------------------------------------------------- quantize

__global__ void k_quant_q8k(const float* __restrict__ x, int64_t nblocks, uint8_t* __restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= nblocks) return;
    warp_quant_q8k(x + b * 256, out + b * 292, lane);
}

__global__ void k_quant_q8_1(const float* __restrict__ x, int64_t nblocks, uint8_t* __restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= nblocks) return;
    warp_quant_q8_1(x + b * 32, out + b * 36, lane);
}

__global__ void k_quant_q8_0(const float* __restrict__ x, int64_t nblocks, uint8_t* __restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= nblocks) return;
    warp_quant_q8_0(x + b * 32, out + b * 34, lane);
}

cudaError_t launch_quantize(int act, const float* x, int64_t T, int64_t K, uint8_t* out, cudaStream_t s) {
    const int64_t nb = T * K / (act == 1 ? 256 : 32);  // act: 0 = Q8_1, 1 = Q8_K, 2 = Q8_0
    if (nb == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (nb * 32 + threads - 1) / threads;
    if (act == 0)
        return launch_pdl(k_quant_q8_1, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s, x, nb, out);
    if (act == 2)
        return launch_pdl(k_quant_q8_0, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s, x, nb, out);
    return launch_pdl(k_quant_q8k, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0, s, x, nb, out);
}

// ---------------------------------------------------------------- dequantize

__device__ __forceinline__ float half_at(const uint8_t* p) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(p[0] | (p[1] << 8))));
}

// One thread per weight block; element formulas of each GGUF format.
template <int F>
__global__ void k_dequant(const uint8_t* __restrict__ blocks, int64_t nblocks, float* __restrict__ out) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= nblocks) return;
    const uint8_t* b = blocks + i * fmt_bytes(F);
    float* y = out + i * fmt_qk(F);
    if constexpr (F == F_Q4_0) {
        const float d = half_at(b);
        for (int j = 0; j < 16; ++j) {
            y[j] = d * static_cast<float>((b[2 + j] & 15) - 8);
            y[j + 16] = d * static_cast<float>((b[2 + j] >> 4) - 8);
        }
    } else if constexpr (F == F_Q8_0) {
        const float d = half_at(b);
        for (int j = 0; j < 32; ++j) y[j] = d * static_cast<float>(static_cast<int8_t>(b[2 + j]));
    } else if constexpr (F == F_MXFP4) {
        const float sc = e8m0_half_scale(b[0]);
        const int tab[16] = {0, 1, 2, 3, 4, 6, 8, 12, 0, -1, -2, -3, -4, -6, -8, -12};
        for (int j = 0; j < 16; ++j) {
            y[j] = sc * static_cast<float>(tab[b[1 + j] & 15]);
            y[j + 16] = sc * static_cast<float>(tab[b[1 + j] >> 4]);
        }
    } else if constexpr (F == F_Q4_K || F == F_Q5_K) {
        const float d = half_at(b), dmin = half_at(b + 2);
        const uint8_t* sc = b + 4;
        const uint8_t* qh = b + 16;
        const uint8_t* qs = b + (F == F_Q4_K ? 16 : 48);
        for (int s = 0; s < 8; ++s) {
            int scv, mv;
            if (s < 4) {
                scv = sc[s] & 63;
                mv = sc[s + 4] & 63;
            } else {
                scv = (sc[s + 4] & 15) | ((sc[s - 4] >> 6) << 4);
                mv = (sc[s + 4] >> 4) | ((sc[s] >> 6) << 4);
            }
            const float a = d * static_cast<float>(scv), m = dmin * static_cast<float>(mv);
            for (int l = 0; l < 32; ++l) {
                const uint8_t byte = qs[32 * (s >> 1) + l];
                int q = (s & 1) ? (byte >> 4) : (byte & 15);
                if constexpr (F == F_Q5_K) q += 16 * ((qh[l] >> s) & 1);
                y[32 * s + l] = a * static_cast<float>(q) - m;
            }
        }
    } else if constexpr (F == F_Q2_K || F == F_Q3_K) {
        // element 128n + 32j + l: bits 2j, 2j+1 of qs[32n + l]; Q3_K: bit 4n + j of hmask[l]
        // clear subtracts 4; Q2_K scale/min nibbles per 16, Q3_K packed 6-bit scales - 32
        const float d = half_at(b + (F == F_Q2_K ? 80 : 108));
        for (int e = 0; e < 256; ++e) {
            const int n = e >> 7, j = (e >> 5) & 3, l = e & 31, g = e >> 4;
            int q = (b[(F == F_Q2_K ? 16 : 32) + 32 * n + l] >> (2 * j)) & 3;
            if constexpr (F == F_Q2_K) {
                y[e] = d * static_cast<float>(b[g] & 15) * static_cast<float>(q) - half_at(b + 82) * static_cast<float>(b[g] >> 4);
            } else {
                if (!((b[l] >> (4 * n + j)) & 1)) q -= 4;
                const int lo = g < 8 ? (b[96 + g] & 15) : (b[96 + g - 8] >> 4);
                const int hi = (b[104 + (g & 3)] >> (2 * (g >> 2))) & 3;
                y[e] = d * static_cast<float>((lo | (hi << 4)) - 32) * static_cast<float>(q);
            }
        }
    } else {  // Q6_K
        const float d = half_at(b + 208);
        for (int e = 0; e < 256; ++e) {
            const int h = e >> 7, g = (e >> 5) & 3, l = e & 31;
            const uint8_t lo = b[64 * h + 32 * (g & 1) + l];
            const int nib = (g < 2) ? (lo & 15) : (lo >> 4);
            const int hi = (b[128 + 32 * h + l] >> (2 * g)) & 3;
            y[e] = d * static_cast<float>(static_cast<int8_t>(b[192 + (e >> 4)])) * static_cast<float>((nib | (hi << 4)) - 32);
        }
    }
}

cudaError_t launch_dequant(int fmt, const uint8_t* blocks, int64_t rows, int64_t K, float* out, cudaStream_t s) {
    const int64_t nb = rows * (K / fmt_qk(fmt));
    if (nb == 0) return cudaSuccess;
    const unsigned grid = static_cast<unsigned>((nb + 127) / 128);
    switch (fmt) {
    case F_Q4_0: return launch_pdl(k_dequant<F_Q4_0>, dim3(grid), dim3(128), 0, s, blocks, nb, out);
    case F_Q8_0: return launch_pdl(k_dequant<F_Q8_0>, dim3(grid), dim3(128), 0, s, blocks, nb, out);
    case F_Q4_K: return launch_pdl(k_dequant<F_Q4_K>, dim3(grid), dim3(128), 0, s, blocks, nb, out);
    case F_Q5_K: return launch_pdl(k_dequant<F_Q5_K>, dim3(grid), dim3(128), 0, s, blocks, nb, out);
    case F_Q6_K: return launch_pdl(k_dequant<F_Q6_K>, dim3(grid), dim3(128), 0, s, blocks, nb, out);
    case F_Q2_K: return launch_pdl(k_dequant<F_Q2_K>, dim3(grid), dim3(128), 0, s, blocks, nb, out);
    case F_Q3_K: return launch_pdl(k_dequant<F_Q3_K>, dim3(grid), dim3(128), 0, s, blocks, nb, out);
    default: return launch_pdl(k_dequant<F_MXFP4>, dim3(grid), dim3(128), 0, s, blocks, nb, out);
    }
    return cudaGetLastError();
}

}  // namespace ggq

// ---------------------------------------------------------------- expert-sorted route (5 tokens and up)

namespace ggq {

// Q8_K rows written pitch bytes apart (the grouped kernel copies whole rows
// with 16-byte bulk copies, so its activation rows start on 16-byte marks).
__global__ void k_quant_q8k_pitched(const float* __restrict__ x, int64_t rows, int nbr, uint8_t* __restrict__ out,
                                    int64_t pitch) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= rows * nbr) return;
    const int64_t r = b / nbr, c = b - r * nbr;
    warp_quant_q8k(x + b * 256, out + r * pitch + c * 292, lane);
}

cudaError_t launch_quantize_pitched(const float* x, int64_t rows, int64_t K, uint8_t* out, int64_t pitch,
                                    cudaStream_t s) {
    const int64_t nb = rows * (K / 256);
    if (nb == 0) return cudaSuccess;
    return launch_pdl(k_quant_q8k_pitched, dim3(static_cast<unsigned>((nb * 32 + 255) / 256)), dim3(256), 0, s, x, rows,
                      static_cast<int>(K / 256), out, pitch);
}

// h = silu(g) * u (the SwiGLU of the gate/up outputs, same rounding steps as the
// grouped kernels' epilogues), then Q8_K: one warp per 256-block of a row.
__global__ void k_quant_silu_q8k(const float* __restrict__ g, const float* __restrict__ u, int64_t rows, int nbr,
                                 uint8_t* __restrict__ out, int64_t pitch, float* __restrict__ h_out) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= rows * nbr) return;
    const int64_t r = b / nbr, c = b - r * nbr;
    const float4* gp = reinterpret_cast<const float4*>(g + b * 256) + 2 * lane;
    const float4* up = reinterpret_cast<const float4*>(u + b * 256) + 2 * lane;
    const float4 g0 = __ldcg(gp), g1 = __ldcg(gp + 1), u0 = __ldcg(up), u1 = __ldcg(up + 1);
    const float gv[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    const float uv[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
    float x[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) x[i] = __fmul_rn(__fdiv_rn(gv[i], 1.0f + expf(-gv[i])), uv[i]);
    if (h_out) {
        float4* hp = reinterpret_cast<float4*>(h_out + b * 256) + 2 * lane;
        hp[0] = make_float4(x[0], x[1], x[2], x[3]);
        hp[1] = make_float4(x[4], x[5], x[6], x[7]);
    }
    warp_quant_q8k_regs(x, out + r * pitch + c * 292, lane);
}

cudaError_t launch_quantize_silu(const float* g, const float* u, int64_t rows, int64_t K, uint8_t* out, int64_t pitch,
                                 float* h_out, cudaStream_t s) {
    const int64_t nb = rows * (K / 256);
    if (nb == 0) return cudaSuccess;
    return launch_pdl(k_quant_silu_q8k, dim3(static_cast<unsigned>((nb * 32 + 255) / 256)), dim3(256), 0, s, g, u,
                      rows, static_cast<int>(K / 256), out, pitch, h_out);
}

// Q8_K rows (pitched) -> the operands of the f16 grouped GEMM: the quants as
// f16 (exact), the 16-element group sums as f16 (|sum| <= 2032: exact) and the
// block scales as f32.  Output row r takes input row map[r] / div (the
// expert-sorted order of the (token, expert) pairs), or row r without a map.
// BF16: the quants as bf16 instead (the MXFP4 operands; exact too).  One warp
// per block.
template <bool BF16>
__global__ void k_q8k_to_f16(const uint8_t* __restrict__ q, int64_t pitch, const int* __restrict__ map, int div,
                             int64_t rows, int nbr, __half* __restrict__ x16, __half* __restrict__ bs16,
                             float* __restrict__ dx, int64_t dx_pitch) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t b = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
    if (b >= rows * nbr) return;
    const int64_t r = b / nbr, c = b - r * nbr;
    const int64_t src = map ? static_cast<int64_t>(__ldg(map + r) / div) : r;
    const uint8_t* blk = q + src * pitch + c * 292;
    const uint32_t* qw = reinterpret_cast<const uint32_t*>(blk + 4);
    uint32_t out[4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        if constexpr (BF16) {
            // an int8 value is exact in bf16: the top half of its f32 bits
            const uint32_t w = __ldcg(qw + 2 * lane + i);
            uint32_t h[4];
#pragma unroll
            for (int k = 0; k < 4; ++k)
                h[k] = __float_as_uint(static_cast<float>(static_cast<int8_t>((w >> (8 * k)) & 0xFFu))) >> 16;
            out[2 * i] = h[0] | (h[1] << 16);
            out[2 * i + 1] = h[2] | (h[3] << 16);
        } else {
            const uint32_t u = __ldcg(qw + 2 * lane + i) ^ 0x80808080u;  // x + 128 in each byte
            const uint32_t a = prmt(u, 0u, 0x4140u) | 0x64006400u, bb = prmt(u, 0u, 0x4342u) | 0x64006400u;
            const __half2 off = __halves2half2(__ushort_as_half(0x6480u), __ushort_as_half(0x6480u));  // 1152
            const __half2 ha = __hsub2(*reinterpret_cast<const __half2*>(&a), off);
            const __half2 hb = __hsub2(*reinterpret_cast<const __half2*>(&bb), off);
            out[2 * i] = *reinterpret_cast<const uint32_t*>(&ha);
            out[2 * i + 1] = *reinterpret_cast<const uint32_t*>(&hb);
        }
    }
    const int64_t K = static_cast<int64_t>(nbr) * 256;
    *reinterpret_cast<uint4*>(x16 + r * K + c * 256 + 8 * lane) = make_uint4(out[0], out[1], out[2], out[3]);
    if (lane < 16) {
        const int v = static_cast<int>(reinterpret_cast<const int16_t*>(blk + 260)[lane]);
        bs16[r * (K / 16) + c * 16 + lane] = __int2half_rn(v);
    }
    if (lane == 0) dx[r * dx_pitch + c] = __ldcg(reinterpret_cast<const float*>(blk));
}

cudaError_t launch_q8k_to_f16(const uint8_t* q, int64_t pitch, const int* map, int div, int64_t rows, int64_t K,
                              __half* x16, __half* bs16, float* dx, int64_t dx_pitch, cudaStream_t s, bool bf16) {
    const int64_t nb = rows * (K / 256);
    if (nb == 0) return cudaSuccess;
    const dim3 grid(static_cast<unsigned>((nb * 32 + 255) / 256));
    if (bf16)
        return launch_pdl(k_q8k_to_f16<true>, grid, dim3(256), 0, s, q, pitch, map, div, rows,
                          static_cast<int>(K / 256), x16, bs16, dx, dx_pitch);
    return launch_pdl(k_q8k_to_f16<false>, grid, dim3(256), 0, s, q, pitch, map, div, rows, static_cast<int>(K / 256),
                      x16, bs16, dx, dx_pitch);
}

// One warp per token: top-k by logit (ties to the lower index) and the
// renormalised softmax weights over the selected experts; or copy given ids.
// Every pair's expert is counted into counts[] (zeroed by the caller).  The
// remaining warps quantize x to Q8_K rows x_pitch bytes apart.
__global__ void __launch_bounds__(256) k_route_sorted(const float* __restrict__ logits,
                                                      const int32_t* __restrict__ ids_in,
                                                      const float* __restrict__ w_in, const float* __restrict__ X,
                                                      int T, int E, int k, int H, uint8_t* __restrict__ xq,
                                                      int64_t x_pitch, int32_t* ids, float* w, int* counts, int* err) {
    pdl_launch_dependents();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nw = (gridDim.x * blockDim.x) >> 5;
    const int nbr = H >> 8;
    // quantize: all warps, one 256-block each (X null: x^ was given)
    for (int b = gw; X && b < T * nbr; b += nw) {
        const int r = b / nbr, c = b - r * nbr;
        warp_quant_q8k(X + static_cast<int64_t>(b) * 256, xq + r * x_pitch + c * 292, lane);
    }
    for (int t = gw; t < T; t += nw) {
        if (logits) {
            const float* l = logits + static_cast<int64_t>(t) * E;
            uint32_t taken[4] = {0u, 0u, 0u, 0u};
            float lmax = 0.0f, wsum = 0.0f;
            float wj[8];
            int idj[8];
            for (int j = 0; j < k; ++j) {
                float bv = -INFINITY;
                int bi = 0x7fffffff;
                for (int i = 0, e = lane; e < E; ++i, e += 32) {
                    if ((taken[i >> 5] >> (i & 31)) & 1u) continue;
                    const float v = l[e];
                    if (v > bv || (v == bv && e < bi)) {
                        bv = v;
                        bi = e;
                    }
                }
#pragma unroll
                for (int sft = 16; sft >= 1; sft >>= 1) {
                    const float ov = __shfl_xor_sync(0xffffffffu, bv, sft);
                    const int oi = __shfl_xor_sync(0xffffffffu, bi, sft);
                    if (ov > bv || (ov == bv && oi < bi)) {
                        bv = ov;
                        bi = oi;
                    }
                }
                if ((bi & 31) == lane) {
                    const int i = bi >> 5;
                    taken[i >> 5] |= 1u << (i & 31);
                }
                if (j == 0) lmax = bv;
                idj[j] = bi;
                wj[j] = expf(bv - lmax);
                wsum += wj[j];
            }
            if (lane < k) {
                int id = 0;
                float wv = 0.0f;
                for (int j = 0; j < k; ++j)
                    if (j == lane) {
                        id = idj[j];
                        wv = wj[j];
                    }
                ids[t * k + lane] = id;
                w[t * k + lane] = wv / wsum;
                atomicAdd(&counts[id], 1);
            }
        } else if (lane < k) {
            const int id = ids_in[t * k + lane];
            ids[t * k + lane] = id;
            w[t * k + lane] = w_in[t * k + lane];
            if (id >= 0 && id < E)
                atomicAdd(&counts[id], 1);
            else
                set_error(err, DEV_ERR_BAD_IDS);
        }
    }
}

cudaError_t launch_route_sorted(const float* logits, const int32_t* ids_in, const float* w_in, const float* X, int T,
                                int E, int k, int H, uint8_t* xq, int64_t x_pitch, int32_t* ids, float* w,
                                int* counts, int* err, cudaStream_t s) {
    const int warps = T > T * (H >> 8) ? T : T * (H >> 8);
    const int grid = (warps + 7) / 8 < 1184 ? (warps + 7) / 8 : 1184;
    return launch_pdl(k_route_sorted, dim3(grid > 0 ? grid : 1), dim3(256), 0, s, logits, ids_in, w_in, X, T, E, k, H,
                      xq, x_pitch, ids, w, counts, err);
}

// One CTA: exclusive scan of the expert counts, the list of non-empty experts
// (the groups of the grouped kernel) and zeroed scatter cursors.
__global__ void __launch_bounds__(1024) k_group_plan(const int* __restrict__ counts, int E, int* offsets, int* cursor,
                                                     int* ngroups, int* group_expert, int* group_off, int* group_cnt,
                                                     unsigned long long* tel_pairs, unsigned long long* tel_calls) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int s_sum[1024];
    __shared__ int s_ne[1024];
    const int tid = threadIdx.x;
    const int per = (E + 1023) / 1024;  // experts per thread (E <= 4096)
    int loc = 0, ne = 0;
    for (int i = 0; i < per; ++i) {
        const int e = tid * per + i;
        if (e < E) {
            loc += counts[e];
            ne += counts[e] > 0;
        }
    }
    s_sum[tid] = loc;
    s_ne[tid] = ne;
    __syncthreads();
    for (int d = 1; d < 1024; d <<= 1) {  // inclusive Hillis-Steele scan
        const int a = tid >= d ? s_sum[tid - d] : 0, b = tid >= d ? s_ne[tid - d] : 0;
        __syncthreads();
        s_sum[tid] += a;
        s_ne[tid] += b;
        __syncthreads();
    }
    int run = s_sum[tid] - loc, grun = s_ne[tid] - ne;
    for (int i = 0; i < per; ++i) {
        const int e = tid * per + i;
        if (e < E) {
            const int c = counts[e];
            offsets[e] = run;
            cursor[e] = 0;
            if (c > 0) {
                group_expert[grun] = e;
                group_off[grun] = run;
                group_cnt[grun] = c;
                ++grun;
                if (tel_pairs) atomicAdd(tel_pairs + e, static_cast<unsigned long long>(c));
            }
            run += c;
        }
    }
    if (tid == 1023) {
        offsets[E] = s_sum[1023];
        *ngroups = s_ne[1023];
        if (tel_calls) {  // expert-load telemetry: one call, its distinct experts
            atomicAdd(tel_calls, 1ull);
            atomicAdd(tel_calls + 1, static_cast<unsigned long long>(s_ne[1023]));
        }
    }
}

// Expert-load telemetry of a call that ran as several direct-route launches:
// from the routed ids of all its pairs, the pairs per expert and one call with
// its distinct experts (ids outside [0, E) are skipped: the launches report them).
__global__ void __launch_bounds__(256) k_moe_count(const int32_t* __restrict__ ids, int P, int E,
                                                   unsigned long long* tel_pairs, unsigned long long* tel_calls) {
    pdl_launch_dependents();
    pdl_wait();
    __shared__ int cnt[4096];
    __shared__ int distinct;
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) cnt[e] = 0;
    if (tid == 0) distinct = 0;
    __syncthreads();
    for (int q = tid; q < P; q += blockDim.x) {
        const int e = ids[q];
        if (e >= 0 && e < E) atomicAdd(&cnt[e], 1);
    }
    __syncthreads();
    int nd = 0;
    for (int e = tid; e < E; e += blockDim.x)
        if (cnt[e] > 0) {
            atomicAdd(tel_pairs + e, static_cast<unsigned long long>(cnt[e]));
            ++nd;
        }
    atomicAdd(&distinct, nd);
    __syncthreads();
    if (tid == 0) {
        atomicAdd(tel_calls, 1ull);
        atomicAdd(tel_calls + 1, static_cast<unsigned long long>(distinct));
    }
}

cudaError_t launch_moe_count(const int32_t* ids, int P, int E, unsigned long long* tel_pairs,
                             unsigned long long* tel_calls, cudaStream_t s) {
    return launch_pdl(k_moe_count, dim3(1), dim3(256), 0, s, ids, P, E, tel_pairs, tel_calls);
}

cudaError_t launch_group_plan(const int* counts, int E, int* offsets, int* cursor, int* ngroups, int* group_expert,
                              int* group_off, int* group_cnt, cudaStream_t s, unsigned long long* tel_pairs,
                              unsigned long long* tel_calls) {
    return launch_pdl(k_group_plan, dim3(1), dim3(1024), 0, s, counts, E, offsets, cursor, ngroups, group_expert,
                      group_off, group_cnt, tel_pairs, tel_calls);
}

// Scatter pair p to its expert's range.  The order inside a range does not
// matter: every column of the grouped kernel is computed on its own.
__global__ void k_scatter(const int32_t* __restrict__ ids, int P, int E, const int* __restrict__ offsets, int* cursor,
                          int* perm) {
    pdl_launch_dependents();
    pdl_wait();
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    const int e = ids[p];
    if (e < 0 || e >= E) return;  // reported by the route kernel
    perm[offsets[e] + atomicAdd(&cursor[e], 1)] = p;
}

cudaError_t launch_scatter(const int32_t* ids, int P, int E, const int* offsets, int* cursor, int* perm,
                           cudaStream_t s) {
    if (P == 0) return cudaSuccess;
    return launch_pdl(k_scatter, dim3((P + 255) / 256), dim3(256), 0, s, ids, P, E, offsets, cursor, perm);
}

// y[t][n] = sum_j w[t][j] * o[t*k + j][n], slots in order.
__global__ void k_combine(const float* __restrict__ o, const float* __restrict__ w, int T, int k, int64_t H,
                          float* __restrict__ Y) {
    pdl_launch_dependents();
    pdl_wait();
    const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (i >= T * H) return;
    const int64_t t = i / H, n = i - t * H;
    float acc = 0.0f;
    for (int j = 0; j < k; ++j) acc += w[t * k + j] * o[(t * k + j) * H + n];
    Y[i] = acc;
}

cudaError_t launch_combine(const float* o, const float* w, int T, int k, int64_t H, float* Y, cudaStream_t s) {
    const int64_t n = T * H;
    if (n == 0) return cudaSuccess;
    return launch_pdl(k_combine, dim3(static_cast<unsigned>((n + 255) / 256)), dim3(256), 0, s, o, w, T, k, H, Y);
}

}  // namespace ggq

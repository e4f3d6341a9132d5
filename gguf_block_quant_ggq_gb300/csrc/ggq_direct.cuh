// ggq_direct.cuh -- the direct tiny-batch MoE route (1 to 4 tokens): two
// kernels per layer, with no cross-CTA counters, fences or extra launches.
//
// ds4 PR #656 "Add ROCm MXFP4 routed expert kernels" (Summary): 2-4 token
// batches go through direct kernels instead of partially filled expert-sorted
// tiles, and gate/up, SwiGLU and down stay register-resident.  Here:
//   gate/up kernel: every CTA routes the tokens itself (top-k of softmax by
//     logit, ties to the lower index), groups the <= 32 (token, slot) pairs by
//     distinct expert with one warp match, and quantizes x to Q8_K straight
//     into shared memory.  Each consumer warp owns one gate row and the same
//     up row of a 16-row tile, so h = silu(g) * u is formed in the warp and
//     written once to global memory (fp32).
//   down kernel: routes again from the same inputs (so its weight stream can
//     start while gate/up finishes), quantizes h to Q8_K into shared memory
//     (bit-exactly the same quantizer), and for each 16-row tile of the output
//     streams that tile of every selected expert, G experts per stage.  A
//     warp's row of the G experts is one concatenated row spread over all 32
//     lanes; each lane adds w_j * (its partial of pair j) straight into the
//     sum of pair j's token, and one reduction per tile gives y, so the
//     result is deterministic.  With a per-pair dump requested, the down
//     kernel instead takes one expert per stage and reduces every pair
//     (o_j) before combining.
// Both kernels stream weights with the producer warp / mbarrier ring of the
// streaming kernel and use its dp4a consumer (row_accumulate).
#pragma once
#include <atomic>
#include <type_traits>
#include "ggq_stream.cuh"

namespace ggq {

constexpr int kDirectMaxPairs = 32;  // 4 tokens x top-8
constexpr int kDownUnits = 8;        // fused down: 64-weight units per lane per stage (G * K/64 <= 256)

struct DirectPlan {
    int D;                                        // distinct experts
    int expert[kDirectMaxPairs];                  // expert of distinct slot u
    int npairs[kDirectMaxPairs];                  // pairs on it
    int pair[kDirectMaxPairs][4];                 // pair indices p = t*k + j (one per token)
    float wt[kDirectMaxPairs];                    // routing weight of pair p
    int ids[kDirectMaxPairs];                     // expert of pair p
    int bad;                                      // a routed id was out of range
    int tok[kDirectMaxPairs];                     // token of pair p (p / top_k)
};

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int n) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(n) : "memory");
}

// Group the P <= 32 pairs (expert ids in s->ids) by distinct expert, in order
// of first appearance.  One warp.
__device__ __forceinline__ void direct_group(DirectPlan* s, int P, int E, int lane) {
    const bool active = lane < P;
    const int e = active ? s->ids[lane] : -1 - lane;
    const unsigned act = __ballot_sync(0xffffffffu, active);
    const unsigned same = __match_any_sync(0xffffffffu, e) & act;
    const unsigned lt = (1u << lane) - 1u;
    const bool leader = active && (same & lt) == 0u;
    const unsigned leaders = __ballot_sync(0xffffffffu, leader);
    const int lead = active ? __ffs(same) - 1 : 0;
    const int u = __popc(leaders & ((1u << lead) - 1u));
    const int slot = __popc(same & lt);
    const bool bad = active && (e < 0 || e >= E || slot >= 4);
    const unsigned anybad = __ballot_sync(0xffffffffu, bad);
    if (active && !anybad) {
        s->pair[u][slot] = lane;
        if (leader) {
            s->expert[u] = e;
            s->npairs[u] = __popc(same);
        }
    }
    if (lane == 0) {
        s->D = anybad ? 0 : __popc(leaders);
        s->bad = anybad != 0u;
    }
}

// Routing of token t by one warp: top-k by logit (ties to the lower expert
// index) and the softmax weights renormalised over the selected experts.
__device__ __forceinline__ void direct_route_token(const float* __restrict__ l, int E, int k, int* ids, float* w,
                                                   int lane) {
    uint32_t taken[4] = {0u, 0u, 0u, 0u};
    float lmax = 0.0f, wsum = 0.0f, myw = 0.0f;
    int myid = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = 0x7fffffff;
        for (int i = 0, e = lane; e < E; ++i, e += 32) {
            if ((taken[i >> 5] >> (i & 31)) & 1u) continue;
            const float v = __ldcg(l + e);
            if (v > bv || (v == bv && e < bi)) {
                bv = v;
                bi = e;
            }
        }
#pragma unroll
        for (int s = 16; s >= 1; s >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, s);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, s);
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
        const float p = expf(bv - lmax);
        wsum += p;
        if (lane == j) {
            myid = bi;
            myw = p;
        }
    }
    if (lane < k) {
        ids[lane] = myid;
        w[lane] = myw / wsum;
    }
}

// The same routing with the token's logits held in registers (E <= 256).  Each
// round is two warp reductions: the largest logit as an order-preserving
// integer key (redux.sync max), then the lowest expert index carrying it
// (redux.sync min) -- the fp32 comparison with ties to the lower index, without
// a shuffle chain.  -0 counts as +0 (they compare equal); NaN and taken experts
// get key 0, which no logit's key reaches.
__device__ __forceinline__ unsigned route_key(float f) {
    if (f != f) return 0u;
    const unsigned b = __float_as_uint(f == 0.0f ? 0.0f : f);
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ void direct_route_token_reg(const float* __restrict__ l, int E, int k, int* ids, float* w,
                                                       int lane) {
    float v[8];
    unsigned key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        v[i] = lane + 32 * i < E ? __ldcg(l + lane + 32 * i) : 0.0f;
        key[i] = lane + 32 * i < E ? route_key(v[i]) : 0u;
    }
    int myid = 0;
    for (int j = 0; j < k; ++j) {
        unsigned km = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) km = key[i] > km ? key[i] : km;
        km = __reduce_max_sync(0xffffffffu, km);
        unsigned im = 0xffffffffu;
#pragma unroll
        for (int i = 7; i >= 0; --i)
            if (key[i] == km) im = static_cast<unsigned>(lane + 32 * i);  // lowest of this lane
        const int bi = static_cast<int>(__reduce_min_sync(0xffffffffu, im));
#pragma unroll
        for (int i = 0; i < 8; ++i)
            if (lane + 32 * i == bi) key[i] = 0u;
        if (lane == j) myid = bi;
    }
    // the softmax over the selected logits, after the rounds (lane j: the j-th
    // selected; the sum taken in selection order)
    float bv = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float t = __shfl_sync(0xffffffffu, v[i], myid & 31);
        if ((myid >> 5) == i) bv = t;
    }
    const float lmax = __shfl_sync(0xffffffffu, bv, 0);
    const float pj = expf(bv - lmax);
    float wsum = 0.0f;
    for (int j = 0; j < k; ++j) wsum += __shfl_sync(0xffffffffu, pj, j);
    if (lane < k) {
        ids[lane] = myid;
        w[lane] = pj / wsum;
    }
}

// Quantize the 256-element block `blk` of an fp32 row (global memory) to Q8_K
// straight into the shared-memory activation region (row `row`), with the
// same arithmetic as warp_quant_q8k.  Optionally also writes the packed block.
// `a`, `b` are the lane's eight values (elements 8 lane .. 8 lane + 7 of the block).
template <bool PERM>
__device__ __forceinline__ void warp_quant_to_smem(float4 a, float4 b, int row, int blk, int K, const XRegion& x,
                                                   uint8_t* packed, int lane) {
    float v[8];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(v[i]));
    const float amax = warp_max(m);
    float id;
    const float d = quant_scale(amax, &id);
    int q[8], s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        q[i] = quant_one(v[i], id);
        s += q[i];
    }
    const uint32_t w0 = (q[0] & 0xFF) | ((q[1] & 0xFF) << 8) | ((q[2] & 0xFF) << 16) | (static_cast<uint32_t>(q[3] & 0xFF) << 24);
    const uint32_t w1 = (q[4] & 0xFF) | ((q[5] & 0xFF) << 8) | ((q[6] & 0xFF) << 16) | (static_cast<uint32_t>(q[7] & 0xFF) << 24);
    int8_t* dq = x.q + static_cast<size_t>(row) * xq_row_bytes(K);
    const int e0 = 256 * blk + 8 * lane;
    if constexpr (!PERM) {
        *reinterpret_cast<uint32_t*>(dq + xq_addr(e0)) = w0;
        *reinterpret_cast<uint32_t*>(dq + xq_addr(e0 + 4)) = w1;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int el = e0 + i, r = el & 31;
            dq[xq_addr((el & ~31) + 2 * (r & 15) + (r >> 4))] = static_cast<int8_t>(q[i]);
        }
    }
    int s16 = s + __shfl_xor_sync(0xffffffffu, s, 1);   // 16-element group: lanes 2g, 2g+1
    int s32 = s16 + __shfl_xor_sync(0xffffffffu, s16, 2);  // 32-element block: lanes 4b..4b+3
    if ((lane & 1) == 0) x.bs[static_cast<size_t>(row) * (K >> 4) + 16 * blk + (lane >> 1)] = static_cast<int16_t>(s16);
    if ((lane & 3) == 0) x.s32[static_cast<size_t>(row) * (K >> 5) + 8 * blk + (lane >> 2)] = s32;
    if (lane == 0) x.d[static_cast<size_t>(row) * (K >> 8) + blk] = d;
    if (packed) {
        uint32_t* pq = reinterpret_cast<uint32_t*>(packed + 4 + 8 * lane);
        pq[0] = w0;
        pq[1] = w1;
        if ((lane & 1) == 0) reinterpret_cast<int16_t*>(packed + 260)[lane >> 1] = static_cast<int16_t>(s16);
        if (lane == 0) *reinterpret_cast<float*>(packed) = d;
    }
}

struct DirectParams {
    const uint8_t* W;    // gate bank (gate/up) or down bank
    const uint8_t* W2;   // up bank
    int64_t rowbytes;
    int64_t N;           // I (gate/up) or H (down)
    int K;               // H (gate/up) or I (down)
    int T, E, top_k;
    const float* X;              // gate/up: x [T][H]
    const float* logits;         // gate/up: [T][E] or null (routed)
    const int32_t* ids_in;       // gate/up routed ids
    const float* w_in;
    int32_t* ids;                // routed ids [T*k] (written by gate/up CTA 0, read by down)
    float* w;                    // routed weights [T*k]
    float* h;                    // [T*k][I]
    uint8_t* xq_dump;            // optional packed Q8_K of x
    const uint8_t* xq_in;        // gate/up: x already quantized, packed Q8_K [T][K/256] (X then unused)
    uint8_t* hq;                 // optional packed Q8_K of h (down CTA 0)
    int early_weights;
    int G;                       // fused down: experts per stage           // 1: stream weights before waiting for the previous kernel
    float* g_dump;
    float* u_dump;
    float* o_dump;               // optional [T*k][H]
    float* Y;                    // down: [T][H]
    int* err;
    int stages, stage_stride, x_bytes;
    int32_t* coefs[2];           // optional integer-core dump [T*k][N][ncoef]: gate and up, or down
    int ncoef;                   // coefficients per row: K/blk * (2 for Q4_K/Q5_K, else 1)
    unsigned long long* tel_pairs;  // optional expert-load telemetry: pairs per expert [E]
    unsigned long long* tel_calls;  // and [calls, distinct experts]
};

// Gate/up (KIND_GATEUP), down with per-pair outputs (KIND_DOWN) or fused
// down (KIND_DOWNF) of the direct route.
template <int KIND, int F, int NT, bool DUMP>
__global__ void __launch_bounds__(kThreads, 1) k_direct(const DirectParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    constexpr bool DOWN = KIND != KIND_GATEUP;
    constexpr int LV = NT == 1 ? 0 : NT == 2 ? 1 : 2;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int K = p.K, P = p.T * p.top_k;
    if constexpr (KIND == KIND_GATEUP) {
        pdl_wait();               // logits (or routed ids) and x come from earlier kernels
        pdl_launch_dependents();  // the down kernel, once it runs, may read them without waiting
    } else {
        pdl_launch_dependents();  // h is read only after pdl_wait below
    }

    uint8_t* ring = smem;
    uint8_t* xreg = smem + static_cast<size_t>(p.stages) * p.stage_stride;
    const int xrows = KIND == KIND_GATEUP ? p.T : P;
    const XRegion xr_ = x_region(xreg, xrows, K, false);
    uint64_t* full = reinterpret_cast<uint64_t*>(xreg + p.x_bytes);
    uint64_t* empty = full + kMaxStages;
    uint64_t* hbar = empty + kMaxStages;  // down: the fp32 h rows have landed (spare stage)
    DirectPlan* plan = reinterpret_cast<DirectPlan*>(hbar + 2);

    // ---- barriers (producer warp), routing (warps < T) and, in the gate/up
    // kernel, the activations (the other consumer warps), side by side.  Named
    // barriers: 3 = every thread (barriers initialised, plan, activations:
    // the consumers wait on it), 4 = warp 0 and the producer warp (the plan:
    // the producer's copies start as soon as it is known), 5 = the routing warps.
    // gate/up: the activations of the T tokens, by consumer warps w0 .. 15
    const auto stage_x = [&](int w0) {
        if (warp >= w0 && warp < kConsumerWarps) {
            const int sw = warp - w0, nsw = kConsumerWarps - w0;
            // x^ given (the "Q8 prequant" entry): staged as it is
            if (p.xq_in) stage_acts<false, F == F_MXFP4>(p.xq_in, xrows, K, xr_, tid - 32 * w0, 32 * nsw);
            // else quantize x (every CTA; a few blocks per warp, their loads issued together)
            const int nbr = K >> 8, nb = p.xq_in ? 0 : xrows * nbr;
            for (int b0 = sw; b0 < nb; b0 += 4 * nsw) {
                float4 va[4], vb[4];
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int b = b0 + h * nsw;
                    if (b < nb) {
                        const float4* src = reinterpret_cast<const float4*>(p.X + static_cast<int64_t>(b) * 256);
                        va[h] = __ldcg(src + 2 * lane);
                        vb[h] = __ldcg(src + 2 * lane + 1);
                    }
                }
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const int b = b0 + h * nsw;
                    if (b < nb) {
                        const int r = b / nbr, c = b - r * nbr;
                        uint8_t* pk = (blockIdx.x == 0 && p.xq_dump) ? p.xq_dump + static_cast<int64_t>(b) * 292 : nullptr;
                        warp_quant_to_smem<F == F_MXFP4>(va[h], vb[h], r, c, K, xr_, pk, lane);
                    }
                }
            }
        }
    };
    const bool single = p.T == 1 && p.logits != nullptr;
    if (warp == kConsumerWarps) {
        if (lane == 0) {
            for (int s = 0; s < p.stages; ++s) {
                mbar_init(&full[s], 1);
                mbar_init(&empty[s], kConsumerWarps);
            }
            mbar_init(hbar, 1);
            fence_barrier_init();
        }
        __syncwarp();
        named_arrive(3, kThreads);
        named_sync(4, 64);
    } else if (warp < p.T) {
        // both kernels route from the same inputs with the same arithmetic
        if (p.logits) {
            if (p.E <= 256)
                direct_route_token_reg(p.logits + static_cast<int64_t>(warp) * p.E, p.E, p.top_k,
                                       plan->ids + warp * p.top_k, plan->wt + warp * p.top_k, lane);
            else
                direct_route_token(p.logits + static_cast<int64_t>(warp) * p.E, p.E, p.top_k,
                                   plan->ids + warp * p.top_k, plan->wt + warp * p.top_k, lane);
        } else if (lane < p.top_k) {
            plan->ids[warp * p.top_k + lane] = __ldcg(p.ids_in + warp * p.top_k + lane);
            plan->wt[warp * p.top_k + lane] = __ldcg(p.w_in + warp * p.top_k + lane);
        }
        if (tid < P) plan->tok[tid] = tid / p.top_k;
        if (single) {
            // one token: its k experts are distinct (routing picks each once), so
            // the routing warp lays out the plan itself -- pair j on expert slot j
            // (routed ids given by the caller are grouped like several tokens')
            __syncwarp();
            const int e = lane < P ? plan->ids[lane] : 0;
            const unsigned anybad = __ballot_sync(0xffffffffu, e < 0 || e >= p.E);
            if (lane < P) {
                plan->expert[lane] = e;
                plan->npairs[lane] = 1;
                plan->pair[lane][0] = lane;
            }
            if (lane == 0) {
                plan->D = anybad ? 0 : P;
                plan->bad = anybad != 0u;
            }
        } else {
            named_sync(5, 32 * p.T);
            if (warp == 0) direct_group(plan, P, p.E, lane);
        }
        if (warp == 0) named_arrive(4, 64);
        named_sync(3, kThreads);
    } else {
        if constexpr (KIND == KIND_GATEUP) stage_x(p.T);
        named_sync(3, kThreads);
    }
    const int D = plan->D;
    if (KIND == KIND_GATEUP && blockIdx.x == 0 && tid < P) {
        p.ids[tid] = plan->ids[tid];
        p.w[tid] = plan->wt[tid];
        if (plan->bad && tid == 0) set_error(p.err, DEV_ERR_BAD_IDS);
        if (p.tel_pairs && tid < D) atomicAdd(p.tel_pairs + plan->expert[tid], static_cast<unsigned long long>(plan->npairs[tid]));
        if (p.tel_calls && tid == 0) {
            atomicAdd(p.tel_calls, 1ull);
            atomicAdd(p.tel_calls + 1, static_cast<unsigned long long>(D));
        }
    }
    const int tiles = static_cast<int>(p.N / kTileRows);
    const int nitems = KIND == KIND_GATEUP ? D * tiles : (D > 0 ? tiles : 0);
    if (static_cast<int>(blockIdx.x) >= nitems) return;
    // stages per item: the gate and up tiles of one expert; G experts' tiles (fused
    // down); one expert's tile (down with per-pair outputs)
    const int per_item = KIND == KIND_GATEUP ? 1 : KIND == KIND_DOWNF ? (D + p.G - 1) / p.G : D;

    if (warp == kConsumerWarps) {
        // ================= producer: lane 0 waits for the slot and posts its bytes,
        // then one lane per tile copy (copies of different experts' tiles are
        // issued side by side)
        const uint64_t pol = policy_evict_first();
        if (DOWN && !p.early_weights) pdl_wait();  // the weights may come from earlier kernels
        const uint32_t bytes = static_cast<uint32_t>(kTileRows * p.rowbytes);  // multiple of 16
        int j = 0, s = 0;
        uint32_t ph = 0u;  // ring slot and phase of stage j
        bool ok = true;
        for (int item = blockIdx.x; ok && item < nitems; item += gridDim.x) {
            for (int q = 0; q < per_item; ++q) {
                if (lane == 0) ok = mbar_wait(&empty[s], ph ^ 1u);
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) {
                    if (lane == 0) set_error(p.err, DEV_ERR_TIMEOUT);
                    break;
                }
                const int ncp = KIND == KIND_GATEUP ? 2 : KIND == KIND_DOWNF ? (D - q * p.G < p.G ? D - q * p.G : p.G) : 1;
                if (lane == 0) mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(ncp) * bytes);
                __syncwarp();
                if (lane < ncp) {
                    const int u = KIND == KIND_GATEUP ? item / tiles : KIND == KIND_DOWNF ? q * p.G + lane : q;
                    const int tile = KIND == KIND_GATEUP ? item - u * tiles : item;
                    const int64_t e = plan->expert[u];
                    const int64_t off = (e * p.N + static_cast<int64_t>(tile) * kTileRows) * p.rowbytes;
                    const uint8_t* src = (KIND == KIND_GATEUP && lane == 1 ? p.W2 : p.W) + off;
                    bulk_g2s(ring + static_cast<size_t>(s) * p.stage_stride + static_cast<size_t>(lane) * bytes, src,
                             bytes, &full[s], pol);
                }
                ++j;
                if (++s == p.stages) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
        // the copies still in flight land before the CTA exits
        if (lane == 0)
            for (int q = (j > p.stages ? j - p.stages : 0); q < j; ++q)
                if (!mbar_wait(&full[q % p.stages], static_cast<uint32_t>(q / p.stages) & 1u)) break;
        return;
    }

    // ================= consumers (down): h^ into shared memory
    if constexpr (DOWN) {
        pdl_wait();  // h comes from the gate/up kernel
        // With a ring stage to spare (this CTA's items take fewer stages than the
        // ring holds), the fp32 h rows come in by one bulk copy into the ring's
        // last stage: every CTA reads all of h, and word loads from every SM
        // queue on the same L2 lines.  Otherwise they are read directly.
        const int my_items = (nitems - static_cast<int>(blockIdx.x) + static_cast<int>(gridDim.x) - 1) /
                             static_cast<int>(gridDim.x);
        const int hbytes = P * K * 4;
        const bool hb = my_items * per_item < p.stages && hbytes <= p.stage_stride && hbytes % 16 == 0 &&
                        (reinterpret_cast<uintptr_t>(p.h) & 15) == 0;
        const float* hsrc = p.h;
        if (hb) {
            uint8_t* const raw = ring + static_cast<size_t>(p.stages - 1) * p.stage_stride;
            if (tid == 0) {
                mbar_arrive_expect_tx(hbar, static_cast<uint32_t>(hbytes));
                bulk_g2s(raw, p.h, static_cast<uint32_t>(hbytes), hbar, policy_evict_last());
            }
            if (!mbar_wait(hbar, 0u)) set_error(p.err, DEV_ERR_TIMEOUT);
            hsrc = reinterpret_cast<const float*>(raw);
        }
        // quantize h (every CTA: all pairs, K/256 blocks each; loads of four blocks in flight)
        const int nbr = K >> 8, nb = xrows * nbr;
        for (int b0 = warp; b0 < nb; b0 += 4 * kConsumerWarps) {
            float4 va[4], vb[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int b = b0 + h * kConsumerWarps;
                if (b < nb) {
                    const float4* src = reinterpret_cast<const float4*>(hsrc + static_cast<int64_t>(b) * 256);
                    va[h] = hb ? src[2 * lane] : __ldcg(src + 2 * lane);
                    vb[h] = hb ? src[2 * lane + 1] : __ldcg(src + 2 * lane + 1);
                }
            }
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const int b = b0 + h * kConsumerWarps;
                if (b < nb) {
                    const int r = b / nbr, c = b - r * nbr;
                    uint8_t* pk = (blockIdx.x == 0 && p.hq) ? p.hq + static_cast<int64_t>(b) * 292 : nullptr;
                    warp_quant_to_smem<F == F_MXFP4>(va[h], vb[h], r, c, K, xr_, pk, lane);
                }
            }
        }
        consumer_sync();
    }
    XS xs;
    xs.q = smem_addr(xr_.q);
    xs.d = smem_addr(xr_.d);
    xs.s32 = smem_addr(xr_.s32);
    xs.bs = smem_addr(xr_.bs);
    xs.K = K;
    const saddr ring_s = smem_addr(ring);
    constexpr int SH = 5 - (LV + (KIND == KIND_GATEUP ? 1 : 0));

    // fused down: the lane's units of a warp's concatenated row (G experts x nu
    // units): slot i is unit lane + 32 i, expert vg[i] (>= G: none), unit vu[i]
    const int nb32 = K >> 5;
    int vg[kDownUnits], vu[kDownUnits];
    if constexpr (KIND == KIND_DOWNF) {
        // v = lane + 32 i = g nu + u, walked without a division per slot
        const int nu = units_per_row(K), q32 = 32 / nu, r32 = 32 - q32 * nu;
        int g = lane / nu, u = lane - g * nu;
#pragma unroll
        for (int i = 0; i < kDownUnits; ++i) {
            const bool in = lane + 32 * i < p.G * nu;
            vg[i] = in ? g : kDirectMaxPairs;
            vu[i] = in ? u : 0;
            g += q32;
            u += r32;
            if (u >= nu) {
                u -= nu;
                ++g;
            }
        }
    }
    // The item loop, in two compiled copies for the gate/up kernel at one token:
    // with rows of at most 32 units, lane l owns unit l of every row and holds
    // its activations in registers (the dumping instance too, so that g and u
    // do not depend on what is dumped); else the generic dot, without those
    // registers held.
    const auto run = [&](auto rx_tag) {
        constexpr bool RX = decltype(rx_tag)::value;
        XUnit xa, xb;
        bool va = false, vb = false;
        if constexpr (RX) {
            va = lane < units_per_row(K);
            vb = lane + 32 < units_per_row(K);
            if (va) load_xunit<F>(xs, lane, xa);
            if (vb) load_xunit<F>(xs, lane + 32, xb);
        }
        int s = 0;
        uint32_t ph = 0u;  // ring slot and phase of the next stage
        const auto next_stage = [&]() {
            if (++s == p.stages) {
                s = 0;
                ph ^= 1u;
            }
        };
        for (int item = blockIdx.x; item < nitems; item += gridDim.x) {
            if constexpr (KIND == KIND_GATEUP) {
                const int u = item / tiles, tile = item - u * tiles;
                const bool ready = __all_sync(0xffffffffu, mbar_wait(&full[s], ph));
                const int np = plan->npairs[u];
                int xr[NT];
#pragma unroll
                for (int t = 0; t < NT; ++t) xr[t] = t < np ? plan->tok[plan->pair[u][t]] : 0;
                const saddr stage = ring_s + static_cast<uint32_t>(s * p.stage_stride);
                const int64_t row = static_cast<int64_t>(tile) * kTileRows + warp;
                if (ready) {
                    float acc[2 * NT];
#pragma unroll
                    for (int i = 0; i < 2 * NT; ++i) acc[i] = 0.0f;
                    const saddr grow = stage + static_cast<uint32_t>(warp * p.rowbytes);
                    const saddr urow = stage + static_cast<uint32_t>((kTileRows + warp) * p.rowbytes);
                    if constexpr (RX) {
                        acc[0] = (va ? unit_dot_rx<F>(grow, lane, nb32, xa) : 0.0f) +
                                 (vb ? unit_dot_rx<F>(grow, lane + 32, nb32, xb) : 0.0f);
                        acc[1] = (va ? unit_dot_rx<F>(urow, lane, nb32, xa) : 0.0f) +
                                 (vb ? unit_dot_rx<F>(urow, lane + 32, nb32, xb) : 0.0f);
                    } else if (np == 1) {
                        // the expert's only pair: its token's activation units in registers
                        // and the register-resident dot (the same integers and epilogue as
                        // the generic path below, fewer instructions)
                        const int nu = units_per_row(K), r = xr[0];
                        XS xp = xs;
                        xp.q = xs.q + static_cast<uint32_t>(r * xq_row_bytes(K));
                        xp.d = xs.d + 4u * static_cast<uint32_t>(r * (K >> 8));
                        xp.s32 = xs.s32 + 4u * static_cast<uint32_t>(r * (K >> 5));
                        xp.bs = xs.bs + 2u * static_cast<uint32_t>(r * (K >> 4));
                        float ag = 0.0f, au = 0.0f;
                        for (int v = lane; v < nu; v += 32) {
                            XUnit xu;
                            load_xunit<F>(xp, v, xu);
                            ag += unit_dot_rx<F>(grow, v, nb32, xu);
                            au += unit_dot_rx<F>(urow, v, nb32, xu);
                        }
                        acc[0] = ag;
                        acc[NT] = au;
                    } else {
                        row_accumulate<F, NT>(grow, xs, xr, np, acc, lane);
                        row_accumulate<F, NT>(urow, xs, xr, np, acc + NT, lane);
                    }
                    const float v = warp_transpose_reduce<LV + 1>(acc, lane);  // index = gate/up * NT + slot
                    const float uval = __shfl_down_sync(0xffffffffu, v, NT << SH);
                    const int idx = lane >> SH;
                    if ((lane & ((1 << SH) - 1)) == 0 && idx < NT && idx < np) {
                        const float hval = __fmul_rn(__fdiv_rn(v, 1.0f + expf(-v)), uval);
                        const int64_t o = static_cast<int64_t>(plan->pair[u][idx]) * p.N + row;
                        p.h[o] = hval;
                        if (p.g_dump) p.g_dump[o] = v;
                        if (p.u_dump) p.u_dump[o] = uval;
                    }
                    if constexpr (DUMP) {  // integer core of the gate and up rows for every pair on this expert
                        for (int j = 0; j < np; ++j) {
                            const int pr = plan->pair[u][j], tk = plan->tok[pr];
                            const int64_t o = (static_cast<int64_t>(pr) * p.N + row) * p.ncoef;
                            row_coefs_one<F>(stage + static_cast<uint32_t>(warp * p.rowbytes), xs, tk, p.coefs[0] + o, lane);
                            row_coefs_one<F>(stage + static_cast<uint32_t>((kTileRows + warp) * p.rowbytes), xs, tk,
                                             p.coefs[1] + o, lane);
                        }
                    }
                } else {
                    set_error(p.err, DEV_ERR_TIMEOUT);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);
                next_stage();
                if (!ready) break;
            } else if constexpr (KIND == KIND_DOWN) {
                const int tile = item;
                const int64_t row = static_cast<int64_t>(tile) * kTileRows + warp;
                // y for the T tokens of this row, accumulated over the experts in plan order
                float yacc = 0.0f;  // lane t (t < T) holds y[t][row] after each reduction
                bool ok = true;
                for (int u = 0; u < D; ++u) {
                    const bool ready = __all_sync(0xffffffffu, mbar_wait(&full[s], ph));
                    const int np = plan->npairs[u];
                    int xr[NT];
#pragma unroll
                    for (int t = 0; t < NT; ++t) xr[t] = t < np ? plan->pair[u][t] : 0;
                    if (ready && ok) {
                        const saddr stage = ring_s + static_cast<uint32_t>(s * p.stage_stride);
                        float acc[NT];
#pragma unroll
                        for (int i = 0; i < NT; ++i) acc[i] = 0.0f;
                        row_accumulate<F, NT>(stage + static_cast<uint32_t>(warp * p.rowbytes), xs, xr, np, acc, lane);
                        const float v = warp_transpose_reduce<LV>(acc, lane);  // lane >> SH = slot
                        const int slot = lane >> SH;
                        const int pp = slot < np ? xr[slot] : -1;
                        if constexpr (DUMP) {  // integer core of this down row for every pair on the expert
                            for (int j = 0; j < np; ++j) {
                                const int pr = plan->pair[u][j];
                                row_coefs_one<F>(stage + static_cast<uint32_t>(warp * p.rowbytes), xs, pr,
                                                 p.coefs[0] + (static_cast<int64_t>(pr) * p.N + row) * p.ncoef, lane);
                            }
                        }
                        if (pp >= 0 && (lane & ((1 << SH) - 1)) == 0 && p.o_dump) p.o_dump[static_cast<int64_t>(pp) * p.N + row] = v;
                        // move each slot's weighted value to the lane of its token
                        const float contrib = pp >= 0 ? plan->wt[pp] * v : 0.0f;
                        const int tok = pp >= 0 ? plan->tok[pp] : -1;
#pragma unroll
                        for (int q = 0; q < NT; ++q) {
                            const float cq = __shfl_sync(0xffffffffu, contrib, q << SH);
                            const int tq = __shfl_sync(0xffffffffu, tok, q << SH);
                            if (q < np && lane == tq) yacc += cq;
                        }
                    } else if (!ready) {
                        set_error(p.err, DEV_ERR_TIMEOUT);
                        ok = false;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    next_stage();
                }
                if (ok && lane < p.T) p.Y[static_cast<int64_t>(lane) * p.N + row] = yacc;
                if (!ok) break;
            } else {
                // fused down: y[t][row] = sum over experts and their pairs of w * (W_e row . h^_pair),
                // each lane adding the weighted partials of its units into its token sums
                const int64_t row = static_cast<int64_t>(item) * kTileRows + warp;
                float acc[NT];
#pragma unroll
                for (int t = 0; t < NT; ++t) acc[t] = 0.0f;
                bool ok = true;
                for (int ug = 0; ug < D; ug += p.G) {
                    const bool ready = __all_sync(0xffffffffu, mbar_wait(&full[s], ph));
                    if (ready && ok) {
                        const int gc = D - ug < p.G ? D - ug : p.G;
                        const saddr stage = ring_s + static_cast<uint32_t>(s * p.stage_stride);
                        if constexpr (NT == 1) {
                            // one token: each expert's pair reads its activation unit into
                            // registers and takes the register-resident dot (the same integers
                            // and epilogue as the path below, fewer instructions); the lane's
                            // units walked in a rolled loop (v = lane + 32 i = g nu + ur)
                            const int nu = units_per_row(K), q32 = 32 / nu, r32 = 32 - q32 * nu;
                            int g = lane / nu, ur = lane - g * nu;
#pragma unroll 1
                            for (int i = 0; i < kDownUnits && g < gc; ++i) {
                                const int u = ug + g;
                                const int pr = plan->pair[u][0];
                                const saddr rowp = stage + static_cast<uint32_t>((g * kTileRows + warp) * p.rowbytes);
                                XS xp = xs;
                                xp.q = xs.q + static_cast<uint32_t>(pr * xq_row_bytes(K));
                                xp.d = xs.d + 4u * static_cast<uint32_t>(pr * (K >> 8));
                                xp.s32 = xs.s32 + 4u * static_cast<uint32_t>(pr * (K >> 5));
                                xp.bs = xs.bs + 2u * static_cast<uint32_t>(pr * (K >> 4));
                                XUnit xu;
                                load_xunit<F>(xp, ur, xu);
                                acc[0] += plan->wt[pr] * unit_dot_rx<F>(rowp, ur, nb32, xu);
                                g += q32;
                                ur += r32;
                                if (ur >= nu) {
                                    ur -= nu;
                                    ++g;
                                }
                            }
                        } else {
#pragma unroll
                            for (int i = 0; i < kDownUnits; ++i) {
                                if (vg[i] < gc) {
                                    const int g = vg[i], ur = vu[i], u = ug + g;
                                    const int np = plan->npairs[u];
                                    const saddr rowp = stage + static_cast<uint32_t>((g * kTileRows + warp) * p.rowbytes);
                                    if (np == 1) {  // the expert's only pair: the register-resident dot
                                        const int pr = plan->pair[u][0];
                                        XS xp = xs;
                                        xp.q = xs.q + static_cast<uint32_t>(pr * xq_row_bytes(K));
                                        xp.d = xs.d + 4u * static_cast<uint32_t>(pr * (K >> 8));
                                        xp.s32 = xs.s32 + 4u * static_cast<uint32_t>(pr * (K >> 5));
                                        xp.bs = xs.bs + 2u * static_cast<uint32_t>(pr * (K >> 4));
                                        XUnit xu;
                                        load_xunit<F>(xp, ur, xu);
                                        const float val = plan->wt[pr] * unit_dot_rx<F>(rowp, ur, nb32, xu);
                                        const int tk = plan->tok[pr];
#pragma unroll
                                        for (int t = 0; t < NT; ++t)
                                            if (t == tk) acc[t] += val;
                                        continue;
                                    }
                                    Unit un;
                                    load_unit<F>(rowp, ur, nb32, un);
                                    int xo[4];
                                    unit_offsets<F>(ur, xo);
#pragma unroll
                                    for (int jj = 0; jj < NT; ++jj) {
                                        if (jj < np) {
                                            const int pr = plan->pair[u][jj];
                                            int A0, A1;
                                            unit_ints<F>(un, xo, xs, pr, ur, A0, A1);
                                            const float val = plan->wt[pr] * unit_value<F>(un, xs, pr, ur, A0, A1);
                                            const int tk = plan->tok[pr];
#pragma unroll
                                            for (int t = 0; t < NT; ++t)
                                                if (t == tk) acc[t] += val;
                                        }
                                    }
                                }
                            }
                        }
                    } else if (!ready) {
                        set_error(p.err, DEV_ERR_TIMEOUT);
                        ok = false;
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[s]);
                    next_stage();
                }
                const float v = warp_transpose_reduce<LV>(acc, lane);  // lane >> SH = token
                const int t = lane >> SH;
                if (ok && (lane & ((1 << SH) - 1)) == 0 && t < p.T) p.Y[static_cast<int64_t>(t) * p.N + row] = v;
                if (!ok) break;
            }
        }
    };
    if constexpr (KIND == KIND_GATEUP && NT == 1) {
        if (units_per_row(K) <= 64) run(std::true_type{});
        else run(std::false_type{});
    } else {
        run(std::false_type{});
    }
}

template <int KIND, int F, int NT, bool DUMP = false>
cudaError_t launch_direct_one(const DirectParams& p, int grid, int smem, cudaStream_t s) {
    static std::atomic<bool> attr_set[kMaxDevices] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (!attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(k_direct<KIND, F, NT, DUMP>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemLimit);
        if (e != cudaSuccess) return e;
        attr_set[dev].store(true, std::memory_order_release);
    }
    return launch_pdl(k_direct<KIND, F, NT, DUMP>, dim3(grid), dim3(kThreads), smem, s, p);
}

}  // namespace ggq

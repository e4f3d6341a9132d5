/*
 * ggq.h -- C ABI of libggq: keep-quant matrix-vector products and MoE
 * routed-expert GEMMs over GGUF block-quantized weights, on one GB300 GPU
 * (sm_103a).
 *
 * Weights stay in their packed GGUF blocks (Q4_0, Q8_0, Q2_K, Q3_K, Q4_K, Q5_K,
 * Q6_K, MXFP4; Q2_K and Q3_K in the matrix-vector product only).  Activations
 * are quantized on the fly to int8 blocks (Q8_1 for Q4_0, Q8_K for every other
 * format) and every dot is an exact integer block dot
 * followed by a floating-point scale epilogue.
 *
 * Pages the operations follow (cited by title and section):
 *   FreeToken PR #136 "feat(rocm): enable native GGUF kernels on ROCm
 *     (validated on RDNA4)", Summary: Q4_0 dequantization, the int8-activation
 *     matvec ggml_mul_mat_vec_a8 and the routed ggml_moe_a8_vec.
 *   vllm.cpp PR #523 "feat(rocm): grouped + non-grouped keep-quant expert
 *     GEMM", What changed: kMatmulBTQuant (op 74, non-grouped) and
 *     kMatmulBTQuantGrouped (op 75, grouped over expert_ids), Q8_0/Q4_K/Q5_K/
 *     Q6_K weights, Q8_0 + Q8_K activation quantizers; Honest gaps: the K-quants
 *     Q2_K and Q3_K follow the same skeleton; review: a per-dtype
 *     availability query instead of a boolean, a refusal that names the
 *     unsupported formats, and a grow-only scratch pool with no per-call
 *     malloc, free or synchronisation (graph capture safe).
 *   ds4 PR #656 "Add ROCm MXFP4 routed expert kernels", Summary: MXFP4 x Q8_K
 *     routed gate/up and down, SwiGLU, and a direct route for 2-4 tokens
 *     instead of partially filled expert-sorted tiles.
 *
 * Conventions for every call:
 *   - All data pointers are caller-owned CUDA DEVICE pointers on the context's
 *     device, 16-byte aligned (cudaMalloc gives 256).  The library owns only its
 *     scratch pool.  Nothing is freed by the library except that pool.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Calls only enqueue work: they never synchronise, except
 *     ggq_sync_status, and never allocate, except ggq_create and ggq_reserve.
 *     So every compute call can be captured into a CUDA graph once the pool
 *     is large enough and the kernel attributes were set by one earlier call
 *     outside capture.
 *   - Block layouts are the GGUF ones: a matrix of `rows` x K is rows of
 *     K/block_elems consecutive blocks, row after row, no padding.
 *   - Errors are returned as ggq_status; no exception crosses the ABI.  The
 *     message of the last error is ggq_last_error(ctx).  A call that returns
 *     an error has enqueued nothing.
 *   - Calls on one context are not thread-safe with each other.
 *   - A call that takes a context runs on the context's device and leaves the
 *     calling thread's current device as it found it.
 */
#ifndef GGQ_H
#define GGQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum ggq_status {
    GGQ_OK = 0,
    GGQ_ERR_INVALID_ARG = 1,   /* null pointer, unknown enum, misaligned pointer */
    GGQ_ERR_SHAPE = 2,         /* size not a multiple of the block, token count out of range */
    GGQ_ERR_UNSUPPORTED = 3,   /* (weight format, activation format, op) not implemented */
    GGQ_ERR_ARCH = 4,          /* device is not compute capability 10.3 (sm_103) */
    GGQ_ERR_CUDA = 5,          /* a CUDA runtime call failed; message has its text */
    GGQ_ERR_CAPACITY = 6,      /* scratch pool too small for this call: ggq_reserve first */
    GGQ_ERR_CAPTURE_ALLOC = 7, /* ggq_reserve would allocate while the stream is capturing */
    GGQ_ERR_DEVICE = 8         /* a kernel reported an error word (bounded wait ran out) */
} ggq_status;

/* Block formats.  The numeric values are the GGUF tensor type ids, so a GGUF
 * reader can pass its type field through unchanged. */
typedef enum ggq_type {
    GGQ_TYPE_Q4_0 = 2,   /* 32 weights: fp16 d, 16 B nibbles; w = (q - 8) d               */
    GGQ_TYPE_Q8_0 = 8,   /* 32 weights or activations: fp16 d, int8[32];  v = q d        */
    GGQ_TYPE_Q8_1 = 9,   /* 32 activations: fp16 d, fp16 s = d*sum(q), int8[32]            */
    GGQ_TYPE_Q2_K = 10,  /* 256: scales[16] (4-bit scale, 4-bit min), 64 B 2-bit quants, d, dmin */
    GGQ_TYPE_Q3_K = 11,  /* 256: 32 B high bits, 64 B 2-bit quants, 12 B 6-bit scales, fp16 d */
    GGQ_TYPE_Q4_K = 12,  /* 256: fp16 d, dmin, 12 B 6-bit scales/mins, 128 B nibbles       */
    GGQ_TYPE_Q5_K = 13,  /* 256: Q4_K header, 32 B high bits, 128 B nibbles                 */
    GGQ_TYPE_Q6_K = 14,  /* 256: 128 B low nibbles, 64 B high 2 bits, int8 scales[16], d   */
    GGQ_TYPE_Q8_K = 15,  /* 256 activations: fp32 d, int8[256], int16 bsums[16]             */
    GGQ_TYPE_MXFP4 = 39  /* 32 weights: E8M0 exponent byte, 16 B E2M1 nibbles               */
} ggq_type;

typedef enum ggq_op {
    GGQ_OP_QUANTIZE_ACT = 0, /* ggq_quantize_act                                  */
    GGQ_OP_DEQUANT = 1,      /* ggq_dequant                                        */
    GGQ_OP_MUL_MAT_VEC = 2,  /* ggq_mul_mat_vec / _q / _qa / ggq_block_dots (op 74) */
    GGQ_OP_MOE = 3           /* ggq_moe_experts / _routed, as gate/up or down (op 75) */
} ggq_op;

typedef struct ggq_ctx ggq_ctx;

/* Worst-case shapes for ggq_reserve.  Zero fields are ignored. */
typedef struct ggq_plan {
    int64_t max_tokens; /* largest T of any call                         */
    int64_t max_k;      /* largest GEMV input width K                     */
    int64_t n_experts;  /* E of the MoE calls                             */
    int64_t hidden;     /* H of the MoE calls                             */
    int64_t inter;      /* I (expert intermediate width) of the MoE calls */
    int64_t top_k;      /* k of the MoE calls                             */
} ggq_plan;

/* Expert banks of one MoE layer.  Each bank is E matrices back to back:
 * gate and up are [E][I rows][H/block], down is [E][H rows][I/block]. */
typedef struct ggq_moe_weights {
    int32_t gate_type, up_type, down_type; /* ggq_type of each bank */
    const void* gate;
    const void* up;
    const void* down;
} ggq_moe_weights;

/* Optional device buffers that receive the MoE intermediates (any may be NULL).
 * For tests and debugging; filling them costs extra stores.  Slot j of token t
 * is pair p = t*k + j.
 * The coefs_* arrays receive the integer core of the kernels that ran the
 * layer: for each pair, each output row and each weight block, the int32
 * coefficients that multiply the block's scale product, laid out
 * [T*k][rows][K/blk * c] exactly as ggq_block_dots writes them (rows = I for
 * gate/up, H for down; K = H for gate/up, I for down; c = 2 for Q4_K/Q5_K,
 * else 1).  They are written by the same launches that compute the outputs
 * (the kernels take a dump variant that also stores what their dp4a or
 * tensor-core integer sums hold); entries of pairs that do not exist are not
 * written. */
typedef struct ggq_moe_dump {
    int32_t* ids;    /* [T][k]   selected experts                         */
    float* weights;  /* [T][k]   renormalised routing weights             */
    void* xq;        /* [T][H/256] Q8_K blocks of x                        */
    float* g;        /* [T*k][I] gate outputs                              */
    float* u;        /* [T*k][I] up outputs                                */
    float* h;        /* [T*k][I] silu(g) * u                               */
    void* hq;        /* [T*k][I/256] Q8_K blocks of h                      */
    float* o;        /* [T*k][H] down outputs before the routing weight   */
    int32_t* coefs_gate; /* [T*k][I][H/blk * c] gate integer core          */
    int32_t* coefs_up;   /* [T*k][I][H/blk * c] up integer core            */
    int32_t* coefs_down; /* [T*k][H][I/blk * c] down integer core (h^)     */
} ggq_moe_dump;

/* Create a context on `device` (a CUDA ordinal).  Refuses any device that is
 * not compute capability 10.3 with GGQ_ERR_ARCH: the kernels are built for
 * sm_103a only (analogue of the fail-fast on non-wave32 targets in FreeToken
 * PR #136, Support scope).  Allocates a small control block (error word,
 * counters).  On error *out is NULL. */
ggq_status ggq_create(ggq_ctx** out, int device);

/* Free the scratch pool (including retired generations) and the context.
 * The caller must make sure no work of the context is still in flight. */
ggq_status ggq_destroy(ggq_ctx* ctx);

/* Text of the last error on this context ("" if none).  Owned by ctx. */
const char* ggq_last_error(const ggq_ctx* ctx);

/* Grow the scratch pool to fit every call whose shapes are within `plan`
 * (vllm.cpp PR #523 review: a grow-only pool replaces per-call malloc/free).
 * Grow-only: a smaller plan is a no-op.  The previous pool generation is
 * retired, not freed, until ggq_destroy, so work already enqueued on it stays
 * valid.  Returns GGQ_ERR_CAPTURE_ALLOC, without allocating, if the pool must
 * grow while `stream` is capturing. */
ggq_status ggq_reserve(ggq_ctx* ctx, const ggq_plan* plan, void* stream);

/* Current pool size in bytes. */
size_t ggq_scratch_bytes(const ggq_ctx* ctx);

/* Declare that no kernel writes any weight buffer passed to this context while
 * calls of the context are in flight (the usual case in inference).  Every
 * kernel of the library is launched with programmatic dependent launch: it
 * may start while the previous kernel in the stream is finishing, and waits
 * for that kernel before it reads activations or writes outputs.  With static
 * weights the GEMV kernels also start streaming their weights before that
 * wait, overlapping one call's weight reads with the previous call's tail.
 * Default 0 (weights are read only after the wait).  Takes effect for calls
 * enqueued after it. */
ggq_status ggq_set_static_weights(ggq_ctx* ctx, int static_weights);

/* Largest token count that ggq_moe_experts serves on the direct route (ds4 PR
 * #656 "Add ROCm MXFP4 routed expert kernels", Summary: the direct kernels
 * take 2-4 tokens, 5 and up go to expert-sorted tiles).  Above 4 tokens the
 * direct route runs as calls of at most 4 tokens each, and only while the
 * (token, expert) pairs number at most twice the experts; beyond that the
 * call takes expert-sorted tiles.  Default 32 (measured faster than the tiles
 * up to there on the decode layers); 4 keeps the page's split exactly.
 * max_tokens outside [4, 32] returns GGQ_ERR_INVALID_ARG.  Takes effect for
 * calls enqueued after it; results agree within the fp32 tolerance either way
 * (the integer dots are the same, the order of the fp32 sums is not). */
ggq_status ggq_set_direct_route_max_tokens(ggq_ctx* ctx, int max_tokens);

/* Per-format availability: 1 if (weight format w, activation format act, op)
 * runs on this library, else 0.  For GGQ_OP_QUANTIZE_ACT w is ignored and act
 * is Q8_1 or Q8_K; for GGQ_OP_DEQUANT act is ignored.  Callers decide at load
 * time whether to keep a tensor packed (vllm.cpp PR #523 review: a per-dtype
 * query, not a boolean, and refusal at load rather than at forward time). */
int ggq_supported(int w, int act, int op);

/* Quantize x [T][K] fp32 to packed activation blocks out [T][K/blk]
 * (act = GGQ_TYPE_Q8_1: K % 32 == 0, 36 B blocks; GGQ_TYPE_Q8_0: K % 32 == 0,
 * 34 B blocks; GGQ_TYPE_Q8_K: K % 256 == 0, 292 B blocks).  Per block:
 * d = amax/127 (fp32), q = round-half-away(x * (1/d)) clamped to +-127; Q8_1
 * stores d and s = d*sum(q) as fp16, Q8_0 stores d as fp16 (the Q8_0 activation
 * quantizer of vllm.cpp PR #523, What changed), Q8_K stores d as fp32 and the
 * 16 sums of 16 quants.  T = 0 or K = 0 is an empty call: it
 * returns GGQ_OK without reading or writing (the pointers may be NULL).
 * Needs no scratch. */
ggq_status ggq_quantize_act(ggq_ctx* ctx, int act, const float* x, int64_t T, int64_t K, void* out, void* stream);

/* Dequantize rows x K weights of format w to fp32 out [rows][K] (FreeToken
 * PR #136, Summary: Q4_0 dequantization; all six weight formats here).
 * rows = 0 or K = 0 is an empty call (GGQ_OK, nothing read or written).
 * Needs no scratch. */
ggq_status ggq_dequant(ggq_ctx* ctx, int w, const void* blocks, int64_t rows, int64_t K, float* out, void* stream);

/* Y[T][N] = X[T][K] . W[N][K]^T with W packed in format w and X fp32
 * ("MatmulBT", vllm.cpp PR #523 op 74; ggml_mul_mat_vec_a8 of FreeToken
 * PR #136).  X is quantized inside the call (Q8_1 for Q4_0, Q8_K otherwise)
 * into the scratch pool.  1 <= T <= 8.  K must be a multiple of the weight
 * block (32 or 256); Q8_K activations also need K % 256 == 0.  Long rows
 * stream in row chunks when a 16-row tile does not fit twice in shared memory;
 * the quantized activations are held whole in shared memory (about 1.52 bytes
 * per input per token), and when those of all T tokens leave too little room
 * the tokens run in groups (each group streams the weights once).  Every
 * format runs K up to 146432; larger K returns GGQ_ERR_SHAPE. */
ggq_status ggq_mul_mat_vec(ggq_ctx* ctx, int w, const void* W, int64_t N, int64_t K, const float* X, int64_t T,
                           float* Y, void* stream);

/* Same as ggq_mul_mat_vec with X already quantized: Xq is [T][K/blk] packed
 * Q8_1 (w = Q4_0) or Q8_K blocks, as ggq_quantize_act writes them (the "Q8
 * prequant" path: quantize once, reuse across calls).  Needs no scratch. */
ggq_status ggq_mul_mat_vec_q(ggq_ctx* ctx, int w, const void* W, int64_t N, int64_t K, const void* Xq, int64_t T,
                             float* Y, void* stream);

/* ggq_mul_mat_vec_q with the activation format named: act = the weight
 * format's default (Q8_1 for Q4_0, Q8_K otherwise), or GGQ_TYPE_Q8_0 with
 * Q4_0 or Q8_0 weights (the Q8_0 x Q8_0 pairing of vllm.cpp PR #523, What
 * changed; Xq [T][K/32] 34-byte blocks from ggq_quantize_act, K % 32 == 0).
 * Other pairings return GGQ_ERR_UNSUPPORTED.  Q8_0 activations run on the dp4a
 * streaming kernel at every token count.  Needs no scratch. */
ggq_status ggq_mul_mat_vec_qa(ggq_ctx* ctx, int w, int act, const void* W, int64_t N, int64_t K, const void* Xq,
                              int64_t T, float* Y, void* stream);

/* Debug dump of the integer core of ggq_mul_mat_vec_q: the int32 coefficients
 * that multiply each block's scale product, out [T][N][K/blk * c]:
 *   Q4_0 x Q8_1, Q8_0 x Q8_K, MXFP4 x Q8_K (c = 1): S = sum of integer products
 *     per 32-block (MXFP4 with doubled E2M1 codes);
 *   Q4_K/Q5_K x Q8_K (c = 2): A = sum_s sc_s S_s and B = sum_s m_s bsum_s per
 *     superblock, y += d_x (d A - dmin B);
 *   Q6_K x Q8_K (c = 1): A = sum_j sc_j S_j per superblock, y += d_x d A;
 *   Q2_K x Q8_K (c = 2): A = sum_j sc_j S_j and B = sum_j m_j bsum_j over the 16
 *     groups of 16, y += d_x (d A - dmin B);
 *   Q3_K x Q8_K (c = 1): A = sum_j (sc_j - 32) S_j over the 16 groups, y += d_x d A.
 * Runs the kernel that ggq_mul_mat_vec_q picks for the same (w, N, K, T) --
 * the dp4a streaming kernel, the tensor-path GEMV (3-8 tokens) or the grouped
 * int8 tensor-core kernel -- in a variant that stores the integers its dp4a or
 * mma units produce instead of the outputs.  The tensor paths hold them in
 * f32 accumulators; every such chain is short enough that its partial sums
 * stay below 2^24, so the stored value is the exact integer.  out must be
 * 4-byte aligned; the call clears it first. */
ggq_status ggq_block_dots(ggq_ctx* ctx, int w, const void* W, int64_t N, int64_t K, const void* Xq, int64_t T,
                          int32_t* coefs, void* stream);

/* ggq_block_dots for the pairings of ggq_mul_mat_vec_qa (Q4_0 x Q8_0 and
 * Q8_0 x Q8_0: S = sum of integer products per 32-block). */
ggq_status ggq_block_dots_qa(ggq_ctx* ctx, int w, int act, const void* W, int64_t N, int64_t K, const void* Xq,
                             int64_t T, int32_t* coefs, void* stream);

/* Routed-expert layer (ggml_moe_a8_vec / vllm.cpp PR #523 op 75 / ds4 PR #656):
 *   ids, weights = top_k of softmax(router_logits[t]) by logit (ties to the
 *     lower expert index), renormalised over the selected experts;
 *   x^ = Q8_K(X[t]);  g = W_gate[e] x^,  u = W_up[e] x^,  h = silu(g) * u;
 *   h^ = Q8_K(h);  o = W_down[e] h^;  Y[t] = sum_j weights[t][j] * o_j.
 * X [T][H] fp32, router_logits [T][E] fp32, Y [T][H] fp32 (overwritten).
 * H and I multiples of 256; gate/up rows and down rows multiples of 8;
 * 1 <= top_k <= 8, top_k <= E <= 4096, 1 <= T.  Routing by token count: T = 1
 * streams the selected experts once; 2 <= T <= 4 is the direct tiny-batch
 * route (each distinct expert's rows are read once for every token that chose
 * it); T >= 5 groups (token, slot) pairs by expert into expert-sorted tiles.
 * Widths are bounded by shared memory (16-row weight tiles and the quantized
 * activations of the tokens or pairs are staged whole): the direct route
 * (T <= 4) runs H up to 6400 for Q8_0 gate/up and 8192-12288 for the 4-6-bit
 * and MXFP4 formats at one token (less at four tokens: 5632-9984), and I up
 * to 3328-3840 at four tokens with top-8; wider shapes return GGQ_ERR_SHAPE.
 * `dump` may be NULL.  Scratch: ggq_reserve with the same E, H, I, top_k, T. */
ggq_status ggq_moe_experts(ggq_ctx* ctx, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I, int top_k,
                           const float* X, const float* router_logits, int64_t T, float* Y, const ggq_moe_dump* dump,
                           void* stream);

/* Same layer with the routing given: ids [T][top_k] int32 in 0..E-1 (distinct
 * per token) and weights [T][top_k] fp32, both device pointers. */
ggq_status ggq_moe_experts_routed(ggq_ctx* ctx, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I,
                                  int top_k, const float* X, const int32_t* ids, const float* weights, int64_t T,
                                  float* Y, const ggq_moe_dump* dump, void* stream);

/* The routed-expert layer of ggq_moe_experts with x already quantized: Xq is
 * [T][H/256] packed Q8_K blocks as ggq_quantize_act writes them (the "Q8
 * prequant" path of ds4 PR #656 "Add ROCm MXFP4 routed expert kernels", A/B
 * notes: quantize the activations once and reuse them, e.g. across the layers
 * or calls that share one input).  Same routing, kernels, shapes, scratch and
 * errors as ggq_moe_experts; Y is bit-identical to ggq_moe_experts on the x
 * that Xq was quantized from.  Xq must be 4-byte aligned.  With a dump, dump->xq
 * receives a copy of Xq. */
ggq_status ggq_moe_experts_q(ggq_ctx* ctx, const ggq_moe_weights* w, int64_t E, int64_t H, int64_t I, int top_k,
                             const void* Xq, const float* router_logits, int64_t T, float* Y, const ggq_moe_dump* dump,
                             void* stream);

/* ggq_mul_mat_vec without a context and without any allocation.  (The pages
 * have no counterpart of this call; it exists for deployment.)
 * For callers that cannot allocate device memory: code that runs while a CUDA
 * graph is being captured in a mode that forbids cudaMalloc, plugins whose
 * host framework owns every device byte through its own allocator, serving
 * processes whose HBM is partitioned up front and whose request path may not
 * allocate, and plain C callers that have nowhere to keep a context (creating
 * one allocates its control block).
 * The quantized activations live in a fixed array of 152 KB in the library's
 * device data, one per device that loads the library, held until the process
 * exits: T * (K/32 * 36) bytes for w = Q4_0, T * (K/256 * 292) otherwise, which
 * allows 8 tokens x 16384 inputs.  Larger shapes return GGQ_ERR_CAPACITY and
 * launch nothing.  Arguments and layouts are those of ggq_mul_mat_vec, on the
 * CURRENT device; other errors: GGQ_ERR_UNSUPPORTED, _INVALID_ARG, _SHAPE,
 * _ARCH (not sm_103), _CUDA.  Every token count runs on the dp4a streaming
 * kernel, whereas ggq_mul_mat_vec takes the tensor-path kernel at 3-8 tokens
 * where it applies: the two agree within the fp32 tolerance of the keep-quant
 * dot (the integer dots are the same; the order of the fp32 sums is not).
 * The first call on a device checks the architecture and looks up the
 * array's device address; make that first call before any stream capture.
 * Every call on a device shares the one array and it keeps the last call's
 * contents: calls whose work overlaps on the GPU (other streams, or other
 * host threads) race on it, so order them on one stream.  The kernels' waits
 * are bounded (about two seconds each); one that runs out is not reported by
 * this entry point, and the output rows of the tiles it gave up keep what Y
 * held before -- callers who need that failure reported use ggq_mul_mat_vec
 * and ggq_sync_status. */
ggq_status ggq_mul_mat_vec_noalloc(int w, const void* W, int64_t N, int64_t K, const float* X, int64_t T, float* Y,
                                   void* stream);

/* Expert-load telemetry of the routed-expert calls (FreeToken PR #260
 * "ROCm: validate native gfx1151 serving on Strix Halo", MoE cache telemetry:
 * active experts per layer).  With buffers set, every later ggq_moe_experts /
 * _routed call on the context adds on the device, in stream order:
 *   pairs[e]  += number of (token, slot) pairs the call routed to expert e
 *                (int64 [n_experts]: how often each expert's weights are read);
 *   calls[0]  += 1 and calls[1] += the number of distinct experts the call
 *                used (int64 [2]: calls[1] / calls[0] = experts per layer).
 * The buffers are caller-owned device memory, 8-byte aligned; the caller
 * clears them and reads them after synchronising.  Calls with E > n_experts
 * return GGQ_ERR_SHAPE while the telemetry is on.  pairs = calls = NULL turns
 * it off.  No allocation, no synchronisation: capture-safe like the calls. */
ggq_status ggq_set_moe_counters(ggq_ctx* ctx, int64_t* pairs, int64_t n_experts, int64_t* calls);

/* Synchronise `stream` and read the device error word: GGQ_OK, or
 * GGQ_ERR_DEVICE (a bounded wait inside a kernel ran out; the word is cleared),
 * or GGQ_ERR_CUDA. */
ggq_status ggq_sync_status(ggq_ctx* ctx, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* GGQ_H */

/*
 * ggq_oracle.c -- the CPU oracle for the keep-quant GEMV / MoE routed-expert path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA path.  Plain C99, double precision wherever the method leaves the
 * precision open, single precision only where the activation quantizer fixes
 * it.  Slow and obvious on purpose: every function follows the definition it
 * names, with no blocking, fusion or reordering beyond that definition.
 *
 * Sources (web pages, cited by title and section):
 *   [FT136] FreeToken PR #136 "feat(rocm): enable native GGUF kernels on ROCm
 *           (validated on RDNA4)" -- Summary: Q4_0 dequantization,
 *           ggml_mul_mat_vec_a8 (int8-activation matvec) and ggml_moe_a8_vec.
 *   [VC523] vllm.cpp PR #523 "feat(rocm): grouped + non-grouped keep-quant
 *           expert GEMM" -- What changed: kMatmulBTQuant / kMatmulBTQuantGrouped,
 *           Q8_0/Q4_K/Q5_K/Q6_K weights, Q8_0 + Q8_K activation quantizers,
 *           integer superblock dots (DotQ8_0/DotQ4K/DotQ5K/DotQ6K) with dp4a;
 *           Honest gaps: Q2_K and Q3_K follow the same skeleton (the review
 *           there lists them among the formats its CPU keep-quant oracle
 *           accepts).
 *   [DS656] ds4 PR #656 "Add ROCm MXFP4 routed expert kernels" -- Summary and
 *           Correctness: MXFP4 x Q8_K routed gate/up, SwiGLU, down.
 * The pages name the block formats but print no layout; the layouts below are
 * the public GGUF block definitions, restated.  Readings of points the pages
 * leave open are marked READING.
 *
 * Parity status: every function is pinned by the CPU tests (closed forms,
 * exhaustive enumeration, integer-form == dequantize-form, brute force) except
 * that agreement of the byte layouts with real GGUF files is unpinned: no such
 * file is available to compare against.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#include "ggq_oracle.h"

static int g_threads = 1;

void orc_set_threads(int n) { g_threads = n < 1 ? 1 : n; }

int orc_get_threads(void) {
#ifdef _OPENMP
    return g_threads;
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- scalars */

/* IEEE-754 binary16 -> double, from the definition of the format. */
double orc_half_to_double(uint16_t h) {
    int s = h >> 15, e = (h >> 10) & 31, m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
    return s ? -v : v;
}

/* float -> IEEE binary16, round to nearest, ties to even. */
uint16_t orc_float_to_half(float f) {
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    double a = fabs((double)f);
    if (isnan(f)) return (uint16_t)(sign | 0x7e00u);
    if (a >= 65520.0) return (uint16_t)(sign | 0x7c00u); /* at or past the tie above 65504 */
    if (a < ldexp(1.0, -14)) {                           /* subnormal range, unit 2^-24 */
        double r = rint(a * 16777216.0);                  /* exact scaling; rint = nearest-even */
        return (uint16_t)(sign | (uint16_t)r);            /* r == 1024 lands on the smallest normal */
    }
    int e;
    (void)frexp(a, &e);               /* a in [2^(e-1), 2^e) */
    double r = rint(ldexp(a, 11 - e)); /* significand in units of the last place: [1024, 2048] */
    int E = e - 1 + 15;
    if (r == 2048.0) { r = 1024.0; E += 1; }
    if (E >= 31) return (uint16_t)(sign | 0x7c00u);
    return (uint16_t)(sign | (uint16_t)(E << 10) | (uint16_t)((int)r - 1024));
}

/* E2M1 (FP4) code -> value: sign bit 3, exponent bits 2..1 (bias 1), mantissa bit 0.
 * Written from the OCP microscaling element definition: e == 0 is subnormal (m * 0.5). */
double orc_e2m1(int code) {
    int s = (code >> 3) & 1, e = (code >> 1) & 3, m = code & 1;
    double v = (e == 0) ? 0.5 * m : ldexp(1.0 + 0.5 * m, e - 1);
    return s ? -v : v;
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static int16_t rds16(const uint8_t* p) { return (int16_t)rd16(p); }
static float rdf32(const uint8_t* p) { float f; memcpy(&f, p, 4); return f; }

/* ---------------------------------------------------------- block layouts */

int orc_block_elems(int type) {
    switch (type) {
    case ORC_Q4_0: case ORC_Q8_0: case ORC_MXFP4: case ORC_Q8_1: return 32;
    case ORC_Q4_K: case ORC_Q5_K: case ORC_Q6_K: case ORC_Q8_K: case ORC_Q2_K: case ORC_Q3_K: return 256;
    default: return 0;
    }
}

int orc_block_bytes(int type) {
    switch (type) {
    case ORC_Q4_0: return 18;  /* fp16 d, 16 B of nibbles */
    case ORC_Q8_0: return 34;  /* fp16 d, int8[32] */
    case ORC_MXFP4: return 17; /* E8M0 exponent byte, 16 B of E2M1 nibbles */
    case ORC_Q8_1: return 36;  /* fp16 d, fp16 s, int8[32] */
    case ORC_Q4_K: return 144; /* fp16 d, fp16 dmin, scales[12], qs[128] */
    case ORC_Q5_K: return 176; /* fp16 d, fp16 dmin, scales[12], qh[32], qs[128] */
    case ORC_Q6_K: return 210; /* ql[128], qh[64], int8 scales[16], fp16 d */
    case ORC_Q8_K: return 292; /* fp32 d, int8[256], int16 bsums[16] */
    case ORC_Q2_K: return 84;  /* scales[16] (low nibble scale, high nibble min), qs[64], fp16 d, fp16 dmin */
    case ORC_Q3_K: return 110; /* hmask[32], qs[64], scales[12] (16 packed 6-bit), fp16 d */
    default: return 0;
    }
}

/* Q4_K / Q5_K: 6-bit scale and min of sub-block s (0..7) from the 12 packed bytes. */
void orc_kq_scale_min(const uint8_t* sc12, int s, int* sc, int* m) {
    if (s < 4) {
        *sc = sc12[s] & 63;
        *m = sc12[s + 4] & 63;
    } else {
        *sc = (sc12[s + 4] & 15) | ((sc12[s - 4] >> 6) << 4);
        *m = (sc12[s + 4] >> 4) | ((sc12[s] >> 6) << 4);
    }
}

/* Q3_K: 6-bit scale of 16-element group s (0..15) from the 12 packed bytes:
 * its low four bits are the low (s < 8) or high (s >= 8) nibble of byte s % 8,
 * its high two bits are bits 2(s/4), 2(s/4)+1 of byte 8 + s % 4.  The group's
 * signed scale is this value - 32. */
int orc_q3k_scale(const uint8_t* sc12, int s) {
    int lo = s < 8 ? (sc12[s] & 15) : (sc12[s - 8] >> 4);
    int hi = (sc12[8 + s % 4] >> (2 * (s / 4))) & 3;
    return lo | (hi << 4);
}

/* Integer quant of element i of one weight block, plus the per-element integer
 * scale factor where the format has one.  Values follow the closed forms:
 *   Q4_0: (nib - 8)                    value = d * q
 *   Q8_0: q                            value = d * q
 *   Q4_K: nib in 0..15, sub-block s     value = d*sc_s*q - dmin*m_s
 *   Q5_K: nib + 16*hbit                 value = d*sc_s*q - dmin*m_s
 *   Q6_K: (6-bit) - 32, group j=i/16    value = d*sc_j*q
 *   Q2_K: 2-bit q in 0..3, group j=i/16  value = d*sc_j*q - dmin*m_j
 *   Q3_K: 2 low bits + high bit, in -4..3 value = d*(sc6_j - 32)*q
 *   MXFP4: doubled E2M1 code (integer)  value = q * 2^(e-128)
 * Q2_K / Q3_K element i = 128n + 32j + l takes bits 2j, 2j+1 of qs[32n + l];
 * Q3_K adds bit 4n + j of hmask[l]: set keeps the value, clear subtracts 4. */
static int elem_q(int type, const uint8_t* b, int i) {
    switch (type) {
    case ORC_Q4_0: {
        const uint8_t* qs = b + 2;
        int nib = i < 16 ? (qs[i] & 15) : (qs[i - 16] >> 4);
        return nib - 8;
    }
    case ORC_Q8_0: return (int8_t)b[2 + i];
    case ORC_MXFP4: {
        const uint8_t* qs = b + 1;
        int code = i < 16 ? (qs[i] & 15) : (qs[i - 16] >> 4);
        return (int)lrint(2.0 * orc_e2m1(code)); /* doubled value is an integer */
    }
    case ORC_Q4_K: case ORC_Q5_K: {
        int s = i / 32, l = i % 32, c = s / 2;
        const uint8_t* qs = b + (type == ORC_Q4_K ? 16 : 48);
        int nib = (s % 2 == 0) ? (qs[32 * c + l] & 15) : (qs[32 * c + l] >> 4);
        if (type == ORC_Q5_K) nib += 16 * ((b[16 + l] >> s) & 1);
        return nib;
    }
    case ORC_Q6_K: {
        int h = i / 128, r = i % 128, g = r / 32, l = r % 32;
        const uint8_t* ql = b;
        const uint8_t* qh = b + 128;
        int lo = ql[64 * h + 32 * (g & 1) + l];
        int nib = (g < 2) ? (lo & 15) : (lo >> 4);
        int hi = (qh[32 * h + l] >> (2 * g)) & 3;
        return (nib | (hi << 4)) - 32;
    }
    case ORC_Q2_K: {
        int n = i / 128, j = (i % 128) / 32, l = i % 32;
        return (b[16 + 32 * n + l] >> (2 * j)) & 3;
    }
    case ORC_Q3_K: {
        int n = i / 128, j = (i % 128) / 32, l = i % 32;
        int lo = (b[32 + 32 * n + l] >> (2 * j)) & 3;
        int hbit = (b[l] >> (4 * n + j)) & 1;
        return lo - (hbit ? 0 : 4);
    }
    default: return 0;
    }
}

/* Dequantize one weight block to doubles (the plain per-element definitions). */
void orc_dequant_block(int type, const uint8_t* b, double* out) {
    int n = orc_block_elems(type);
    for (int i = 0; i < n; ++i) {
        int q = elem_q(type, b, i);
        switch (type) {
        case ORC_Q4_0: case ORC_Q8_0: out[i] = orc_half_to_double(rd16(b)) * q; break;
        case ORC_MXFP4: out[i] = ldexp((double)q, (int)b[0] - 128); break;
        case ORC_Q4_K: case ORC_Q5_K: {
            int sc, m;
            orc_kq_scale_min(b + 4, i / 32, &sc, &m);
            out[i] = orc_half_to_double(rd16(b)) * sc * q - orc_half_to_double(rd16(b + 2)) * m;
            break;
        }
        case ORC_Q6_K: out[i] = orc_half_to_double(rd16(b + 208)) * (int8_t)b[192 + i / 16] * q; break;
        case ORC_Q2_K:
            out[i] = orc_half_to_double(rd16(b + 80)) * (b[i / 16] & 15) * q -
                     orc_half_to_double(rd16(b + 82)) * (b[i / 16] >> 4);
            break;
        case ORC_Q3_K: out[i] = orc_half_to_double(rd16(b + 108)) * (orc_q3k_scale(b + 96, i / 16) - 32) * q; break;
        case ORC_Q8_1: out[i] = orc_half_to_double(rd16(b)) * (int8_t)b[4 + i]; break;
        case ORC_Q8_K: out[i] = (double)rdf32(b) * (int8_t)b[4 + i]; break;
        }
    }
}

/* Dequantize rows x K elements (rows of consecutive blocks). */
void orc_dequant(int type, const uint8_t* blocks, int64_t rows, int64_t K, double* out) {
    int be = orc_block_elems(type), bb = orc_block_bytes(type);
    int64_t nb = K / be;
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t j = 0; j < nb; ++j)
            orc_dequant_block(type, blocks + (r * nb + j) * bb, out + r * K + j * be);
}

/* ------------------------------------------------- activation quantizers */

/* READING (the pages give only the names; the per-block rule d = amax/127 with
 * int8 round-to-nearest is fixed by the workload definition).  Same IEEE fp32
 * sequence for both activation formats:
 *   amax = max |x| over the block;  d = amax / 127.0f;  id = d != 0 ? 1/d : 0;
 *   q = clamp(roundf(x * id), -127, 127)  (ties away from zero).
 * Q8_1 stores d as fp16 (nearest-even) and s = fp16(d * sum q) with d the fp32
 * value; Q8_K stores d as fp32 and bsums[j] = sum of q over elements 16j..16j+15. */
static void quant_block_f32(const float* x, int n, int8_t* q, float* d_out) {
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    float d = amax / 127.0f;
    float id = (d != 0.0f) ? 1.0f / d : 0.0f;
    for (int i = 0; i < n; ++i) {
        float v = x[i] * id;
        float r = roundf(v);
        if (r > 127.0f) r = 127.0f;
        if (r < -127.0f) r = -127.0f;
        q[i] = (int8_t)r;
    }
    *d_out = d;
}

void orc_quantize_q8_1(const float* x, int64_t T, int64_t K, uint8_t* out) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < K / 32; ++j) {
            uint8_t* b = out + (t * (K / 32) + j) * 36;
            int8_t q[32];
            float d;
            quant_block_f32(x + t * K + j * 32, 32, q, &d);
            int sum = 0;
            for (int i = 0; i < 32; ++i) sum += q[i];
            float s = d * (float)sum;
            uint16_t hd = orc_float_to_half(d), hs = orc_float_to_half(s);
            b[0] = hd & 255; b[1] = hd >> 8; b[2] = hs & 255; b[3] = hs >> 8;
            memcpy(b + 4, q, 32);
        }
}

/* Q8_0 activation blocks ([VC523] What changed: the Q8_0 activation quantizer
 * that pairs with Q8_0 weights): the same fp32 sequence per 32 elements, d
 * stored as fp16 (nearest-even) followed by the 32 quants -- the Q8_0 weight
 * layout. */
void orc_quantize_q8_0(const float* x, int64_t T, int64_t K, uint8_t* out) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < K / 32; ++j) {
            uint8_t* b = out + (t * (K / 32) + j) * 34;
            int8_t q[32];
            float d;
            quant_block_f32(x + t * K + j * 32, 32, q, &d);
            uint16_t hd = orc_float_to_half(d);
            b[0] = hd & 255; b[1] = hd >> 8;
            memcpy(b + 2, q, 32);
        }
}

void orc_quantize_q8_k(const float* x, int64_t T, int64_t K, uint8_t* out) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t j = 0; j < K / 256; ++j) {
            uint8_t* b = out + (t * (K / 256) + j) * 292;
            int8_t q[256];
            float d;
            quant_block_f32(x + t * K + j * 256, 256, q, &d);
            memcpy(b, &d, 4);
            memcpy(b + 4, q, 256);
            for (int g = 0; g < 16; ++g) {
                int s = 0;
                for (int i = 0; i < 16; ++i) s += q[16 * g + i];
                int16_t s16 = (int16_t)s;
                memcpy(b + 260 + 2 * g, &s16, 2);
            }
        }
}

/* ------------------------------------------------- integer block dots */

/* Activation format paired with each weight format ([FT136] Summary: Q4_0 with
 * the "a8" Q8_1 blocks; [VC523] What changed and [DS656] Summary: Q8_K). */
int orc_act_type(int wtype) { return wtype == ORC_Q4_0 ? ORC_Q8_1 : ORC_Q8_K; }

/* Number of int32 coefficients per weight block that the block dot produces:
 * 32-element formats: one S per block; Q4_K/Q5_K/Q2_K: (A, B) per superblock;
 * Q6_K/Q3_K: A. */
int orc_coefs_per_block(int wtype) {
    return (wtype == ORC_Q4_K || wtype == ORC_Q5_K || wtype == ORC_Q2_K) ? 2 : 1;
}

/* Whether the library pairs weight format wtype with activation format atype:
 * every weight format with its default activation, and the Q8_0 activation
 * blocks with the Q4_0 and Q8_0 weights ([VC523] What changed: Q8_0 x Q8_0). */
int orc_pair_ok(int wtype, int atype) {
    if (atype == orc_act_type(wtype)) return 1;
    return atype == ORC_Q8_0 && (wtype == ORC_Q4_0 || wtype == ORC_Q8_0);
}

/* The 32 int8 quants and the scale of 32-element block j of an activation row. */
static const int8_t* act_q32(int atype, const uint8_t* xrow, int64_t j) {
    switch (atype) {
    case ORC_Q8_1: return (const int8_t*)(xrow + j * 36 + 4);
    case ORC_Q8_0: return (const int8_t*)(xrow + j * 34 + 2);
    default: return (const int8_t*)(xrow + (j / 8) * 292 + 4 + (j % 8) * 32);
    }
}
static double act_d32(int atype, const uint8_t* xrow, int64_t j) {
    switch (atype) {
    case ORC_Q8_1: return orc_half_to_double(rd16(xrow + j * 36));
    case ORC_Q8_0: return orc_half_to_double(rd16(xrow + j * 34));
    default: return (double)rdf32(xrow + (j / 8) * 292);
    }
}

/* Integer coefficients of one weight row against one quantized activation row
 * ([VC523] What changed: the keep-quant dot is an integer core per superblock
 * followed by the scale epilogue).  For each weight block b:
 *   Q4_0 x Q8_1/Q8_0 : S_b = sum_j (nib_j - 8) * qx_j
 *   Q8_0 x Q8_K/Q8_0 : S_b = sum_j qw_j * qx_j
 *   MXFP4 x Q8_K: S_b = sum_j code2_j * qx_j          (doubled E2M1 codes)
 *   Q4_K/Q5_K x Q8_K: A = sum_s sc_s * S_s,  B = sum_s m_s * (bsum_2s + bsum_2s+1)
 *   Q6_K x Q8_K : A = sum_j sc_j * S_j,  S_j over 16 elements of q6 - 32
 *   Q2_K x Q8_K : A = sum_j sc_j * S_j,  B = sum_j m_j * bsum_j   (16-element groups j)
 *   Q3_K x Q8_K : A = sum_j (sc6_j - 32) * S_j,  S_j over 16 elements of q3     */
void orc_row_coefs_a(int wtype, int atype, const uint8_t* wrow, const uint8_t* xrow, int64_t K, int32_t* coefs) {
    int be = orc_block_elems(wtype), bb = orc_block_bytes(wtype), nc = orc_coefs_per_block(wtype);
    for (int64_t j = 0; j < K / be; ++j) {
        const uint8_t* b = wrow + j * bb;
        int32_t* out = coefs + j * nc;
        if (be == 32) {
            const int8_t* qx = act_q32(atype, xrow, j);
            int32_t S = 0;
            for (int i = 0; i < 32; ++i) S += elem_q(wtype, b, i) * qx[i];
            out[0] = S;
        } else {
            const uint8_t* xb = xrow + j * 292;
            const int8_t* qx = (const int8_t*)(xb + 4);
            if (wtype == ORC_Q6_K) {
                int32_t A = 0;
                for (int g = 0; g < 16; ++g) {
                    int32_t S = 0;
                    for (int i = 0; i < 16; ++i) S += elem_q(wtype, b, 16 * g + i) * qx[16 * g + i];
                    A += (int8_t)b[192 + g] * S;
                }
                out[0] = A;
            } else if (wtype == ORC_Q2_K) {
                int32_t A = 0, B = 0;
                for (int g = 0; g < 16; ++g) {
                    int32_t S = 0;
                    for (int i = 0; i < 16; ++i) S += elem_q(wtype, b, 16 * g + i) * qx[16 * g + i];
                    A += (b[g] & 15) * S;
                    B += (b[g] >> 4) * rds16(xb + 260 + 2 * g);
                }
                out[0] = A;
                out[1] = B;
            } else if (wtype == ORC_Q3_K) {
                int32_t A = 0;
                for (int g = 0; g < 16; ++g) {
                    int32_t S = 0;
                    for (int i = 0; i < 16; ++i) S += elem_q(wtype, b, 16 * g + i) * qx[16 * g + i];
                    A += (orc_q3k_scale(b + 96, g) - 32) * S;
                }
                out[0] = A;
            } else {
                int32_t A = 0, B = 0;
                for (int s = 0; s < 8; ++s) {
                    int sc, m;
                    orc_kq_scale_min(b + 4, s, &sc, &m);
                    int32_t S = 0;
                    for (int i = 0; i < 32; ++i) S += elem_q(wtype, b, 32 * s + i) * qx[32 * s + i];
                    A += sc * S;
                    B += m * (rds16(xb + 260 + 2 * (2 * s)) + rds16(xb + 260 + 2 * (2 * s + 1)));
                }
                out[0] = A;
                out[1] = B;
            }
        }
    }
}

void orc_row_coefs(int wtype, const uint8_t* wrow, const uint8_t* xrow, int64_t K, int32_t* coefs) {
    orc_row_coefs_a(wtype, orc_act_type(wtype), wrow, xrow, K, coefs);
}

/* Scale epilogue: the dot of one weight row with one quantized activation row,
 * in double, from the integer coefficients (form A of the oracle). */
static double row_dot_int(int wtype, int atype, const uint8_t* wrow, const uint8_t* xrow, int64_t K,
                          int32_t* scratch) {
    int be = orc_block_elems(wtype), bb = orc_block_bytes(wtype), nc = orc_coefs_per_block(wtype);
    orc_row_coefs_a(wtype, atype, wrow, xrow, K, scratch);
    double y = 0.0;
    for (int64_t j = 0; j < K / be; ++j) {
        const uint8_t* b = wrow + j * bb;
        const int32_t* c = scratch + j * nc;
        switch (wtype) {
        case ORC_Q4_0: case ORC_Q8_0:
            y += orc_half_to_double(rd16(b)) * act_d32(atype, xrow, j) * c[0];
            break;
        case ORC_MXFP4:
            y += ldexp(1.0, (int)b[0] - 128) * act_d32(atype, xrow, j) * c[0];
            break;
        case ORC_Q4_K: case ORC_Q5_K:
            y += (double)rdf32(xrow + j * 292) *
                 (orc_half_to_double(rd16(b)) * c[0] - orc_half_to_double(rd16(b + 2)) * c[1]);
            break;
        case ORC_Q6_K:
            y += (double)rdf32(xrow + j * 292) * orc_half_to_double(rd16(b + 208)) * c[0];
            break;
        case ORC_Q2_K:
            y += (double)rdf32(xrow + j * 292) *
                 (orc_half_to_double(rd16(b + 80)) * c[0] - orc_half_to_double(rd16(b + 82)) * c[1]);
            break;
        case ORC_Q3_K:
            y += (double)rdf32(xrow + j * 292) * orc_half_to_double(rd16(b + 108)) * c[0];
            break;
        }
    }
    return y;
}

/* Y[t][n] = sum_k W[n][k] * Xq[t][k]  ("MatmulBT": [VC523] What changed, op 74;
 * [FT136] Summary, ggml_mul_mat_vec_a8), Xq in activation format atype.
 * Integer-dot form, double epilogue. */
void orc_gemv_a(int wtype, int atype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T,
                double* Y) {
    int64_t wrow = K / orc_block_elems(wtype) * orc_block_bytes(wtype);
    int64_t xrow = K / orc_block_elems(atype) * orc_block_bytes(atype);
    int64_t ncoef = K / orc_block_elems(wtype) * orc_coefs_per_block(wtype);
#pragma omp parallel num_threads(g_threads)
    {
        int32_t* scratch = (int32_t*)__builtin_alloca(sizeof(int32_t) * (size_t)ncoef);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n)
            for (int64_t t = 0; t < T; ++t)
                Y[t * N + n] = row_dot_int(wtype, atype, W + n * wrow, Xq + t * xrow, K, scratch);
    }
}

void orc_gemv(int wtype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T, double* Y) {
    orc_gemv_a(wtype, orc_act_type(wtype), W, N, K, Xq, T, Y);
}

/* Per-block integer coefficients of every (t, n) pair: out[t][n][K/blk * ncoef]. */
void orc_gemv_coefs_a(int wtype, int atype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T,
                      int32_t* out) {
    int64_t wrow = K / orc_block_elems(wtype) * orc_block_bytes(wtype);
    int64_t xrow = K / orc_block_elems(atype) * orc_block_bytes(atype);
    int64_t ncoef = K / orc_block_elems(wtype) * orc_coefs_per_block(wtype);
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < N; ++n)
            orc_row_coefs_a(wtype, atype, W + n * wrow, Xq + t * xrow, K, out + (t * N + n) * ncoef);
}

void orc_gemv_coefs(int wtype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T, int32_t* out) {
    orc_gemv_coefs_a(wtype, orc_act_type(wtype), W, N, K, Xq, T, out);
}

/* Form B: dequantize both operands to double and take the plain dot.
 * If absdot is non-null it receives sum_k |w_k * x_k| (the tolerance scale). */
void orc_gemv_dequant(int wtype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T, double* Y,
                      double* absdot) {
    orc_gemv_dequant_a(wtype, orc_act_type(wtype), W, N, K, Xq, T, Y, absdot);
}

void orc_gemv_dequant_a(int wtype, int atype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T,
                        double* Y, double* absdot) {
    int64_t wrow = K / orc_block_elems(wtype) * orc_block_bytes(wtype);
    int64_t xrow = K / orc_block_elems(atype) * orc_block_bytes(atype);
#pragma omp parallel num_threads(g_threads)
    {
        double* w = (double*)__builtin_alloca(sizeof(double) * (size_t)K);
        double* x = (double*)__builtin_alloca(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; ++n) {
            orc_dequant(wtype, W + n * wrow, 1, K, w);
            for (int64_t t = 0; t < T; ++t) {
                orc_dequant(atype, Xq + t * xrow, 1, K, x);
                double s = 0.0, a = 0.0;
                for (int64_t k = 0; k < K; ++k) {
                    s += w[k] * x[k];
                    a += fabs(w[k] * x[k]);
                }
                Y[t * N + n] = s;
                if (absdot) absdot[t * N + n] = a;
            }
        }
    }
}

/* ------------------------------------------------------------------ MoE */

/* Router (READING: the workload definition gives softmax -> top-k -> renormalise;
 * [VC523] and [FT260] name the router and the MoE combine/gate chain only).
 * Selection is by logit in fp32 comparisons, largest first, ties to the lower
 * expert index; weights are p_i / sum over the selected p, in double. */
void orc_router(const float* logits, int64_t T, int64_t E, int k, int32_t* ids, double* weights) {
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * E;
        double mx = -INFINITY;
        for (int64_t e = 0; e < E; ++e)
            if ((double)l[e] > mx) mx = l[e];
        double Z = 0.0;
        for (int64_t e = 0; e < E; ++e) Z += exp((double)l[e] - mx);
        double psel = 0.0;
        for (int j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                int taken = 0;
                for (int i = 0; i < j; ++i)
                    if (ids[t * k + i] == e) taken = 1;
                if (taken) continue;
                if (best < 0 || l[e] > l[best]) best = e;
            }
            ids[t * k + j] = (int32_t)best;
            weights[t * k + j] = exp((double)l[best] - mx) / Z;
            psel += weights[t * k + j];
        }
        for (int j = 0; j < k; ++j) weights[t * k + j] /= psel;
    }
}

/* silu(z) = z / (1 + e^-z); SwiGLU h = silu(g) * u ([DS656] Correctness: gate/up,
 * SwiGLU, down).  READING: no clamp, no bias, separate gate and up matrices. */
double orc_silu(double z) { return z / (1.0 + exp(-z)); }

/* Gate/up stage for every (token, slot): g, u, h = silu(g) * u, in double.
 * Banks are [E][rows][blocks]; xq is Q8_K of x, [T][H/256]. */
void orc_moe_gate_up(int gtype, const uint8_t* gate_bank, int utype, const uint8_t* up_bank, int64_t H, int64_t I,
                     const uint8_t* xq, int64_t T, const int32_t* ids, int k, double* g, double* u, double* h) {
    int64_t grow = H / orc_block_elems(gtype) * orc_block_bytes(gtype);
    int64_t urow = H / orc_block_elems(utype) * orc_block_bytes(utype);
    int64_t xrow = H / 256 * 292;
    int64_t nc = H / 32 * 2;
#pragma omp parallel num_threads(g_threads)
    {
        int32_t* scratch = (int32_t*)__builtin_alloca(sizeof(int32_t) * (size_t)nc);
#pragma omp for schedule(static) collapse(2)
        for (int64_t tk = 0; tk < T * k; ++tk)
            for (int64_t i = 0; i < I; ++i) {
                int64_t t = tk / k, e = ids[tk];
                double gv = row_dot_int(gtype, orc_act_type(gtype), gate_bank + (e * I + i) * grow, xq + t * xrow, H,
                                        scratch);
                double uv = row_dot_int(utype, orc_act_type(utype), up_bank + (e * I + i) * urow, xq + t * xrow, H,
                                        scratch);
                if (g) g[tk * I + i] = gv;
                if (u) u[tk * I + i] = uv;
                h[tk * I + i] = orc_silu(gv) * uv;
            }
    }
}

/* Down stage: o[t*k+j][n] = W_d[ids[t*k+j]][n] . hq[t*k+j]; hq is Q8_K of h. */
void orc_moe_down(int dtype, const uint8_t* down_bank, int64_t H, int64_t I, const uint8_t* hq, int64_t T,
                  const int32_t* ids, int k, double* o) {
    int64_t drow = I / orc_block_elems(dtype) * orc_block_bytes(dtype);
    int64_t hrow = I / 256 * 292;
    int64_t nc = I / 32 * 2;
#pragma omp parallel num_threads(g_threads)
    {
        int32_t* scratch = (int32_t*)__builtin_alloca(sizeof(int32_t) * (size_t)nc);
#pragma omp for schedule(static) collapse(2)
        for (int64_t tk = 0; tk < T * k; ++tk)
            for (int64_t n = 0; n < H; ++n)
                o[tk * H + n] = row_dot_int(dtype, orc_act_type(dtype), down_bank + (ids[tk] * H + n) * drow,
                                            hq + tk * hrow, I, scratch);
    }
}

/* Weighted combine y[t][n] = sum_j w[t][j] * o[t*k+j][n]
 * ([VC523] header: the MoE combine/gate chain). */
void orc_moe_combine(const double* o, const double* weights, int64_t T, int k, int64_t H, double* y) {
    for (int64_t t = 0; t < T; ++t)
        for (int64_t n = 0; n < H; ++n) {
            double s = 0.0;
            for (int j = 0; j < k; ++j) s += weights[t * k + j] * o[(t * k + j) * H + n];
            y[t * H + n] = s;
        }
}

/* The whole routed-expert layer, steps in order:
 *   router -> x^ = Q8_K(x) -> g, u -> h = silu(g) u -> h^ = Q8_K(fp32(h)) -> o -> y.
 * Intermediate buffers are caller-provided so that tests can inspect them:
 *   xq [T][H/256*292], hq [T*k][I/256*292], h [T*k][I] double, o [T*k][H] double. */
void orc_moe(int gtype, const uint8_t* gate_bank, int utype, const uint8_t* up_bank, int dtype,
             const uint8_t* down_bank, int64_t E, int64_t H, int64_t I, int k, const float* x, const float* logits,
             int64_t T, int32_t* ids, double* weights, uint8_t* xq, double* h, uint8_t* hq, double* o, double* y) {
    (void)E;
    orc_router(logits, T, E, k, ids, weights);
    orc_quantize_q8_k(x, T, H, xq);
    orc_moe_gate_up(gtype, gate_bank, utype, up_bank, H, I, xq, T, ids, k, 0, 0, h);
    for (int64_t tk = 0; tk < T * k; ++tk) {
        /* the quantizer consumes fp32 activations: h is rounded to fp32 first */
        float hf[4096];
        for (int64_t base = 0; base < I; base += 4096) {
            int64_t n = I - base < 4096 ? I - base : 4096;
            for (int64_t i = 0; i < n; ++i) hf[i] = (float)h[tk * I + base + i];
            orc_quantize_q8_k(hf, 1, n, hq + tk * (I / 256) * 292 + (base / 256) * 292);
        }
    }
    orc_moe_down(dtype, down_bank, H, I, hq, T, ids, k, o);
    orc_moe_combine(o, weights, T, k, H, y);
}

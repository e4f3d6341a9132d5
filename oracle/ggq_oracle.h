/*
 * ggq_oracle.h -- declarations of the CPU oracle (test infrastructure only).
 * See ggq_oracle.c for the definitions each function follows.
 */
#ifndef GGQ_ORACLE_H
#define GGQ_ORACLE_H
#include <stdint.h>

/* The oracle's own format tags (independent of the library's enum). */
enum {
    ORC_Q4_0 = 0, ORC_Q8_0 = 1, ORC_Q4_K = 2, ORC_Q5_K = 3, ORC_Q6_K = 4, ORC_MXFP4 = 5, ORC_Q8_1 = 6, ORC_Q8_K = 7,
    ORC_Q2_K = 8, ORC_Q3_K = 9
};

void orc_set_threads(int n);
int orc_get_threads(void);

double orc_half_to_double(uint16_t h);
uint16_t orc_float_to_half(float f);
double orc_e2m1(int code);

int orc_block_elems(int type);
int orc_block_bytes(int type);
int orc_act_type(int wtype);
int orc_coefs_per_block(int wtype);
void orc_kq_scale_min(const uint8_t* sc12, int s, int* sc, int* m);
int orc_q3k_scale(const uint8_t* sc12, int s);

void orc_dequant_block(int type, const uint8_t* b, double* out);
void orc_dequant(int type, const uint8_t* blocks, int64_t rows, int64_t K, double* out);

void orc_quantize_q8_1(const float* x, int64_t T, int64_t K, uint8_t* out);
void orc_quantize_q8_0(const float* x, int64_t T, int64_t K, uint8_t* out);
void orc_quantize_q8_k(const float* x, int64_t T, int64_t K, uint8_t* out);

int orc_pair_ok(int wtype, int atype);
void orc_row_coefs(int wtype, const uint8_t* wrow, const uint8_t* xrow, int64_t K, int32_t* coefs);
void orc_row_coefs_a(int wtype, int atype, const uint8_t* wrow, const uint8_t* xrow, int64_t K, int32_t* coefs);
void orc_gemv_a(int wtype, int atype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T,
                double* Y);
void orc_gemv_coefs_a(int wtype, int atype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T,
                      int32_t* out);
void orc_gemv_dequant_a(int wtype, int atype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T,
                        double* Y, double* absdot);
void orc_gemv(int wtype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T, double* Y);
void orc_gemv_coefs(int wtype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T, int32_t* out);
void orc_gemv_dequant(int wtype, const uint8_t* W, int64_t N, int64_t K, const uint8_t* Xq, int64_t T, double* Y,
                      double* absdot);

void orc_router(const float* logits, int64_t T, int64_t E, int k, int32_t* ids, double* weights);
double orc_silu(double z);
void orc_moe_gate_up(int gtype, const uint8_t* gate_bank, int utype, const uint8_t* up_bank, int64_t H, int64_t I,
                     const uint8_t* xq, int64_t T, const int32_t* ids, int k, double* g, double* u, double* h);
void orc_moe_down(int dtype, const uint8_t* down_bank, int64_t H, int64_t I, const uint8_t* hq, int64_t T,
                  const int32_t* ids, int k, double* o);
void orc_moe_combine(const double* o, const double* weights, int64_t T, int k, int64_t H, double* y);
void orc_moe(int gtype, const uint8_t* gate_bank, int utype, const uint8_t* up_bank, int dtype,
             const uint8_t* down_bank, int64_t E, int64_t H, int64_t I, int k, const float* x, const float* logits,
             int64_t T, int32_t* ids, double* weights, uint8_t* xq, double* h, uint8_t* hq, double* o, double* y);

#endif

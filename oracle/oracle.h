/*
 * oracle.h -- fp64 CPU reference for the quantised decode GEMV.
 * TEST INFRASTRUCTURE ONLY: see oracle.c for what it computes and why.
 *
 * Layouts (all row-major):
 *   NVFP4: codes u8[N][K/2] (low nibble = even k), scales u8[N][K/16] (E4M3),
 *          global scale g.
 *   Q4/Q5: q_lo u8[N][K/2], q_hi u8[N][K/8] (Q5 only; bit k%8 of byte k/8),
 *          scale and min as fp16 bit patterns u16[N][K/32].
 *   x: bf16 bit patterns u16[M][K]; residual r: u16[M][N]; y: double[M][N].
 */
#ifndef QGEMV_ORACLE_H
#define QGEMV_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

double orc_e2m1(unsigned code);
double orc_e4m3(unsigned code);
double orc_f16(unsigned bits);
double orc_bf16(unsigned bits);
double orc_round_bf16(double v);
unsigned orc_bf16_bits(double v);
double orc_silu(double v);

void orc_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales, double g,
                       int64_t N, int64_t K, double* w);
void orc_dequant_q45(const uint8_t* q_lo, const uint8_t* q_hi, const uint16_t* scale,
                     const uint16_t* mn, int bits, int64_t N, int64_t K, double* w);

void orc_gemv_nvfp4(const uint8_t* codes, const uint8_t* scales, double g,
                    const uint16_t* x, const uint16_t* r, int64_t M, int64_t N, int64_t K,
                    int64_t n0, int64_t n1, double* y, double* absacc);
void orc_gemv_q45(const uint8_t* q_lo, const uint8_t* q_hi, const uint16_t* scale,
                  const uint16_t* mn, int bits, const uint16_t* x, const uint16_t* r,
                  int64_t M, int64_t N, int64_t K, int64_t n0, int64_t n1,
                  double* y, double* absacc);

void orc_swiglu(const double* gate, const double* up, int64_t n, double* out);
void orc_rmsnorm(const uint16_t* x, const uint16_t* gamma, double eps, int64_t M, int64_t K,
                 double* r, double* v, uint16_t* h);
void orc_round_bf16_array(const double* v, int64_t n, double* out);
void orc_bf16_bits_array(const double* v, int64_t n, uint16_t* out);
void orc_bf16_array(const uint16_t* bits, int64_t n, double* out);
void orc_f16_array(const uint16_t* bits, int64_t n, double* out);
void orc_e4m3_array(const uint8_t* codes, int64_t n, double* out);

void orc_route_topk(const float* logits, int64_t M, int64_t E, int topk,
                    int32_t* ids, double* w);
void orc_moe_gate_up(const uint8_t* gu_codes, const uint8_t* gu_scales, const double* gu_g,
                     const uint16_t* x, const int32_t* ids, int64_t H, int64_t I, int topk,
                     int64_t p0, int64_t p1, double* gate, double* up,
                     double* abs_gate, double* abs_up, uint16_t* h_bits);
void orc_moe_down(const uint8_t* dn_codes, const uint8_t* dn_scales, const double* dn_g,
                  const double* v, const int32_t* ids, const double* w,
                  int64_t M, int64_t H, int64_t I, int topk, int use_abs,
                  int64_t j0, int64_t j1, double* y);

#ifdef __cplusplus
}
#endif
#endif

/*
 * oracle.c -- plain, slow, fp64 CPU reference for the quantised decode GEMV.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or
 * call this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg use it. It shares no source with the CUDA library.
 *
 * What it computes, and where each definition comes from:
 *   - The pages name the weight formats but print no bit layout: NVFP4 in the
 *     NInfer article (section 2, "自研 CUDA 算子 混合量化权重": NVFP4 artefacts
 *     and a groupwise-int Q4/Q5 recipe) and in the Decapybara README
 *     ("Blackwell CUDA 内核套件", mx_gemv.cu: NVFP4/MXFP8 block mat-vec).
 *   - E2M1 and E4M3 element encodings follow the OCP Microscaling Formats
 *     (MX) specification v1.0 (FP4 E2M1: bias 1, no inf/NaN; FP8 E4M3: bias 7,
 *     S.1111.111 is NaN, no infinities). NVFP4 = E2M1 codes, one E4M3 scale per
 *     16 consecutive weights along K, one FP32 per-tensor scale g.
 *   - Groupwise int: unsigned code q, fp16 scale and min per group of 32 along
 *     K, w = scale * q + min. Q5 keeps the 5th bit in a separate bit plane.
 *   - The GEMV is y[m][n] = sum_k w[n][k] * x[m][k] (decode is a
 *     memory-bound mat-vec: NInfer article, section 2), with optional fused
 *     residual add and SwiGLU epilogues (same section: "矩阵乘、残差加、SwiGLU
 *     ... 一次读、一次写").
 *   - RMSNorm ahead of a projection (same section: normalisation fused with
 *     the matmul): r = 1/sqrt(mean(x^2) + eps), h = bf16(x * r * gamma).
 *   - MoE: softmax over expert logits, top-8, renormalised weights (Decapybara
 *     README, moe.cu "Top-8 门控和 softmax"); each selected expert runs
 *     gate/up + SwiGLU then down, and the outputs are summed with the weights.
 *
 * Arithmetic: every decode is exact in fp64; every sum is a plain sequential
 * fp64 loop in k order. Built with -ffp-contract=off so no fused multiply-add
 * changes a result between machines.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   low nibble of a code byte holds the even k; scales/mins are row-major
 *   [N][K/16] or [N][K/32]; the Q5 bit plane is LSB-first (bit k%8 of byte
 *   k/8); SwiGLU rows are gate [0, I) then up [I, 2I); silu(v) = v/(1+e^-v);
 *   the MoE intermediate h is rounded to bf16 (it is a bf16 activation between
 *   two projections); ties in top-k go to the lower expert id.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* element decodes                                                          */
/* ------------------------------------------------------------------------ */

/* FP4 E2M1 (OCP MX v1.0): bit 3 sign, bits 2-1 exponent (bias 1), bit 0
 * mantissa. Exponent 0 is subnormal: value = m * 2^(1-1) * 0.5. */
double orc_e2m1(unsigned code)
{
    unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
    double mag = (e == 0) ? 0.5 * (double)m : ldexp(1.0 + 0.5 * (double)m, (int)e - 1);
    return s ? -mag : mag;
}

/* FP8 E4M3 (OCP MX v1.0, the "FN" variant used by NVFP4 scales): bit 7 sign,
 * bits 6-3 exponent (bias 7), bits 2-0 mantissa; exponent 0 is subnormal
 * (2^-6 * m/8); S.1111.111 is NaN; there is no infinity (max 448). */
double orc_e4m3(unsigned code)
{
    unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
    double mag;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return s ? -mag : mag;
}

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 mantissa bits. */
double orc_f16(unsigned bits)
{
    unsigned s = (bits >> 15) & 1u, e = (bits >> 10) & 31u, m = bits & 1023u;
    double mag;
    if (e == 31u) mag = m ? NAN : INFINITY;
    else if (e == 0) mag = ldexp((double)m, -24);
    else mag = ldexp(1.0 + (double)m / 1024.0, (int)e - 15);
    return s ? -mag : mag;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 mantissa bits. */
double orc_bf16(unsigned bits)
{
    unsigned s = (bits >> 15) & 1u, e = (bits >> 7) & 255u, m = bits & 127u;
    double mag;
    if (e == 255u) mag = m ? NAN : INFINITY;
    else if (e == 0) mag = ldexp((double)m, -133);
    else mag = ldexp(1.0 + (double)m / 128.0, (int)e - 127);
    return s ? -mag : mag;
}

/* Round an fp64 value to the nearest bfloat16 value, ties to even, in one
 * step (no intermediate fp32 rounding). A bf16 normal has 8 significant bits;
 * below 2^-126 the spacing is fixed at 2^-133. */
double orc_round_bf16(double v)
{
    if (isnan(v) || isinf(v) || v == 0.0) return v;
    int e;
    double a = fabs(v);
    (void)frexp(a, &e);                 /* a = f * 2^e, f in [0.5, 1) */
    int qexp = e - 8;
    if (qexp < -133) qexp = -133;
    double r = ldexp(nearbyint(ldexp(a, -qexp)), qexp);   /* ties-to-even */
    const double bf16_max = ldexp(255.0, 120);              /* (2 - 2^-7) * 2^127 */
    if (r > bf16_max) r = INFINITY;
    return v < 0 ? -r : r;
}

unsigned orc_bf16_bits(double v)
{
    double r = orc_round_bf16(v);
    if (isnan(r)) return 0x7FC0u;
    unsigned s = signbit(r) ? 0x8000u : 0u;
    double a = fabs(r);
    if (isinf(a)) return s | 0x7F80u;
    if (a == 0.0) return s;
    int e;
    double f = frexp(a, &e);            /* a = f * 2^e */
    int be = e - 1 + 127;               /* biased exponent of 1.xxx form */
    if (be <= 0) {                      /* subnormal: a = m * 2^-133 */
        return s | (unsigned)ldexp(a, 133);
    }
    unsigned mant = (unsigned)ldexp(f * 2.0 - 1.0, 7);
    return s | ((unsigned)be << 7) | mant;
}

/* ------------------------------------------------------------------------ */
/* weight decodes                                                           */
/* ------------------------------------------------------------------------ */

static inline unsigned nvfp4_code(const uint8_t* codes, int64_t K, int64_t n, int64_t k)
{
    uint8_t b = codes[n * (K / 2) + k / 2];
    return (k % 2 == 0) ? (b & 0x0Fu) : (b >> 4);
}

static inline double nvfp4_weight(const uint8_t* codes, const uint8_t* scales, double g,
                                  int64_t K, int64_t n, int64_t k)
{
    double c = orc_e2m1(nvfp4_code(codes, K, n, k));
    double s = orc_e4m3(scales[n * (K / 16) + k / 16]);
    return c * s * g;
}

static inline unsigned q45_code(const uint8_t* q_lo, const uint8_t* q_hi, int bits,
                                int64_t K, int64_t n, int64_t k)
{
    uint8_t b = q_lo[n * (K / 2) + k / 2];
    unsigned q = (k % 2 == 0) ? (b & 0x0Fu) : (b >> 4);
    if (bits == 5) {
        unsigned hb = (q_hi[n * (K / 8) + k / 8] >> (k % 8)) & 1u;
        q |= hb << 4;
    }
    return q;
}

static inline double q45_weight(const uint8_t* q_lo, const uint8_t* q_hi, const uint16_t* scale,
                                const uint16_t* mn, int bits, int64_t K, int64_t n, int64_t k)
{
    double q = (double)q45_code(q_lo, q_hi, bits, K, n, k);
    double s = orc_f16(scale[n * (K / 32) + k / 32]);
    double m = orc_f16(mn[n * (K / 32) + k / 32]);
    return s * q + m;
}

void orc_dequant_nvfp4(const uint8_t* codes, const uint8_t* scales, double g,
                       int64_t N, int64_t K, double* w)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = nvfp4_weight(codes, scales, g, K, n, k);
}

void orc_dequant_q45(const uint8_t* q_lo, const uint8_t* q_hi, const uint16_t* scale,
                     const uint16_t* mn, int bits, int64_t N, int64_t K, double* w)
{
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            w[n * K + k] = q45_weight(q_lo, q_hi, scale, mn, bits, K, n, k);
}

/* ------------------------------------------------------------------------ */
/* GEMV                                                                     */
/* ------------------------------------------------------------------------ */

/* y[m][n] = sum_k w[n][k] * x[m][k] (+ r[m][n]); absacc[m][n] = sum_k |w x|.
 * Rows [n0, n1) only. x, r are bf16 bit patterns; r may be NULL. */
void orc_gemv_nvfp4(const uint8_t* codes, const uint8_t* scales, double g,
                    const uint16_t* x, const uint16_t* r, int64_t M, int64_t N, int64_t K,
                    int64_t n0, int64_t n1, double* y, double* absacc)
{
    for (int64_t n = n0; n < n1; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = nvfp4_weight(codes, scales, g, K, n, k) * orc_bf16(x[m * K + k]);
                acc += t;
                aacc += fabs(t);
            }
            if (r) acc += orc_bf16(r[m * N + n]);
            y[m * N + n] = acc;
            if (absacc) absacc[m * N + n] = aacc;
        }
    }
}

void orc_gemv_q45(const uint8_t* q_lo, const uint8_t* q_hi, const uint16_t* scale,
                  const uint16_t* mn, int bits, const uint16_t* x, const uint16_t* r,
                  int64_t M, int64_t N, int64_t K, int64_t n0, int64_t n1,
                  double* y, double* absacc)
{
    for (int64_t n = n0; n < n1; ++n) {
        for (int64_t m = 0; m < M; ++m) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double t = q45_weight(q_lo, q_hi, scale, mn, bits, K, n, k) * orc_bf16(x[m * K + k]);
                acc += t;
                aacc += fabs(t);
            }
            if (r) acc += orc_bf16(r[m * N + n]);
            y[m * N + n] = acc;
            if (absacc) absacc[m * N + n] = aacc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* epilogues                                                                */
/* ------------------------------------------------------------------------ */

/* SiLU (Swish-1): silu(v) = v * sigmoid(v) = v / (1 + e^-v). */
double orc_silu(double v)
{
    return v / (1.0 + exp(-v));
}

/* SwiGLU epilogue: out[i] = silu(gate[i]) * up[i]. */
void orc_swiglu(const double* gate, const double* up, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_silu(gate[i]) * up[i];
}

/* RMSNorm, the normalisation that decode engines fuse ahead of a projection
 * (NInfer article, section 2: normalisation and matmul in one read and one
 * write). For each token m, with a plain sequential fp64 sum in k order:
 *   r_m   = 1 / sqrt( (sum_k x_mk^2) / K + eps )
 *   v_mk  = x_mk * r_m * gamma_k
 *   h_mk  = bf16_rne(v_mk)      -- the bf16 activation the projection reads
 * The pages give no formula; this is the standard RMSNorm with a weight
 * vector gamma, and h is a bf16 activation as between any two layers. */
void orc_rmsnorm(const uint16_t* x, const uint16_t* gamma, double eps, int64_t M, int64_t K,
                 double* r, double* v, uint16_t* h)
{
    for (int64_t m = 0; m < M; ++m) {
        double ss = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double xv = orc_bf16(x[m * K + k]);
            ss += xv * xv;
        }
        const double rm = 1.0 / sqrt(ss / (double)K + eps);
        r[m] = rm;
        for (int64_t k = 0; k < K; ++k) {
            const double vk = orc_bf16(x[m * K + k]) * rm * orc_bf16(gamma[k]);
            v[m * K + k] = vk;
            h[m * K + k] = (uint16_t)orc_bf16_bits(vk);
        }
    }
}

void orc_round_bf16_array(const double* v, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_round_bf16(v[i]);
}

void orc_bf16_bits_array(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = (uint16_t)orc_bf16_bits(v[i]);
}

void orc_bf16_array(const uint16_t* bits, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_bf16(bits[i]);
}

void orc_f16_array(const uint16_t* bits, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_f16(bits[i]);
}

void orc_e4m3_array(const uint8_t* codes, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; ++i) out[i] = orc_e4m3(codes[i]);
}

/* ------------------------------------------------------------------------ */
/* MoE                                                                      */
/* ------------------------------------------------------------------------ */

/* Router: p = softmax(logits[m]) over E experts; the topk largest p (ties to
 * the lower expert id) in descending order; w = p_top / sum(p_top). */
void orc_route_topk(const float* logits, int64_t M, int64_t E, int topk,
                    int32_t* ids, double* w)
{
    double* p = (double*)malloc(sizeof(double) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    for (int64_t m = 0; m < M; ++m) {
        const float* l = logits + m * E;
        double mx = -INFINITY, z = 0.0;
        for (int64_t e = 0; e < E; ++e) if ((double)l[e] > mx) mx = (double)l[e];
        for (int64_t e = 0; e < E; ++e) { p[e] = exp((double)l[e] - mx); z += p[e]; }
        for (int64_t e = 0; e < E; ++e) p[e] /= z;
        memset(taken, 0, (size_t)E);
        double sel = 0.0;
        for (int i = 0; i < topk; ++i) {
            int64_t best = -1;
            for (int64_t e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || p[e] > p[best]) best = e;   /* strict: ties keep lower id */
            }
            taken[best] = 1;
            ids[m * topk + i] = (int32_t)best;
            w[m * topk + i] = p[best];
            sel += p[best];
        }
        for (int i = 0; i < topk; ++i) w[m * topk + i] /= sel;
    }
    free(p);
    free(taken);
}

/* First MoE stage for the (token, slot) pairs [p0, p1) of an M x topk
 * routing: e = ids[pair]; gate = G_e x_m, up = U_e x_m (rows [0, I) and
 * [I, 2I) of expert e's gate/up weights); h = bf16_RNE(silu(gate) * up).
 * Outputs per pair: gate, up, |gate|-sum, |up|-sum (each [I]) and h bits. */
void orc_moe_gate_up(const uint8_t* gu_codes, const uint8_t* gu_scales, const double* gu_g,
                     const uint16_t* x, const int32_t* ids, int64_t H, int64_t I, int topk,
                     int64_t p0, int64_t p1, double* gate, double* up,
                     double* abs_gate, double* abs_up, uint16_t* h_bits)
{
    const int64_t rows = 2 * I;
    for (int64_t pr = p0; pr < p1; ++pr) {
        int64_t m = pr / topk;
        int64_t e = ids[pr];
        const uint8_t* c = gu_codes + e * rows * (H / 2);
        const uint8_t* s = gu_scales + e * rows * (H / 16);
        for (int64_t i = 0; i < rows; ++i) {
            double acc = 0.0, aacc = 0.0;
            for (int64_t k = 0; k < H; ++k) {
                double t = nvfp4_weight(c, s, gu_g[e], H, i, k) * orc_bf16(x[m * H + k]);
                acc += t;
                aacc += fabs(t);
            }
            if (i < I) { gate[pr * I + i] = acc; abs_gate[pr * I + i] = aacc; }
            else { up[pr * I + (i - I)] = acc; abs_up[pr * I + (i - I)] = aacc; }
        }
        for (int64_t i = 0; i < I; ++i)
            h_bits[pr * I + i] = (uint16_t)orc_bf16_bits(orc_silu(gate[pr * I + i]) * up[pr * I + i]);
    }
}

/* Second MoE stage, output rows [j0, j1): for each token m,
 * y[m][j] = sum_{i < topk} c_i * sum_q f(d_{e_i}[j][q]) * v[m][i][q]
 * with c_i = w[m][i] and f = identity when use_abs == 0, and
 * c_i = |w[m][i]|, f = |.| when use_abs != 0 (used for error bounds).
 * Slots are combined in slot order i = 0, 1, ... */
void orc_moe_down(const uint8_t* dn_codes, const uint8_t* dn_scales, const double* dn_g,
                  const double* v, const int32_t* ids, const double* w,
                  int64_t M, int64_t H, int64_t I, int topk, int use_abs,
                  int64_t j0, int64_t j1, double* y)
{
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t j = j0; j < j1; ++j) {
            double acc = 0.0;
            for (int i = 0; i < topk; ++i) {
                int64_t e = ids[m * topk + i];
                const uint8_t* c = dn_codes + e * H * (I / 2);
                const uint8_t* s = dn_scales + e * H * (I / 16);
                const double* vv = v + (m * topk + i) * I;
                double d = 0.0;
                for (int64_t q = 0; q < I; ++q) {
                    double wt = nvfp4_weight(c, s, dn_g[e], I, j, q);
                    d += (use_abs ? fabs(wt) : wt) * vv[q];
                }
                double ci = w[m * topk + i];
                acc += (use_abs ? fabs(ci) : ci) * d;
            }
            y[m * H + j] = acc;
        }
    }
}

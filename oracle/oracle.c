/*
 * oracle.c -- CPU reference of the W8A8 block-FP8 linear path.
 * TEST INFRASTRUCTURE ONLY (see oracle.h): used by tests, the smoke check and
 * the benchmark's CPU-baseline leg; never by the product path.
 *
 * Written as plain C11, single-threaded, fp64 where the method does not fix a
 * precision.  Compile with -ffp-contract=off so no multiply-add is fused.
 */
#include "oracle.h"

#include <math.h>
#include <string.h>

/* ---------------------------------------------------------------- codecs -- */

/* E4M3 (OCP 8-bit floating point, E4M3 variant): value of a code.
 *   exponent field e (4 bits), mantissa field f (3 bits), bias 7
 *   e == 0          : subnormal, f/8 * 2^(1-7)
 *   e in 1..15      : (1 + f/8) * 2^(e-7), except e == 15 && f == 7 -> NaN
 */
double oracle_e4m3_decode(uint8_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int f = code & 0x7;
    double v;
    if (e == 0xF && f == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)f / 8.0, 1 - 7);
    else
        v = ldexp(1.0 + (double)f / 8.0, e - 7);
    return sign ? -v : v;
}

/* Round-to-nearest, ties-to-even, onto the E4M3 grid.  Input finite with
 * |y| <= 448 (the caller clamps).  Works in double, where every step below
 * (scaling by a power of two, rint) is exact. */
uint8_t oracle_e4m3_encode(float y) {
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: grid step 2^-9; count steps, round half-even.
         * A result of 8 steps is exactly the smallest normal, code 0x08. */
        double steps = rint(a / ldexp(1.0, -9)); /* default rounding: half-even */
        return (uint8_t)(sign | (uint8_t)steps);
    }
    int ex; /* a = fr * 2^ex with fr in [0.5, 1) */
    (void)frexp(a, &ex);
    int e_unb = ex - 1;                         /* a in [2^e_unb, 2^(e_unb+1)) */
    double steps = rint(a / ldexp(1.0, e_unb - 3)); /* in [8, 16] */
    if (steps == 16.0) { steps = 8.0; e_unb += 1; }
    int efield = e_unb + 7;
    int ffield = (int)steps - 8;
    return (uint8_t)(sign | (uint8_t)(efield << 3) | (uint8_t)ffield);
}

float oracle_bf16_to_f32(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16; /* bf16 is the top half of an fp32 */
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
float oracle_f16_to_f32(uint16_t bits) {
    int sign = (bits >> 15) & 1;
    int e = (bits >> 10) & 0x1F;
    int f = bits & 0x3FF;
    double v;
    if (e == 0x1F)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, -24);
    else
        v = ldexp(1.0 + (double)f / 1024.0, e - 15);
    return (float)(sign ? -v : v); /* exact: every binary16 value is an fp32 */
}

static float load_elem(const void* base, int dtype, int64_t idx) {
    if (dtype == ORACLE_FP32) return ((const float*)base)[idx];
    uint16_t b = ((const uint16_t*)base)[idx];
    return dtype == ORACLE_BF16 ? oracle_bf16_to_f32(b) : oracle_f16_to_f32(b);
}

/* -------------------------------------------------------------- scales -- */

static const float kEps = 1e-10f;   /* reading: eps = 1e-10 */
static const float kFp8Max = 448.0f; /* largest finite E4M3 value */

float oracle_group_scale(float amax, int ue8m0) {
    float m = amax > kEps ? amax : kEps;
    float s = m / kFp8Max; /* fp32 IEEE division */
    if (ue8m0) {
        /* 2^ceil(log2 s): a positive normal fp32 is 2^(E-127) * 1.f; it is
         * already a power of two iff f == 0, otherwise the next one up is
         * 2^(E-127+1). */
        uint32_t u;
        memcpy(&u, &s, 4);
        uint32_t E = (u >> 23) & 0xFF;
        uint32_t f = u & 0x7FFFFF;
        if (f != 0) E += 1;
        u = E << 23;
        memcpy(&s, &u, 4);
    }
    return s;
}

uint8_t oracle_quant_value(float x, float s) {
    float y = x / s; /* fp32 IEEE division */
    if (y > kFp8Max) y = kFp8Max;
    if (y < -kFp8Max) y = -kFp8Max;
    return oracle_e4m3_encode(y);
}

static int64_t pad4(int64_t m) { return (m + 3) / 4 * 4; }

int64_t oracle_act_scale_bytes(int64_t M, int64_t K, int group, int ue8m0) {
    if (M < 0 || K < 0 || group <= 0 || K % group) return -1;
    int64_t G = K / group;
    int64_t cols = ue8m0 ? (G + 3) / 4 : G;
    return 4 * cols * pad4(M);
}

/* ------------------------------------------------------- activation quant -- */

int oracle_quant_act(const uint16_t* x, int x_dtype, int64_t M, int64_t K, int group,
                     int ue8m0, uint8_t* q, void* s) {
    if (M < 0 || K < 0 || group <= 0 || K % group) return -1;
    if (x_dtype != ORACLE_BF16 && x_dtype != ORACLE_FP16) return -1;
    int64_t G = K / group, Mp = pad4(M);
    memset(s, 0, (size_t)oracle_act_scale_bytes(M, K, group, ue8m0));
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < G; ++g) {
            const int64_t base = m * K + g * group;
            float amax = 0.0f;
            for (int64_t i = 0; i < group; ++i) {
                float v = fabsf(load_elem(x, x_dtype, base + i));
                if (v > amax) amax = v;
            }
            float sc = oracle_group_scale(amax, ue8m0);
            for (int64_t i = 0; i < group; ++i)
                q[base + i] = oracle_quant_value(load_elem(x, x_dtype, base + i), sc);
            if (ue8m0) {
                uint32_t u;
                memcpy(&u, &sc, 4);
                uint32_t* w = (uint32_t*)s + (g / 4) * Mp + m;
                *w |= ((u >> 23) & 0xFFu) << (8 * (g % 4)); /* byte g%4 = biased exponent */
            } else {
                ((float*)s)[g * Mp + m] = sc;
            }
        }
    }
    return 0;
}

/* ----------------------------------------------------------- weight quant -- */

int oracle_quant_weight(const void* w, int w_dtype, int64_t N, int64_t K, int bn, int bk,
                        int ue8m0, uint8_t* q, float* s) {
    if (N < 0 || K < 0 || bn <= 0 || bk <= 0 || K % bk) return -1;
    if (w_dtype != ORACLE_FP32 && w_dtype != ORACLE_BF16 && w_dtype != ORACLE_FP16) return -1;
    int64_t NB = (N + bn - 1) / bn, KB = K / bk;
    for (int64_t nb = 0; nb < NB; ++nb) {
        int64_t n0 = nb * bn, n1 = n0 + bn < N ? n0 + bn : N;
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = kb * bk; k < (kb + 1) * bk; ++k) {
                    float v = fabsf(load_elem(w, w_dtype, n * K + k));
                    if (v > amax) amax = v;
                }
            float sc = oracle_group_scale(amax, ue8m0);
            s[nb * KB + kb] = sc;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = kb * bk; k < (kb + 1) * bk; ++k)
                    q[n * K + k] = oracle_quant_value(load_elem(w, w_dtype, n * K + k), sc);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------ GEMM -- */

double oracle_act_scale(const void* s, int ue8m0, int64_t M, int64_t K, int group,
                        int64_t m, int64_t g) {
    (void)K;
    (void)group;
    int64_t Mp = pad4(M);
    if (ue8m0) {
        uint32_t w = ((const uint32_t*)s)[(g / 4) * Mp + m];
        int byte = (int)((w >> (8 * (g % 4))) & 0xFF);
        return ldexp(1.0, byte - 127);
    }
    return (double)((const float*)s)[g * Mp + m];
}

static double dec_table[256];
static int dec_table_ready = 0;

static void init_dec_table(void) {
    if (dec_table_ready) return;
    for (int c = 0; c < 256; ++c) dec_table[c] = oracle_e4m3_decode((uint8_t)c);
    dec_table_ready = 1;
}

static double gemm_one(int64_t M, int64_t N, int64_t K, const uint8_t* qa, const void* sa,
                       int ue8m0, const uint8_t* qw, const float* sw, int group, int bn, int bk,
                       int64_t m, int64_t n) {
    (void)N;
    int64_t G = K / bk;
    double acc = 0.0;
    for (int64_t kb = 0; kb < G; ++kb) {
        double slab = 0.0; /* exact: <= 128 products of 4-bit significands */
        for (int64_t k = kb * bk; k < (kb + 1) * bk; ++k)
            slab += dec_table[qa[m * K + k]] * dec_table[qw[n * K + k]];
        double scale = oracle_act_scale(sa, ue8m0, M, K, group, m, kb) *
                       (double)sw[(n / bn) * G + kb];
        acc += slab * scale;
    }
    return acc;
}

static int gemm_args_ok(int64_t M, int64_t N, int64_t K, int group, int bn, int bk) {
    return M >= 0 && N >= 0 && K > 0 && group == bk && bn > 0 && bk > 0 && K % bk == 0;
}

int oracle_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* qa, const void* sa, int ue8m0,
                const uint8_t* qw, const float* sw, int group, int bn, int bk,
                int64_t row0, int64_t rows, double* out) {
    if (!gemm_args_ok(M, N, K, group, bn, bk) || row0 < 0 || rows < 0 || row0 + rows > M)
        return -1;
    init_dec_table();
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t n = 0; n < N; ++n)
            out[r * N + n] = gemm_one(M, N, K, qa, sa, ue8m0, qw, sw, group, bn, bk, row0 + r, n);
    return 0;
}

double oracle_gemm_elem(int64_t M, int64_t N, int64_t K, const uint8_t* qa, const void* sa,
                        int ue8m0, const uint8_t* qw, const float* sw, int group, int bn, int bk,
                        int64_t m, int64_t n) {
    if (!gemm_args_ok(M, N, K, group, bn, bk) || m < 0 || m >= M || n < 0 || n >= N) return NAN;
    init_dec_table();
    return gemm_one(M, N, K, qa, sa, ue8m0, qw, sw, group, bn, bk, m, n);
}

/* --------------------------------------------- per-token x per-channel -- */

static const float kInt8Max = 127.0f; /* symmetric int8 range */

int8_t oracle_int8_value(float x, float s) {
    float y = x / s; /* fp32 IEEE division */
    if (y > kInt8Max) y = kInt8Max;
    if (y < -kInt8Max) y = -kInt8Max;
    return (int8_t)rintf(y); /* default rounding mode: half to even */
}

int oracle_quant_rows(const void* x, int x_dtype, int64_t R, int64_t K, int int8, uint8_t* q,
                      float* s) {
    if (R < 0 || K <= 0) return -1;
    if (x_dtype != ORACLE_FP32 && x_dtype != ORACLE_BF16 && x_dtype != ORACLE_FP16) return -1;
    for (int64_t r = 0; r < R; ++r) {
        float amax = 0.0f;
        for (int64_t k = 0; k < K; ++k) {
            float v = fabsf(load_elem(x, x_dtype, r * K + k));
            if (v > amax) amax = v;
        }
        float m = amax > kEps ? amax : kEps;
        float sc = m / (int8 ? kInt8Max : kFp8Max); /* fp32 IEEE division */
        s[r] = sc;
        for (int64_t k = 0; k < K; ++k) {
            float v = load_elem(x, x_dtype, r * K + k);
            q[r * K + k] = int8 ? (uint8_t)oracle_int8_value(v, sc) : oracle_quant_value(v, sc);
        }
    }
    return 0;
}

int oracle_gemm_rowcol(int64_t M, int64_t N, int64_t K, const uint8_t* qa, const float* sa,
                       const uint8_t* qw, const float* sw, int int8, int64_t row0, int64_t rows,
                       double* out) {
    if (M < 0 || N < 0 || K <= 0 || row0 < 0 || rows < 0 || row0 + rows > M) return -1;
    init_dec_table();
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t m = row0 + r;
        for (int64_t n = 0; n < N; ++n) {
            double S;
            if (int8) {
                int64_t acc = 0;
                for (int64_t k = 0; k < K; ++k)
                    acc += (int64_t)(int8_t)qa[m * K + k] * (int64_t)(int8_t)qw[n * K + k];
                S = (double)acc; /* |acc| <= K * 127^2 < 2^53 */
            } else {
                S = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    S += dec_table[qa[m * K + k]] * dec_table[qw[n * K + k]];
            }
            out[r * N + n] = ((double)sa[m] * (double)sw[n]) * S;
        }
    }
    return 0;
}

/* ------------------------------------------------------------ block INT8 -- */

int oracle_quant_act_int8(const uint16_t* x, int x_dtype, int64_t M, int64_t K, int group,
                          int8_t* q, float* s) {
    if (M < 0 || K < 0 || group <= 0 || K % group) return -1;
    if (x_dtype != ORACLE_BF16 && x_dtype != ORACLE_FP16) return -1;
    int64_t G = K / group, Mp = pad4(M);
    memset(s, 0, (size_t)(4 * G * Mp));
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t g = 0; g < G; ++g) {
            const int64_t base = m * K + g * group;
            float amax = 0.0f;
            for (int64_t i = 0; i < group; ++i) {
                float v = fabsf(load_elem(x, x_dtype, base + i));
                if (v > amax) amax = v;
            }
            float mx = amax > kEps ? amax : kEps;
            float sc = mx / kInt8Max; /* fp32 IEEE division */
            for (int64_t i = 0; i < group; ++i)
                q[base + i] = oracle_int8_value(load_elem(x, x_dtype, base + i), sc);
            s[g * Mp + m] = sc;
        }
    }
    return 0;
}

int oracle_quant_weight_int8(const void* w, int w_dtype, int64_t N, int64_t K, int bn, int bk,
                             int8_t* q, float* s) {
    if (N < 0 || K < 0 || bn <= 0 || bk <= 0 || K % bk) return -1;
    if (w_dtype != ORACLE_FP32 && w_dtype != ORACLE_BF16 && w_dtype != ORACLE_FP16) return -1;
    int64_t NB = (N + bn - 1) / bn, KB = K / bk;
    for (int64_t nb = 0; nb < NB; ++nb) {
        int64_t n0 = nb * bn, n1 = n0 + bn < N ? n0 + bn : N;
        for (int64_t kb = 0; kb < KB; ++kb) {
            float amax = 0.0f;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = kb * bk; k < (kb + 1) * bk; ++k) {
                    float v = fabsf(load_elem(w, w_dtype, n * K + k));
                    if (v > amax) amax = v;
                }
            float mx = amax > kEps ? amax : kEps;
            float sc = mx / kInt8Max; /* fp32 IEEE division */
            s[nb * KB + kb] = sc;
            for (int64_t n = n0; n < n1; ++n)
                for (int64_t k = kb * bk; k < (kb + 1) * bk; ++k)
                    q[n * K + k] = oracle_int8_value(load_elem(w, w_dtype, n * K + k), sc);
        }
    }
    return 0;
}

int oracle_gemm_int8_block(int64_t M, int64_t N, int64_t K, const int8_t* qa, const float* sa,
                           const int8_t* qw, const float* sw, int group, int bn, int bk,
                           int64_t row0, int64_t rows, double* out) {
    if (!gemm_args_ok(M, N, K, group, bn, bk) || row0 < 0 || rows < 0 || row0 + rows > M)
        return -1;
    const int64_t G = K / bk, Mp = pad4(M);
    for (int64_t r = 0; r < rows; ++r) {
        const int64_t m = row0 + r;
        for (int64_t n = 0; n < N; ++n) {
            double acc = 0.0;
            for (int64_t kb = 0; kb < G; ++kb) {
                int64_t S = 0; /* exact */
                for (int64_t k = kb * bk; k < (kb + 1) * bk; ++k)
                    S += (int64_t)qa[m * K + k] * (int64_t)qw[n * K + k];
                acc += ((double)sa[kb * Mp + m] * (double)sw[(n / bn) * G + kb]) * (double)S;
            }
            out[r * N + n] = acc;
        }
    }
    return 0;
}

/* -------------------------------------------------------------- calc_diff -- */

double oracle_calc_diff(const double* x, const double* y, int64_t n) {
    double xy = 0.0, den = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        xy += x[i] * y[i];
        den += x[i] * x[i] + y[i] * y[i];
    }
    return 1.0 - 2.0 * xy / den;
}

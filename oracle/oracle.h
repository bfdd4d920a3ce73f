/*
 * oracle.h -- plain, slow, single-threaded CPU reference of the W8A8 block-FP8
 * linear path (per-token-group activation quant, 128x128 weight block quant,
 * block-scaled GEMM accumulated in fp64).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this code; only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or constant generator with
 * the CUDA path.
 *
 * Sources (web pages; cited by title and section):
 *   [DG]  "vLLM DeepGEMM FP8 Block GEMM 基准测试：DeepSeek DeepGEMM 对比 Triton 与
 *          CUTLASS 的块量化 GEMM 内核解析" (blog.gitcode.com), §4.1 (quant layouts:
 *          per_block_cast_to_fp8, per_token_group_quant_fp8), §4.2 (the Triton
 *          kernel's per-K-block scale multiply), §4.3 (metrics), §4.4 (calc_diff).
 *   [PR]  "vllm-project/vllm PR 42153" (prhub.com.cn), 实现拆解 (the packed
 *          UE8M0 per-token-group quant kernel: eps, min/max 8-bit bounds,
 *          packed int32 scales, TMA-aligned rows).
 *   [CFG] "vLLM 量化 Kernel 配置机制" (blog.gitcode.com), §2 (M grid).
 * Readings of points the pages leave open (eps = 1e-10, fp8 max = 448,
 * IEEE division x/s, ceil on the fp32-rounded scale, biased-exponent UE8M0
 * byte, little-endian packing, zero padding) are listed in the design notes;
 * each function below states the one it uses.
 *
 * Parity status: every function here is pinned by tests under tests/ that do
 * not call the function's own formula (brute force, exact rationals, closed
 * forms, invariants, library special cases).  calc_diff is pinned only by its
 * closed-form special cases; the pages' printed 0.000684 depends on their RNG
 * and is not reproducible (parity unpinned for that one number).
 */
#ifndef FP8BQ_ORACLE_H
#define FP8BQ_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* dtype codes for raw 16/32-bit inputs */
enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1, ORACLE_FP32 = 2 };

/* OCP FP8 E4M3 ("e4m3fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits, no
 * infinities, S.1111.111 is NaN, largest finite 448.  decode() returns the
 * exact value (NaN for 0x7F/0xFF). */
double oracle_e4m3_decode(uint8_t code);
/* Round-to-nearest-even of a finite fp32 value with |y| <= 448 (callers clamp
 * first, see oracle_quant_value); the sign of zero is kept (-0 -> 0x80). */
uint8_t oracle_e4m3_encode(float y);

float oracle_bf16_to_f32(uint16_t bits);
float oracle_f16_to_f32(uint16_t bits);

/* Scale of one group/block from its amax: s = fp32(max(amax, 1e-10) / 448);
 * with ue8m0 != 0, s is rounded up to the next power of two (2^ceil(log2 s)),
 * computed on the fp32 bits of s.  [DG §4.1], [PR 实现拆解]. */
float oracle_group_scale(float amax, int ue8m0);
/* code of one element: e4m3_rne(clamp(fp32(x / s), -448, 448)). */
uint8_t oracle_quant_value(float x, float s);

/* Bytes of the activation-scale buffer: Mp = ceil(M/4)*4 rows;
 * fp32: 4*G*Mp; ue8m0 packed: 4*ceil(G/4)*Mp.  G = K/group. */
int64_t oracle_act_scale_bytes(int64_t M, int64_t K, int group, int ue8m0);

/* Per-token-group activation quant.  x: [M,K] row-major bf16/fp16 bits.
 * q: [M,K] e4m3 codes.  s: column-major scales, element (g, m) at g*Mp + m
 * (fp32 mode) or byte (g%4) of u32 word (g/4)*Mp + m (ue8m0 mode; byte =
 * biased fp32 exponent of the power-of-two scale).  Rows m in [M, Mp) and
 * unused bytes of the last word are 0.  Returns 0, or -1 on bad arguments. */
int oracle_quant_act(const uint16_t* x, int x_dtype, int64_t M, int64_t K, int group,
                     int ue8m0, uint8_t* q, void* s);

/* 128x128 weight block quant.  w: [N,K] row-major (fp32, bf16 or fp16).
 * q: [N,K] codes; s: fp32 [ceil(N/bn)][K/bk] row-major.  A partial last row
 * block takes its amax over the rows that exist.  [DG §4.1] */
int oracle_quant_weight(const void* w, int w_dtype, int64_t N, int64_t K, int bn, int bk,
                        int ue8m0, uint8_t* q, float* s);

/* Activation scale (m, g) decoded to a double (fp32 value or 2^(byte-127)). */
double oracle_act_scale(const void* s, int ue8m0, int64_t M, int64_t K, int group,
                        int64_t m, int64_t g);

/* Block-scaled GEMM, exact-in-fp64 slab sums:
 *   ref[m,n] = sum_kb sa[m,kb] * sw[n/bn,kb] * S_kb,
 *   S_kb     = sum_{k in slab kb} dec(qa[m,k]) * dec(qw[n,k])
 * accumulated in fp64 in the order kb = 0..G-1 ([DG §4.2]: each K block's
 * dot product is multiplied by the two scales and added to the accumulator).
 * Rows [row0, row0+rows) of the [M,N] result are written to out (rows x N). */
int oracle_gemm(int64_t M, int64_t N, int64_t K, const uint8_t* qa, const void* sa, int ue8m0,
                const uint8_t* qw, const float* sw, int group, int bn, int bk,
                int64_t row0, int64_t rows, double* out);
/* One element of the same result. */
double oracle_gemm_elem(int64_t M, int64_t N, int64_t K, const uint8_t* qa, const void* sa,
                        int ue8m0, const uint8_t* qw, const float* sw, int group, int bn, int bk,
                        int64_t m, int64_t n);

/* ------------------------------------------------------------------------
 * Per-token x per-channel formats.  [HL] ("用 Helion 为 vLLM 构建高性能可移植
 * 线性后端", 范围) lists, beside Block_FP8, FP8_Dynamic (FP8 codes, one scale
 * per activation token and one per weight output channel) and W8A8_INT8 (the
 * same scaling with INT8 codes).  The pages give no formula for them; the
 * readings taken are the block path's with the block widened to a whole row:
 *   e4m3: s = fp32(max(amax_row, 1e-10) / 448), q = e4m3_rne(clamp(x/s, +-448))
 *   int8: s = fp32(max(amax_row, 1e-10) / 127), q = rne(clamp(x/s, +-127))
 * x/s is the IEEE fp32 division, rne rounds half to even, int8 is symmetric
 * (-128 is never produced).
 * ------------------------------------------------------------------------ */

/* One scale per row of x [R,K] (fp32, bf16 or fp16): per-token activation
 * scales, or per-channel weight scales when x is a weight [N,K].
 * q: [R,K] codes (e4m3, or int8 two's complement when int8 != 0); s: fp32 [R].
 * Returns 0, or -1 on bad arguments. */
int oracle_quant_rows(const void* x, int x_dtype, int64_t R, int64_t K, int int8, uint8_t* q,
                      float* s);
/* The int8 code of one element with scale s: rne(clamp(fp32(x / s), -127, 127)). */
int8_t oracle_int8_value(float x, float s);

/* Per-token x per-channel GEMM, rows [row0, row0+rows) of
 *   ref[m,n] = (sa[m] * sw[n]) * S[m,n],   S[m,n] = sum_k dec(qa[m,k]) * dec(qw[n,k])
 * (dec = e4m3 value, or the int8 integer).  S is exact in fp64 for the sizes
 * used (e4m3 products are multiples of 2^-18 below 2^18, so a K <= 2^16 sum
 * needs at most 52 bits; int8 sums are accumulated in int64), sa*sw is exact
 * (two fp32 significands), so ref is the correctly rounded value of the exact
 * product.  [HL] 内核实现: the quantised kernels apply the scales after the
 * matmul's dot product. */
int oracle_gemm_rowcol(int64_t M, int64_t N, int64_t K, const uint8_t* qa, const float* sa,
                       const uint8_t* qw, const float* sw, int int8, int64_t row0, int64_t rows,
                       double* out);

/* ------------------------------------------------------------------------
 * Block INT8 ("vLLM 量化 Kernel 配置机制" §1: int8_w8a8 tables with
 * block_shape [128,128], the block-quantised path of GPUs without FP8 tensor
 * cores).  The page gives the layout but no formula; the reading taken is the
 * block FP8 path's with int8 codes: per 1 x group activation group and per
 * bn x bk weight block,
 *   s = fp32(max(amax, 1e-10) / 127),  q = rne(clamp(fp32(x / s), -127, 127))
 * (fp32 scales only), and the GEMM promotes every K slab's exact integer sum:
 *   ref[m,n] = sum_kb sa[m,kb] * sw[n/bn,kb] * S_kb,
 *   S_kb = sum_{k in slab kb} qa[m,k] * qw[n,k]     (int64, exact)
 * accumulated in fp64 in the order kb = 0..G-1.
 * ------------------------------------------------------------------------ */

/* Activation quant with int8 codes: x [M,K] bf16/fp16 bits; q [M,K] int8;
 * s fp32 column-major [G][Mp] (Mp = ceil(M/4)*4, padding rows 0), as the
 * fp32 mode of oracle_quant_act. */
int oracle_quant_act_int8(const uint16_t* x, int x_dtype, int64_t M, int64_t K, int group,
                          int8_t* q, float* s);
/* Weight block quant with int8 codes: w [N,K] fp32/bf16/fp16; q [N,K] int8;
 * s fp32 [ceil(N/bn)][K/bk]. */
int oracle_quant_weight_int8(const void* w, int w_dtype, int64_t N, int64_t K, int bn, int bk,
                             int8_t* q, float* s);
/* Rows [row0, row0+rows) of the block INT8 GEMM above (sa as written by
 * oracle_quant_act_int8, sw by oracle_quant_weight_int8). */
int oracle_gemm_int8_block(int64_t M, int64_t N, int64_t K, const int8_t* qa, const float* sa,
                           const int8_t* qw, const float* sw, int group, int bn, int bk,
                           int64_t row0, int64_t rows, double* out);

/* calc_diff of [DG §4.4]: 1 - 2*sum(x*y) / sum(x*x + y*y), in fp64. */
double oracle_calc_diff(const double* x, const double* y, int64_t n);

#ifdef __cplusplus
}
#endif
#endif

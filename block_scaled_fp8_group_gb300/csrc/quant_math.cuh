// quant_math.cuh -- the per-group quantisation arithmetic, shared by the
// standalone quant kernels (quant.cu) and the GEMM that quantises its own
// activation tiles (gemm.cu), so both produce the same codes and scales.
//
// "vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.1: s = max(amax, eps) / fp8_max,
// rounded up to a power of two for UE8M0; codes = e4m3 RNE of clamp(x/s, +-448).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "internal.h"

namespace fp8bq {

// Power-of-two round-up of a positive normal fp32 scale, on its bits.
__device__ __forceinline__ float ceil_pow2(float s) {
    uint32_t u = __float_as_uint(s);
    uint32_t e = (u >> 23) & 0xFFu;
    if (u & 0x7FFFFFu) e += 1u;
    return __uint_as_float(e << 23);
}

__device__ __forceinline__ float group_scale(float amax, int ue8m0) {
    float s = __fdiv_rn(fmaxf(amax, kEps), kFp8Max);
    return ue8m0 ? ceil_pow2(s) : s;
}

// Two fp32 values -> two e4m3 codes (low byte = first), saturating RNE.
__device__ __forceinline__ uint32_t cvt2_e4m3(float a, float b) {
    a = fminf(fmaxf(a, -kFp8Max), kFp8Max);
    b = fminf(fmaxf(b, -kFp8Max), kFp8Max);
    return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE,
                                                          __NV_E4M3));
}

// fp32(x / s) for an activation value x (bf16 or fp16: at most 11 significant
// bits) and its group or row scale s = fp32(max(amax, eps) / Q) (amax of the
// same format, Q = 448 or 127), from r = fp32(1 / s): the product
// q0 = fp32(x * r), its exact residual x - q0 * s (one FMA) and one
// correction fp32(q0 + residual * r) -- the division step of P. Markstein,
// "Computation of elementary functions on the IBM RISC System/6000
// processor", IBM J. Res. Develop. 34(1), 1990.  For every pair of input and
// scale significands these formats allow, the result is the correctly
// rounded quotient (the scaling by powers of two commutes with each step
// while the values stay normal, and quotients below 2^-126 give a zero code
// either way); a zero quotient takes the sign of x, as the division gives it.
// It costs three FP operations where the IEEE division needs a reciprocal
// iteration and a range check per value.
__device__ __forceinline__ float act_quotient(float x, float s, float r) {
    const float q0 = __fmul_rn(x, r);
    const float e = __fmaf_rn(-q0, s, x);
    return copysignf(__fmaf_rn(e, r, q0), x);
}

// Four activation values -> four int8 codes, as cvt4_int8 with the quotient
// of act_quotient (r = fp32(1 / s)).
__device__ __forceinline__ uint32_t cvt4_int8_act(float a, float b, float c, float d, float s,
                                                  float r) {
    const float v[4] = {a, b, c, d};
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float y = fminf(fmaxf(act_quotient(v[j], s, r), -kInt8Max), kInt8Max);
        w |= (static_cast<uint32_t>(__float2int_rn(y)) & 0xFFu) << (8 * j);
    }
    return w;
}

// Four fp32 values -> four int8 codes (byte j = value j): round half to even
// of clamp(v / s, -127, 127), with the IEEE division.
__device__ __forceinline__ uint32_t cvt4_int8(float a, float b, float c, float d, float s) {
    const float v[4] = {a, b, c, d};
    uint32_t w = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const float y = fminf(fmaxf(__fdiv_rn(v[j], s), -kInt8Max), kInt8Max);
        w |= (static_cast<uint32_t>(__float2int_rn(y)) & 0xFFu) << (8 * j);
    }
    return w;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ float f16_lo(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w & 0xFFFFu)));
}
__device__ __forceinline__ float f16_hi(uint32_t w) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(w >> 16)));
}

}  // namespace fp8bq

// quant.cu -- per-token-group activation quant and 128x128 weight block quant.
//
// Method ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.1; "vllm-project/vllm PR
// 42153" 实现拆解): per group amax, s = max(amax, 1e-10)/448 (rounded up to a
// power of two for UE8M0), codes = e4m3 round-to-nearest-even of
// clamp(x/s, +-448).  Both kernels are HBM streams on the CUDA cores.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8bq {

namespace {

// -------------------------------------------------------- activation quant
//
// One warp owns 4 consecutive groups (512 elements, 1 KB of bf16) of one row:
// lane l holds elements [16 l, 16 l + 16) of that span, i.e. lanes 8j..8j+7
// hold group j.  The group amax is a 3-step xor shuffle inside those 8 lanes,
// and the 4 UE8M0 exponents of the warp form exactly one packed u32 word, so
// packing needs no traffic between warps.
//
// Grid without runtime division: blockIdx.x picks kRows rows (one per warp),
// blockIdx.y the 4-group column and, for grouped rows, blockIdx.z the expert
// (rows then counted within it); every index below is a product or sum of
// those with compile-time constants or kernel arguments.
constexpr int kQuantRows = 8;  // warps per CTA = rows per CTA

// Eight resident CTAs per SM (at most 32 registers a thread): the kernel is a
// load-latency-bound stream, and the full 64 warps keep more loads in flight
// than the 48 that 40 registers allow (16384 x 18432: 0.84 -> 0.89 of the
// measured copy bandwidth with UE8M0 scales, 0.78 -> 0.82 with fp32 scales).
template <bool kFp16, bool kGrouped>
__global__ void __launch_bounds__(kQuantRows * 32, 8) quant_act_kernel(const QuantActArgs a) {
    const int lane = threadIdx.x & 31;
    const int64_t wrow = static_cast<int64_t>(blockIdx.x) * kQuantRows + (threadIdx.x >> 5);
    const int64_t row = kGrouped ? static_cast<int64_t>(blockIdx.z) * a.m_max + wrow : wrow;
    const int quad = blockIdx.y;             // 4-group column index
    const int g = quad * 4 + (lane >> 3);    // this lane's group
    const bool active = row < a.M && g < a.G;

    // Programmatic dependent launch: wait for the previous kernel (it may
    // produce x or still read q/s), then let the next one start its set-up.
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    if (row >= a.Mp) return;
    if (kGrouped) {
        // grouped rows: skip the rows past the expert's count (warp-uniform)
        if (wrow >= a.m_max) return;
        const int c = __ldg(a.counts + blockIdx.z);
        if (wrow >= (c < 0 ? 0 : c)) return;
    }

    const int64_t off = row * a.K + static_cast<int64_t>(quad) * 512 + lane * 16;
    uint4 v0 = make_uint4(0, 0, 0, 0), v1 = make_uint4(0, 0, 0, 0);
    if (active) {
        const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(a.x) + off);
        v0 = __ldcs(src);
        v1 = __ldcs(src + 1);
    }
    float f[16];
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = kFp16 ? f16_lo(w[i]) : bf16_lo(w[i]);
        f[2 * i + 1] = kFp16 ? f16_hi(w[i]) : bf16_hi(w[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    const float s = a.int8 ? __fdiv_rn(fmaxf(amax, kEps), kInt8Max) : group_scale(amax, a.ue8m0);

    if (active && a.int8) {
        // block INT8: 16 int8 codes
        const float r = __fdiv_rn(1.0f, s);
        *reinterpret_cast<uint4*>(a.q + off) =
            make_uint4(cvt4_int8_act(f[0], f[1], f[2], f[3], s, r),
                       cvt4_int8_act(f[4], f[5], f[6], f[7], s, r),
                       cvt4_int8_act(f[8], f[9], f[10], f[11], s, r),
                       cvt4_int8_act(f[12], f[13], f[14], f[15], s, r));
    } else if (active) {
        uint32_t c[8];
        if (a.ue8m0) {
            // s = 2^e exactly, so x * (1/s) is the same correctly rounded
            // value as x / s.
            const float r = __fdiv_rn(1.0f, s);
#pragma unroll
            for (int i = 0; i < 8; ++i) c[i] = cvt2_e4m3(f[2 * i] * r, f[2 * i + 1] * r);
        } else {
            // fp32 scales: fp32(x / s) from the reciprocal and one residual
            // correction (act_quotient: exact for these inputs)
            const float r = __fdiv_rn(1.0f, s);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                c[i] = cvt2_e4m3(act_quotient(f[2 * i], s, r), act_quotient(f[2 * i + 1], s, r));
        }
        uint4 out;
        out.x = c[0] | (c[1] << 16);
        out.y = c[2] | (c[3] << 16);
        out.z = c[4] | (c[5] << 16);
        out.w = c[6] | (c[7] << 16);
        *reinterpret_cast<uint4*>(a.q + off) = out;
    }

    // Scales: padding rows (row >= M) and groups past G store 0.
    if (a.ue8m0) {
        const uint32_t byte = (row < a.M && g < a.G) ? ((__float_as_uint(s) >> 23) & 0xFFu) : 0u;
        const uint32_t b0 = __shfl_sync(0xFFFFFFFFu, byte, 0);
        const uint32_t b1 = __shfl_sync(0xFFFFFFFFu, byte, 8);
        const uint32_t b2 = __shfl_sync(0xFFFFFFFFu, byte, 16);
        const uint32_t b3 = __shfl_sync(0xFFFFFFFFu, byte, 24);
        if (lane == 0)
            static_cast<uint32_t*>(a.s)[static_cast<int64_t>(quad) * a.Mp + row] =
                b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    } else if ((lane & 7) == 0 && g < a.G) {
        static_cast<float*>(a.s)[static_cast<int64_t>(g) * a.Mp + row] = row < a.M ? s : 0.0f;
    }
}

// ------------------------------------------------------------ weight quant
//
// One CTA per 128x128 block; 256 threads, thread t covers columns
// 16*(t%8) .. +16 of rows t/8 + 32*i (i = 0..3).  The block amax is a warp
// shuffle reduction followed by a shared-memory one across the 8 warps.
template <typename T>
__device__ __forceinline__ void load16(const T* p, float (&f)[16]);

template <>
__device__ __forceinline__ void load16<float>(const float* p, float (&f)[16]) {
    const float4* s = reinterpret_cast<const float4*>(p);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float4 v = s[i];
        f[4 * i] = v.x;
        f[4 * i + 1] = v.y;
        f[4 * i + 2] = v.z;
        f[4 * i + 3] = v.w;
    }
}

template <>
__device__ __forceinline__ void load16<__nv_bfloat16>(const __nv_bfloat16* p, float (&f)[16]) {
    const uint4* s = reinterpret_cast<const uint4*>(p);
    uint4 v0 = s[0], v1 = s[1];
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = bf16_lo(w[i]);
        f[2 * i + 1] = bf16_hi(w[i]);
    }
}

template <>
__device__ __forceinline__ void load16<__half>(const __half* p, float (&f)[16]) {
    const uint4* s = reinterpret_cast<const uint4*>(p);
    uint4 v0 = s[0], v1 = s[1];
    const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = f16_lo(w[i]);
        f[2 * i + 1] = f16_hi(w[i]);
    }
}

template <typename T>
__global__ void __launch_bounds__(256) quant_weight_kernel(const QuantWeightArgs a) {
    __shared__ float warp_max[8];
    const int t = threadIdx.x;
    const int kb = blockIdx.x, nb = blockIdx.y;
    const int64_t col = static_cast<int64_t>(kb) * kGroup + (t & 7) * 16;
    const T* w = static_cast<const T*>(a.w);

    float f[4][16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t n = static_cast<int64_t>(nb) * kGroup + (t >> 3) + 32 * i;
        if (n < a.N) {
            load16<T>(w + n * a.K + col, f[i]);
#pragma unroll
            for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[i][j]));
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((t & 31) == 0) warp_max[t >> 5] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < 8; ++i) amax = fmaxf(amax, warp_max[i]);
    const float s = a.int8 ? __fdiv_rn(fmaxf(amax, kEps), kInt8Max) : group_scale(amax, a.ue8m0);
    if (t == 0) a.s[static_cast<int64_t>(nb) * a.KB + kb] = s;

#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int64_t n = static_cast<int64_t>(nb) * kGroup + (t >> 3) + 32 * i;
        if (n >= a.N) continue;
        if (a.int8) {
            const float* v = f[i];
            *reinterpret_cast<uint4*>(a.q + n * a.K + col) =
                make_uint4(cvt4_int8(v[0], v[1], v[2], v[3], s), cvt4_int8(v[4], v[5], v[6], v[7], s),
                           cvt4_int8(v[8], v[9], v[10], v[11], s),
                           cvt4_int8(v[12], v[13], v[14], v[15], s));
            continue;
        }
        uint32_t c[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
            c[j] = cvt2_e4m3(__fdiv_rn(f[i][2 * j], s), __fdiv_rn(f[i][2 * j + 1], s));
        uint4 out;
        out.x = c[0] | (c[1] << 16);
        out.y = c[2] | (c[3] << 16);
        out.z = c[4] | (c[5] << 16);
        out.w = c[6] | (c[7] << 16);
        *reinterpret_cast<uint4*>(a.q + n * a.K + col) = out;
    }
}

// ------------------------------------------------------------ per-row quant
//
// FP8_Dynamic / W8A8_INT8 ("用 Helion 为 vLLM 构建高性能可移植线性后端", 范围):
// one scale per row, s = max(amax_row, eps) / 448 (e4m3) or / 127 (int8),
// codes = round-half-even of clamp(x / s).  One CTA per row: 256 threads take
// 16-element chunks round robin (16 B bf16 loads, 16 B code stores), keep up
// to kRowCache chunks in registers between the amax pass and the code pass and
// re-read any further ones (an L2 hit: the row was just read).
constexpr int kRowThreads = 256;
constexpr int kRowCache = 5;  // rows up to 5 * 256 * 16 = 20480 elements stay in registers

template <bool kInt8>
__device__ __forceinline__ uint4 encode16(const float (&f)[16], float s) {
    uint32_t c[4];
    if constexpr (kInt8) {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            c[i] = cvt4_int8(f[4 * i], f[4 * i + 1], f[4 * i + 2], f[4 * i + 3], s);
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
            c[i] = cvt2_e4m3(__fdiv_rn(f[4 * i], s), __fdiv_rn(f[4 * i + 1], s)) |
                   (cvt2_e4m3(__fdiv_rn(f[4 * i + 2], s), __fdiv_rn(f[4 * i + 3], s)) << 16);
    }
    return make_uint4(c[0], c[1], c[2], c[3]);
}

template <typename T, bool kInt8>
__global__ void __launch_bounds__(kRowThreads) quant_rows_kernel(const QuantRowsArgs a) {
    __shared__ float warp_max[kRowThreads / 32];
    const int t = threadIdx.x;
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    const int64_t row = blockIdx.x;
    const T* x = static_cast<const T*>(a.x) + row * a.K;
    uint8_t* q = a.q + row * a.K;
    const int nc = static_cast<int>(a.K / 16);

    float f[kRowCache][16];
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < kRowCache; ++i) {
        const int c = t + i * kRowThreads;
        if (c < nc) {
            load16<T>(x + static_cast<int64_t>(c) * 16, f[i]);
#pragma unroll
            for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(f[i][j]));
        }
    }
    for (int c = t + kRowCache * kRowThreads; c < nc; c += kRowThreads) {
        float g[16];
        load16<T>(x + static_cast<int64_t>(c) * 16, g);
#pragma unroll
        for (int j = 0; j < 16; ++j) amax = fmaxf(amax, fabsf(g[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((t & 31) == 0) warp_max[t >> 5] = amax;
    __syncthreads();
    amax = warp_max[0];
#pragma unroll
    for (int i = 1; i < kRowThreads / 32; ++i) amax = fmaxf(amax, warp_max[i]);
    const float s = __fdiv_rn(fmaxf(amax, kEps), kInt8 ? kInt8Max : kFp8Max);
    if (t == 0) a.s[row] = s;

#pragma unroll
    for (int i = 0; i < kRowCache; ++i) {
        const int c = t + i * kRowThreads;
        if (c < nc) *reinterpret_cast<uint4*>(q + static_cast<int64_t>(c) * 16) = encode16<kInt8>(f[i], s);
    }
    for (int c = t + kRowCache * kRowThreads; c < nc; c += kRowThreads) {
        float g[16];
        load16<T>(x + static_cast<int64_t>(c) * 16, g);
        *reinterpret_cast<uint4*>(q + static_cast<int64_t>(c) * 16) = encode16<kInt8>(g, s);
    }
}

// ------------------------------------------------------------ int8 planes
//
// One CTA per row; a thread turns 16 int8 codes (one 16-byte load) into 16
// codes of 16 h and 16 codes of l (two 16-byte stores).  Each nibble indexes
// a 16-entry table of e4m3 codes, four bytes at a time with byte permutes:
//   l = q & 15        -> e4m3(l):          0, 1, 2, ..., 15
//   h = q >> 4 (signed) -> e4m3(16 h) for the nibble 0..7 (h = 0..7) and
//                        8..15 (h = -8..-1)
// (the entries are the OCP e4m3 encodings of those exact integers: bias 7,
// three mantissa bits).
__device__ __forceinline__ uint32_t nibble_lut(uint32_t n, uint32_t t0, uint32_t t1, uint32_t t2,
                                               uint32_t t3) {
    // n: four nibbles, one in the low half of each byte
    const uint32_t sel = (n & 0x7u) | ((n >> 4) & 0x70u) | ((n >> 8) & 0x700u) |
                         ((n >> 12) & 0x7000u);  // low three index bits, a nibble per byte
    const uint32_t lo = __byte_perm(t0, t1, sel);  // entries 0..7
    const uint32_t hi = __byte_perm(t2, t3, sel);  // entries 8..15
    const uint32_t m = ((n >> 3) & 0x01010101u) * 0xFFu;  // bytes whose index is >= 8
    return (lo & ~m) | (hi & m);
}

__global__ void __launch_bounds__(kRowThreads) int8_planes_kernel(const Int8PlanesArgs a) {
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    const int64_t row = blockIdx.x;
    const int8_t* q = a.q + row * a.K;
    uint8_t* out = a.planes + row * 2 * a.Kp;
    const int nc = static_cast<int>(a.Kp / 16);
    for (int c = threadIdx.x; c < nc; c += kRowThreads) {
        const int64_t k = static_cast<int64_t>(c) * 16;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (k < a.K) v = __ldcs(reinterpret_cast<const uint4*>(q + k));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            lo[i] = nibble_lut(w[i] & 0x0F0F0F0Fu, 0x44403800u, 0x4E4C4A48u, 0x53525150u,
                               0x57565554u);
            hi[i] = nibble_lut((w[i] >> 4) & 0x0F0F0F0Fu, 0x64605800u, 0x6E6C6A68u, 0xEAECEEF0u,
                               0xD8E0E4E8u);
        }
        // slab kb = c / 8 starts at 256 kb; the chunk sits at 16 (c % 8) inside
        const int64_t o = static_cast<int64_t>(c >> 3) * 256 + (c & 7) * 16;
        *reinterpret_cast<uint4*>(out + o) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(out + o + 128) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// ------------------------------------------------------ bounded-wait test

__global__ void wait_selftest_kernel(int* status, uint64_t timeout_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);
        fence_barrier_init();
        // Nothing ever arrives on `bar`: the wait must give up by itself.
        mbar_wait_bounded(&bar, 0, &abort_flag, status, timeout_ns,
                          static_cast<int>(FP8BQ_ERR_DEVICE_TIMEOUT));
    }
}

}  // namespace

cudaError_t launch_quant_act(const QuantActArgs& a, cudaStream_t stream) {
    const int quads = (a.G + 3) / 4;
    cudaLaunchConfig_t cfg = {};
    if (a.counts != nullptr) {
        // one grid layer per expert (M = E * m_max rows, m_max a multiple of 4)
        const int64_t E = a.m_max > 0 ? a.M / a.m_max : 0;
        if (E <= 0 || E > 65535) return cudaErrorInvalidConfiguration;
        cfg.gridDim = dim3(static_cast<unsigned>((a.m_max + kQuantRows - 1) / kQuantRows),
                           static_cast<unsigned>(quads), static_cast<unsigned>(E));
    } else {
        cfg.gridDim = dim3(static_cast<unsigned>((a.Mp + kQuantRows - 1) / kQuantRows),
                           static_cast<unsigned>(quads));
    }
    cfg.blockDim = dim3(kQuantRows * 32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (a.counts != nullptr) {
        if (a.fp16) return cudaLaunchKernelEx(&cfg, quant_act_kernel<true, true>, a);
        return cudaLaunchKernelEx(&cfg, quant_act_kernel<false, true>, a);
    }
    if (a.fp16) return cudaLaunchKernelEx(&cfg, quant_act_kernel<true, false>, a);
    return cudaLaunchKernelEx(&cfg, quant_act_kernel<false, false>, a);
}

cudaError_t launch_quant_weight(const QuantWeightArgs& a, cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>(a.KB), static_cast<unsigned>(a.NB));
    if (a.dtype == FP8BQ_FP32)
        quant_weight_kernel<float><<<grid, 256, 0, stream>>>(a);
    else if (a.dtype == FP8BQ_BF16)
        quant_weight_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(a);
    else
        quant_weight_kernel<__half><<<grid, 256, 0, stream>>>(a);
    return cudaGetLastError();
}

namespace {
template <bool kInt8>
cudaError_t launch_rows(const QuantRowsArgs& a, cudaLaunchConfig_t* cfg) {
    if (a.dtype == FP8BQ_FP32) return cudaLaunchKernelEx(cfg, quant_rows_kernel<float, kInt8>, a);
    if (a.dtype == FP8BQ_BF16)
        return cudaLaunchKernelEx(cfg, quant_rows_kernel<__nv_bfloat16, kInt8>, a);
    return cudaLaunchKernelEx(cfg, quant_rows_kernel<__half, kInt8>, a);
}
}  // namespace

cudaError_t launch_quant_rows(const QuantRowsArgs& a, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.R));
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return a.int8 ? launch_rows<true>(a, &cfg) : launch_rows<false>(a, &cfg);
}

cudaError_t launch_int8_planes(const Int8PlanesArgs& a, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(a.R));
    cfg.blockDim = dim3(kRowThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, int8_planes_kernel, a);
}

cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(status, timeout_ns);
    return cudaGetLastError();
}

}  // namespace fp8bq

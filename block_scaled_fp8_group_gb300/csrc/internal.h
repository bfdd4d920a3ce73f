// internal.h -- declarations shared by the library's translation units (not
// part of the public ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/fp8bq.h"

namespace fp8bq {

constexpr int kGroup = 128;  // activation group / weight block edge
constexpr float kEps = 1e-10f;
constexpr float kFp8Max = 448.0f;
constexpr float kInt8Max = 127.0f;  // symmetric int8 codes

inline int64_t pad_rows4(int64_t m) { return (m + 3) / 4 * 4; }

// Every workspace starts with this many bytes of split-K tile counters.  The
// region must be zero before first use and every call leaves it zero, so one
// workspace can serve calls of any shape in turn (data goes after it).
constexpr size_t kCounterRegion = 65536;

// ---------------------------------------------------------------- quant

struct QuantActArgs {
    const void* x;
    uint8_t* q;
    void* s;
    int64_t M;   // rows
    int64_t Mp;  // rows rounded up to a multiple of 4
    int64_t K;
    int G;       // groups per row
    int ue8m0;
    int fp16;    // input is fp16 (else bf16)
    int int8 = 0;  // int8 codes, s = max(amax, eps) / 127 (fp32 scales; block INT8)
    // Grouped rows (optional): M = E * m_max rows, expert e owning rows
    // [e * m_max, (e + 1) * m_max), of which the first counts[e] (device
    // array, clamped to [0, m_max]) are quantised; other rows are neither
    // read nor written.  The launch gives every expert its own grid layer.
    const int* counts = nullptr;
    int64_t m_max = 0;
};
cudaError_t launch_quant_act(const QuantActArgs& a, cudaStream_t stream);

struct QuantWeightArgs {
    const void* w;
    uint8_t* q;
    float* s;
    int64_t N, K;
    int NB, KB;
    int dtype;  // fp8bq_dtype
    int ue8m0;
    int int8 = 0;  // int8 codes (block INT8)
};
cudaError_t launch_quant_weight(const QuantWeightArgs& a, cudaStream_t stream);

// One scale per row of x [R, K] (per-token activations, per-channel weights).
struct QuantRowsArgs {
    const void* x;
    uint8_t* q;  // [R, K] e4m3 or int8 codes
    float* s;    // [R]
    int64_t R, K;
    int dtype;   // fp8bq_dtype of x
    int int8;    // codes are int8 (else e4m3)
};
cudaError_t launch_quant_rows(const QuantRowsArgs& a, cudaStream_t stream);

// INT8 codes as two e4m3 planes for the tcgen05 FP8 MMA: q = 16 h + l with
// h = q >> 4 in [-8, 7] and l = q & 15 in [0, 15], both exact in e4m3.  Row r
// of the output ([R, 2 Kp], Kp = K rounded up to 128) holds, for every
// 128-wide K slab kb, the codes of 16 h at [256 kb, 256 kb + 128) and of l at
// [256 kb + 128, 256 kb + 256); columns past K are zero codes.  Then
//   q_a q_w = (16 h_a)(16 h_w) + (16 h_a) l_w + l_a (16 h_w) + l_a l_w.
struct Int8PlanesArgs {
    const int8_t* q;  // [R, K]
    uint8_t* planes;  // [R, 2 Kp]
    int64_t R, K, Kp;
};
cudaError_t launch_int8_planes(const Int8PlanesArgs& a, cudaStream_t stream);

// ----------------------------------------------------------------- GEMM

struct GemmPlan {
    int kind;      // fp8bq_kind
    int bn;        // MMA N
    int split;     // K splits per tile
    int mx;        // 1: UE8M0 scales applied by the block-scaled MMA (gemm_mx_kernel)
    int grid;      // CTAs
    int tiles_tok; // token tiles
    int tiles_w;   // weight tiles
    int num_items; // tiles * split
    int experts;   // grouped: experts (0: one plain problem)
    int rowwise;   // one scale per token and per weight row: 1 e4m3 (gemm_mx_kernel, RW 1),
                   // 2 int8 (gemm_i8_kernel), 3 int8 as two e4m3 planes (gemm_mx_kernel,
                   // RW 2; K is then the logical K, a multiple of 128); 4 block INT8 on
                   // the warp-level MMA (gemm_i8_kernel, BLK), 5 block INT8 as two e4m3
                   // planes on the promotion kernel (gemm_kernel, PL 2; K logical); 0 block
                   // FP8 scales
    size_t ws_bytes;
};

// Fills the derived fields of a plan for (M, N, K) and the chosen variant;
// returns false if the variant is not supported.  With experts > 0 the plan
// is for a grouped problem: `experts` independent (M, N, K) problems whose
// token rows, weight rows and outputs are stacked (M is the rows per expert).
// With rowwise != 0 the plan is for the rowwise-scaled GEMM (1: e4m3, 2:
// int8; 128-row tiles, promotion-free; K in whole 16-byte rows, the last
// slab zero-filled).
bool make_gemm_plan(int64_t M, int64_t N, int64_t K, const fp8bq_variant& v, int num_sms,
                    GemmPlan* plan, int64_t experts = 0, int rowwise = 0);

struct GemmLaunch {
    int64_t M, N, K;
    const void* a_q;
    const void* a_s;
    const void* w_q;
    const float* w_s;
    int ue8m0;
    int out_dtype;
    void* out;
    void* workspace;        // counter prefix at offset 0
    size_t ws_data_offset;  // partials start at kCounterRegion + this offset
    int* status;
    uint64_t timeout_ns;
    // Weights may be read before the previous kernel in the stream has
    // finished (the linear path; see fp8bq_linear's contract).
    int prefetch_w;
    // Fused quant (linear path, UE8M0, swap-AB token tiles of 16/32): raw
    // bf16/fp16 activations [M, K] instead of a_q / a_s.
    const void* x;
    int x_fp16;
    // Grouped problem (E > 0): M = E * m_max stacked token rows, w_q/w_s hold
    // E stacked [N, K] weights, out is [E * m_max, N]; expert e's valid rows
    // are [e * m_max, e * m_max + counts[e]) (device array, clamped to
    // [0, m_max]).
    int64_t E = 0;
    int64_t m_max = 0;
    const int* counts = nullptr;
    // Rowwise scales (plan.rowwise): a_s is fp32 [M] (one per token), w_s
    // fp32 [N] (one per weight row).
};
cudaError_t launch_gemm(const GemmPlan& plan, const GemmLaunch& g, cudaStream_t stream);

// Bounded-wait self test (one CTA, one thread).
cudaError_t launch_wait_selftest(int* status, uint64_t timeout_ns, cudaStream_t stream);

// Driver entry point for tensor-map encoding (resolved once through the runtime).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn get_encode_tiled();

// One line to stderr when FP8BQ_LOG=1 (diagnostics only).
void log_error(const char* what);

}  // namespace fp8bq

/*
 * fp8bq.h -- C ABI of the W8A8 block-FP8 linear path for GB300 (sm_103a).
 *
 * Two steps, as the pages describe them:
 *   1. per-token-group activation quant: bf16/fp16 rows -> float8_e4m3fn codes
 *      with one scale per 1x128 group, fp32 or UE8M0 (power of two, four
 *      exponent bytes packed per int32), in a TMA-aligned column-major layout
 *      ("vLLM DeepGEMM FP8 Block GEMM 基准测试", §4.1; "vllm-project/vllm PR
 *      42153", 实现拆解);
 *   2. a dense GEMM of those codes against weights quantised in 128x128
 *      blocks, where each 128-wide K slab's partial sum is promoted by
 *      sa[m,kb]*sw[nb,kb] into an fp32 accumulator and the result is written as
 *      bf16, fp16 or fp32 ("vLLM DeepGEMM FP8 Block GEMM 基准测试", §4.2 and
 *      §4.3; split-K and swap-AB variants: "用 Helion 为 vLLM 构建高性能可移植
 *      线性后端", 内核实现).
 *
 * Conventions for every entry point below:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the library
 *     never allocates device memory and never frees anything it is given.
 *   - Calls are asynchronous on `stream` (0 = legacy default stream) and never
 *     synchronise, except fp8bq_device_status.
 *   - Errors are returned as fp8bq_status, never thrown or aborted on.  All
 *     argument checks run on the host before any launch; a call that returns
 *     an argument error has written nothing.
 *   - Shapes: int64 sizes; M (tokens) >= 0 arbitrary, K a positive multiple of
 *     128, N a multiple of 64 for the GEMM (the DeepGEMM dispatch predicate of
 *     "vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.2: bf16 output, N % 64 == 0,
 *     K % 128 == 0 -- fp16/fp32 outputs are accepted here as well).  M == 0 or
 *     N == 0 is a no-op that returns FP8BQ_OK.
 *   - Inputs must hold finite values; outputs for NaN/Inf inputs are
 *     unspecified.
 *   - Calls sharing one workspace must not overlap on the GPU (same stream, or
 *     ordered by events).
 */
#ifndef FP8BQ_H
#define FP8BQ_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FP8BQ_OK = 0,
    FP8BQ_ERR_INVALID_ARG = 1,    /* null pointer, negative size, bad enum */
    FP8BQ_ERR_SHAPE = 2,          /* K % 128 != 0 or K <= 0, N % 64 != 0, size overflow */
    FP8BQ_ERR_ALIGNMENT = 3,      /* a pointer not 16-byte aligned */
    FP8BQ_ERR_UNSUPPORTED = 4,    /* group/block != 128, dtype not accepted, GPU not sm_103 */
    FP8BQ_ERR_WORKSPACE = 5,      /* workspace null or smaller than required */
    FP8BQ_ERR_LAUNCH = 6,         /* the kernel launch itself failed */
    FP8BQ_ERR_DEVICE_TIMEOUT = 7, /* a kernel's bounded wait gave up (see fp8bq_device_status) */
    FP8BQ_ERR_CUDA = 8            /* another CUDA runtime error (no device, ...) */
} fp8bq_status;

typedef enum {
    FP8BQ_SCALE_FP32 = 0,  /* one fp32 scale per group */
    FP8BQ_SCALE_UE8M0 = 1  /* power-of-two scales; activation scales packed 4 per u32 */
} fp8bq_scale_fmt;

typedef enum { FP8BQ_BF16 = 0, FP8BQ_FP16 = 1, FP8BQ_FP32 = 2 } fp8bq_dtype;

/* GEMM variant (kernel shape) -- what the per-shape table stores.
 * "用 Helion 为 vLLM 构建高性能可移植线性后端", 内核实现: Standard, Split-K and
 * Swap-AB exposed as tunable choices; "vLLM 量化 Kernel 配置机制" §4.2: per-M
 * configs, nearest-M lookup. */
typedef enum {
    FP8BQ_KIND_NORMAL = 0, /* MMA M = 128 tokens, MMA N = block_n weight rows */
    FP8BQ_KIND_SWAP_AB = 1, /* D^T = W A^T: MMA M = 128 weight rows, MMA N = block_n tokens */
    FP8BQ_KIND_SWAP_AB_64 = 2 /* swap-AB with 64 weight rows per tile (MMA M = 64), twice the
                               * tiles of kind 1 for narrow N; block_n 16 or 32 */
} fp8bq_kind;

typedef struct {
    int32_t kind;       /* fp8bq_kind */
    int32_t block_n;    /* MMA N: swap-AB {16,32,64,128}; normal {128,256} */
    int32_t split;      /* K splits per output tile, 1..64 (1 = no split-K) */
    int32_t grid;       /* CTAs to launch; 0 = one per SM, capped by the work items */
    int32_t from_table; /* output of fp8bq_select_variant: 1 = measured table, 0 = default */
    int32_t mma_scale;  /* 0: each K slab's fp32 product is promoted by sa*sw on the CUDA
                         * cores; 1: the tensor core applies the scales (block-scaled MMA,
                         * E8M0 factors in TMEM) and accumulates all slabs itself -- either
                         * orientation (kinds 0 and 1; not kind 2), UE8M0 scales only, K a
                         * multiple of 512 (FP8BQ_ERR_UNSUPPORTED otherwise) */
} fp8bq_variant;

/* ------------------------------------------------------------ size queries */

/* Bytes of the activation scale buffer for an [M,K] input with 1 x `group`
 * groups (G = K/group): rows are padded to Mp = ceil(M/4)*4 (TMA-aligned);
 * FP32: 4*G*Mp bytes, element (g, m) at float index g*Mp + m;
 * UE8M0: 4*ceil(G/4)*Mp bytes, group g of row m in byte (g%4) of the u32 at
 * index (g/4)*Mp + m (byte = biased fp32 exponent of the scale, 127 = 1.0).
 * Returns 0 on invalid arguments. */
size_t fp8bq_act_scale_bytes(int64_t M, int64_t K, int group, fp8bq_scale_fmt fmt);

/* Bytes of the weight scale buffer: fp32 [ceil(N/block_n)][K/block_k]. */
size_t fp8bq_weight_scale_bytes(int64_t N, int64_t K, int block_n, int block_k);

/* Workspace bytes fp8bq_gemm needs for this shape (0 when none is needed:
 * no split-K).  Every workspace starts with a 65536-byte prefix of split-K
 * tile counters, followed by fp32 partial tiles.  The prefix must be zero
 * before the first use; every successful call leaves it zero again (the
 * counters reset themselves), so one workspace can serve calls of any shape
 * in turn.  After an FP8BQ_ERR_DEVICE_TIMEOUT, zero the prefix again. */
size_t fp8bq_gemm_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_scale_fmt fmt,
                                  fp8bq_dtype out_dtype);
/* Same for an explicit variant (fp8bq_gemm_variant). */
size_t fp8bq_variant_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                     const fp8bq_variant* variant);
/* Workspace bytes of fp8bq_linear: the 65536-byte counter prefix, then the
 * activation codes (M*K bytes), the activation scales and the split-K
 * partials, each at a 256-byte aligned offset. */
size_t fp8bq_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_scale_fmt fmt,
                                    fp8bq_dtype out_dtype);

/* ------------------------------------------------------------------ quant */

/* Per-token-group activation quant ("vLLM DeepGEMM FP8 Block GEMM 基准测试"
 * §4.1 per_token_group_quant_fp8 with column_major_scales and
 * tma_aligned_scales; packed UE8M0 scales as in "vllm-project/vllm PR 42153").
 * For each row m and group g (128 consecutive k):
 *   amax = max |x|;  s = fp32(max(amax, 1e-10) / 448);
 *   UE8M0: s = 2^ceil(log2 s);
 *   q = e4m3 round-to-nearest-even of clamp(fp32(x / s), -448, 448).
 * x: [M,K] row-major, x_dtype FP8BQ_BF16 or FP8BQ_FP16, 16-byte aligned.
 * q: [M,K] e4m3 codes row-major, 16-byte aligned.
 * s: fp8bq_act_scale_bytes(M,K,group,fmt) bytes, 16-byte aligned; padding rows
 *    [M, Mp) and unused bytes of the last packed word are written as 0.
 * group must be 128.  Results are bit-exact functions of the input. */
fp8bq_status fp8bq_quant_act(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t K,
                             int group, fp8bq_scale_fmt fmt, void* q, void* s,
                             cudaStream_t stream);

/* 128x128 weight block quant ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.1
 * per_block_cast_to_fp8(B, [128,128], use_ue8m0)): per block (nb, kb) the same
 * scale and rounding rules as fp8bq_quant_act, over the block's 128x128
 * elements (a partial last row block uses the rows that exist).
 * w: [N,K] row-major, FP8BQ_FP32, FP8BQ_BF16 or FP8BQ_FP16, 16-byte aligned.
 * q: [N,K] e4m3 codes, 16-byte aligned.
 * s: fp32 [ceil(N/128)][K/128] row-major (powers of two in UE8M0 mode).
 * block_n and block_k must be 128.  Meant for offline use. */
fp8bq_status fp8bq_quant_weight(const void* w, fp8bq_dtype w_dtype, int64_t N, int64_t K,
                                int block_n, int block_k, fp8bq_scale_fmt fmt, void* q,
                                float* s, cudaStream_t stream);

/* ------------------------------------------------------------------- GEMM */

/* out[m,n] = sum_kb sa[m,kb] * sw[n/128,kb] * sum_{k in slab kb} a_q[m,k]*w_q[n,k]
 * ("vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.2: fp8_gemm_nt, A [M,K] and W
 * [N,K] both K-major; the per-K-block scale multiply into the accumulator).
 * Each slab's FP8 products are summed by the tensor cores in fp32.  With
 * mma_scale = 0 (every fp32-scale shape, and the UE8M0 shapes the table
 * picks so) the slab sum is promoted by sa*sw into an fp32 register
 * accumulator; with mma_scale = 1 (UE8M0 only) the tensor core multiplies
 * every 32-wide K block's products by the power-of-two factors as it
 * accumulates, and all slabs build up in one fp32 TMEM accumulator.  The
 * result is rounded to nearest even into out_dtype.
 * a_q: [M,K] e4m3 row-major, 16-byte aligned.
 * a_s: activation scales in the fp8bq_quant_act layout for `fmt`.
 * w_q: [N,K] e4m3 row-major, 16-byte aligned.  w_s: fp32 [ceil(N/128)][K/128].
 * out: [M,N] row-major out_dtype (BF16, FP16 or FP32), 16-byte aligned.
 * workspace: fp8bq_gemm_workspace_bytes(...) bytes (may be NULL when that is
 * 0), zero-filled before first use, 256-byte aligned.
 * group, block_n, block_k must be 128.  The kernel shape comes from the
 * per-shape table (fp8bq_select_variant). */
fp8bq_status fp8bq_gemm(int64_t M, int64_t N, int64_t K, const void* a_q, const void* a_s,
                        const void* w_q, const float* w_s, int group, int block_n, int block_k,
                        fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype, void* out,
                        void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* fp8bq_gemm with an explicit kernel shape (used by the tuner and the tests).
 * The workspace size is fp8bq_variant_workspace_bytes for that variant. */
fp8bq_status fp8bq_gemm_variant(int64_t M, int64_t N, int64_t K, const void* a_q,
                                const void* a_s, const void* w_q, const float* w_s,
                                fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype, void* out,
                                const fp8bq_variant* variant, void* workspace,
                                size_t workspace_bytes, cudaStream_t stream);
/* Host-only check of an explicit kernel shape before fp8bq_gemm_variant:
 * FP8BQ_OK when the kernels have this tile/split/schedule for (M, N, K) and
 * the scale format (the block-scaled MMA, mma_scale 1, needs UE8M0 scales and
 * K % 512 == 0) on this GPU (152 SMs when none is visible); the argument
 * errors of fp8bq_gemm, or FP8BQ_ERR_UNSUPPORTED.  Launches nothing. */
fp8bq_status fp8bq_variant_supported(int64_t M, int64_t N, int64_t K, fp8bq_scale_fmt fmt,
                                     const fp8bq_variant* variant);

/* ---------------------------------------------------------- grouped GEMM */

/* Grouped (mixture-of-experts) GEMM, masked layout: E independent
 * fp8bq_gemm problems of the same (N, K), one per expert, in one launch.
 * The pages apply the same per-shape kernel-config scheme to the MoE
 * kernels, with the expert count added to the key ("vLLM 量化 Kernel
 * 配置机制" §5, 同构机制的延伸), and name an MoE backend as the next target
 * ("用 Helion 为 vLLM 构建高性能可移植线性后端", 未来工作); neither spells the
 * kernel out.  The reading taken: expert e multiplies its own token rows by
 * its own 128x128-block-quantised weights, exactly as fp8bq_gemm does.
 *   rows of expert e: [e*M_max, e*M_max + c_e), c_e = counts[e] clamped to
 *   [0, M_max]; out[e*M_max + m, n] = fp8bq_gemm of (a rows, w_q[e], w_s[e]).
 * counts: int32 [E] in DEVICE memory (a routing kernel may write it just
 *   before; it is read after the preceding work in `stream` has finished).
 * a_q: [E*M_max, K] e4m3; a_s: fp8bq_quant_act scales of all E*M_max rows.
 * w_q: [E][N][K] e4m3 (E stacked fp8bq_quant_weight outputs);
 * w_s: fp32 [E][N/128][K/128].
 * out: [E*M_max, N]; rows of an expert at or past its count are not written.
 * Preconditions (else FP8BQ_ERR_SHAPE): M_max % 4 == 0 (each expert's scale
 * rows start 16-byte aligned), N % 128 == 0, K % 128 == 0.  E >= 1.
 * M_max == 0 or N == 0 is a no-op.  The kernel shape comes from
 * fp8bq_select_grouped_variant (every expert counted as full). */
fp8bq_status fp8bq_grouped_gemm(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                const int32_t* counts, const void* a_q, const void* a_s,
                                const void* w_q, const float* w_s, int group, int block_n,
                                int block_k, fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype,
                                void* out, void* workspace, size_t workspace_bytes,
                                cudaStream_t stream);

/* fp8bq_grouped_gemm with an explicit kernel shape.  Stream-K (split 0) is
 * not accepted for grouped problems (FP8BQ_ERR_UNSUPPORTED). */
fp8bq_status fp8bq_grouped_gemm_variant(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                        const int32_t* counts, const void* a_q,
                                        const void* a_s, const void* w_q, const float* w_s,
                                        fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype, void* out,
                                        const fp8bq_variant* variant, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream);

/* Grouped W8A8 linear layer: the activation quant of the experts' occupied
 * rows followed by fp8bq_grouped_gemm, one call, two launches on `stream`.
 * x: [E*M_max, K] bf16/fp16, 16-byte aligned; rows of expert e at or past
 * counts[e] are not read.  The codes and scales go to the front of
 * `workspace` (fp8bq_grouped_linear_workspace_bytes; counter prefix, codes,
 * scales, split-K partials, as fp8bq_linear); their padding rows are not
 * written.  E at most 65535 (FP8BQ_ERR_UNSUPPORTED otherwise: the quant
 * kernel's grid has one layer per expert).  Other arguments and
 * preconditions as fp8bq_grouped_gemm. */
fp8bq_status fp8bq_grouped_linear(const void* x, fp8bq_dtype x_dtype, int64_t E, int64_t M_max,
                                  int64_t N, int64_t K, const int32_t* counts, const void* w_q,
                                  const float* w_s, int group, int block_n, int block_k,
                                  fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype, void* out,
                                  void* workspace, size_t workspace_bytes, cudaStream_t stream);
size_t fp8bq_grouped_linear_workspace_bytes(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                            fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype);

/* The kernel shape fp8bq_grouped_gemm uses, and workspace sizes. */
fp8bq_status fp8bq_select_grouped_variant(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                          fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype,
                                          fp8bq_variant* variant);
size_t fp8bq_grouped_gemm_workspace_bytes(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                          fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype);
size_t fp8bq_grouped_variant_workspace_bytes(int64_t E, int64_t M_max, int64_t N, int64_t K,
                                             const fp8bq_variant* variant);

/* Activation quant followed by the GEMM, one call, two launches on `stream`
 * (the whole W8A8 linear layer for a bf16/fp16 input x [M,K]).  The codes and
 * scales go to the front of `workspace`; see fp8bq_linear_workspace_bytes.
 * With the environment variable FP8BQ_LINEAR_FUSE=1, UE8M0 problems whose
 * selected variant is swap-AB with a 16/32-token tile run as one block-scaled
 * launch that quantises its own activation tiles instead (bit-identical
 * output; slower on GB300 at the shapes measured, hence off by default). */
fp8bq_status fp8bq_linear(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t N, int64_t K,
                          const void* w_q, const float* w_s, int group, int block_n,
                          int block_k, fp8bq_scale_fmt fmt, fp8bq_dtype out_dtype, void* out,
                          void* workspace, size_t workspace_bytes, cudaStream_t stream);

/* fp8bq_gemm for callers that cannot allocate device memory.  (The pages
 * have no counterpart: this exists for integration, not for the method.)
 * Some callers cannot call cudaMalloc where they run a layer -- runtimes that
 * hand out all device memory from their own pool at start-up and forbid
 * allocations later, code that must not risk the device synchronisation an
 * allocation can cause, plug-ins that only receive tensors and a stream -- so
 * they cannot provide the split-K workspace fp8bq_gemm may need.  This entry
 * point takes the same arguments minus the workspace and allocates nothing:
 * no cudaMalloc, no cudaFree, no allocating library call.  Its scratch is one
 * array of 32 MiB (33554432 bytes) built into the library; every GPU on which
 * it is first used holds it from then until the process exits.
 *   - Problems whose chosen kernel needs more split-K scratch than 32 MiB are
 *     rejected with FP8BQ_ERR_WORKSPACE (nothing is launched); use fp8bq_gemm
 *     with a workspace for those.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current.  Under the CUDA
 *     runtime's default lazy module loading, that lookup is also what loads
 *     the array's module on the device: it reserves the 32 MiB there and may
 *     synchronise the device.  So make that first call once at start-up,
 *     outside any region where allocation or synchronisation is not allowed,
 *     and before any stream capture.
 *   - All calls share the one array, and each call clears the counters at its
 *     start (cudaMemsetAsync on `stream`): calls that overlap on the GPU
 *     (different streams without ordering) race and give wrong results. */
fp8bq_status fp8bq_gemm_noalloc(int64_t M, int64_t N, int64_t K, const void* a_q,
                                const void* a_s, const void* w_q, const float* w_s, int group,
                                int block_n, int block_k, fp8bq_scale_fmt fmt,
                                fp8bq_dtype out_dtype, void* out, cudaStream_t stream);

/* ------------------------------------- per-token x per-channel formats
 *
 * "用 Helion 为 vLLM 构建高性能可移植线性后端", 范围, lists two more W8A8
 * formats beside Block_FP8: FP8_Dynamic (FP8 codes, one scale per activation
 * token and one per weight output channel) and W8A8_INT8 (the same scaling
 * with INT8 codes).  The pages give no formulas; the rule used is the block
 * path's with the block widened to a whole row:
 *   s[r] = fp32(max(amax of row r, 1e-10) / Q), Q = 448 (e4m3) or 127 (int8)
 *   q    = round-half-even(clamp(x / s, -Q, Q))   (IEEE fp32 division)
 *   out[m,n] = a_s[m] * w_s[n] * sum_k dec(a_q[m,k]) * dec(w_q[n,k])
 * Shapes: K > 0 and K % 16 == 0 (16-byte code rows), N % 16 == 0 for the
 * GEMM (FP8BQ_ERR_SHAPE otherwise); M (or R) >= 0 arbitrary, 0 is a no-op. */
typedef enum {
    FP8BQ_CODE_E4M3 = 0, /* FP8_Dynamic: float8_e4m3fn codes, tcgen05 FP8 MMA */
    FP8BQ_CODE_INT8 = 1  /* W8A8_INT8: two's-complement int8 codes in [-127, 127]; exact
                          * int32 sums on the warp-level int8 tensor-core MMA (sm_103a's
                          * tcgen05 has no integer kind) */
} fp8bq_code;

/* One scale per row of x [R,K] (bf16, fp16 or fp32, 16-byte aligned):
 * per-token activation scales, or per-channel scales when x is a weight
 * [N,K].  q: [R,K] codes (16-byte aligned); s: fp32 [R] (4-byte aligned).
 * One launch on `stream`. */
fp8bq_status fp8bq_quant_rows(const void* x, fp8bq_dtype x_dtype, int64_t R, int64_t K,
                              fp8bq_code code, void* q, float* s, cudaStream_t stream);

/* Rowwise-scaled GEMM: a_q [M,K] codes with a_s fp32 [M]; w_q [N,K] codes
 * with w_s fp32 [N]; out [M,N] bf16/fp16/fp32.  The workspace
 * (fp8bq_rowwise_workspace_bytes, 256-byte aligned) follows the rules of
 * fp8bq_gemm_workspace_bytes: the counter prefix, then split parts, then (int8
 * on the FP8 MMA) the two operands' planes.  The kernel shape comes from
 * fp8bq_select_rowwise_variant. */
fp8bq_status fp8bq_gemm_rowwise(int64_t M, int64_t N, int64_t K, const void* a_q,
                                const float* a_s, const void* w_q, const float* w_s,
                                fp8bq_code code, fp8bq_dtype out_dtype, void* out,
                                void* workspace, size_t workspace_bytes, cudaStream_t stream);
/* The same with an explicit kernel shape.  e4m3: swap-AB (block_n 16..128) or
 * normal (128, 256) tiles, split >= 0 (0 = stream-K), mma_scale 0.  int8 has
 * two kernels, chosen by mma_scale:
 *   0 -- the warp-level int8 tensor-core MMA (exact int32 sums), swap-AB
 *        tiles only, block_n 8, 16, 32, 64 or 128;
 *   1 -- the codes split exactly into two e4m3 planes (q = 16h + l, h = q >> 4,
 *        l = q & 15) on the tcgen05 FP8 MMA, four cross products per K step;
 *        swap-AB or normal tiles as for e4m3.  Both operands are rewritten into
 *        the workspace first (2 bytes per code, K rounded up to 128), so this
 *        form needs a workspace even without split-K.
 * fp8bq_gemm_rowwise takes the kernel and shape from the measured table's
 * "ri8" entry for the problem (nearest M) when there is one, else the
 * warp-level kernel up to 64 tokens and the planes above.  Other shapes:
 * FP8BQ_ERR_UNSUPPORTED. */
fp8bq_status fp8bq_gemm_rowwise_variant(int64_t M, int64_t N, int64_t K, const void* a_q,
                                        const float* a_s, const void* w_q, const float* w_s,
                                        fp8bq_code code, fp8bq_dtype out_dtype, void* out,
                                        const fp8bq_variant* variant, void* workspace,
                                        size_t workspace_bytes, cudaStream_t stream);
fp8bq_status fp8bq_select_rowwise_variant(int64_t M, int64_t N, int64_t K, fp8bq_code code,
                                          fp8bq_dtype out_dtype, fp8bq_variant* variant);
size_t fp8bq_rowwise_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_code code,
                                     fp8bq_dtype out_dtype);
size_t fp8bq_rowwise_variant_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_code code,
                                             const fp8bq_variant* variant);

/* The rowwise linear layer: fp8bq_quant_rows of x [M,K] (bf16/fp16) followed
 * by fp8bq_gemm_rowwise, one call, two launches on `stream`.  The codes and
 * scales go to the front of `workspace`: [65536-byte counter prefix][codes
 * M*K][scales 4*M][split parts], each part at a 256-byte aligned offset. */
fp8bq_status fp8bq_linear_rowwise(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t N,
                                  int64_t K, const void* w_q, const float* w_s, fp8bq_code code,
                                  fp8bq_dtype out_dtype, void* out, void* workspace,
                                  size_t workspace_bytes, cudaStream_t stream);
size_t fp8bq_linear_rowwise_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_code code,
                                            fp8bq_dtype out_dtype);

/* ------------------------------------------------------------ block INT8
 *
 * "vLLM 量化 Kernel 配置机制" §1 lists int8_w8a8 tables with block_shape
 * [128,128]: the block-quantised path with INT8 codes.  The rule used is the
 * block FP8 path's with int8 codes and fp32 scales:
 *   s = fp32(max(amax, 1e-10) / 127) per 1 x 128 activation group and per
 *       128 x 128 weight block, q = round-half-even(clamp(x / s, -127, 127));
 *   out[m,n] = sum_kb sa[m,kb] * sw[n/128,kb] * S_kb,  S_kb the exact integer
 *       sum of slab kb's products (int32 on the warp-level int8 MMA, promoted
 *       per slab in fp32).
 * Layouts as the FP8 block path with fp32 scales: activation scales fp32
 * column-major [K/128][Mp] (Mp = ceil(M/4)*4, padding rows 0), weight scales
 * fp32 [ceil(N/128)][K/128], codes int8 row-major.  K % 128 == 0; N % 16 == 0
 * for the GEMM; group/block sizes 128 (FP8BQ_ERR_UNSUPPORTED otherwise). */
fp8bq_status fp8bq_quant_act_int8(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t K,
                                  int group, void* q, float* s, cudaStream_t stream);
fp8bq_status fp8bq_quant_weight_int8(const void* w, fp8bq_dtype w_dtype, int64_t N, int64_t K,
                                     int block_n, int block_k, void* q, float* s,
                                     cudaStream_t stream);
/* The block INT8 GEMM; workspace rules as fp8bq_gemm (counter prefix, then
 * split parts, then, for the planes kernel, both operands' e4m3 planes).  The
 * _variant form chooses the kernel by mma_scale, as fp8bq_gemm_rowwise_variant
 * does for int8: 0 -- the warp-level int8 MMA with per-slab promotion, swap-AB
 * tiles with block_n 8, 16, 32, 64 or 128; 1 -- two e4m3 planes on the
 * promotion kernel, swap-AB (16..128) or normal (128, 256) tiles.  split >= 0
 * (0 = stream-K).  fp8bq_gemm_int8_block takes the measured table's "bi8"
 * entry when there is one, else the warp-level kernel up to 64 tokens and the
 * planes above. */
fp8bq_status fp8bq_gemm_int8_block(int64_t M, int64_t N, int64_t K, const void* a_q,
                                   const float* a_s, const void* w_q, const float* w_s,
                                   int group, int block_n, int block_k, fp8bq_dtype out_dtype,
                                   void* out, void* workspace, size_t workspace_bytes,
                                   cudaStream_t stream);
fp8bq_status fp8bq_gemm_int8_block_variant(int64_t M, int64_t N, int64_t K, const void* a_q,
                                           const float* a_s, const void* w_q, const float* w_s,
                                           fp8bq_dtype out_dtype, void* out,
                                           const fp8bq_variant* variant, void* workspace,
                                           size_t workspace_bytes, cudaStream_t stream);
fp8bq_status fp8bq_select_int8_block_variant(int64_t M, int64_t N, int64_t K,
                                             fp8bq_dtype out_dtype, fp8bq_variant* variant);
size_t fp8bq_int8_block_workspace_bytes(int64_t M, int64_t N, int64_t K, fp8bq_dtype out_dtype);
size_t fp8bq_int8_block_variant_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                                const fp8bq_variant* variant);
/* Block INT8 linear layer: fp8bq_quant_act_int8 of x [M,K] (bf16/fp16), then
 * the GEMM, one call, two launches.  Workspace: [65536-byte counter prefix]
 * [codes M*K][scales 4*(K/128)*Mp][split parts], each at a 256-byte aligned
 * offset. */
fp8bq_status fp8bq_linear_int8_block(const void* x, fp8bq_dtype x_dtype, int64_t M, int64_t N,
                                     int64_t K, const void* w_q, const float* w_s, int group,
                                     int block_n, int block_k, fp8bq_dtype out_dtype, void* out,
                                     void* workspace, size_t workspace_bytes,
                                     cudaStream_t stream);
size_t fp8bq_linear_int8_block_workspace_bytes(int64_t M, int64_t N, int64_t K,
                                               fp8bq_dtype out_dtype);

/* ------------------------------------------------------------ host queries */

/* The variant fp8bq_gemm would run for this shape (host only, no GPU work):
 * the measured table for (device, N, K, fmt, out_dtype) is searched for the
 * M grid point nearest to M (a tie goes to the smaller M); without a table
 * entry a default variant is used and, with FP8BQ_LOG=1 in the environment,
 * one line is logged per (N, K, fmt, out_dtype) ("vLLM 量化 Kernel 配置机制"
 * §4.1-§4.2).  The table file is FP8BQ_TABLE if set, else
 * <package>/tables/<device name, spaces as '_'>.tbl. */
fp8bq_status fp8bq_select_variant(int64_t M, int64_t N, int64_t K, fp8bq_scale_fmt fmt,
                                  fp8bq_dtype out_dtype, fp8bq_variant* variant);

/* Reloads the table (after FP8BQ_TABLE changed); host only. */
fp8bq_status fp8bq_reload_table(void);

/* Synchronises `stream`, reads and clears the library's device status word:
 * *code = FP8BQ_OK, or FP8BQ_ERR_DEVICE_TIMEOUT if a kernel's bounded wait
 * gave up since the last read.  Bounded waits give up after
 * FP8BQ_WAIT_TIMEOUT_MS milliseconds (environment, default 2000). */
fp8bq_status fp8bq_device_status(int* code, cudaStream_t stream);

/* Self-test of the bounded-wait machinery: launches one CTA that waits on an
 * mbarrier nothing arrives at, for at most timeout_ns nanoseconds, then
 * records FP8BQ_ERR_DEVICE_TIMEOUT in the status word and returns.  Never
 * hangs.  Read the result with fp8bq_device_status. */
fp8bq_status fp8bq_selftest_wait_timeout(uint64_t timeout_ns, cudaStream_t stream);

const char* fp8bq_status_string(fp8bq_status status);
int fp8bq_abi_version(void); /* 1 */

#ifdef __cplusplus
}
#endif
#endif /* FP8BQ_H */

// gemm.cu -- block-scaled FP8 GEMM on tcgen05 tensor cores (sm_103a).
//
//   out[m,n] = sum_kb sa[m,kb] * sw[n/128,kb] * P_kb[m,n],
//   P_kb[m,n] = sum_{k in slab kb} a[m,k] * w[n,k]        (FP8 x FP8 -> fp32)
//
// "vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.2 describes the promotion (each
// K block's dot product times a_s[:,None]*b_s[None,:] added to an fp32
// accumulator); "用 Helion 为 vLLM 构建高性能可移植线性后端", 内核实现, the
// Split-K and Swap-AB variants.
//
// Design (one CTA per SM, persistent over work items):
//   warp 0     TMA producer: per K slab, one 128x128 tile of the MMA-M operand
//              and one BNx128 tile of the MMA-N operand into a STAGES-deep
//              shared-memory ring (128-byte swizzle, K-major).
//   warp 1     MMA issuer: four tcgen05.mma (K = 32 each) per slab into a
//              fresh TMEM accumulator buffer; commits free the smem stage and
//              publish the TMEM buffer.  Warp 1 also owns the TMEM allocation.
//   warps 2..  promotion/epilogue: per slab, tcgen05.ld the slab's fp32 sums,
//              release the TMEM buffer, and fold them into a register
//              accumulator with fma(P, sa*sw, acc).  NBUF TMEM buffers let the
//              MMA of slab kb+1 overlap the promotion of slab kb.
// Work item = (output tile, K split).  split == 1 is the plain (Standard)
// GEMM; split > 1 writes fp32 partial tiles to the workspace and the last CTA
// to finish a tile (atomic ticket; no CTA waits for another) sums the splits
// in fixed order 0..S-1, so results are run-to-run bit-stable.
// Swap-AB (decode): the MMA-M operand is the weight (128 rows of n), the
// MMA-N operand the tokens (BN = 16..128), so small M does not waste a
// 128-row MMA; the epilogue writes the transposed tile back into [M,N].
//
// Every wait is bounded (global-timer limit); on expiry the CTA records
// FP8BQ_ERR_DEVICE_TIMEOUT in the status word, lets its in-flight copies and
// MMAs land (again bounded), frees its TMEM and returns.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace fp8bq {

namespace {

constexpr int BM = 128;  // MMA M
constexpr int BK = 128;  // K slab (one scale block)
constexpr int kCountersPerTile = 8;  // one split-K ticket per epilogue warp

template <int BN>
struct Cfg {
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN <= 16 ? 10 : BN <= 32 ? 9 : BN <= 64 ? 8 : BN <= 128 ? 6 : 4;
    static constexpr int NBUF = BN <= 64 ? 4 : 2;
    static constexpr int TMEM_NEED = NBUF * BN;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32    ? 32
                                     : TMEM_NEED <= 64  ? 64
                                     : TMEM_NEED <= 128 ? 128
                                     : TMEM_NEED <= 256 ? 256
                                                        : 512;
    static constexpr int EPI_WARPS = BN >= 128 ? 8 : 4;
    static constexpr int CPT = BN / (EPI_WARPS / 4);  // accumulator columns per thread
    static constexpr int THREADS = 64 + 32 * EPI_WARPS;
    static constexpr int BAR_BYTES = 8 * (2 * STAGES + 2 * NBUF + 1) + 16;
    static constexpr int SMEM = 1024 + STAGES * STAGE_BYTES + BAR_BYTES;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
    static_assert(CPT % 16 == 0, "TMEM loads are 16 columns wide");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct KArgs {
    int M, N, G;
    int Mp;          // activation-scale column stride (rows padded to 4)
    int swap;        // MMA-M operand is the weight
    int tiles_tok;   // token tiles (MMA-M tiles when !swap, MMA-N tiles when swap)
    int split;
    int num_items;
    int ue8m0;
    int out_dtype;
    const void* sa;
    const float* sw;
    void* out;
    float* partials;
    unsigned* counters;
    int* status;
    unsigned long long timeout_ns;
};

struct Item {
    int tile;     // linear tile index
    int tok0;     // first token of the tile
    int w0;       // first weight row (n) of the tile
    int kb0, kb1; // K slab range
    int split;    // index of this split
};

template <int BN>
__device__ __forceinline__ Item decode_item(const KArgs& a, int item) {
    Item it;
    it.tile = item / a.split;
    it.split = item - it.tile * a.split;
    const int wt = it.tile / a.tiles_tok;        // weight tile (slow)
    const int tt = it.tile - wt * a.tiles_tok;   // token tile (fast: neighbours share weights)
    if (a.swap) {
        it.w0 = wt * BM;
        it.tok0 = tt * BN;
    } else {
        it.w0 = wt * BN;
        it.tok0 = tt * BM;
    }
    it.kb0 = static_cast<int>((static_cast<long long>(it.split) * a.G) / a.split);
    it.kb1 = static_cast<int>((static_cast<long long>(it.split + 1) * a.G) / a.split);
    return it;
}

__device__ __forceinline__ float act_scale(const KArgs& a, int m, int kb) {
    if (m >= a.M) return 0.0f;
    if (a.ue8m0) {
        const uint32_t w =
            __ldg(static_cast<const uint32_t*>(a.sa) + static_cast<int64_t>(kb >> 2) * a.Mp + m);
        return __uint_as_float(((w >> (8 * (kb & 3))) & 0xFFu) << 23);
    }
    return __ldg(static_cast<const float*>(a.sa) + static_cast<int64_t>(kb) * a.Mp + m);
}

__device__ __forceinline__ void store_out1(void* out, int dtype, int64_t idx, float v) {
    if (dtype == FP8BQ_BF16)
        static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
    else if (dtype == FP8BQ_FP16)
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
    else
        static_cast<float*>(out)[idx] = v;
}

// Stores 8 consecutive columns starting at out[idx] (16- or 32-byte chunk).
__device__ __forceinline__ void store_out8(void* out, int dtype, int64_t idx, float v0, float v1,
                                           float v2, float v3, float v4, float v5, float v6,
                                           float v7) {
    const float v[8] = {v0, v1, v2, v3, v4, v5, v6, v7};
    if (dtype == FP8BQ_FP32) {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
        p[0] = make_float4(v[0], v[1], v[2], v[3]);
        p[1] = make_float4(v[4], v[5], v[6], v[7]);
        return;
    }
    uint32_t w[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (dtype == FP8BQ_BF16) {
            __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        } else {
            __half2 h = __floats2half2_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&h);
        }
    }
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(out) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
}

// Wait with only a time limit (used while draining after an abort).
__device__ __forceinline__ void mbar_wait_drain(uint64_t* bar, uint32_t parity,
                                                uint64_t timeout_ns) {
    const uint64_t t0 = global_timer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (global_timer_ns() - t0 > timeout_ns) return;
    }
}

template <int BN>
__global__ void __launch_bounds__(Cfg<BN>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_mma_m,  // MMA-M operand [rows, K]
                const __grid_constant__ CUtensorMap tm_mma_n,  // MMA-N operand [rows, K]
                const KArgs a) {
    using C = Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                                // STAGES x [128 rows x 128 B]
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;       // STAGES x [BN rows x 128 B]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::STAGES * C::STAGE_BYTES);
    uint64_t* empty = full + C::STAGES;
    uint64_t* tfull = empty + C::STAGES;
    uint64_t* tempty = tfull + C::NBUF;
    uint64_t* mma_done = tempty + C::NBUF;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < C::NBUF; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], C::EPI_WARPS);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_mma_m);
        tma_prefetch_desc(&tm_mma_n);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    // Programmatic dependent launch: everything above overlapped the tail of
    // the previous kernel; inputs are read only after it has finished.
    pdl_wait_prior_grid();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t tmo = a.timeout_ns;
    const int code = static_cast<int>(FP8BQ_ERR_DEVICE_TIMEOUT);

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            // weights stream once; activations are re-read by other tiles
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            const uint64_t pol_m = a.swap ? pol_w : pol_a;
            const uint64_t pol_n = a.swap ? pol_a : pol_w;
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            for (int item = blockIdx.x; item < a.num_items; item += gridDim.x) {
                const Item it = decode_item<BN>(a, item);
                const int row_m = a.swap ? it.w0 : it.tok0;
                const int row_n = a.swap ? it.tok0 : it.w0;
                bool ok = true;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status, tmo,
                                           code)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    tma_load_2d_hint(sA + stage * C::A_BYTES, &tm_mma_m, &full[stage], kb * BK,
                                     row_m, pol_m);
                    tma_load_2d_hint(sB + stage * C::B_BYTES, &tm_mma_n, &full[stage], kb * BK,
                                     row_n, pol_n);
                    ++fills;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            // Let every issued copy land before the CTA can exit.
            const long long first = fills > C::STAGES ? fills - C::STAGES : 0;
            for (long long f = first; f < fills; ++f)
                mbar_wait_drain(&full[f % C::STAGES], static_cast<uint32_t>((f / C::STAGES) & 1),
                                tmo);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
            int stage = 0, buf = 0;
            uint32_t phase = 0, bphase = 0;
            for (int item = blockIdx.x; item < a.num_items; item += gridDim.x) {
                const Item it = decode_item<BN>(a, item);
                bool ok = true;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (!mbar_wait_bounded(&tempty[buf], bphase ^ 1u, abort_flag, a.status, tmo,
                                           code) ||
                        !mbar_wait_bounded(&full[stage], phase, abort_flag, a.status, tmo, code)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_addr(sA + stage * C::A_BYTES);
                    const uint32_t b_addr = smem_addr(sB + stage * C::B_BYTES);
                    const uint32_t d_addr = tmem_base + static_cast<uint32_t>(buf * BN);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; ++kk)
                        mma_f8f6f4(d_addr, smem_desc_k128_sw128(a_addr + kk * 32),
                                   smem_desc_k128_sw128(b_addr + kk * 32), idesc, kk > 0 ? 1u : 0u);
                    mma_commit(&empty[stage]);
                    mma_commit(&tfull[buf]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (++buf == C::NBUF) {
                        buf = 0;
                        bphase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            mma_commit(mma_done);
            mbar_wait_drain(mma_done, 0, tmo);
        }
    } else {
        // ------------------------------------------------ promotion/epilogue
        const int ew = warp - 2;
        const int quad = warp & 3;   // TMEM lanes this warp may access
        const int chalf = ew >> 2;   // column half (8 epilogue warps)
        const int row = quad * 32 + lane;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                static_cast<uint32_t>(chalf * C::CPT);
        constexpr int SA_REGS = C::CPT >= 32 ? C::CPT / 32 : 1;
        int buf = 0;
        uint32_t bphase = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < a.num_items && ok; item += gridDim.x) {
            const Item it = decode_item<BN>(a, item);
            float acc[C::CPT];
#pragma unroll
            for (int j = 0; j < C::CPT; ++j) acc[j] = 0.0f;

            // Per-slab scale factors.  Normal: one factor per thread (its row
            // is a token m, its columns lie in one 128-wide weight block).
            // Swap-AB: sw is uniform over the tile (128 weight rows = one
            // block); sa varies per column (token), held one per lane and
            // broadcast by shuffles.
            const int m_row = it.tok0 + row;                       // normal
            const int nb_norm = (it.w0 + chalf * C::CPT) / BK;     // normal
            const int nb_swap = it.w0 / BK;                        // swap
            const int tok_col0 = it.tok0 + chalf * C::CPT;         // swap
            const int NB = (a.N + BK - 1) / BK;

            auto load_factor = [&](int kb, float (&sreg)[SA_REGS], float& sw) {
                if (!a.swap) {
                    const float s_w = nb_norm < NB ? __ldg(a.sw + static_cast<int64_t>(nb_norm) * a.G + kb) : 0.0f;
                    sreg[0] = act_scale(a, m_row, kb);
                    sw = s_w;
                } else {
                    sw = __ldg(a.sw + static_cast<int64_t>(nb_swap) * a.G + kb);
#pragma unroll
                    for (int r = 0; r < SA_REGS; ++r) {
                        const int c = r * 32 + lane;
                        sreg[r] = c < C::CPT ? act_scale(a, tok_col0 + c, kb) : 0.0f;
                    }
                }
            };

            float sa_next[SA_REGS], sw_next;
            load_factor(it.kb0, sa_next, sw_next);
            for (int kb = it.kb0; kb < it.kb1; ++kb) {
                float sa_cur[SA_REGS];
#pragma unroll
                for (int r = 0; r < SA_REGS; ++r) sa_cur[r] = sa_next[r];
                const float sw_cur = sw_next;
                if (kb + 1 < it.kb1) load_factor(kb + 1, sa_next, sw_next);

                // lane 0 waits (bounded), the warp follows its verdict, so the
                // warp-collective TMEM loads below are always reached together
                int got = 1;
                if (lane == 0)
                    got = mbar_wait_bounded(&tfull[buf], bphase, abort_flag, a.status, tmo, code)
                              ? 1
                              : 0;
                got = __shfl_sync(0xFFFFFFFFu, got, 0);
                if (!got) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t t_buf = t_lane + static_cast<uint32_t>(buf * BN);
                const float f_norm = sa_cur[0] * sw_cur;
#pragma unroll
                for (int c0 = 0; c0 < C::CPT; c0 += 16) {
                    uint32_t r[16];
                    tmem_ld16(t_buf + c0, r);
                    tmem_ld_wait();
                    if (c0 + 16 == C::CPT) {
                        // all of this buffer is in registers: hand it back
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tempty[buf]);
                    }
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int col = c0 + j;
                        float f;
                        if (!a.swap) {
                            f = f_norm;
                        } else {
                            f = __shfl_sync(0xFFFFFFFFu, sa_cur[col >> 5], col & 31) * sw_cur;
                        }
                        acc[col] = fmaf(__uint_as_float(r[j]), f, acc[col]);
                    }
                }
                if (++buf == C::NBUF) {
                    buf = 0;
                    bphase ^= 1u;
                }
            }
            if (!ok) break;

            // ---------------------------------------------- split-K reduction
            // Each epilogue warp owns a fixed 32-row x CPT-column sub-block of
            // the tile and takes its own ticket for it, so no barrier between
            // warps is needed (and none can be left waiting after an abort).
            if (a.split > 1) {
                float* part = a.partials + static_cast<int64_t>(it.tile) * a.split * (BM * BN);
                float* mine = part + static_cast<int64_t>(it.split) * (BM * BN);
#pragma unroll
                for (int j = 0; j < C::CPT; ++j)
                    __stcg(mine + (chalf * C::CPT + j) * BM + row, acc[j]);
                __threadfence();
                __syncwarp();
                unsigned* ctr = a.counters + static_cast<int64_t>(it.tile) * kCountersPerTile + ew;
                unsigned prev = 0;
                if (lane == 0) prev = atomicAdd(ctr, 1u);
                prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
                if (prev != static_cast<unsigned>(a.split - 1)) continue;
                __threadfence();
#pragma unroll
                for (int j = 0; j < C::CPT; ++j) {
                    const int64_t off = (chalf * C::CPT + j) * BM + row;
                    float v = it.split == 0 ? acc[j] : __ldcg(part + off);
                    for (int s = 1; s < a.split; ++s)
                        v += (s == it.split) ? acc[j]
                                             : __ldcg(part + static_cast<int64_t>(s) * (BM * BN) + off);
                    acc[j] = v;
                }
                if (lane == 0) *ctr = 0u;  // ready for the next call
            }

            // ------------------------------------------------------- store
            if (!a.swap) {
                const int m = it.tok0 + row;
                if (m < a.M) {
                    const int n0 = it.w0 + chalf * C::CPT;
#pragma unroll
                    for (int j = 0; j < C::CPT; j += 8)
                        if (n0 + j < a.N)
                            store_out8(a.out, a.out_dtype, static_cast<int64_t>(m) * a.N + n0 + j,
                                       acc[j], acc[j + 1], acc[j + 2], acc[j + 3], acc[j + 4],
                                       acc[j + 5], acc[j + 6], acc[j + 7]);
                }
            } else {
                const int n = it.w0 + row;
                if (n < a.N) {
#pragma unroll
                    for (int j = 0; j < C::CPT; ++j) {
                        const int t = tok_col0 + j;
                        if (t < a.M) store_out1(a.out, a.out_dtype, static_cast<int64_t>(t) * a.N + n, acc[j]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------------ host

bool encode_map(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows, uint32_t box_rows) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int BN>
cudaError_t launch_bn(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    using C = Cfg<BN>;
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        err = cudaFuncSetAttribute(gemm_kernel<BN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   C::SMEM);
        if (err != cudaSuccess) return err;
        attr_done[dev] = 1;
    }
    const bool swap = p.kind == FP8BQ_KIND_SWAP_AB;
    CUtensorMap tm_m, tm_n;
    const uint64_t K = static_cast<uint64_t>(g.K);
    bool ok;
    if (swap) {
        ok = encode_map(&tm_m, g.w_q, K, static_cast<uint64_t>(g.N), BM) &&
             encode_map(&tm_n, g.a_q, K, static_cast<uint64_t>(g.M), BN);
    } else {
        ok = encode_map(&tm_m, g.a_q, K, static_cast<uint64_t>(g.M), BM) &&
             encode_map(&tm_n, g.w_q, K, static_cast<uint64_t>(g.N), BN);
    }
    if (!ok) return cudaErrorInvalidValue;

    KArgs a;
    a.M = static_cast<int>(g.M);
    a.N = static_cast<int>(g.N);
    a.G = static_cast<int>(g.K / BK);
    a.Mp = static_cast<int>(pad_rows4(g.M));
    a.swap = swap ? 1 : 0;
    a.tiles_tok = p.tiles_tok;
    a.split = p.split;
    a.num_items = p.num_items;
    a.ue8m0 = g.ue8m0;
    a.out_dtype = g.out_dtype;
    a.sa = g.a_s;
    a.sw = g.w_s;
    a.out = g.out;
    // workspace: [tile counters: fixed kCounterRegion prefix] [fp32 partial tiles]
    a.counters = p.split > 1 ? static_cast<unsigned*>(g.workspace) : nullptr;
    a.partials = p.split > 1 ? reinterpret_cast<float*>(static_cast<uint8_t*>(g.workspace) +
                                                        kCounterRegion + g.ws_data_offset)
                             : nullptr;
    a.status = g.status;
    a.timeout_ns = g.timeout_ns;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(p.grid));
    cfg.blockDim = dim3(C::THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = g.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_kernel<BN>, tm_m, tm_n, a);
}

}  // namespace

static size_t workspace_for(int tiles, int split, int bn) {
    if (split <= 1) return 0;
    return kCounterRegion + static_cast<size_t>(tiles) * split * BM * bn * sizeof(float);
}

bool make_gemm_plan(int64_t M, int64_t N, int64_t K, const fp8bq_variant& v, int num_sms,
                    GemmPlan* p) {
    const int G = static_cast<int>(K / BK);
    const bool swap = v.kind == FP8BQ_KIND_SWAP_AB;
    if (v.kind != FP8BQ_KIND_SWAP_AB && v.kind != FP8BQ_KIND_NORMAL) return false;
    if (swap) {
        if (v.block_n != 16 && v.block_n != 32 && v.block_n != 64 && v.block_n != 128) return false;
    } else {
        if (v.block_n != 128 && v.block_n != 256) return false;
    }
    if (v.split < 1 || v.split > 64 || v.split > G) return false;
    if (v.grid < 0) return false;
    p->kind = v.kind;
    p->bn = v.block_n;
    p->split = v.split;
    if (swap) {
        p->tiles_tok = static_cast<int>((M + v.block_n - 1) / v.block_n);
        p->tiles_w = static_cast<int>((N + BM - 1) / BM);
    } else {
        p->tiles_tok = static_cast<int>((M + BM - 1) / BM);
        p->tiles_w = static_cast<int>((N + v.block_n - 1) / v.block_n);
    }
    const long long tiles = static_cast<long long>(p->tiles_tok) * p->tiles_w;
    const long long items = tiles * v.split;
    if (items <= 0 || items > (1LL << 30)) return false;
    // split-K tickets live in the fixed counter prefix of the workspace
    if (v.split > 1 && tiles * kCountersPerTile * 4 > kCounterRegion) return false;
    p->num_items = static_cast<int>(items);
    const int g = v.grid > 0 ? v.grid : num_sms;
    p->grid = static_cast<int>(items < g ? items : g);
    p->ws_bytes = workspace_for(static_cast<int>(tiles), v.split, v.block_n);
    return true;
}

cudaError_t launch_gemm(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    if (p.kind == FP8BQ_KIND_SWAP_AB) {
        switch (p.bn) {
            case 16: return launch_bn<16>(p, g, stream);
            case 32: return launch_bn<32>(p, g, stream);
            case 64: return launch_bn<64>(p, g, stream);
            case 128: return launch_bn<128>(p, g, stream);
        }
    } else {
        switch (p.bn) {
            case 128: return launch_bn<128>(p, g, stream);
            case 256: return launch_bn<256>(p, g, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace fp8bq

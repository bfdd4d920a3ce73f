// gemm_impl.cuh -- the GEMM kernels and their host-side launchers (template
// code).  Each gemm_*.cu translation unit includes this file and instantiates
// the launchers of a few tile shapes, so the shapes compile in parallel;
// gemm.cu holds the planner and the dispatch over those launchers.
//
// block-scaled FP8 GEMM on tcgen05 tensor cores (sm_103a).
//
//   out[m,n] = sum_kb sa[m,kb] * sw[n/128,kb] * P_kb[m,n],
//   P_kb[m,n] = sum_{k in slab kb} a[m,k] * w[n,k]        (FP8 x FP8 -> fp32)
//
// "vLLM DeepGEMM FP8 Block GEMM 基准测试" §4.2 describes the promotion (each
// K block's dot product times a_s[:,None]*b_s[None,:] added to an fp32
// accumulator); "用 Helion 为 vLLM 构建高性能可移植线性后端", 内核实现, the
// Split-K and Swap-AB variants.
//
// Kernels in this file (the host picks one per plan, GemmPlan::rowwise/mx):
//   gemm_kernel     promotion on the CUDA cores (fp32 or UE8M0 scales);
//                   GR: grouped (MoE) tiles; PL = 2: block INT8 as two e4m3
//                   planes (four cross products per K step)
//   gemm_mx_kernel  block-scaled MMA for UE8M0 scales; FQ: activation quant
//                   fused into the producer; RW = 1: rowwise (FP8_Dynamic)
//                   scales applied in the epilogue; RW = 2: rowwise INT8 as
//                   two e4m3 planes
//   gemm_i8_kernel  warp-level int8 MMA (mma.sync), rowwise INT8 or (BLK)
//                   block INT8 with per-slab promotion
// All share the work schedule (WorkIter: split-K items or stream-K shares),
// the tile origins, the bounded waits and the split-part ticket protocol.
//
// Design (one CTA per SM, persistent over its work):
//   warp 0     TMA producer: per K slab, one 128x128 tile of the MMA-M operand
//              and one BNx128 tile of the MMA-N operand into a STAGES-deep
//              shared-memory ring (128-byte swizzle, K-major), and the slab's
//              scales (activation scales of the tile's tokens, the weight
//              block's scale) into a separate SR-deep scale ring.
//   warp 1     MMA issuer: four tcgen05.mma (K = 32 each) per slab into a
//              fresh TMEM accumulator buffer; commits free the smem stage and
//              publish the TMEM buffer.  Warp 1 also owns the TMEM allocation.
//   warps 2..  promotion/epilogue: per slab, tcgen05.ld the slab's fp32 sums,
//              release the TMEM buffer, and fold them into a register
//              accumulator with fma(P, sa*sw, acc), the scales read from the
//              scale ring.  NBUF TMEM buffers let the MMA of slab kb+1 overlap
//              the promotion of slab kb.
//
// Work: the output is cut into tiles; a tile's K slabs are split into
// segments processed by different CTAs when the tiles alone cannot fill the
// GPU.  Two schedules:
//   split-K (split >= 1): work item = (tile, split s), items dealt round-robin
//       over the CTAs, split s covering slabs [s*G/S, (s+1)*G/S);
//   stream-K (split == 0): the tiles x G (tile, slab) units are divided into
//       equal contiguous ranges, one per CTA, so every CTA streams the same
//       number of slabs; a range holds at most two partial tiles.
// A tile finished by one segment is stored directly.  Otherwise every segment
// writes an fp32 partial tile to the workspace and takes a ticket (one per
// epilogue warp and tile); the last to arrive sums the partials in K order
// and stores, so results are run-to-run bit-stable and no CTA ever waits for
// another.
// Swap-AB (decode): the MMA-M operand is the weight (128 rows of n), the
// MMA-N operand the tokens (BN = 16..128), so small M does not waste a
// 128-row MMA; the epilogue writes the transposed tile back into [M,N].
//
// Every wait is bounded (global-timer limit); on expiry the CTA records
// FP8BQ_ERR_DEVICE_TIMEOUT in the status word, lets its in-flight copies and
// MMAs land (again bounded), frees its TMEM and returns.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8bq {

namespace {

constexpr int BM = 128;              // MMA M
constexpr int BK = 128;              // K slab (one scale block)
constexpr int kCountersPerTile = 8;  // one split-K ticket per epilogue warp
constexpr int SR = 16;               // scale ring depth (slabs)
constexpr int SLOT_BYTES = 768;      // per slab: 128 act scales, 2 weight-scale chunks
constexpr int SLOT_SW = 512;         // weight-scale chunk c at SLOT_SW + c * SLOT_SW_STEP
constexpr int SLOT_SW_STEP = 128;    // (TMA destinations 128-byte aligned)

// PL = 2 (block INT8 as two e4m3 planes, 128-row tiles): a stage holds both
// planes of both operands of one logical K slab, and the slab's MMA is the
// four cross products per 32-wide K step into its TMEM buffer (see MxCfg).
template <bool SWAP, int BN, int WM = BM, int PL = 1>
struct Cfg {
    // MMA-M rows of a tile: tokens (normal, always 128) or weight rows (swap:
    // 128, or 64 with the M = 64 MMA, whose accumulator row r sits at TMEM
    // lane 32*(r/16) + r%16, i.e. lanes 0-15 of each 32-lane quarter)
    static constexpr int MR = SWAP ? WM : BM;
    static_assert(MR == 128 || (SWAP && MR == 64), "tile rows");
    static constexpr int ROWS_PER_QUAD = MR / 4;
    static_assert(PL == 1 || MR == 128, "planes: 128-row tiles");
    static constexpr int A_BYTES = MR * BK;  // one plane of one slab
    static constexpr int B_BYTES = BN * BK;
    static constexpr int A_STAGE = PL * A_BYTES;
    static constexpr int B_STAGE = PL * B_BYTES;
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE;
    // 64-row weight tiles carry half the bytes per stage, so twice the stages
    // keep the same bytes in flight; two planes take twice the room
    static constexpr int STAGES_128 = BN <= 16 ? 10 : BN <= 32 ? 9 : BN <= 64 ? 8 : BN <= 128 ? 6 : 4;
    static constexpr int STAGES_PL = STAGES_128 / PL < 2 ? 2 : STAGES_128 / PL;
    static constexpr int STAGES = MR == 128 ? STAGES_PL : (BN <= 16 ? 18 : 15);
    // TMEM accumulator buffers: as many as fit in the 512 columns (at most 8)
    static constexpr int NBUF = 512 / BN >= 8 ? 8 : 512 / BN;
    static constexpr int TMEM_NEED = NBUF * BN;
    static constexpr int TMEM_COLS = TMEM_NEED <= 32    ? 32
                                     : TMEM_NEED <= 64  ? 64
                                     : TMEM_NEED <= 128 ? 128
                                     : TMEM_NEED <= 256 ? 256
                                                        : 512;
    // 4 epilogue warps (one per TMEM lane quadrant) below 64 columns; wider
    // tiles split their columns over 8 warps
    static constexpr int EPI_WARPS = BN >= 64 ? 8 : 4;
    static constexpr int CPT = BN / (EPI_WARPS / 4);  // accumulator columns per thread
    // 128 accumulators per thread do not fit the 168 registers a 320-thread
    // CTA gets; such tiles run warpgroup 0 (producer, MMA, 2 idle warps) on
    // few registers and hand the rest to the two epilogue warpgroups
    // (setmaxnreg).  The shares must add up to at most the launch total.
    static constexpr bool REGSPLIT = CPT >= 128;
    static constexpr int EPI_FIRST = REGSPLIT ? 4 : 2;  // first epilogue warp
    static constexpr int THREADS = 32 * EPI_FIRST + 32 * EPI_WARPS;
    static constexpr int REG_ROLE = 64;   // per thread, warpgroup 0
    static constexpr int REG_EPI = 208;   // per thread, epilogue warpgroups
    static constexpr int REG_MIN_LAUNCH =  // registers per thread the launch must provide
        (REG_ROLE * 128 + REG_EPI * 32 * EPI_WARPS + THREADS - 1) / THREADS;
    static constexpr int SRC = STAGES + 4 > SR ? STAGES + 4 : SR;  // scale ring depth
    static constexpr int RING_OFF = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = RING_OFF + SRC * SLOT_BYTES;
    static constexpr int BAR_BYTES = 8 * (2 * STAGES + 2 * SRC + 2 * NBUF + 1) + 16;
    static constexpr int FACT_OFF = (BAR_OFF + BAR_BYTES + 15) / 16 * 16;  // per-warp factors
    static constexpr int SMEM = 1024 + FACT_OFF + EPI_WARPS * CPT * 4;
    static constexpr int CHUNK = (REGSPLIT || CPT == 32) ? 32 : 16;  // TMEM columns per load
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
    static_assert(CPT % 16 == 0, "TMEM loads are 16 columns wide");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

struct KArgs {
    int M, N, G;
    int NB;          // weight row blocks
    int swap;        // MMA-M operand is the weight
    int tiles_tok;   // token tiles (MMA-M tiles when !swap, MMA-N tiles when swap)
    int tiles;
    int split;       // >= 1: split-K round robin; 0: stream-K
    int num_items;   // split-K: tiles * split
    long long units; // stream-K: tiles * G
    int ue8m0;
    int out_dtype;
    int prefetch_w;  // weights may be read before the previous grid finishes
    const float* w_s;  // weight scales [NB][G] (read directly by the fused-quant path);
                       // rowwise scales: one per weight row [N]
    const float* s_tok;  // rowwise scales: one per token [M]
    void* out;
    float* partials;
    unsigned* counters;
    int* status;
    unsigned long long timeout_ns;
    // grouped problem (E > 0): E stacked problems of m_max token rows each;
    // M = E * m_max, N is one expert's width (and the output row length)
    int E;
    int m_max;
    int tiles_e;        // tiles per expert (tiles_tok * tiles_w)
    int tiles_w;        // weight tiles per expert
    int tok_tile;       // tokens per tile (BN when swap, BM otherwise)
    const int* counts;  // valid token rows of each expert (device)
};

// One contiguous run of K slabs of one tile.
struct Seg {
    int tile;
    int kb0, kb1;
    int part;    // index of this segment among the tile's segments (K order)
    int nparts;  // segments of this tile (1: the tile is stored directly)
};

// Stream-K ownership: CTA c owns units [c*T/P, (c+1)*T/P).
__device__ __forceinline__ long long sk_begin(long long c, long long T, long long P) {
    return c * T / P;
}
__device__ __forceinline__ int sk_owner(long long u, long long T, long long P) {
    return static_cast<int>(((u + 1) * P - 1) / T);
}

// Grouped problems: valid token rows of expert e (its count clamped to
// [0, m_max]).
__device__ __forceinline__ int expert_rows(const KArgs& a, int e) {
    const int c = __ldg(a.counts + e);
    return c < 0 ? 0 : (c > a.m_max ? a.m_max : c);
}

// Iterates this CTA's segments in order (identically in every role).
//
// Grouped problems number only the tiles that hold rows: expert by expert,
// within an expert weight tile by weight tile and its occupied token tiles,
// and (tile, split part) items go round robin over the CTAs, so every CTA
// gets the same number of items to within one whatever the counts are.  An
// iterator walks the experts forward as its item index grows.  GR (grouped)
// is a template parameter, so the plain kernels carry none of this.
template <bool GR>
struct WorkIter {
    long long u, u_end;  // stream-K
    int item;            // split-K
    int ge;              // grouped: expert of the current items
    int gbase;           // grouped: index of expert ge's first item
    int gnt;             // grouped: token tiles of expert ge holding rows

    __device__ void init(const KArgs& a) {
        if (a.split == 0) {
            u = sk_begin(blockIdx.x, a.units, gridDim.x);
            u_end = sk_begin(blockIdx.x + 1, a.units, gridDim.x);
        } else {
            item = blockIdx.x;
            ge = -1;
            gbase = 0;
            gnt = 0;
        }
    }

    __device__ bool next(const KArgs& a, Seg& s) {
        if (a.split == 0) {
            if (u >= u_end) return false;
            s.tile = static_cast<int>(u / a.G);
            s.kb0 = static_cast<int>(u - static_cast<long long>(s.tile) * a.G);
            const long long left = u_end - u;
            s.kb1 = left < a.G - s.kb0 ? s.kb0 + static_cast<int>(left) : a.G;
            const long long t0 = static_cast<long long>(s.tile) * a.G;
            const int c_first = sk_owner(t0, a.units, gridDim.x);
            const int c_last = sk_owner(t0 + a.G - 1, a.units, gridDim.x);
            s.nparts = c_last - c_first + 1;
            s.part = static_cast<int>(blockIdx.x) - c_first;
            u += s.kb1 - s.kb0;
            return true;
        }
        if constexpr (GR) {
            if (ge >= a.E) return false;
            for (;;) {
                if (ge >= 0) {
                    const int n_items = gnt * a.tiles_w * a.split;
                    if (item < gbase + n_items) break;
                    gbase += n_items;
                }
                if (ge >= a.E - 1) {
                    ge = a.E;
                    return false;
                }
                ++ge;
                gnt = (expert_rows(a, ge) + a.tok_tile - 1) / a.tok_tile;
            }
            const int local = item - gbase;
            const int tl = local / a.split;
            s.part = local - tl * a.split;
            const int wt = tl / gnt;
            s.tile = ge * a.tiles_e + wt * a.tiles_tok + (tl - wt * gnt);
        } else {
            if (item >= a.num_items) return false;
            s.tile = item / a.split;
            s.part = item - s.tile * a.split;
        }
        item += gridDim.x;
        s.nparts = a.split;
        s.kb0 = static_cast<int>((static_cast<long long>(s.part) * a.G) / a.split);
        s.kb1 = static_cast<int>((static_cast<long long>(s.part + 1) * a.G) / a.split);
        return true;
    }
};

// Workspace slot of segment `p` of `tile`.
__device__ __forceinline__ int64_t part_slot(const KArgs& a, int tile, int p) {
    if (a.split == 0) {
        const long long t0 = static_cast<long long>(tile) * a.G;
        const int c = sk_owner(t0, a.units, gridDim.x) + p;
        const long long b = sk_begin(c, a.units, gridDim.x);
        return 2 * static_cast<int64_t>(c) + ((b / a.G) == tile ? 0 : 1);
    }
    return static_cast<int64_t>(tile) * a.split + p;
}

struct TileOrigin {
    int tok0;     // first token (row of the stacked operand)
    int w0;       // first weight row (row of the stacked weights)
    int tok_end;  // tokens [tok0, tok_end) are stored
    int w_end;    // weight rows [w0, w_end) are stored
    int col0;     // output column of weight row n: n - col0
};

template <bool SWAP, int BN, int WM, bool GR>
__device__ __forceinline__ TileOrigin tile_origin(const KArgs& a, int tile) {
    int tok_base = 0, w_base = 0;
    TileOrigin o;
    o.tok_end = a.M;
    if constexpr (GR) {
        const int e = tile / a.tiles_e;
        tile -= e * a.tiles_e;
        tok_base = e * a.m_max;
        w_base = e * a.N;
        o.tok_end = tok_base + expert_rows(a, e);
    }
    o.w_end = w_base + a.N;
    o.col0 = w_base;
    const int wt = tile / a.tiles_tok;       // weight tile (slow)
    const int tt = tile - wt * a.tiles_tok;  // token tile (fast: neighbours share weights)
    if (SWAP) {
        o.w0 = w_base + wt * WM;
        o.tok0 = tok_base + tt * BN;
    } else {
        o.w0 = w_base + wt * BN;
        o.tok0 = tok_base + tt * BM;
    }
    return o;
}

// Rowwise scales: v[j] *= s_tok[token] * w_s[weight row] for accumulator row
// `row` and columns [c0, c0 + NC) of the tile (positions outside the tile's
// stored range get 0 and are not stored).
template <bool SWAP, int NC>
__device__ __forceinline__ void rowwise_scale(const KArgs& a, const TileOrigin& o, int row,
                                              int c0, float* v) {
    if constexpr (SWAP) {
        const int n = o.w0 + row;
        const float sw = n < o.w_end ? __ldg(a.w_s + n) : 0.0f;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            const int t = o.tok0 + c0 + j;
            v[j] *= (t < o.tok_end ? __ldg(a.s_tok + t) : 0.0f) * sw;
        }
    } else {
        const int m = o.tok0 + row;
        const float st = m < o.tok_end ? __ldg(a.s_tok + m) : 0.0f;
#pragma unroll
        for (int j = 0; j < NC; ++j) {
            const int n = o.w0 + c0 + j;
            v[j] *= st * (n < o.w_end ? __ldg(a.w_s + n) : 0.0f);
        }
    }
}

// The PL planes of K slab kb of one operand (PL = 2: the two e4m3 planes of
// INT8 codes, at K columns 256 kb and 256 kb + 128 of the planar operand).
template <int PL>
__device__ __forceinline__ void tma_load_slab(uint8_t* dst, const CUtensorMap* map,
                                              uint64_t* bar, int kb, int row, uint64_t pol,
                                              int plane_bytes) {
#pragma unroll
    for (int p = 0; p < PL; ++p)
        tma_load_2d_hint(dst + p * plane_bytes, map, bar, (PL * kb + p) * BK, row, pol);
}

__device__ __forceinline__ float ue8m0_value(uint32_t word, int kb) {
    return __uint_as_float(((word >> (8 * (kb & 3))) & 0xFFu) << 23);
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
    if (dtype == FP8BQ_FP32) {
        float4* p = reinterpret_cast<float4*>(static_cast<float*>(out) + idx);
        p[0] = make_float4(v0, v1, v2, v3);
        p[1] = make_float4(v4, v5, v6, v7);
        return;
    }
    const float v[8] = {v0, v1, v2, v3, v4, v5, v6, v7};
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

// Warp-uniform bounded wait: lane 0 waits, the warp follows its verdict, so
// the warp-collective instructions after it are always reached together.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          int* status, uint64_t tmo, int code) {
    int got = 1;
    if ((threadIdx.x & 31) == 0) got = mbar_wait_bounded(bar, parity, abort, status, tmo, code);
    return __shfl_sync(0xFFFFFFFFu, got, 0) != 0;
}

template <bool SWAP, int BN, int WM, bool GR, int PL = 1>
__global__ void __launch_bounds__(Cfg<SWAP, BN, WM, PL>::THREADS, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tm_mma_m,  // MMA-M operand [rows, K] e4m3
                const __grid_constant__ CUtensorMap tm_mma_n,  // MMA-N operand [rows, K] e4m3
                const __grid_constant__ CUtensorMap tm_sa,     // act scales [cols][Mp] 4-byte
                const __grid_constant__ CUtensorMap tm_sw,     // weight scales, flat fp32
                const KArgs a) {
    using C = Cfg<SWAP, BN, WM, PL>;
    constexpr int SR = C::SRC;  // scale ring depth of this configuration
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                            // STAGES x PL x [MR rows x 128 B]
    uint8_t* sB = smem + C::STAGES * C::A_STAGE;   // STAGES x PL x [BN rows x 128 B]
    uint8_t* ring = smem + C::RING_OFF;            // SR x SLOT_BYTES
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* empty = full + C::STAGES;
    uint64_t* sfull = empty + C::STAGES;
    uint64_t* sempty = sfull + SR;
    uint64_t* tfull = sempty + SR;
    uint64_t* tempty = tfull + C::NBUF;
    uint64_t* mma_done = tempty + C::NBUF;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* fact = reinterpret_cast<float*>(smem + C::FACT_OFF);  // EPI_WARPS x CPT

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int s = 0; s < SR; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sempty[s], C::EPI_WARPS);
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
        tma_prefetch_desc(&tm_sa);
        tma_prefetch_desc(&tm_sw);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    // Every warp reconverges before a CTA barrier: bar.sync counts warps, so a
    // warp must reach it with all its lanes at once.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t tmo = a.timeout_ns;
    const int code = static_cast<int>(FP8BQ_ERR_DEVICE_TIMEOUT);
    if constexpr (C::REGSPLIT) {
        // warpgroup 0 gives registers back; the epilogue warpgroups take
        // them at the start of their branch (so the compiler budgets that
        // code with REG_EPI registers)
        if (warp < 4) asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(C::REG_ROLE));
    }

    // Programmatic dependent launch: the set-up above overlapped the tail of
    // the previous kernel.  When the caller guarantees that the weights were
    // complete before the previous kernel started (the fused linear path),
    // the producer starts streaming the first weight tiles now; everything
    // else is read or written only after the previous grid has finished.
    int prefetched = 0;
    if (a.prefetch_w && warp == 0 && lane == 0) {
        WorkIter<GR> wi;
        wi.init(a);
        Seg sg;
        if (wi.next(a, sg)) {
            const TileOrigin o = tile_origin<SWAP, BN, WM, GR>(a, sg.tile);
            const int nslab = sg.kb1 - sg.kb0;
            prefetched = nslab < C::STAGES ? nslab : C::STAGES;
            for (int i = 0; i < prefetched; ++i) {
                mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
                if (SWAP)
                    tma_load_slab<PL>(sA + i * C::A_STAGE, &tm_mma_m, &full[i], sg.kb0 + i, o.w0,
                                      policy_evict_first(), C::A_BYTES);
                else
                    tma_load_slab<PL>(sB + i * C::B_STAGE, &tm_mma_n, &full[i], sg.kb0 + i, o.w0,
                                      policy_evict_first(), C::B_BYTES);
            }
        }
    }
    pdl_wait_prior_grid();
    pdl_launch_dependents();
    // bytes one scale slot receives: the activation scales of the tile's
    // tokens plus one (swap-AB, 128-row weight tile) or two (256-wide weight
    // tile) 16-byte chunks of weight scales
    const int sw_chunks = (!SWAP && BN > BM) ? 2 : 1;
    const uint32_t slot_tx = 4u * (SWAP ? BN : BM) + 16u * sw_chunks;

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            // weights stream once; activations are re-read by other tiles
            const uint64_t pol_w = policy_evict_first();
            const uint64_t pol_a = policy_evict_last();
            const uint64_t pol_m = SWAP ? pol_w : pol_a;
            const uint64_t pol_n = SWAP ? pol_a : pol_w;
            int stage = 0, slot = 0;
            uint32_t phase = 0, sphase = 0;
            long long fills = 0, sfills = 0;
            WorkIter<GR> wi;
            wi.init(a);
            Seg sg;
            bool ok = true;
            while (ok && wi.next(a, sg)) {
                const TileOrigin o = tile_origin<SWAP, BN, WM, GR>(a, sg.tile);
                const int row_m = SWAP ? o.w0 : o.tok0;
                const int row_n = SWAP ? o.tok0 : o.w0;
                const int nb = o.w0 / BK;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (fills < prefetched) {
                        // the weight tile of this stage is already on its way
                        if (SWAP)
                            tma_load_slab<PL>(sB + stage * C::B_STAGE, &tm_mma_n, &full[stage], kb,
                                              row_n, pol_n, C::B_BYTES);
                        else
                            tma_load_slab<PL>(sA + stage * C::A_STAGE, &tm_mma_m, &full[stage], kb,
                                              row_m, pol_m, C::A_BYTES);
                    } else {
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status,
                                               tmo, code)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        tma_load_slab<PL>(sA + stage * C::A_STAGE, &tm_mma_m, &full[stage], kb,
                                          row_m, pol_m, C::A_BYTES);
                        tma_load_slab<PL>(sB + stage * C::B_STAGE, &tm_mma_n, &full[stage], kb,
                                          row_n, pol_n, C::B_BYTES);
                    }
                    ++fills;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (!mbar_wait_bounded(&sempty[slot], sphase ^ 1u, abort_flag, a.status, tmo,
                                           code)) {
                        ok = false;
                        break;
                    }
                    uint8_t* sl = ring + slot * SLOT_BYTES;
                    mbar_arrive_expect_tx(&sfull[slot], slot_tx);
                    tma_load_2d(sl, &tm_sa, &sfull[slot], o.tok0, a.ue8m0 ? (kb >> 2) : kb);
                    const int e0 = nb * a.G + kb;
                    tma_load_2d(sl + SLOT_SW, &tm_sw, &sfull[slot], e0 & ~3, 0);
                    if (sw_chunks == 2)
                        tma_load_2d(sl + SLOT_SW + SLOT_SW_STEP, &tm_sw, &sfull[slot],
                                    (e0 + a.G) & ~3, 0);
                    ++sfills;
                    if (++slot == SR) {
                        slot = 0;
                        sphase ^= 1u;
                    }
                }
            }
            // Let every issued copy land before the CTA can exit.
            for (long long f = fills > C::STAGES ? fills - C::STAGES : 0; f < fills; ++f)
                mbar_wait_drain(&full[f % C::STAGES], static_cast<uint32_t>((f / C::STAGES) & 1),
                                tmo);
            for (long long f = sfills > SR ? sfills - SR : 0; f < sfills; ++f)
                mbar_wait_drain(&sfull[f % SR], static_cast<uint32_t>((f / SR) & 1), tmo);
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_e4m3_f32(C::MR, BN);
            int stage = 0, buf = 0;
            uint32_t phase = 0, bphase = 0;
            WorkIter<GR> wi;
            wi.init(a);
            Seg sg;
            bool ok = true;
            while (ok && wi.next(a, sg)) {
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!mbar_wait_bounded(&tempty[buf], bphase ^ 1u, abort_flag, a.status, tmo,
                                           code) ||
                        !mbar_wait_bounded(&full[stage], phase, abort_flag, a.status, tmo, code)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_addr(sA + stage * C::A_STAGE);
                    const uint32_t b_addr = smem_addr(sB + stage * C::B_STAGE);
                    const uint32_t d_addr = tmem_base + static_cast<uint32_t>(buf * BN);
#pragma unroll
                    for (int kk = 0; kk < BK / 32; ++kk)
#pragma unroll
                        for (int pq = 0; pq < PL * PL; ++pq)  // PL = 2: the four cross products
                            mma_f8f6f4(d_addr,
                                       smem_desc_k128_sw128(a_addr + (pq / PL) * C::A_BYTES + kk * 32),
                                       smem_desc_k128_sw128(b_addr + (pq % PL) * C::B_BYTES + kk * 32),
                                       idesc, (kk > 0 || pq > 0) ? 1u : 0u);
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
            }
            mma_commit(mma_done);
            mbar_wait_drain(mma_done, 0, tmo);
        }
    } else if (warp >= C::EPI_FIRST) {
        // ------------------------------------------------ promotion/epilogue
        if constexpr (C::REGSPLIT)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(C::REG_EPI));
        const int ew = warp - C::EPI_FIRST;
        const int quad = warp & 3;   // TMEM lanes this warp may access
        const int chalf = ew >> 2;   // column half (8 epilogue warps)
        // MMA-M row of this lane; with 64-row tiles lanes 16-31 hold none
        // and skip every store and partial access
        const int row = quad * C::ROWS_PER_QUAD + lane;
        const bool row_ok = lane < C::ROWS_PER_QUAD;
        const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                static_cast<uint32_t>(chalf * C::CPT);
        int buf = 0, slot = 0;
        uint32_t bphase = 0, sphase = 0;
        WorkIter<GR> wi;
        wi.init(a);
        Seg sg;
        bool ok = true;
        while (ok && wi.next(a, sg)) {
            const TileOrigin o = tile_origin<SWAP, BN, WM, GR>(a, sg.tile);
            const int nb = o.w0 / BK;
            float acc[C::CPT];
#pragma unroll
            for (int j = 0; j < C::CPT; ++j) acc[j] = 0.0f;

            for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                if (!warp_wait(&sfull[slot], sphase, abort_flag, a.status, tmo, code) ||
                    !warp_wait(&tfull[buf], bphase, abort_flag, a.status, tmo, code)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint8_t* sl = ring + slot * SLOT_BYTES;
                // weight scale of this warp's columns (swap: the tile's block;
                // normal: block of this column half)
                const int e = (nb + (SWAP ? 0 : (chalf * C::CPT) / BK)) * a.G + kb;
                const int chunk = (SWAP || chalf * C::CPT < BK) ? 0 : 1;
                const float swv =
                    reinterpret_cast<const float*>(sl + SLOT_SW + SLOT_SW_STEP * chunk)[e & 3];
                float f_norm = 0.0f;
                float* fw = fact + ew * C::CPT;
                if (!SWAP) {
                    const float sam = a.ue8m0
                                          ? ue8m0_value(reinterpret_cast<const uint32_t*>(sl)[row], kb)
                                          : reinterpret_cast<const float*>(sl)[row];
                    f_norm = (o.tok0 + row < o.tok_end) ? sam * swv : 0.0f;
                } else {
                    // per-column (token) factors sa[t] * sw, computed once per
                    // slab by the warp's lanes and read back as broadcasts
                    for (int c = lane; c < C::CPT; c += 32) {
                        const int t = chalf * C::CPT + c;
                        const uint32_t w = reinterpret_cast<const uint32_t*>(sl)[t];
                        const float sv = a.ue8m0 ? ue8m0_value(w, kb) : __uint_as_float(w);
                        fw[c] = (o.tok0 + t < o.tok_end) ? sv * swv : 0.0f;
                    }
                    __syncwarp();
                }
                const uint32_t t_buf = t_lane + static_cast<uint32_t>(buf * BN);
                // double-buffered TMEM loads: chunk c+1 is in flight while the
                // FMAs of chunk c run (tcgen05.wait::ld waits for all loads)
                constexpr int NCH = C::CPT / C::CHUNK;
                uint32_t rr[2][C::CHUNK];
                if constexpr (C::CHUNK == 32)
                    tmem_ld32(t_buf, rr[0]);
                else
                    tmem_ld16(t_buf, rr[0]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    const int c0 = c * C::CHUNK;
                    if (c + 1 < NCH) {
                        if constexpr (C::CHUNK == 32)
                            tmem_ld32(t_buf + c0 + C::CHUNK, rr[(c + 1) & 1]);
                        else
                            tmem_ld16(t_buf + c0 + C::CHUNK, rr[(c + 1) & 1]);
                    } else {
                        // all of this buffer is in registers: hand it back
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&tempty[buf]);
                    }
                    const uint32_t* r = rr[c & 1];
#pragma unroll
                    for (int j = 0; j < C::CHUNK; j += 4) {
                        float4 f4;
                        if (SWAP)
                            f4 = *reinterpret_cast<const float4*>(fw + c0 + j);
                        else
                            f4 = make_float4(f_norm, f_norm, f_norm, f_norm);
                        acc[c0 + j] = fmaf(__uint_as_float(r[j]), f4.x, acc[c0 + j]);
                        acc[c0 + j + 1] = fmaf(__uint_as_float(r[j + 1]), f4.y, acc[c0 + j + 1]);
                        acc[c0 + j + 2] = fmaf(__uint_as_float(r[j + 2]), f4.z, acc[c0 + j + 2]);
                        acc[c0 + j + 3] = fmaf(__uint_as_float(r[j + 3]), f4.w, acc[c0 + j + 3]);
                    }
                    if (c + 1 < NCH) tmem_ld_wait();
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&sempty[slot]);
                if (++buf == C::NBUF) {
                    buf = 0;
                    bphase ^= 1u;
                }
                if (++slot == SR) {
                    slot = 0;
                    sphase ^= 1u;
                }
            }
            if (!ok) break;

            // -------------------------------------------- split reduction
            // Each epilogue warp owns a fixed 32-row x CPT-column sub-block of
            // the tile and takes its own ticket for it, so no barrier between
            // warps is needed (and none can be left waiting after an abort).
            if (sg.nparts > 1) {
                constexpr int64_t TILE = C::MR * BN;
                float* mine = a.partials + part_slot(a, sg.tile, sg.part) * TILE;
                if (row_ok) {
#pragma unroll
                    for (int j = 0; j < C::CPT; ++j)
                        __stcg(mine + (chalf * C::CPT + j) * C::MR + row, acc[j]);
                }
                __threadfence();
                __syncwarp();
                unsigned* ctr = a.counters + static_cast<int64_t>(sg.tile) * kCountersPerTile + ew;
                unsigned prev = 0;
                if (lane == 0) prev = atomicAdd(ctr, 1u);
                prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
                if (prev != static_cast<unsigned>(sg.nparts - 1)) continue;
                __threadfence();
                // Sum the segments in K order (own segment from registers).
                // The loads of PB segments are all issued before the first
                // add, so PB parts cost one L2 round trip per RC-column
                // chunk instead of one each; PB is as large as the
                // registers allow without spilling (1 from 64 columns a thread).
                constexpr int RC = C::CPT >= 128 ? 8 : (C::EPI_WARPS == 8 || C::CPT < 32) ? 16 : 32;
                constexpr int PB = C::CPT == 16 ? 4 : C::CPT == 32 ? 2 : 1;
#pragma unroll
                for (int c0 = 0; c0 < C::CPT; c0 += RC) {
                    float r[RC];
                    for (int p0 = 0; p0 < sg.nparts; p0 += PB) {
                        float t[PB][RC];
#pragma unroll
                        for (int q = 0; q < PB; ++q) {
                            const int p = p0 + q;
                            if (p < sg.nparts && p != sg.part) {
                                const float* src = a.partials + part_slot(a, sg.tile, p) * TILE +
                                                   (chalf * C::CPT + c0) * C::MR + row;
#pragma unroll
                                for (int j = 0; j < RC; ++j)
                                    t[q][j] = row_ok ? __ldcg(src + j * C::MR) : 0.0f;
                            }
                        }
#pragma unroll
                        for (int q = 0; q < PB; ++q) {
                            const int p = p0 + q;
                            if (p < sg.nparts) {
#pragma unroll
                                for (int j = 0; j < RC; ++j) {
                                    const float v = (p == sg.part) ? acc[c0 + j] : t[q][j];
                                    r[j] = (p == 0) ? v : r[j] + v;
                                }
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < RC; ++j) acc[c0 + j] = r[j];
                }
                if (lane == 0) *ctr = 0u;  // ready for the next call
            }

            // ------------------------------------------------------- store
            // (the tile's bounds are recomputed here rather than held in
            // registers across the slab loop)
            const TileOrigin os = tile_origin<SWAP, BN, WM, GR>(a, sg.tile);
            if (!SWAP) {
                const int m = os.tok0 + row;
                if (m < os.tok_end) {
                    const int n0 = os.w0 + chalf * C::CPT;
#pragma unroll
                    for (int j = 0; j < C::CPT; j += 8)
                        if (n0 + j < os.w_end)
                            store_out8(a.out, a.out_dtype,
                                       static_cast<int64_t>(m) * a.N + (n0 + j - os.col0), acc[j],
                                       acc[j + 1], acc[j + 2], acc[j + 3], acc[j + 4], acc[j + 5],
                                       acc[j + 6], acc[j + 7]);
                }
            } else {
                const int n = os.w0 + row;
                const int t0 = os.tok0 + chalf * C::CPT;
                if (row_ok && n < os.w_end) {
#pragma unroll
                    for (int j = 0; j < C::CPT; ++j)
                        if (t0 + j < os.tok_end)
                            store_out1(a.out, a.out_dtype,
                                       static_cast<int64_t>(t0 + j) * a.N + (n - os.col0), acc[j]);
                }
            }
        }
    }

    // Reconverge each warp (its lane 0 may have run a role loop alone), then
    // wait for the whole CTA before giving the TMEM back.
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------ block-scaled path
//
// UE8M0 scales applied by the tensor core (both orientations): the E8M0
// factors of the weights (one per 128x128 block) and of the tokens (one per
// 1x128 group) go to TMEM, and tcgen05.mma.kind::mxf8f6f4.block_scale multiplies each
// 32-wide K block's products by 2^(ea+ew) as it accumulates, so a segment's
// sum of promoted slab products builds up in one TMEM accumulator and is read
// once.  A slab's four K blocks share its group's factors.  The packed UE8M0
// activation words (four groups per u32) are the TMEM factor words as they
// are: slab kb uses byte kb % 4 (the instruction's factor ids) of word kb / 4.
//
//   warp 0     TMA: per slab the weight and token tiles (as gemm_kernel);
//              per 4-slab group the tile's token factor words and the four
//              fp32 scales of each weight block of the tile into the scale
//              ring.
//   warp 1     MMA issuer; owns TMEM.  Per slab four block-scaled MMAs into
//              the segment's accumulator (two alternating by segment, one for
//              256-wide tiles).
//   warps 2-5  factor writers: per group, tcgen05.st of the factor words into
//              a TMEM ring entry, each warp into its 32-lane quarter (every
//              quarter holds a full copy).  MMA-M operand factors at columns
//              0-3 (row r: lane r%32, column r/32), MMA-N operand factors from
//              column 8: swap-AB -- weight word x4, then token 32c+l at lane
//              l, column 8+c; normal -- token words x4, then the word of
//              weight block c/4 in column 8+c.
//   warps 6-9  epilogue: per segment, read the accumulator, store or reduce
//              the split parts (same workspace protocol as gemm_kernel).
//
// Requires K % 512 == 0 (whole groups of four slabs, so the four weight
// scales of a group are one aligned 16-byte chunk).
//
// FQ (fused quant; fp8bq_linear, UE8M0, swap-AB token tiles of 16/32): the
// operand tile of the tokens is quantised inside the kernel.  Warp 0 streams
// the raw bf16/fp16 activation tile of each slab beside the weight tile.
// Warps 2-5 each take a quarter of the token rows: group amax and E8M0 scale
// with the standalone quant's arithmetic (quant_math.cuh), the e4m3 codes into
// the 128-byte-swizzled operand tile, the exponents into a per-stage array.
// Warps 6-9 (idle until a segment ends) gather each 4-slab group's exponents
// into the same factor words as the unfused path (byte kb % 4) and write the
// group's TMEM ring entry, each into its own lane quarter.  K % 128 suffices:
// a group cut by a segment boundary is written when the segment ends.
//
// RW (rowwise scales; FP8_Dynamic of "用 Helion 为 vLLM 构建高性能可移植线性
// 后端", 范围: one fp32 scale per token and one per weight output channel):
// no factors at all.  Warp 1 issues plain kind::f8f6f4 MMAs that accumulate a
// whole segment in TMEM, warps 2-5 idle, and the epilogue multiplies each
// finished sum by s_tok[m] * w_s[n] before it stores (split parts are summed
// unscaled, then scaled once).  K needs only whole 16-byte rows: the last
// slab's columns past K are TMA zero fill.
//
// RW == 2 (W8A8_INT8 on the FP8 tensor core): both operands come as two e4m3
// planes per 128-wide K slab (16 h and l of q = 16 h + l; launch_int8_planes
// writes them), a stage holds both planes of both operands, and warp 1 issues
// the four cross products per 32-wide K step into the one accumulator:
// (16 h_a)(16 h_w) + (16 h_a) l_w + l_a (16 h_w) + l_a l_w = q_a q_w.
template <bool SWAP, int BN, int FQ = 0, int RW = 0>
struct MxCfg {
    static_assert(FQ == 0 || (SWAP && BN <= 32), "fused quant: swap-AB token tiles of 16/32");
    static_assert(!(FQ && RW), "rowwise scales take quantised tokens");
    static constexpr int A_BYTES = BM * BK;  // one plane of one slab
    static constexpr int B_BYTES = BN * BK;
    static constexpr int PL = RW == 2 ? 2 : 1;  // planes per operand and slab
    static constexpr int A_STAGE = PL * A_BYTES;
    static constexpr int B_STAGE = PL * B_BYTES;
    static constexpr int X_BYTES = FQ ? BN * BK * 2 : 0;  // raw activation tile (fused quant)
    static constexpr int E_BYTES = FQ ? BN * 4 : 0;       // the tile rows' scale exponents
    static constexpr int STAGE_BYTES = A_STAGE + B_STAGE + X_BYTES + E_BYTES;
    static constexpr int STAGES_X = (200 * 1024) / STAGE_BYTES > 8 ? 8 : (200 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = FQ ? (BN <= 16 ? 9 : 7) : RW == 2 ? STAGES_X : Cfg<SWAP, BN>::STAGES;
    static constexpr int SRM = (FQ || RW) ? 0 : SR;  // scale-ring slots (fused, rowwise: none)
    static constexpr int NC = (BN + 31) / 32;       // factor columns of the MMA-N operand
    static constexpr int TOK_WORDS = SWAP ? BN : BM;  // token factor words per group
    static constexpr int WBLK = SWAP ? 1 : BN / BK;   // weight blocks per tile
    // one factor-ring entry: weight factors at columns +0..3, token factors at
    // +8..8+NC-1; both start on an 8-column boundary (tcgen05.st.x4 and the
    // MMA's factor addresses need aligned columns)
    static constexpr int SF_B = 8;
    static constexpr int SF_COLS = 16;
    static constexpr int RF = 8;                    // factor-ring entries (groups in flight)
    // accumulators: two (the next segment's MMAs overlap this one's read-out)
    // when they fit beside the factor ring
    static constexpr int NACC = (RW || 2 * BN + RF * SF_COLS <= 512) ? 2 : 1;
    static constexpr int SF_BASE = NACC * BN;       // after the accumulators
    static constexpr int TMEM_NEED = SF_BASE + (RW ? 0 : RF * SF_COLS);
    static constexpr int TMEM_COLS = TMEM_NEED <= 32    ? 32
                                     : TMEM_NEED <= 64  ? 64
                                     : TMEM_NEED <= 128 ? 128
                                     : TMEM_NEED <= 256 ? 256
                                                        : 512;
    static constexpr int EPI_FIRST = 6;             // factor writers 2..5, epilogue 6..9
    static constexpr int THREADS = 32 * 10;
    static constexpr int CHUNK = BN >= 32 ? 32 : 16;  // accumulator columns per TMEM load
    static constexpr int RING_OFF = STAGES * STAGE_BYTES;
    static constexpr int BAR_OFF = RING_OFF + SRM * SLOT_BYTES;
    static constexpr int BAR_BYTES = 8 * (4 * STAGES + 2 * SRM + 2 * RF + 2 * NACC + 1) + 16;
    static constexpr int SMEM = 1024 + BAR_OFF + BAR_BYTES;
    static_assert(TMEM_NEED <= 512, "TMEM columns");
    static_assert(SF_BASE % 16 == 0 && NC <= SF_COLS - SF_B, "factor-ring column alignment");
    static_assert(SMEM <= 227 * 1024, "shared memory");
    static_assert(4 * TOK_WORDS <= SLOT_SW && SLOT_SW + WBLK * SLOT_SW_STEP <= SLOT_BYTES,
                  "scale slot layout");
};

template <bool SWAP, int BN, int FQ, bool GR, int RW = 0>
__global__ void __launch_bounds__(MxCfg<SWAP, BN, FQ, RW>::THREADS, 1)
    gemm_mx_kernel(const __grid_constant__ CUtensorMap tm_mma_m,  // MMA-M operand [rows, K] e4m3
                   const __grid_constant__ CUtensorMap tm_mma_n,  // MMA-N operand [rows, K] e4m3
                                                                  // (FQ: raw activations, 2-byte)
                   const __grid_constant__ CUtensorMap tm_sa,     // packed act words [G/4][Mp]
                   const __grid_constant__ CUtensorMap tm_sw,     // weight scales, flat fp32
                   const KArgs a) {
    using C = MxCfg<SWAP, BN, FQ, RW>;
    constexpr int SR = C::SRM;  // scale-ring slots of this configuration
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                           // STAGES x PL x [128 MMA-M rows x 128 B]
    uint8_t* sB = smem + C::STAGES * C::A_STAGE;  // STAGES x PL x [BN MMA-N rows x 128 B]
    uint8_t* sX = sB + C::STAGES * C::B_STAGE;    // FQ: STAGES x [BN tokens x 256 B raw]
    uint32_t* sE = reinterpret_cast<uint32_t*>(sX + C::STAGES * C::X_BYTES);  // FQ: STAGES x BN
    uint8_t* ring = smem + C::RING_OFF;           // SR x SLOT_BYTES
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* empty = full + C::STAGES;
    uint64_t* sfull = empty + C::STAGES;
    uint64_t* sempty = sfull + SR;
    uint64_t* ffull = sempty + SR;   // factor-ring entry written
    uint64_t* fempty = ffull + C::RF;  // factor-ring entry consumed by its MMAs
    uint64_t* tfull = fempty + C::RF;     // accumulator complete
    uint64_t* tempty = tfull + C::NACC;   // accumulator read out
    uint64_t* mma_done = tempty + C::NACC;
    uint64_t* xfull = mma_done + 1;       // FQ: raw activation tile landed
    uint64_t* qdone = xfull + C::STAGES;  // FQ: the stage's codes and exponents written
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(qdone + C::STAGES);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            // FQ: the weight tile's bytes plus the four quantising warps' codes
            mbar_init(&full[s], FQ ? 5 : 1);
            mbar_init(&empty[s], 1);
            mbar_init(&xfull[s], 1);
            mbar_init(&qdone[s], 4);
        }
        for (int s = 0; s < SR; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sempty[s], 4);
        }
        for (int r = 0; r < C::RF; ++r) {
            mbar_init(&ffull[r], 4);
            mbar_init(&fempty[r], 1);
        }
        for (int b = 0; b < C::NACC; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_mma_m);
        tma_prefetch_desc(&tm_mma_n);
        tma_prefetch_desc(&tm_sa);
        tma_prefetch_desc(&tm_sw);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const uint64_t tmo = a.timeout_ns;
    const int code = static_cast<int>(FP8BQ_ERR_DEVICE_TIMEOUT);

    // Programmatic dependent launch, as in gemm_kernel: only weight tiles may
    // be read before the previous grid has finished.
    int prefetched = 0;
    if (a.prefetch_w && warp == 0 && lane == 0) {
        WorkIter<GR> wi;
        wi.init(a);
        Seg sg;
        if (wi.next(a, sg)) {
            const TileOrigin o = tile_origin<SWAP, BN, BM, GR>(a, sg.tile);
            const int nslab = sg.kb1 - sg.kb0;
            prefetched = nslab < C::STAGES ? nslab : C::STAGES;
            for (int i = 0; i < prefetched; ++i) {
                mbar_arrive_expect_tx(&full[i], FQ ? C::A_BYTES : C::STAGE_BYTES);
                if (SWAP)
                    tma_load_slab<C::PL>(sA + i * C::A_STAGE, &tm_mma_m, &full[i], sg.kb0 + i,
                                         o.w0, policy_evict_first(), C::A_BYTES);
                else
                    tma_load_slab<C::PL>(sB + i * C::B_STAGE, &tm_mma_n, &full[i], sg.kb0 + i,
                                         o.w0, policy_evict_first(), C::B_BYTES);
            }
        }
    }
    pdl_wait_prior_grid();
    pdl_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------ TMA producer
        if (lane == 0) {
            // weights stream once; activations are re-read by other tiles
            const uint64_t pol_m = SWAP ? policy_evict_first() : policy_evict_last();
            const uint64_t pol_n = SWAP ? policy_evict_last() : policy_evict_first();
            int stage = 0, slot = 0;
            uint32_t phase = 0, sphase = 0;
            long long fills = 0, sfills = 0;
            WorkIter<GR> wi;
            wi.init(a);
            Seg sg;
            bool ok = true;
            while (ok && wi.next(a, sg)) {
                const TileOrigin o = tile_origin<SWAP, BN, BM, GR>(a, sg.tile);
                const int row_m = SWAP ? o.w0 : o.tok0;
                const int row_n = SWAP ? o.tok0 : o.w0;
                const int nb = o.w0 / BK;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!FQ && !RW && (kb == sg.kb0 || (kb & 3) == 0)) {
                        // the group's factors: BN token words, four weight scales
                        if (!mbar_wait_bounded(&sempty[slot], sphase ^ 1u, abort_flag, a.status,
                                               tmo, code)) {
                            ok = false;
                            break;
                        }
                        uint8_t* sl = ring + slot * SLOT_BYTES;
                        mbar_arrive_expect_tx(&sfull[slot], 4u * C::TOK_WORDS + 16u * C::WBLK);
                        tma_load_2d(sl, &tm_sa, &sfull[slot], o.tok0, kb >> 2);
#pragma unroll
                        for (int b = 0; b < C::WBLK; ++b)
                            tma_load_2d(sl + SLOT_SW + b * SLOT_SW_STEP, &tm_sw, &sfull[slot],
                                        (nb + b) * a.G + (kb & ~3), 0);
                        ++sfills;
                        if (++slot == SR) {
                            slot = 0;
                            sphase ^= 1u;
                        }
                    }
                    if (FQ) {
                        // weight tile to the operand stage, raw activations to sX
                        if (fills >= prefetched) {
                            if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag,
                                                   a.status, tmo, code)) {
                                ok = false;
                                break;
                            }
                            mbar_arrive_expect_tx(&full[stage], C::A_BYTES);
                            tma_load_2d_hint(sA + stage * C::A_BYTES, &tm_mma_m, &full[stage],
                                             kb * BK, row_m, pol_m);
                        }
                        mbar_arrive_expect_tx(&xfull[stage], C::X_BYTES);
                        tma_load_2d_hint(sX + stage * C::X_BYTES, &tm_mma_n, &xfull[stage],
                                         kb * BK, row_n, pol_n);
                    } else if (fills < prefetched) {
                        // the weight tile of this stage is already on its way
                        if (SWAP)
                            tma_load_slab<C::PL>(sB + stage * C::B_STAGE, &tm_mma_n, &full[stage],
                                                 kb, row_n, pol_n, C::B_BYTES);
                        else
                            tma_load_slab<C::PL>(sA + stage * C::A_STAGE, &tm_mma_m, &full[stage],
                                                 kb, row_m, pol_m, C::A_BYTES);
                    } else {
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status,
                                               tmo, code)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        tma_load_slab<C::PL>(sA + stage * C::A_STAGE, &tm_mma_m, &full[stage], kb,
                                             row_m, pol_m, C::A_BYTES);
                        tma_load_slab<C::PL>(sB + stage * C::B_STAGE, &tm_mma_n, &full[stage], kb,
                                             row_n, pol_n, C::B_BYTES);
                    }
                    ++fills;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (long long f = fills > C::STAGES ? fills - C::STAGES : 0; f < fills; ++f) {
                if (FQ)
                    mbar_wait_drain(&xfull[f % C::STAGES],
                                    static_cast<uint32_t>((f / C::STAGES) & 1), tmo);
                mbar_wait_drain(&full[f % C::STAGES], static_cast<uint32_t>((f / C::STAGES) & 1),
                                tmo);
            }
            if constexpr (SR > 0) {
                for (long long f = sfills > SR ? sfills - SR : 0; f < sfills; ++f)
                    mbar_wait_drain(&sfull[f % SR], static_cast<uint32_t>((f / SR) & 1), tmo);
            }
        }
    } else if (warp == 1) {
        // -------------------------------------------------------- MMA issuer
        if (lane == 0) {
            int stage = 0, r = 0, acc = 0;
            uint32_t phase = 0, rphase = 0, aphase = 0;
            WorkIter<GR> wi;
            wi.init(a);
            Seg sg;
            bool ok = true;
            while (ok && wi.next(a, sg)) {
                if (!mbar_wait_bounded(&tempty[acc], aphase ^ 1u, abort_flag, a.status, tmo,
                                       code)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_addr = tmem_base + static_cast<uint32_t>(acc * BN);
                int cur = 0;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!RW && (kb == sg.kb0 || (kb & 3) == 0)) {
                        if (!mbar_wait_bounded(&ffull[r], rphase, abort_flag, a.status, tmo,
                                               code)) {
                            ok = false;
                            break;
                        }
                        cur = r;
                        if (++r == C::RF) {
                            r = 0;
                            rphase ^= 1u;
                        }
                    }
                    if (!mbar_wait_bounded(&full[stage], phase, abort_flag, a.status, tmo, code)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_addr = smem_addr(sA + stage * C::A_STAGE);
                    const uint32_t b_addr = smem_addr(sB + stage * C::B_STAGE);
                    if constexpr (RW == 2) {
                        // INT8 as two e4m3 planes: the four cross products
                        constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
#pragma unroll
                        for (int kk = 0; kk < BK / 32; ++kk)
#pragma unroll
                            for (int pq = 0; pq < 4; ++pq)
                                mma_f8f6f4(d_addr,
                                           smem_desc_k128_sw128(a_addr + (pq >> 1) * C::A_BYTES +
                                                                kk * 32),
                                           smem_desc_k128_sw128(b_addr + (pq & 1) * C::B_BYTES +
                                                                kk * 32),
                                           idesc, (kb > sg.kb0 || kk > 0 || pq > 0) ? 1u : 0u);
                    } else if constexpr (RW) {
                        // rowwise scales: the plain FP8 MMA, scaled in the epilogue
                        constexpr uint32_t idesc = idesc_e4m3_f32(BM, BN);
#pragma unroll
                        for (int kk = 0; kk < BK / 32; ++kk)
                            mma_f8f6f4(d_addr, smem_desc_k128_sw128(a_addr + kk * 32),
                                       smem_desc_k128_sw128(b_addr + kk * 32), idesc,
                                       (kb > sg.kb0 || kk > 0) ? 1u : 0u);
                    } else {
                        const uint32_t sfa =
                            tmem_base + static_cast<uint32_t>(C::SF_BASE + cur * C::SF_COLS);
                        // factor byte kb % 4 of the group's words
                        const uint32_t idesc =
                            idesc_mx_e4m3(BM, BN, static_cast<uint32_t>(kb & 3));
#pragma unroll
                        for (int kk = 0; kk < BK / 32; ++kk)
                            mma_mxf8(d_addr, smem_desc_k128_sw128(a_addr + kk * 32),
                                     smem_desc_k128_sw128(b_addr + kk * 32), idesc, sfa,
                                     sfa + C::SF_B, (kb > sg.kb0 || kk > 0) ? 1u : 0u);
                    }
                    mma_commit(&empty[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                    if (!RW && ((kb & 3) == 3 || kb == sg.kb1 - 1)) mma_commit(&fempty[cur]);
                }
                if (!ok) break;
                mma_commit(&tfull[acc]);
                if (++acc == C::NACC) {
                    acc = 0;
                    aphase ^= 1u;
                }
            }
            mma_commit(mma_done);
            mbar_wait_drain(mma_done, 0, tmo);
        }
    } else if (warp < C::EPI_FIRST) {
        const int quarter = warp & 3;  // TMEM lanes this warp may access
        const uint32_t t_quarter = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        if constexpr (FQ) {
            // ----------------------------------------- quantising warps (FQ)
            // Per slab: the BN x 128 raw tile in sX (row-major, 256 B a row).
            // Warp q takes rows [q*BN/4, (q+1)*BN/4): pass p covers 4 of them,
            // 8 lanes a row, 16 elements a lane.
            constexpr int RPW = BN / 4;      // rows per warp
            constexpr int PASSES = RPW / 4;  // 1 (16 tokens) or 2 (32 tokens)
            const int g = lane >> 3;         // row within the pass
            const int c16 = lane & 7;        // 16-element chunk within the row
            int stage = 0;
            uint32_t phase = 0;
            WorkIter<GR> wi;
            wi.init(a);
            Seg sg;
            bool ok = true;
            while (ok && wi.next(a, sg)) {
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!warp_wait(&xfull[stage], phase, abort_flag, a.status, tmo, code)) {
                        ok = false;
                        break;
                    }
                    const uint8_t* xs = sX + stage * C::X_BYTES;
                    uint8_t* bs = sB + stage * C::B_BYTES;
                    uint32_t* es = sE + stage * BN;
#pragma unroll
                    for (int p = 0; p < PASSES; ++p) {
                        const int row = quarter * RPW + 4 * p + g;
                        const uint4* src = reinterpret_cast<const uint4*>(xs + row * (2 * BK) + c16 * 32);
                        const uint4 v0 = src[0], v1 = src[1];
                        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
                        float f[16];
#pragma unroll
                        for (int i = 0; i < 8; ++i) {
                            f[2 * i] = FQ == 2 ? f16_lo(w[i]) : bf16_lo(w[i]);
                            f[2 * i + 1] = FQ == 2 ? f16_hi(w[i]) : bf16_hi(w[i]);
                        }
                        float amax = 0.0f;
#pragma unroll
                        for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
                        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
                        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
                        amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
                        const float sc = group_scale(amax, 1);
                        // sc = 2^e exactly: x * (1/sc) is the correctly rounded x / sc
                        const float rs = __fdiv_rn(1.0f, sc);
                        uint32_t cw[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) cw[i] = cvt2_e4m3(f[2 * i] * rs, f[2 * i + 1] * rs);
                        // 128-byte swizzle: chunk c of row r at chunk c ^ (r % 8)
                        *reinterpret_cast<uint4*>(bs + row * BK + ((c16 ^ (row & 7)) << 4)) =
                            make_uint4(cw[0] | (cw[1] << 16), cw[2] | (cw[3] << 16),
                                       cw[4] | (cw[5] << 16), cw[6] | (cw[7] << 16));
                        if (c16 == 0) es[row] = (__float_as_uint(sc) >> 23) & 0xFFu;
                    }
                    // the codes are read by the tensor core (async proxy)
                    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&full[stage]);
                        mbar_arrive(&qdone[stage]);
                    }
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        } else if constexpr (!RW) {
            // -------------------------------------------------- factor writers
            int slot = 0, r = 0;
            uint32_t sphase = 0, rphase = 0;
            WorkIter<GR> wi;
            wi.init(a);
            Seg sg;
            bool ok = true;
            while (ok && wi.next(a, sg)) {
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (kb != sg.kb0 && (kb & 3) != 0) continue;
                    if (!warp_wait(&sfull[slot], sphase, abort_flag, a.status, tmo, code) ||
                        !warp_wait(&fempty[r], rphase ^ 1u, abort_flag, a.status, tmo, code)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t* sl = ring + slot * SLOT_BYTES;
                    // weight words: byte j = E8M0 exponent of the block's scale of
                    // slab 4*(kb/4)+j (the fp32 scales are powers of two)
                    uint32_t ww[C::WBLK];
    #pragma unroll
                    for (int b = 0; b < C::WBLK; ++b) {
                        const float* swc = reinterpret_cast<const float*>(sl + SLOT_SW + b * SLOT_SW_STEP);
                        ww[b] = 0;
    #pragma unroll
                        for (int j = 0; j < 4; ++j)
                            ww[b] |= ((__float_as_uint(swc[j]) >> 23) & 0xFFu) << (8 * j);
                    }
                    const uint32_t* tw = reinterpret_cast<const uint32_t*>(sl);
                    const uint32_t col = static_cast<uint32_t>(C::SF_BASE + r * C::SF_COLS);
                    if constexpr (SWAP) {
                        tmem_st4(t_quarter + col, ww[0], ww[0], ww[0], ww[0]);
    #pragma unroll
                        for (int c = 0; c < C::NC; ++c) {
                            const int t = 32 * c + lane;
                            tmem_st1(t_quarter + col + C::SF_B + c, t < BN ? tw[t] : 0u);
                        }
                    } else {
                        tmem_st4(t_quarter + col, tw[lane], tw[32 + lane], tw[64 + lane], tw[96 + lane]);
    #pragma unroll
                        for (int b = 0; b < C::WBLK; ++b)
                            tmem_st4(t_quarter + col + C::SF_B + 4 * b, ww[b], ww[b], ww[b], ww[b]);
                    }
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) {
                        mbar_arrive(&ffull[r]);
                        mbar_arrive(&sempty[slot]);
                    }
                    if (++slot == SR) {
                        slot = 0;
                        sphase ^= 1u;
                    }
                    if (++r == C::RF) {
                        r = 0;
                        rphase ^= 1u;
                    }
                }
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int quad = warp & 3;
        const int row = quad * 32 + lane;  // MMA-M row: weight row (swap-AB) or token
        int acc = 0;
        uint32_t aphase = 0;
        WorkIter<GR> wi;
        wi.init(a);
        Seg sg;
        bool ok = true;
        constexpr int NCH = BN / C::CHUNK;
        // stores one chunk of this row's columns [c0, c0 + CHUNK) of the tile
        auto store_chunk = [&](const TileOrigin& o, int c0, const float* v) {
            if constexpr (SWAP) {
                const int n = o.w0 + row;
                if (n < o.w_end) {
#pragma unroll
                    for (int j = 0; j < C::CHUNK; ++j) {
                        const int t = o.tok0 + c0 + j;
                        if (t < o.tok_end)
                            store_out1(a.out, a.out_dtype,
                                       static_cast<int64_t>(t) * a.N + (n - o.col0), v[j]);
                    }
                }
            } else {
                const int m = o.tok0 + row;
                if (m < o.tok_end) {
#pragma unroll
                    for (int j = 0; j < C::CHUNK; j += 8) {
                        const int n0 = o.w0 + c0 + j;
                        if (n0 < o.w_end)
                            store_out8(a.out, a.out_dtype,
                                       static_cast<int64_t>(m) * a.N + (n0 - o.col0), v[j],
                                       v[j + 1], v[j + 2], v[j + 3], v[j + 4], v[j + 5], v[j + 6],
                                       v[j + 7]);
                    }
                }
            }
        };
        // stores 16 columns [c0, c0 + 16) of this row (the split reduction's unit)
        auto store_rc = [&](const TileOrigin& o, int c0, const float* v) {
            if constexpr (SWAP) {
                const int n = o.w0 + row;
                if (n < o.w_end) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = o.tok0 + c0 + j;
                        if (t < o.tok_end)
                            store_out1(a.out, a.out_dtype,
                                       static_cast<int64_t>(t) * a.N + (n - o.col0), v[j]);
                    }
                }
            } else {
                const int m = o.tok0 + row;
                if (m < o.tok_end) {
#pragma unroll
                    for (int j = 0; j < 16; j += 8) {
                        const int n0 = o.w0 + c0 + j;
                        if (n0 < o.w_end)
                            store_out8(a.out, a.out_dtype,
                                       static_cast<int64_t>(m) * a.N + (n0 - o.col0), v[j],
                                       v[j + 1], v[j + 2], v[j + 3], v[j + 4], v[j + 5], v[j + 6],
                                       v[j + 7]);
                    }
                }
            }
        };
        // FQ: the factor ring, written here slab by slab
        int fstage = 0, fr = 0;
        uint32_t fphase = 0, frphase = 0;
        while (ok && wi.next(a, sg)) {
            const TileOrigin o = tile_origin<SWAP, BN, BM, GR>(a, sg.tile);
            if constexpr (FQ > 0) {
                // per 4-slab group (as the packed words of the unfused path):
                // byte j of the weight word = the block's exponent of slab
                // 4w+j, byte j of token t's word = its exponent in that slab
                const uint32_t t_quarter = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);
                const float* wrow = a.w_s + static_cast<int64_t>(o.w0 / BK) * a.G;
                auto wload = [&](int kb) { return kb < sg.kb1 ? __ldg(wrow + kb) : 0.0f; };
                float w_cur = wload(sg.kb0 + lane);
                float w_nxt = wload(sg.kb0 + 32 + lane);
                uint32_t ww = 0, tw = 0;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    const int wi32 = (kb - sg.kb0) & 31;
                    if (wi32 == 0 && kb != sg.kb0) {
                        w_cur = w_nxt;
                        w_nxt = wload(kb + 32 + lane);
                    }
                    if (!warp_wait(&qdone[fstage], fphase, abort_flag, a.status, tmo, code)) {
                        ok = false;
                        break;
                    }
                    const int byte = 8 * (kb & 3);
                    ww |= ((__float_as_uint(__shfl_sync(0xFFFFFFFFu, w_cur, wi32)) >> 23) & 0xFFu)
                          << byte;
                    if (lane < BN) tw |= sE[fstage * BN + lane] << byte;
                    if (++fstage == C::STAGES) {
                        fstage = 0;
                        fphase ^= 1u;
                    }
                    if ((kb & 3) != 3 && kb != sg.kb1 - 1) continue;
                    // the group is complete: write its ring entry
                    if (!warp_wait(&fempty[fr], frphase ^ 1u, abort_flag, a.status, tmo, code)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t col = static_cast<uint32_t>(C::SF_BASE + fr * C::SF_COLS);
                    tmem_st4(t_quarter + col, ww, ww, ww, ww);
                    tmem_st1(t_quarter + col + C::SF_B, tw);
                    tmem_st_wait();
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&ffull[fr]);
                    ww = 0;
                    tw = 0;
                    if (++fr == C::RF) {
                        fr = 0;
                        frphase ^= 1u;
                    }
                }
                if (!ok) break;
            }
            if (!warp_wait(&tfull[acc], aphase, abort_flag, a.status, tmo, code)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t t_acc = tmem_base + (static_cast<uint32_t>(quad * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            constexpr int64_t TILE = BM * BN;
            float* mine = sg.nparts > 1 ? a.partials + part_slot(a, sg.tile, sg.part) * TILE
                                        : nullptr;
#pragma unroll
            for (int c = 0; c < NCH; ++c) {
                uint32_t v[C::CHUNK];
                if constexpr (C::CHUNK == 32)
                    tmem_ld32(t_acc + c * C::CHUNK, v);
                else
                    tmem_ld16(t_acc + c * C::CHUNK, v);
                tmem_ld_wait();
                if (c + 1 == NCH) {
                    // the accumulator is in registers: hand it back
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tempty[acc]);
                }
                if (sg.nparts > 1) {
#pragma unroll
                    for (int j = 0; j < C::CHUNK; ++j)
                        __stcg(mine + (c * C::CHUNK + j) * BM + row, __uint_as_float(v[j]));
                } else {
                    float f[C::CHUNK];
#pragma unroll
                    for (int j = 0; j < C::CHUNK; ++j) f[j] = __uint_as_float(v[j]);
                    if constexpr (RW) rowwise_scale<SWAP, C::CHUNK>(a, o, row, c * C::CHUNK, f);
                    store_chunk(o, c * C::CHUNK, f);
                }
            }
            if (++acc == C::NACC) {
                acc = 0;
                aphase ^= 1u;
            }
            if (sg.nparts == 1) continue;
            // split parts: per-warp ticket; the last to arrive sums all parts
            // in K order and stores (every warp owns its 32 rows)
            __threadfence();
            __syncwarp();
            unsigned* ctr = a.counters + static_cast<int64_t>(sg.tile) * kCountersPerTile + quad;
            unsigned prev = 0;
            if (lane == 0) prev = atomicAdd(ctr, 1u);
            prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
            if (prev != static_cast<unsigned>(sg.nparts - 1)) continue;
            __threadfence();
            if constexpr (BN <= 32) {
                // narrow tiles split many ways: 16 columns at a time, the loads
                // of PB parts go out before the first add (one L2 round trip
                // per PB parts); the sum runs in K order
                constexpr int RC = 16;
                constexpr int PB = 4;
#pragma unroll 1
                for (int c0 = 0; c0 < BN; c0 += RC) {
                    float r[RC];
                    for (int p0 = 0; p0 < sg.nparts; p0 += PB) {
                        float t[PB][RC];
#pragma unroll
                        for (int q = 0; q < PB; ++q) {
                            if (p0 + q < sg.nparts) {
                                const float* src = a.partials +
                                                   part_slot(a, sg.tile, p0 + q) * TILE + c0 * BM +
                                                   row;
#pragma unroll
                                for (int j = 0; j < RC; ++j) t[q][j] = __ldcg(src + j * BM);
                            }
                        }
#pragma unroll
                        for (int q = 0; q < PB; ++q) {
                            if (p0 + q < sg.nparts) {
#pragma unroll
                                for (int j = 0; j < RC; ++j)
                                    r[j] = (p0 + q == 0) ? t[q][j] : r[j] + t[q][j];
                            }
                        }
                    }
                    if constexpr (RW) rowwise_scale<SWAP, RC>(a, o, row, c0, r);
                    store_rc(o, c0, r);
                }
            } else {
                // wide tiles split at most a few ways: part by part, in K order
#pragma unroll
                for (int c = 0; c < NCH; ++c) {
                    float r[C::CHUNK];
                    for (int p = 0; p < sg.nparts; ++p) {
                        const float* src = a.partials + part_slot(a, sg.tile, p) * TILE +
                                           (c * C::CHUNK) * BM + row;
                        float t[C::CHUNK];
#pragma unroll
                        for (int j = 0; j < C::CHUNK; ++j) t[j] = __ldcg(src + j * BM);
#pragma unroll
                        for (int j = 0; j < C::CHUNK; ++j) r[j] = (p == 0) ? t[j] : r[j] + t[j];
                    }
                    if constexpr (RW) rowwise_scale<SWAP, C::CHUNK>(a, o, row, c * C::CHUNK, r);
                    store_chunk(o, c * C::CHUNK, r);
                }
            }
            if (lane == 0) *ctr = 0u;  // ready for the next call
        }
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

// ------------------------------------------------------------- INT8 GEMM
//
// W8A8_INT8 ("用 Helion 为 vLLM 构建高性能可移植线性后端", 范围): int8 codes with
// one scale per token and one per weight output channel,
//   out[m,n] = s_tok[m] * w_s[n] * sum_k a[m,k] * w[n,k]    (int32 sums, exact).
// tcgen05 has no integer kind on sm_103a, so the products run on the
// warp-level int8 tensor-core instruction (mma.sync m16n8k32, s8 x s8 -> s32).
// Tiles are swap-AB shaped, 128 weight rows x BN tokens:
//   warp 0      TMA producer: per K slab the 128x128 weight tile and the
//               BNx128 token tile (128-byte swizzle) into a STAGES-deep ring;
//   warps 1-8   consumer warp w owns weight rows 16(w-1)..16(w-1)+15: per
//               32-byte K step one ldmatrix.x4 of its rows, one per 16 tokens,
//               and BN/8 MMAs into int32 registers.  At a segment's end it
//               scales and stores its 16 x BN block, or writes it as an int32
//               split part; the last part to arrive (ticket per warp and tile,
//               as in the FP8 kernels) adds the parts in K order and stores.
// The swizzle puts 16-byte chunk c of row r at chunk c ^ (r % 8), so the eight
// row addresses of every ldmatrix fall in distinct bank groups.
template <int BN>
struct I8Cfg {
    static constexpr int CW = 8;  // consumer warps
    static constexpr int THREADS = 32 * (1 + CW);
    static constexpr int A_BYTES = BM * BK;
    static constexpr int B_BYTES = BN * BK;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES_FIT = (200 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_FIT > 12 ? 12 : STAGES_FIT;
    static constexpr int BAR_OFF = STAGES * STAGE_BYTES;
    static constexpr int SMEM = 1024 + BAR_OFF + 8 * 2 * STAGES + 16;
    static_assert((BN % 16 == 0 || BN == 8) && BN <= 128, "token tile");
    static_assert(SMEM <= 227 * 1024, "shared memory");
};

// BLK (block INT8: int8_w8a8 with 1x128 activation groups and 128x128 weight
// blocks, fp32 scales): after every K slab each thread converts its exact
// int32 slab sums (|S| < 2^21) to fp32 exactly and promotes them by
// sa[kb][t] * sw[nb][kb] into fp32 accumulators, as the FP8 block path does;
// split parts are then fp32 and stores need no further scaling.
__device__ __forceinline__ float exact_i2f(int v) {
    // |v| < 2^22: v + 1.5 * 2^23 has the fp32 exponent of 2^23, so its low
    // mantissa bits are v; subtracting 1.5 * 2^23 leaves exactly v
    return __int_as_float(v + 0x4B400000) - 12582912.0f;
}

template <int BN, bool BLK = false>
__global__ void __launch_bounds__(I8Cfg<BN>::THREADS, 1)
    gemm_i8_kernel(const __grid_constant__ CUtensorMap tm_w,  // weights [N, K] int8
                   const __grid_constant__ CUtensorMap tm_t,  // tokens [M, K] int8
                   const KArgs a) {
    using C = I8Cfg<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                           // STAGES x [128 weight rows x 128 B]
    uint8_t* sB = smem + C::STAGES * C::A_BYTES;  // STAGES x [BN tokens x 128 B]
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::BAR_OFF);
    uint64_t* empty = full + C::STAGES;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + C::STAGES);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], C::CW);
        }
        *abort_flag = 0;
        fence_barrier_init();
        tma_prefetch_desc(&tm_w);
        tma_prefetch_desc(&tm_t);
    }
    __syncthreads();
    const uint64_t tmo = a.timeout_ns;
    const int code = static_cast<int>(FP8BQ_ERR_DEVICE_TIMEOUT);

    // Programmatic dependent launch, as in the FP8 kernels: only weight tiles
    // may be read before the previous grid has finished.
    int prefetched = 0;
    if (a.prefetch_w && warp == 0 && lane == 0) {
        WorkIter<false> wi;
        wi.init(a);
        Seg sg;
        if (wi.next(a, sg)) {
            const TileOrigin o = tile_origin<true, BN, BM, false>(a, sg.tile);
            const int nslab = sg.kb1 - sg.kb0;
            prefetched = nslab < C::STAGES ? nslab : C::STAGES;
            for (int i = 0; i < prefetched; ++i) {
                mbar_arrive_expect_tx(&full[i], C::STAGE_BYTES);
                tma_load_2d_hint(sA + i * C::A_BYTES, &tm_w, &full[i], (sg.kb0 + i) * BK, o.w0,
                                 policy_evict_first());
            }
        }
    }
    pdl_wait_prior_grid();
    pdl_launch_dependents();

    if (warp == 0) {
        // ---------------------------------------------------- TMA producer
        if (lane == 0) {
            const uint64_t pol_w = policy_evict_first(), pol_t = policy_evict_last();
            int stage = 0;
            uint32_t phase = 0;
            long long fills = 0;
            WorkIter<false> wi;
            wi.init(a);
            Seg sg;
            bool ok = true;
            while (ok && wi.next(a, sg)) {
                const TileOrigin o = tile_origin<true, BN, BM, false>(a, sg.tile);
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (fills >= prefetched) {
                        if (!mbar_wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status,
                                               tmo, code)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        tma_load_2d_hint(sA + stage * C::A_BYTES, &tm_w, &full[stage], kb * BK,
                                         o.w0, pol_w);
                    }
                    tma_load_2d_hint(sB + stage * C::B_BYTES, &tm_t, &full[stage], kb * BK,
                                     o.tok0, pol_t);
                    ++fills;
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            for (long long f = fills > C::STAGES ? fills - C::STAGES : 0; f < fills; ++f)
                mbar_wait_drain(&full[f % C::STAGES], static_cast<uint32_t>((f / C::STAGES) & 1),
                                tmo);
        }
    } else {
        // ------------------------------------------------------- consumers
        const int cw = warp - 1;  // weight rows 16 cw .. 16 cw + 15 of the tile
        const int g = lane >> 2, t4 = lane & 3;
        // ldmatrix row addresses: weight matrices (rows 0-7 | 8-15) x (bytes
        // 0-15 | 16-31) of the K step; token matrices (tokens 0-7 | 8-15) x
        // (bytes 0-15 | 16-31)
        const int a_row = cw * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int a_half = lane >> 4;
        const int b_row = (lane >> 4) * 8 + (lane & 7);
        const int b_half = (lane >> 3) & 1;
        int stage = 0;
        uint32_t phase = 0;
        WorkIter<false> wi;
        wi.init(a);
        Seg sg;
        bool ok = true;
        const int64_t Mp = (static_cast<int64_t>(a.M) + 3) / 4 * 4;  // BLK: act scale rows
        while (ok && wi.next(a, sg)) {
            int acc[BN / 8][4];
            float accf[BLK ? BN / 8 : 1][4];
#pragma unroll
            for (int j = 0; j < BN / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0;
            if constexpr (BLK) {
#pragma unroll
                for (int j = 0; j < BN / 8; ++j)
                    accf[j][0] = accf[j][1] = accf[j][2] = accf[j][3] = 0.0f;
            }
            const TileOrigin ot = tile_origin<true, BN, BM, false>(a, sg.tile);
            for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                if (!warp_wait(&full[stage], phase, abort_flag, a.status, tmo, code)) {
                    ok = false;
                    break;
                }
                const uint32_t a_base = smem_addr(sA + stage * C::A_BYTES) + a_row * BK;
                const uint32_t b_base = smem_addr(sB + stage * C::B_BYTES);
#pragma unroll
                for (int kk = 0; kk < BK / 32; ++kk) {
                    uint32_t af[4];
                    ldmatrix_x4(af, a_base + (((2 * kk + a_half) ^ (a_row & 7)) << 4));
                    if constexpr (BN == 8) {
                        // one 8-token block: lanes 0-7 give bytes 0-15 of the
                        // step, lanes 8-15 bytes 16-31
                        const int tr = lane & 7;
                        uint32_t bf[2];
                        ldmatrix_x2(bf, b_base + tr * BK + (((2 * kk + b_half) ^ (tr & 7)) << 4));
                        mma_s8_16x8x32(acc[0], af, bf[0], bf[1]);
                    } else {
#pragma unroll
                        for (int j = 0; j < BN / 16; ++j) {
                            const int tr = j * 16 + b_row;
                            uint32_t bf[4];
                            ldmatrix_x4(bf,
                                        b_base + tr * BK + (((2 * kk + b_half) ^ (tr & 7)) << 4));
                            mma_s8_16x8x32(acc[2 * j], af, bf[0], bf[1]);
                            mma_s8_16x8x32(acc[2 * j + 1], af, bf[2], bf[3]);
                        }
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                if (++stage == C::STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
                if constexpr (BLK) {
                    // promote the slab: sa of this thread's token columns,
                    // sw of the tile's weight block
                    const float swv = __ldg(a.w_s + static_cast<int64_t>(ot.w0 / BK) * a.G + kb);
                    const float* sak = a.s_tok + static_cast<int64_t>(kb) * Mp;
#pragma unroll
                    for (int j = 0; j < BN / 8; ++j) {
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int t = ot.tok0 + 8 * j + 2 * t4 + c;
                            const float f = (t < ot.tok_end ? __ldg(sak + t) : 0.0f) * swv;
                            accf[j][c] = fmaf(exact_i2f(acc[j][c]), f, accf[j][c]);
                            accf[j][c + 2] = fmaf(exact_i2f(acc[j][c + 2]), f, accf[j][c + 2]);
                            acc[j][c] = acc[j][c + 2] = 0;
                        }
                    }
                }
            }
            if (!ok) break;

            const TileOrigin o = ot;
            // element (j, i) of this thread: weight row w0 + 16 cw + g + 8 (i / 2),
            // token tok0 + 8 j + 2 t4 + (i % 2)
            auto store = [&](int j, int i, int v) {
                const int n = o.w0 + cw * 16 + g + 8 * (i >> 1);
                const int t = o.tok0 + 8 * j + 2 * t4 + (i & 1);
                if (n < o.w_end && t < o.tok_end)
                    store_out1(a.out, a.out_dtype, static_cast<int64_t>(t) * a.N + n,
                               static_cast<float>(v) * (__ldg(a.s_tok + t) * __ldg(a.w_s + n)));
            };
            auto store_f = [&](int j, int i, float v) {  // BLK: already promoted
                const int n = o.w0 + cw * 16 + g + 8 * (i >> 1);
                const int t = o.tok0 + 8 * j + 2 * t4 + (i & 1);
                if (n < o.w_end && t < o.tok_end)
                    store_out1(a.out, a.out_dtype, static_cast<int64_t>(t) * a.N + n, v);
            };
            if (sg.nparts == 1) {
#pragma unroll
                for (int j = 0; j < BN / 8; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if constexpr (BLK)
                            store_f(j, i, accf[j][i]);
                        else
                            store(j, i, acc[j][i]);
                    }
                continue;
            }
            // split parts: int32 [column][row] tiles in the workspace
            constexpr int64_t TILE = BM * BN;
            int* mine = reinterpret_cast<int*>(a.partials) + part_slot(a, sg.tile, sg.part) * TILE;
            auto pidx = [&](int j, int i) {
                return (8 * j + 2 * t4 + (i & 1)) * BM + cw * 16 + g + 8 * (i >> 1);
            };
#pragma unroll
            for (int j = 0; j < BN / 8; ++j)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    if constexpr (BLK)  // fp32 parts (promoted)
                        __stcg(reinterpret_cast<float*>(mine) + pidx(j, i), accf[j][i]);
                    else
                        __stcg(mine + pidx(j, i), acc[j][i]);
                }
            __threadfence();
            __syncwarp();
            unsigned* ctr = a.counters + static_cast<int64_t>(sg.tile) * kCountersPerTile + cw;
            unsigned prev = 0;
            if (lane == 0) prev = atomicAdd(ctr, 1u);
            prev = __shfl_sync(0xFFFFFFFFu, prev, 0);
            if (prev != static_cast<unsigned>(sg.nparts - 1)) continue;
            __threadfence();
            if constexpr (BLK) {
                // fp32 parts, summed in K order
                for (int p = 0; p < sg.nparts; ++p) {
                    const float* src = a.partials + part_slot(a, sg.tile, p) * TILE;
#pragma unroll
                    for (int j = 0; j < BN / 8; ++j)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float v = __ldcg(src + pidx(j, i));
                            accf[j][i] = p == 0 ? v : accf[j][i] + v;
                        }
                }
#pragma unroll
                for (int j = 0; j < BN / 8; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) store_f(j, i, accf[j][i]);
            } else {
#pragma unroll
                for (int j = 0; j < BN / 8; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) acc[j][i] = 0;
                for (int p = 0; p < sg.nparts; ++p) {
                    const int* src =
                        reinterpret_cast<const int*>(a.partials) + part_slot(a, sg.tile, p) * TILE;
#pragma unroll
                    for (int j = 0; j < BN / 8; ++j)
#pragma unroll
                        for (int i = 0; i < 4; ++i) acc[j][i] += __ldcg(src + pidx(j, i));
                }
#pragma unroll
                for (int j = 0; j < BN / 8; ++j)
#pragma unroll
                    for (int i = 0; i < 4; ++i) store(j, i, acc[j][i]);
            }
            if (lane == 0) *ctr = 0u;  // ready for the next call
        }
    }
}

// ------------------------------------------------------------------ host

bool encode(CUtensorMap* map, CUtensorMapDataType dt, int rank, const void* base,
            const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
            CUtensorMapSwizzle swz) {
    EncodeTiledFn enc = get_encode_tiled();
    if (!enc) return false;
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, dt, rank, const_cast<void*>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [rows, K] e4m3 operand, 128-byte swizzled boxes of box_rows x 128.
bool encode_operand(CUtensorMap* map, const void* base, uint64_t K, uint64_t rows,
                    uint32_t box_rows) {
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), box_rows};
    return encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box,
                  CU_TENSOR_MAP_SWIZZLE_128B);
}

template <bool SWAP, int BN, int WM = BM>
cudaError_t launch_bn(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    using C = Cfg<SWAP, BN, WM>;
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        for (auto fn : {gemm_kernel<SWAP, BN, WM, false>, gemm_kernel<SWAP, BN, WM, true>}) {
            err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
            if (err != cudaSuccess) return err;
            if (C::REGSPLIT) {
                // the register split asks for REG_ROLE/REG_EPI per warpgroup;
                // a launch that provides fewer registers in total would never
                // satisfy setmaxnreg.inc, so refuse it
                cudaFuncAttributes fa;
                err = cudaFuncGetAttributes(&fa, fn);
                if (err != cudaSuccess) return err;
                if (fa.numRegs < C::REG_MIN_LAUNCH) {
                    log_error("GEMM kernel compiled with too few registers for its register split");
                    return cudaErrorInvalidConfiguration;
                }
            }
        }
        attr_done[dev] = 1;
    }
    if constexpr (WM == BM) {
        // block INT8 as two planes (rowwise 5): the PL = 2 promotion kernel
        static int pl_attr_done[64] = {0};
        if (p.rowwise == 5 && dev >= 0 && dev < 64 && !pl_attr_done[dev]) {
            using C2 = Cfg<SWAP, BN, BM, 2>;
            const auto fn = gemm_kernel<SWAP, BN, BM, false, 2>;
            err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C2::SMEM);
            if (err != cudaSuccess) return err;
            if (C2::REGSPLIT) {
                cudaFuncAttributes fa;
                err = cudaFuncGetAttributes(&fa, fn);
                if (err != cudaSuccess) return err;
                if (fa.numRegs < C2::REG_MIN_LAUNCH) {
                    log_error("GEMM kernel compiled with too few registers for its register split");
                    return cudaErrorInvalidConfiguration;
                }
            }
            pl_attr_done[dev] = 1;
        }
    }
    if constexpr (WM == BM) {
        static int mx_attr_done[64] = {0};
        if (p.mx && dev >= 0 && dev < 64 && !mx_attr_done[dev]) {
            for (auto fn : {gemm_mx_kernel<SWAP, BN, 0, false>, gemm_mx_kernel<SWAP, BN, 0, true>}) {
                err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           MxCfg<SWAP, BN, 0>::SMEM);
                if (err != cudaSuccess) return err;
            }
            if constexpr (SWAP && BN <= 32) {
                err = cudaFuncSetAttribute(gemm_mx_kernel<SWAP, BN, 1, false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           MxCfg<SWAP, BN, 1>::SMEM);
                if (err != cudaSuccess) return err;
                err = cudaFuncSetAttribute(gemm_mx_kernel<SWAP, BN, 2, false>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           MxCfg<SWAP, BN, 2>::SMEM);
                if (err != cudaSuccess) return err;
            }
            mx_attr_done[dev] = 1;
        }
        static int rw_attr_done[64] = {0};
        if ((p.rowwise == 1 || p.rowwise == 3) && dev >= 0 && dev < 64 && !rw_attr_done[dev]) {
            err = cudaFuncSetAttribute(gemm_mx_kernel<SWAP, BN, 0, false, 1>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       MxCfg<SWAP, BN, 0, 1>::SMEM);
            if (err != cudaSuccess) return err;
            err = cudaFuncSetAttribute(gemm_mx_kernel<SWAP, BN, 0, false, 2>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       MxCfg<SWAP, BN, 0, 2>::SMEM);
            if (err != cudaSuccess) return err;
            rw_attr_done[dev] = 1;
        }
    }
    const bool swap = SWAP;
    // K columns of the operands: INT8 planes (rowwise 3) hold two per code
    // column (g.K is then the logical K, a multiple of 128)
    const uint64_t K = static_cast<uint64_t>((p.rowwise == 3 || p.rowwise == 5) ? 2 * g.K : g.K);
    const int G = static_cast<int>(p.rowwise ? (g.K + BK - 1) / BK : g.K / BK);
    // grouped: E stacked [N, K] weights (N % 128 == 0), E * m_max token rows
    const int64_t w_rows = g.E > 0 ? g.E * g.N : g.N;
    const int NB = static_cast<int>((w_rows + BK - 1) / BK);
    const uint64_t Mp = static_cast<uint64_t>(pad_rows4(g.M));
    CUtensorMap tm_m, tm_n, tm_sa, tm_sw;
    bool ok;
    if (swap) {
        ok = encode_operand(&tm_m, g.w_q, K, static_cast<uint64_t>(w_rows), WM);
        if (g.x) {
            // fused quant: raw 2-byte activations [M, K], boxes of BN rows x 128
            // elements (256 bytes, unswizzled), rows past M read as zero
            const cuuint64_t dims[2] = {K, static_cast<cuuint64_t>(g.M)};
            const cuuint64_t strides[1] = {K * 2};
            const cuuint32_t box[2] = {static_cast<cuuint32_t>(BK), static_cast<cuuint32_t>(BN)};
            ok = ok && encode(&tm_n, CU_TENSOR_MAP_DATA_TYPE_UINT16, 2, g.x, dims, strides, box,
                              CU_TENSOR_MAP_SWIZZLE_NONE);
        } else {
            ok = ok && encode_operand(&tm_n, g.a_q, K, static_cast<uint64_t>(g.M), BN);
        }
    } else {
        ok = encode_operand(&tm_m, g.a_q, K, static_cast<uint64_t>(g.M), BM) &&
             encode_operand(&tm_n, g.w_q, K, static_cast<uint64_t>(w_rows), BN);
    }
    if (p.rowwise && p.rowwise != 5) {
        // rowwise scales are read by the epilogue directly: no scale maps
        tm_sa = tm_m;
        tm_sw = tm_m;
    } else {
        // activation scales: [cols][Mp] of 4-byte words; box = the tile's tokens of one column
        const cuuint64_t dims[2] = {Mp, static_cast<cuuint64_t>(g.ue8m0 ? (G + 3) / 4 : G)};
        const cuuint64_t strides[1] = {Mp * 4};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(swap ? BN : BM), 1};
        if (g.x)
            tm_sa = tm_n;  // fused quant: the kernel computes the scales itself
        else
            ok = ok && encode(&tm_sa, g.ue8m0 ? CU_TENSOR_MAP_DATA_TYPE_UINT32
                                              : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                              2, g.a_s, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
        // weight scales: the flat [NB*G] fp32 array as one row, 16-byte boxes
        const cuuint64_t flat = static_cast<cuuint64_t>(NB) * G;
        const cuuint64_t wdims[2] = {flat, 1};
        const cuuint64_t wstrides[1] = {(flat * 4 + 15) / 16 * 16};
        const cuuint32_t wbox[2] = {4, 1};
        ok = ok && encode(&tm_sw, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, g.w_s, wdims, wstrides, wbox,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
    }
    if (!ok) {
        log_error("tensor-map encoding failed for the GEMM operands or scales");
        return cudaErrorInvalidValue;
    }

    KArgs a;
    a.M = static_cast<int>(g.M);
    a.N = static_cast<int>(g.N);
    a.G = G;
    a.NB = NB;
    a.swap = swap ? 1 : 0;
    a.tiles_tok = p.tiles_tok;
    a.tiles_e = p.tiles_tok * p.tiles_w;
    a.tiles_w = p.tiles_w;
    a.tiles = a.tiles_e * (p.experts > 0 ? p.experts : 1);
    a.split = p.split;
    a.num_items = p.num_items;
    a.units = static_cast<long long>(a.tiles) * G;
    a.ue8m0 = g.ue8m0;
    a.out_dtype = g.out_dtype;
    // grouped tiles are skipped by the counts, which the previous kernel may
    // write: nothing is read before the dependency wait
    a.prefetch_w = g.E > 0 ? 0 : g.prefetch_w;
    a.E = static_cast<int>(g.E);
    a.m_max = static_cast<int>(g.m_max);
    a.tok_tile = swap ? BN : BM;
    a.counts = g.counts;
    a.w_s = g.w_s;
    a.s_tok = p.rowwise ? static_cast<const float*>(g.a_s) : nullptr;
    a.out = g.out;
    // workspace: [tile counters: fixed kCounterRegion prefix] [fp32 partial tiles]
    a.counters = p.ws_bytes ? static_cast<unsigned*>(g.workspace) : nullptr;
    a.partials = p.ws_bytes ? reinterpret_cast<float*>(static_cast<uint8_t*>(g.workspace) +
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
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (WM == BM) {
        if (p.rowwise == 1) {
            cfg.blockDim = dim3(MxCfg<SWAP, BN, 0, 1>::THREADS);
            cfg.dynamicSmemBytes = MxCfg<SWAP, BN, 0, 1>::SMEM;
            return cudaLaunchKernelEx(&cfg, gemm_mx_kernel<SWAP, BN, 0, false, 1>, tm_m, tm_n,
                                      tm_sa, tm_sw, a);
        }
        if (p.rowwise == 3) {
            cfg.blockDim = dim3(MxCfg<SWAP, BN, 0, 2>::THREADS);
            cfg.dynamicSmemBytes = MxCfg<SWAP, BN, 0, 2>::SMEM;
            return cudaLaunchKernelEx(&cfg, gemm_mx_kernel<SWAP, BN, 0, false, 2>, tm_m, tm_n,
                                      tm_sa, tm_sw, a);
        }
        if (p.mx) {
            if constexpr (SWAP && BN <= 32) {
                if (g.x) {
                    if (g.x_fp16) {
                        cfg.blockDim = dim3(MxCfg<SWAP, BN, 2>::THREADS);
                        cfg.dynamicSmemBytes = MxCfg<SWAP, BN, 2>::SMEM;
                        return cudaLaunchKernelEx(&cfg, gemm_mx_kernel<SWAP, BN, 2, false>, tm_m, tm_n,
                                                  tm_n, tm_n, a);
                    }
                    cfg.blockDim = dim3(MxCfg<SWAP, BN, 1>::THREADS);
                    cfg.dynamicSmemBytes = MxCfg<SWAP, BN, 1>::SMEM;
                    return cudaLaunchKernelEx(&cfg, gemm_mx_kernel<SWAP, BN, 1, false>, tm_m, tm_n, tm_n,
                                              tm_n, a);
                }
            }
            cfg.blockDim = dim3(MxCfg<SWAP, BN, 0>::THREADS);
            cfg.dynamicSmemBytes = MxCfg<SWAP, BN, 0>::SMEM;
            if (g.E > 0)
                return cudaLaunchKernelEx(&cfg, gemm_mx_kernel<SWAP, BN, 0, true>, tm_m, tm_n,
                                          tm_sa, tm_sw, a);
            return cudaLaunchKernelEx(&cfg, gemm_mx_kernel<SWAP, BN, 0, false>, tm_m, tm_n, tm_sa,
                                      tm_sw, a);
        }
    }
    if constexpr (WM == BM) {
        if (p.rowwise == 5) {
            cfg.blockDim = dim3(Cfg<SWAP, BN, BM, 2>::THREADS);
            cfg.dynamicSmemBytes = Cfg<SWAP, BN, BM, 2>::SMEM;
            return cudaLaunchKernelEx(&cfg, gemm_kernel<SWAP, BN, BM, false, 2>, tm_m, tm_n, tm_sa,
                                      tm_sw, a);
        }
    }
    if (g.E > 0)
        return cudaLaunchKernelEx(&cfg, gemm_kernel<SWAP, BN, WM, true>, tm_m, tm_n, tm_sa, tm_sw,
                                  a);
    return cudaLaunchKernelEx(&cfg, gemm_kernel<SWAP, BN, WM, false>, tm_m, tm_n, tm_sa, tm_sw, a);
}

// INT8 GEMM on the warp-level MMA (plan.rowwise 2: rowwise scales; 4: block
// scales): swap-AB tiles of 128 weight rows x BN tokens.
template <int BN>
cudaError_t launch_i8(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    using C = I8Cfg<BN>;
    static int attr_done[64] = {0};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        for (auto fn : {gemm_i8_kernel<BN, false>, gemm_i8_kernel<BN, true>}) {
            err = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
            if (err != cudaSuccess) return err;
        }
        attr_done[dev] = 1;
    }
    const uint64_t K = static_cast<uint64_t>(g.K);
    const int G = static_cast<int>((g.K + BK - 1) / BK);
    CUtensorMap tm_w, tm_t;
    if (!encode_operand(&tm_w, g.w_q, K, static_cast<uint64_t>(g.N), BM) ||
        !encode_operand(&tm_t, g.a_q, K, static_cast<uint64_t>(g.M), BN)) {
        log_error("tensor-map encoding failed for the INT8 GEMM operands");
        return cudaErrorInvalidValue;
    }
    KArgs a = {};
    a.M = static_cast<int>(g.M);
    a.N = static_cast<int>(g.N);
    a.G = G;
    a.NB = static_cast<int>((g.N + BK - 1) / BK);
    a.swap = 1;
    a.tiles_tok = p.tiles_tok;
    a.tiles_w = p.tiles_w;
    a.tiles_e = p.tiles_tok * p.tiles_w;
    a.tiles = a.tiles_e;
    a.split = p.split;
    a.num_items = p.num_items;
    a.units = static_cast<long long>(a.tiles) * G;
    a.out_dtype = g.out_dtype;
    a.prefetch_w = g.prefetch_w;
    a.tok_tile = BN;
    a.w_s = g.w_s;
    a.s_tok = static_cast<const float*>(g.a_s);
    a.out = g.out;
    a.counters = p.ws_bytes ? static_cast<unsigned*>(g.workspace) : nullptr;
    a.partials = p.ws_bytes ? reinterpret_cast<float*>(static_cast<uint8_t*>(g.workspace) +
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
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.rowwise == 4) return cudaLaunchKernelEx(&cfg, gemm_i8_kernel<BN, true>, tm_w, tm_t, a);
    return cudaLaunchKernelEx(&cfg, gemm_i8_kernel<BN, false>, tm_w, tm_t, a);
}

}  // namespace
}  // namespace fp8bq

// gemm.cu -- the GEMM planner (tiles, split-K / stream-K items, workspace)
// and the dispatch of a plan to the launcher of its tile shape.  The kernels
// themselves are in gemm_impl.cuh, instantiated by the gemm_*.cu units.
#include "internal.h"

namespace fp8bq {

namespace {
constexpr int BM = 128;              // MMA M
constexpr int BK = 128;              // K slab (one scale block)
constexpr int kCountersPerTile = 8;  // one split-K ticket per epilogue warp
}  // namespace

cudaError_t launch_gemm_swap16(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_swap16_w64(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_swap32(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_swap32_w64(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_swap64(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_swap128(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_normal128(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_normal256(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_i8_8(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_i8_16(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_i8_32(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_i8_64(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);
cudaError_t launch_gemm_i8_128(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream);

bool make_gemm_plan(int64_t M, int64_t N, int64_t K, const fp8bq_variant& v, int num_sms,
                    GemmPlan* p, int64_t experts, int rowwise) {
    // K slabs (rowwise: the last one may be partly past K, read as zeros)
    const int G = static_cast<int>(rowwise ? (K + BK - 1) / BK : K / BK);
    if (rowwise && (experts != 0 || v.kind == FP8BQ_KIND_SWAP_AB_64)) return false;
    // e4m3 (1) and INT8 on the warp-level MMA (2, swap-AB tiles only) have no
    // block-scaled form; INT8 as FP8 planes (3) is selected by mma_scale = 1
    if ((rowwise == 1 || rowwise == 2 || rowwise == 4) && v.mma_scale != 0) return false;
    if ((rowwise == 2 || rowwise == 4) && v.kind != FP8BQ_KIND_SWAP_AB) return false;
    if (rowwise == 4 && K % BK != 0) return false;
    // block INT8 as two planes on the promotion kernel (5): mma_scale = 1, as 3
    if ((rowwise == 3 || rowwise == 5) && (v.mma_scale != 1 || K % BK != 0)) return false;
    const bool swap = v.kind == FP8BQ_KIND_SWAP_AB || v.kind == FP8BQ_KIND_SWAP_AB_64;
    const int wm = v.kind == FP8BQ_KIND_SWAP_AB_64 ? 64 : BM;  // weight rows per swap tile
    if (v.kind != FP8BQ_KIND_SWAP_AB && v.kind != FP8BQ_KIND_NORMAL &&
        v.kind != FP8BQ_KIND_SWAP_AB_64)
        return false;
    if (v.kind == FP8BQ_KIND_SWAP_AB_64) {
        if (v.block_n != 16 && v.block_n != 32) return false;
    } else if (swap) {
        // (8-token tiles: the INT8 kernel on the warp-level MMA only)
        if (v.block_n != 16 && v.block_n != 32 && v.block_n != 64 && v.block_n != 128 &&
            !(v.block_n == 8 && (rowwise == 2 || rowwise == 4)))
            return false;
    } else {
        if (v.block_n != 128 && v.block_n != 256) return false;
    }
    if (v.split < 0 || v.split > 64 || v.split > G) return false;
    if (v.grid < 0) return false;
    if (v.mma_scale != 0 && v.mma_scale != 1) return false;
    // block-scaled MMA: 128-row tiles (swap-AB or normal), M = 128 MMAs only
    if (v.mma_scale && v.kind == FP8BQ_KIND_SWAP_AB_64) return false;
    // grouped: split-K round robin only (stream-K shares would include the
    // tiles of empty experts), weights in whole 128-row blocks per expert
    if (experts < 0 || experts > (1 << 20)) return false;
    if (experts > 0 && (v.split == 0 || N % BK != 0 || M % 4 != 0)) return false;
    p->experts = static_cast<int>(experts);
    p->rowwise = rowwise;
    p->mx = rowwise ? 0 : v.mma_scale;
    p->kind = v.kind;
    p->bn = v.block_n;
    p->split = v.split;
    if (swap) {
        p->tiles_tok = static_cast<int>((M + v.block_n - 1) / v.block_n);
        p->tiles_w = static_cast<int>((N + wm - 1) / wm);
    } else {
        p->tiles_tok = static_cast<int>((M + BM - 1) / BM);
        p->tiles_w = static_cast<int>((N + v.block_n - 1) / v.block_n);
    }
    const long long tiles =
        static_cast<long long>(p->tiles_tok) * p->tiles_w * (experts > 0 ? experts : 1);
    if (tiles <= 0 || tiles > (1LL << 30)) return false;
    const int g = v.grid > 0 ? v.grid : num_sms;
    const size_t tile_bytes = static_cast<size_t>(swap ? wm : BM) * v.block_n * sizeof(float);
    if (v.split == 0) {
        // stream-K: one CTA per equal share of the tiles x G (tile, slab) units
        const long long units = tiles * G;
        p->num_items = 0;
        p->grid = static_cast<int>(units < g ? units : g);
        p->ws_bytes = kCounterRegion + static_cast<size_t>(2) * p->grid * tile_bytes;
    } else {
        const long long items = tiles * v.split;
        if (items > (1LL << 30)) return false;
        p->num_items = static_cast<int>(items);
        p->grid = static_cast<int>(items < g ? items : g);
        p->ws_bytes = v.split > 1 ? kCounterRegion + static_cast<size_t>(items) * tile_bytes : 0;
    }
    // split tickets live in the fixed counter prefix of the workspace
    if (p->ws_bytes && tiles * kCountersPerTile * 4 > static_cast<long long>(kCounterRegion))
        return false;
    return true;
}

cudaError_t launch_gemm(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    if (p.rowwise == 2 || p.rowwise == 4) {
        switch (p.bn) {
            case 8: return launch_gemm_i8_8(p, g, stream);
            case 16: return launch_gemm_i8_16(p, g, stream);
            case 32: return launch_gemm_i8_32(p, g, stream);
            case 64: return launch_gemm_i8_64(p, g, stream);
            case 128: return launch_gemm_i8_128(p, g, stream);
        }
        return cudaErrorInvalidValue;
    }
    if (p.kind == FP8BQ_KIND_SWAP_AB_64) {
        switch (p.bn) {
            case 16: return launch_gemm_swap16_w64(p, g, stream);
            case 32: return launch_gemm_swap32_w64(p, g, stream);
        }
    } else if (p.kind == FP8BQ_KIND_SWAP_AB) {
        switch (p.bn) {
            case 16: return launch_gemm_swap16(p, g, stream);
            case 32: return launch_gemm_swap32(p, g, stream);
            case 64: return launch_gemm_swap64(p, g, stream);
            case 128: return launch_gemm_swap128(p, g, stream);
        }
    } else {
        switch (p.bn) {
            case 128: return launch_gemm_normal128(p, g, stream);
            case 256: return launch_gemm_normal256(p, g, stream);
        }
    }
    return cudaErrorInvalidValue;
}

}  // namespace fp8bq

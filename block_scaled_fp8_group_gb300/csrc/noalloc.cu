// noalloc.cu -- fp8bq_gemm_noalloc: the block-scaled GEMM for callers that
// cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run a layer: a
// runtime that hands out all device memory up front from its own fixed pool
// and forbids allocations afterwards, code running inside a region where an
// allocation could block or synchronise the device, or a plug-in that only
// receives tensors and a stream.  fp8bq_gemm needs a caller-provided
// workspace when the chosen kernel splits K; this entry point instead uses a
// scratch array that lives in the library itself.  The CUDA runtime loads
// the array's module on a device lazily, at the first lookup of its address
// (the first call of this entry point on that device): that is when the
// device's copy is reserved, and it is kept until the process exits.  That
// first call may synchronise the device, so it belongs at start-up, before
// any stream capture and outside any no-allocation region.
#include <mutex>

#include "internal.h"

namespace fp8bq {
namespace {

// The scratch: split-K tile counters (a fixed prefix that must be zero when
// a kernel starts) followed by fp32 partial tiles.  Its size bounds the
// problems this entry point accepts.
constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device.  In host code the
// array's name only stands for the symbol; the address a kernel can use must
// be asked for, once per device, with that device current.
fp8bq_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return FP8BQ_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return FP8BQ_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) {
            cudaGetLastError();
            log_error("fp8bq_gemm_noalloc: cudaGetSymbolAddress of the scratch array failed");
            return FP8BQ_ERR_CUDA;
        }
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return FP8BQ_OK;
}

}  // namespace
}  // namespace fp8bq

extern "C" {

fp8bq_status fp8bq_gemm_noalloc(int64_t M, int64_t N, int64_t K, const void* a_q,
                                const void* a_s, const void* w_q, const float* w_s, int group,
                                int block_n, int block_k, fp8bq_scale_fmt fmt,
                                fp8bq_dtype out_dtype, void* out, cudaStream_t stream) {
    using namespace fp8bq;
    if (group != kGroup || block_n != kGroup || block_k != kGroup) return FP8BQ_ERR_UNSUPPORTED;
    fp8bq_variant v;
    fp8bq_status st = fp8bq_select_variant(M, N, K, fmt, out_dtype, &v);
    if (st != FP8BQ_OK) return st;
    if (M == 0 || N == 0) return FP8BQ_OK;
    const size_t need = fp8bq_variant_workspace_bytes(M, N, K, &v);
    if (need > kNoAllocScratchBytes) {
        log_error("fp8bq_gemm_noalloc: the problem needs more split-K scratch than the "
                  "library's fixed 32 MiB array; call fp8bq_gemm with a workspace instead");
        return FP8BQ_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    if (need > 0) {
        st = scratch_address(&scratch);
        if (st != FP8BQ_OK) return st;
        // The array keeps whatever the last call left in it; the tile
        // counters at its start must be zero when the kernel begins.
        if (cudaMemsetAsync(scratch, 0, kCounterRegion, stream) != cudaSuccess) {
            cudaGetLastError();
            return FP8BQ_ERR_LAUNCH;
        }
    }
    return fp8bq_gemm_variant(M, N, K, a_q, a_s, w_q, w_s, fmt, out_dtype, out, &v, scratch,
                              need > 0 ? kNoAllocScratchBytes : 0, stream);
}

}  // extern "C"

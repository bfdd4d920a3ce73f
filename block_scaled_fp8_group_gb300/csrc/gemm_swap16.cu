// gemm_swap16.cu -- instantiates the GEMM launchers of: launch_bn<true, 16>, launch_bn<true, 16, 64>.
#include "gemm_impl.cuh"

namespace fp8bq {

cudaError_t launch_gemm_swap16(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_bn<true, 16>(p, g, stream);
}

cudaError_t launch_gemm_swap16_w64(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_bn<true, 16, 64>(p, g, stream);
}

}  // namespace fp8bq

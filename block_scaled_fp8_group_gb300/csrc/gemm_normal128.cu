// gemm_normal128.cu -- instantiates the GEMM launchers of: launch_bn<false, 128>.
#include "gemm_impl.cuh"

namespace fp8bq {

cudaError_t launch_gemm_normal128(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_bn<false, 128>(p, g, stream);
}

}  // namespace fp8bq

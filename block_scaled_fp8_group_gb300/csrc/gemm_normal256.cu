// gemm_normal256.cu -- instantiates the GEMM launchers of: launch_bn<false, 256>.
#include "gemm_impl.cuh"

namespace fp8bq {

cudaError_t launch_gemm_normal256(const GemmPlan& p, const GemmLaunch& g, cudaStream_t stream) {
    return launch_bn<false, 256>(p, g, stream);
}

}  // namespace fp8bq
